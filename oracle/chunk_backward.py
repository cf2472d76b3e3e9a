"""fp64 chunk-form gradients of KDA -- TEST INFRASTRUCTURE ONLY.

The chunked backward of kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, "Backward" ("The
seven launches"), written out plainly in numpy fp64 for one (sequence, value head)
at a time, stage by stage in the pages' order, with every chain-rule step taken
through the chunk form's own formulas (ALGORITHM.md, "Forward", Stages 1-4):

    g2 = chunk-local cumsum of g_scale g (log2), G its last row
    Aqk[r,s] = scale sum_d q_r k_s 2^(g2_r - g2_s)        (s <= r)
    L[r,s]   = beta_r sum_d k_r k_s 2^(g2_r - g2_s)       (s <  r),  Akk = (I + L)^-1
    w = Akk (beta k 2^g2),  u = Akk (beta v),  qg = q 2^g2,  kg = k 2^(G - g2)
    v' = u - w h,  o = scale qg h + Aqk v',  h_next = Diag(2^G) h + kg^T v'

    1 recompute   w, u, qg, kg, Aqk, Akk of every chunk
    2 re-scan     the state h_c at the start of every chunk and v'_c
    3 dAv         dAqk = do v'^T (lower, diagonal included); dv' = Aqk^T do
    4 dhu         reverse scan: dv' += kg dh_{c+1};  dh_c = 2^G dh_{c+1} + scale qg^T do - w^T dv'
    5 wy_dqkg     through qg, kg, 2^G and w, u: dq, dk, dbeta, dAkk and the gate terms
    6 intra       dL = -Akk^T dAkk Akk^T (strictly lower), then the two grams
    7 dg cumsum   per-token gate gradient = g_scale x chunk-local reverse cumsum of dg2

The pages print some of these formulas and not others; each step here is derived
from the forward formulas above (2^x contributes ln 2 to its exponent's gradient).
The op's options wrap this core exactly as they wrap the forward: with `l2norm` the
core sees q / sqrt(sum q^2 + 1e-6) (and the same of k) per (token, head), and the
raw rows' gradients are r (dx^ - x^ (x^ . dx^)), r the row's inverse norm; with
`A_log` the core's gate is -exp(A_log) softplus(g + dt_bias) (natural log; kernel-fun
wheel, kda/chain.py, gate_backward) and the raw gate's gradient is the core's times
-exp(A_log) sigmoid(g + dt_bias), plus dA_log = sum dg' g' and dt_bias's sum over
tokens; with `beta_scale` > 0 the core's beta is sigmoid(beta) beta_scale (rounded to
bf16 in value when `beta_bf16`, the gradient passing straight through).
tests/test_oracle_chunk_backward.py pins every gradient against
oracle/backward.py, the reverse-mode derivative of the token recurrence -- an
independent derivation of the same numbers -- at chunk sizes from 1 to past T, with
packing, empty slots, partial chunks and grouped value heads.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = ["chunk_grads"]

LN2 = math.log(2.0)


def _reverse_cumsum(x):
    """Inclusive reverse cumsum along axis 0: out[r] = sum_{r' >= r} x[r']."""
    return np.cumsum(x[::-1], axis=0)[::-1]


def _chunk_forward(qc, kc, vc, bc, gc, scale, h):
    """Stages 1 and 2 for one chunk: its forward quantities and the state after it."""
    nr = qc.shape[0]
    g2 = np.cumsum(gc, axis=0)
    G = g2[-1]
    E = np.exp2(g2[:, None, :] - g2[None, :, :])            # [r, s, d]; used where s <= r
    incl = np.tril(np.ones((nr, nr)))
    strict = np.tril(np.ones((nr, nr)), -1)
    Aqk = scale * np.einsum("rd,sd,rsd->rs", qc, kc, E) * incl
    P = np.einsum("rd,sd,rsd->rs", kc, kc, E) * strict      # L = diag(beta) P
    Akk = np.linalg.inv(np.eye(nr) + bc[:, None] * P)
    kgate = kc * np.exp2(g2)
    w = Akk @ (bc[:, None] * kgate)
    u = Akk @ (bc[:, None] * vc)
    qg = qc * np.exp2(g2)
    kg = kc * np.exp2(G[None, :] - g2)
    vp = u - w @ h
    h_next = np.exp2(G)[:, None] * h + kg.T @ vp
    return dict(g2=g2, G=G, E=E, incl=incl, strict=strict, Aqk=Aqk, P=P, Akk=Akk,
                kgate=kgate, w=w, u=u, qg=qg, kg=kg, h=h, vp=vp), h_next


def _chunk_backward(f, qc, kc, vc, bc, do_c, dh_next, scale):
    """Stages 3-6 for one chunk given dL/dh_{c+1}: the chunk's input gradients (dg2
    still with respect to the cumsum) and dL/dh_c."""
    Aqk, Akk, E, w, kg, qg, h, vp = (f[x] for x in ("Aqk", "Akk", "E", "w", "kg", "qg", "h", "vp"))
    G, g2, kgate, P = f["G"], f["g2"], f["kgate"], f["P"]
    # 3. dAv
    dAqk = (do_c @ vp.T) * f["incl"]
    dvp = Aqk.T @ do_c
    # 4. dhu: the state update and the readout
    dvp = dvp + kg @ dh_next
    dG = LN2 * np.exp2(G) * np.sum(h * dh_next, axis=1)     # h_next's factor 2^G
    dqg = scale * do_c @ h.T
    dkg = vp @ dh_next.T
    du = dvp
    dw = -dvp @ h.T
    dh = np.exp2(G)[:, None] * dh_next + scale * qg.T @ do_c - w.T @ dvp
    # 5. wy_dqkg: through u, w, qg, kg
    dq = dqg * np.exp2(g2)
    dg2 = LN2 * dqg * qg
    dk = dkg * np.exp2(G[None, :] - g2)
    dG = dG + LN2 * np.sum(dkg * kg, axis=0)
    dg2 = dg2 - LN2 * dkg * kg
    dAkk = du @ (bc[:, None] * vc).T + dw @ (bc[:, None] * kgate).T
    t_u = Akk.T @ du
    t_w = Akk.T @ dw
    dv = bc[:, None] * t_u
    dbeta = np.sum(t_u * vc, axis=1) + np.sum(t_w * kgate, axis=1)
    dkgate = bc[:, None] * t_w
    dk = dk + dkgate * np.exp2(g2)
    dg2 = dg2 + LN2 * dkgate * kgate
    # 6. intra: through Akk = (I + L)^-1 and the grams
    dL = -(Akk.T @ dAkk @ Akk.T) * f["strict"]
    dbeta = dbeta + np.sum(dL * P, axis=1)
    dP = dL * bc[:, None]
    dk = dk + np.einsum("rs,sd,rsd->rd", dP, kc, E) + np.einsum("rs,rd,rsd->sd", dP, kc, E)
    X = np.einsum("rs,rd,sd,rsd->rsd", dP, kc, kc, E)
    dg2 = dg2 + LN2 * (X.sum(axis=1) - X.sum(axis=0))
    dq = dq + scale * np.einsum("rs,sd,rsd->rd", dAqk, kc, E)
    dk = dk + scale * np.einsum("rs,rd,rsd->sd", dAqk, qc, E)
    Y = scale * np.einsum("rs,rd,sd,rsd->rsd", dAqk, qc, kc, E)
    dg2 = dg2 + LN2 * (Y.sum(axis=1) - Y.sum(axis=0))
    dg2[-1] = dg2[-1] + dG                                   # G is the last row of g2
    return dict(dq=dq, dk=dk, dv=dv, dbeta=dbeta, dg2=dg2, dAqk=dAqk, dAkk=dAkk), dh


def _l2norm_rows(x):
    """x / sqrt(sum x^2 + 1e-6) over the last axis, and the inverse norms."""
    r = 1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + 1e-6)
    return x * r, r


def _l2norm_bwd(xh, r, dxh):
    """Gradient of the raw rows from that of the normalised rows xh = r x."""
    return r * (dxh - xh * np.sum(xh * dxh, axis=-1, keepdims=True))


def chunk_grads(q, k, v, g, beta, do, h0=None, dht=None, cu_seqlens=None, scale=None,
                g_scale=1.0, chunk_size=64, stages=False, l2norm=False, A_log=None,
                dt_bias=None, beta_scale=0.0, beta_bf16=False):
    """The chunk-form gradients with the op's options (see the module docstring):
    the plain core (`_core_grads`) between the options' forward transforms and their
    chain rules.  Adds dA_log [HV] and ddt_bias [HV, K] (None when not given)."""
    f64 = lambda x: None if x is None else np.asarray(x, dtype=np.float64)
    q, k, g, beta = f64(q), f64(k), f64(g), f64(beta)
    if cu_seqlens is not None:
        # rows past the last offset belong to no sequence and are never read: they
        # enter neither the core nor the options' sums over tokens
        end = int(np.asarray(cu_seqlens)[-1])
        q, k, g, beta = (x.copy() for x in (q, k, g, beta))
        for x in (q, k, g, beta):
            x[:, end:] = 0.0
    if l2norm:
        qh, rq = _l2norm_rows(q)
        kh, rk = _l2norm_rows(k)
    else:
        qh, kh = q, k
    ga, bact = g, beta
    if A_log is not None:
        a = np.exp(f64(A_log))[None, None, :, None]
        x = g if dt_bias is None else g + f64(dt_bias)[None, None]
        ga = -a * np.logaddexp(0.0, x)
        sig = 0.5 * (1.0 + np.tanh(0.5 * x))
    if beta_scale > 0:
        sb = 0.5 * (1.0 + np.tanh(0.5 * beta))
        bact = beta_scale * sb
        if beta_bf16:
            import torch

            bact = torch.from_numpy(bact).to(torch.bfloat16).to(torch.float64).numpy()
    out = _core_grads(qh, kh, v, ga, bact, do, h0, dht, cu_seqlens, scale, g_scale, chunk_size,
                      stages)
    if l2norm:
        out["dq"] = _l2norm_bwd(qh, rq, out["dq"])
        out["dk"] = _l2norm_bwd(kh, rk, out["dk"])
    out["dA_log"] = out["ddt_bias"] = None
    if A_log is not None:
        dga = out["dg"]
        out["dg"] = dga * (-a) * sig
        out["dA_log"] = np.sum(dga * ga, axis=(0, 1, 3))
        if dt_bias is not None:
            out["ddt_bias"] = np.sum(out["dg"], axis=(0, 1))
    if beta_scale > 0:
        out["dbeta"] = out["dbeta"] * beta_scale * sb * (1.0 - sb)
    return out


def _core_grads(q, k, v, g, beta, do, h0=None, dht=None, cu_seqlens=None, scale=None,
                g_scale=1.0, chunk_size=64, stages=False):
    """Gradients of sum(o * do) + sum(ht * dht) by the chunk form, in fp64 (plain op).

    Shapes as oracle.backward.recurrent_grads: q, k [B,T,H,K]; v, do [B,T,HV,V];
    g [B,T,HV,K] per-token log gate (times g_scale: log2 units after it); beta
    [B,T,HV]; h0, dht [N,HV,K,V] or None; cu_seqlens [N+1] or None (then N = B).
    Chunks of `chunk_size` rows restart at every sequence start; a sequence's last
    chunk may be shorter.  Returns dq, dk, dv, dg, dbeta, dh0 (None without h0) as
    float64 arrays; rows outside every sequence get zero.  With `stages`, also
    "chunks": per (n, hv) the list of per-chunk dicts with the state h_c at the
    chunk's start, dL/dh_{c+1} ("dh_next"), dAqk and dAkk.
    """
    f64 = lambda x: None if x is None else np.asarray(x, dtype=np.float64)
    q, k, v, g, beta, do, h0, dht = (f64(x) for x in (q, k, v, g, beta, do, h0, dht))
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    grp = HV // H
    if scale is None:
        scale = 1.0 / math.sqrt(K)
    cu = None if cu_seqlens is None else [int(x) for x in np.asarray(cu_seqlens)]
    N = B if cu is None else len(cu) - 1
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dg=np.zeros_like(g), dbeta=np.zeros_like(beta),
               dh0=None if h0 is None else np.zeros_like(h0))
    chunks = {}
    for n in range(N):
        b, bos, eos = (n, 0, T) if cu is None else (0, cu[n], cu[n + 1])
        bounds = [(r0, min(r0 + chunk_size, eos)) for r0 in range(bos, eos, chunk_size)]
        for hv in range(HV):
            h = hv // grp
            S = np.zeros((K, V)) if h0 is None else h0[n, hv].copy()
            fwd = []
            for r0, r1 in bounds:                            # stages 1, 2
                f, S = _chunk_forward(q[b, r0:r1, h], k[b, r0:r1, h], v[b, r0:r1, hv],
                                      beta[b, r0:r1, hv], g_scale * g[b, r0:r1, hv], scale, S)
                fwd.append(f)
            dS = np.zeros((K, V)) if dht is None else dht[n, hv].copy()
            rec = []
            for (r0, r1), f in reversed(list(zip(bounds, fwd))):   # stages 3-6, reverse
                gr, dS_prev = _chunk_backward(f, q[b, r0:r1, h], k[b, r0:r1, h],
                                              v[b, r0:r1, hv], beta[b, r0:r1, hv],
                                              do[b, r0:r1, hv], dS, scale)
                out["dq"][b, r0:r1, h] += gr["dq"]
                out["dk"][b, r0:r1, h] += gr["dk"]
                out["dv"][b, r0:r1, hv] = gr["dv"]
                out["dbeta"][b, r0:r1, hv] = gr["dbeta"]
                out["dg"][b, r0:r1, hv] = g_scale * _reverse_cumsum(gr["dg2"])   # stage 7
                if stages:
                    rec.append(dict(h=f["h"], dh_next=dS, dAqk=gr["dAqk"], dAkk=gr["dAkk"]))
                dS = dS_prev
            if h0 is not None:
                out["dh0"][n, hv] = dS
            if stages:
                chunks[(n, hv)] = rec[::-1]
    if stages:
        out["chunks"] = chunks
    return out
