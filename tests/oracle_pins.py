"""Pins for the oracle: checks against what the pages and the mathematics fix.

Each check takes `rec`, a callable with the signature of `oracle.recurrent`, so
the same checks run against the real oracle (tests/test_oracle_pins.py) and
against deliberately broken copies of it (tests/test_oracle_mutants.py).  Every
check raises AssertionError on failure.

The sources of truth:
* the update and readout of the gated delta rule with per-channel decay, and the
  packed-sequence contract (attention-gym PR #317, PR description);
* the chunked formulation (kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, "Forward");
* closed forms the mathematics gives for special inputs (pure decay at beta = 0,
  linear attention to first order in beta, the delta-rule overwrite at beta = 1),
  linearity in v, exact rational brute force on a scalar state, and the literal
  matrix form of the update on a tiny state.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

RTOL = 1e-12


def _rng(seed):
    return np.random.default_rng(seed)


def _rand_inputs(seed, B=1, T=9, H=1, HV=1, K=3, V=5, unit_k=True, g_lo=0.05, g_hi=0.7):
    r = _rng(seed)
    q = r.standard_normal((B, T, H, K))
    k = r.standard_normal((B, T, H, K))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = r.standard_normal((B, T, HV, V))
    g = -r.uniform(g_lo, g_hi, (B, T, HV, K))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((B, T, HV))))
    return q, k, v, g, beta


def _close(a, b, rtol=RTOL, what=""):
    a, b = np.asarray(a), np.asarray(b)
    scale = max(1.0, float(np.max(np.abs(b))))
    err = float(np.max(np.abs(a - b)))
    assert err <= rtol * scale, f"{what}: max abs err {err:.3e} > {rtol:.1e} * {scale:.3e}"


# ---------------------------------------------------------------- P1: chunked form
def check_chunked_equals_recurrent(rec):
    """The chunked WY formulation (ALGORITHM.md Stage 1..3+4) reaches the same
    result as the token recurrence, for chunk sizes 1, 16, 64 and the whole
    sequence, with GVA, packing, empty slots, h0 and the L2-norm option."""
    from oracle.chunk_form import chunk_forward

    r = _rng(11)
    B, T, H, HV, K, V = 2, 70, 2, 4, 6, 5
    q, k, v, g, beta = _rand_inputs(11, B, T, H, HV, K, V)
    h0 = 0.1 * r.standard_normal((B, HV, K, V))
    for l2 in (False, True):
        o_r, h_r = rec(q, k, v, g, beta, h0=h0, l2norm=l2)
        for BT in (1, 16, 64, T):
            o_c, h_c = chunk_forward(q, k, v, g, beta, h0=h0, BT=BT, l2norm=l2)
            _close(o_r, o_c, what=f"o BT={BT} l2={l2}")
            _close(h_r, h_c, what=f"ht BT={BT} l2={l2}")
    # packed with empty slots, one batch row
    cu = np.array([0, 0, 17, 17, 50, 81, 81], dtype=np.int32)
    q, k, v, g, beta = _rand_inputs(12, 1, 90, H, HV, K, V)
    h0 = 0.1 * r.standard_normal((6, HV, K, V))
    o_r, h_r = rec(q, k, v, g, beta, h0=h0, cu_seqlens=cu)
    o_c, h_c = chunk_forward(q, k, v, g, beta, h0=h0, cu_seqlens=cu, BT=16)
    _close(o_r[:, :81], o_c[:, :81], what="packed o")
    _close(h_r, h_c, what="packed ht")


# ---------------------------------------------------------------- P2: pure decay
def check_beta_zero_is_pure_decay(rec):
    """beta = 0: S_t = Diag(2^{sum_{s<=t} g_s}) S_0 and o_t = scale * S_t^T q_t.
    K != V so a transposed state fails; HV = 2H so a wrong head mapping fails."""
    B, T, H, HV, K, V = 1, 7, 2, 4, 3, 5
    q, k, v, g, beta = _rand_inputs(21, B, T, H, HV, K, V)
    beta[:] = 0.0
    h0 = _rng(22).standard_normal((B, HV, K, V))
    scale = 0.37
    o, ht = rec(q, k, v, g, beta, h0=h0, scale=scale)
    cum = np.cumsum(g, axis=1)                           # [B,T,HV,K]
    for hv in range(HV):
        h = hv // (HV // H)
        for t in range(T):
            St = np.exp2(cum[0, t, hv])[:, None] * h0[0, hv]
            _close(o[0, t, hv], scale * St.T @ q[0, t, h], what=f"o t={t} hv={hv}")
        _close(ht[0, hv], np.exp2(cum[0, -1, hv])[:, None] * h0[0, hv], what="ht")
    # g_scale multiplies the gate before exponentiation (natural-log callers)
    o2, _ = rec(q, k, v, g, beta, h0=h0, scale=scale, g_scale=1.0 / math.log(2))
    S1 = np.exp(cum[0, 0, 0])[:, None] * h0[0, 0]
    _close(o2[0, 0, 0], scale * S1.T @ q[0, 0, 0], what="g_scale")


# ---------------------------------------------------------------- P3: linear attention
def check_literal_and_first_order_linear_attention(rec):
    """g = 0, beta = 0 freezes the state: o_t = scale * h0^T q_t (the literal
    reading).  With h0 = 0, g = 0 and beta = eps, o_t / eps tends to causal
    linear attention scale * sum_{j<=t} (q_t . k_j) v_j with O(eps) error."""
    B, T, H, HV, K, V = 1, 6, 1, 1, 4, 3
    q, k, v, g, beta = _rand_inputs(31, B, T, H, HV, K, V)
    g[:] = 0.0
    beta[:] = 0.0
    h0 = _rng(32).standard_normal((B, HV, K, V))
    o, _ = rec(q, k, v, g, beta, h0=h0)
    sc = 1.0 / math.sqrt(K)
    for t in range(T):
        _close(o[0, t, 0], sc * h0[0, 0].T @ q[0, t, 0], what=f"frozen t={t}")
    eps = 1e-6
    beta[:] = eps
    o, _ = rec(q, k, v, g, beta)
    for t in range(T):
        want = sc * sum(float(q[0, t, 0] @ k[0, j, 0]) * v[0, j, 0] for j in range(t + 1))
        _close(o[0, t, 0] / eps, want, rtol=1e-5, what=f"linear attention t={t}")


# ---------------------------------------------------------------- P4: linearity
def check_linear_in_v(rec):
    """With h0 = 0 the outputs are linear in v; jointly linear in (h0, v)."""
    B, T, H, HV, K, V = 1, 11, 1, 2, 4, 3
    q, k, v1, g, beta = _rand_inputs(41, B, T, H, HV, K, V)
    v2 = _rng(42).standard_normal(v1.shape)
    a, b = 0.7, -1.9
    o1, s1 = rec(q, k, v1, g, beta)
    o2, s2 = rec(q, k, v2, g, beta)
    o3, s3 = rec(q, k, a * v1 + b * v2, g, beta)
    _close(o3, a * o1 + b * o2, what="o linear in v")
    _close(s3, a * s1 + b * s2, what="ht linear in v")
    h1 = _rng(43).standard_normal((B, HV, K, V))
    h2 = _rng(44).standard_normal((B, HV, K, V))
    p1 = rec(q, k, v1, g, beta, h0=h1)
    p2 = rec(q, k, v2, g, beta, h0=h2)
    p3 = rec(q, k, a * v1 + b * v2, g, beta, h0=a * h1 + b * h2)
    _close(p3[0], a * p1[0] + b * p2[0], what="o jointly linear")
    _close(p3[1], a * p1[1] + b * p2[1], what="ht jointly linear")


# ---------------------------------------------------------------- P5: overwrite
def check_delta_rule_overwrite(rec):
    """beta = 1, g = 0, unit k: the write makes S_t^T k_t = v_t exactly, so a
    query equal to the key reads back scale * v_t whatever the history."""
    B, T, H, HV, K, V = 1, 8, 1, 1, 5, 4
    q, k, v, g, beta = _rand_inputs(51, B, T, H, HV, K, V)
    g[:] = 0.0
    beta[:] = 1.0
    h0 = _rng(52).standard_normal((B, HV, K, V))
    o, _ = rec(k.copy(), k, v, g, beta, h0=h0, scale=0.5)
    _close(o[0, :, 0], 0.5 * v[0, :, 0], rtol=1e-12, what="overwrite")


# ---------------------------------------------------------------- P6: empty slots
def check_empty_slots_pass_state_bitwise(rec):
    """Repeated offsets are empty slots: their final state equals h0 bit for bit
    (and is +0.0 without h0)."""
    HV, K, V = 2, 3, 4
    q, k, v, g, beta = _rand_inputs(61, 1, 12, 1, HV, K, V)
    cu = np.array([0, 5, 5, 5, 12, 12], dtype=np.int32)
    h0 = _rng(62).standard_normal((5, HV, K, V))
    _, ht = rec(q, k, v, g, beta, h0=h0, cu_seqlens=cu)
    for n in (1, 2, 4):
        assert ht[n].tobytes() == h0[n].tobytes(), f"slot {n} state changed"
    _, ht0 = rec(q, k, v, g, beta, cu_seqlens=cu)
    for n in (1, 2, 4):
        assert np.all(ht0[n] == 0.0) and not np.any(np.signbit(ht0[n])), f"slot {n} not +0"
    assert not np.array_equal(ht[0], h0[0]), "non-empty slot must change"


# ---------------------------------------------------------------- P7: brute force
def _scalar_fraction_recurrence(q, k, v, a, beta, s0, scale):
    """K = V = 1 with decay factors a_t = 2^{g_t} given exactly: s_t =
    (1 - beta k^2) a s_{t-1} + beta k v, o_t = scale * s_t * q, in exact rationals."""
    s, out = s0, []
    for qt, kt, vt, at, bt in zip(q, k, v, a, beta):
        s = (1 - bt * kt * kt) * at * s + bt * kt * vt
        out.append(scale * s * qt)
    return out, s


def check_scalar_brute_force(rec):
    """A one-channel state over four tokens, against exact rational arithmetic
    (decays 2^-1, 2^-2, 2^0, 2^-3 are exact in binary)."""
    F = Fraction
    q = [F(1, 2), F(-3, 4), F(5, 8), F(1)]
    k = [F(3, 4), F(1, 2), F(-1), F(1, 4)]
    v = [F(2), F(-1, 2), F(3, 8), F(5)]
    gs = [-1, -2, 0, -3]
    beta = [F(1, 2), F(1, 4), F(3, 4), F(1)]
    s0, scale = F(3, 2), F(1, 2)
    want_o, want_s = _scalar_fraction_recurrence(q, k, v, [F(2) ** x for x in gs], beta, s0,
                                                 scale)
    arr = lambda xs: np.array([float(x) for x in xs]).reshape(1, 4, 1, 1)
    o, ht = rec(arr(q), arr(k), arr(v), arr(gs), np.array([float(b) for b in beta]).reshape(1, 4, 1),
                h0=np.array([[[[float(s0)]]]]), scale=float(scale))
    for t in range(4):
        assert abs(o[0, t, 0, 0] - float(want_o[t])) <= 1e-15, f"scalar o[{t}]"
    assert abs(ht[0, 0, 0, 0] - float(want_s)) <= 1e-15, "scalar state"


def check_literal_matrix_update(rec):
    """The update exactly as written, S_t = (I - b k k^T) Diag(2^g) S_{t-1} + b k v^T,
    with explicit matrices on a 3x2 state (K != V), no unit-norm keys."""
    B, T, H, HV, K, V = 1, 5, 1, 1, 3, 2
    q, k, v, g, beta = _rand_inputs(71, B, T, H, HV, K, V, unit_k=False)
    h0 = _rng(72).standard_normal((B, HV, K, V))
    sc = 0.8
    o, ht = rec(q, k, v, g, beta, h0=h0, scale=sc)
    S = h0[0, 0].copy()
    for t in range(T):
        kt, bt = k[0, t, 0], beta[0, t, 0]
        S = (np.eye(K) - bt * np.outer(kt, kt)) @ np.diag(np.exp2(g[0, t, 0])) @ S \
            + bt * np.outer(kt, v[0, t, 0])
        _close(o[0, t, 0], sc * S.T @ q[0, t, 0], what=f"matrix form t={t}")
    _close(ht[0, 0], S, what="matrix form ht")


# ---------------------------------------------------------------- P9 / P10
def check_gva_equals_repeated_heads(rec):
    """HV = G*H value heads sharing q/k equal H' = HV heads with q/k repeated."""
    B, T, H, HV, K, V = 1, 9, 2, 6, 4, 3
    q, k, v, g, beta = _rand_inputs(81, B, T, H, HV, K, V)
    o1, s1 = rec(q, k, v, g, beta)
    G = HV // H
    o2, s2 = rec(np.repeat(q, G, axis=2), np.repeat(k, G, axis=2), v, g, beta)
    _close(o1, o2, rtol=0, what="GVA o")
    _close(s1, s2, rtol=0, what="GVA ht")


def check_packed_equals_dense_slices(rec):
    """Each packed sequence equals a dense single-sequence call on its slice,
    including its own h0 row."""
    HV, K, V = 2, 4, 3
    q, k, v, g, beta = _rand_inputs(91, 1, 40, 1, HV, K, V)
    cu = np.array([0, 13, 13, 29, 37], dtype=np.int32)
    h0 = _rng(92).standard_normal((4, HV, K, V))
    o, ht = rec(q, k, v, g, beta, h0=h0, cu_seqlens=cu)
    for n in range(4):
        a, b = cu[n], cu[n + 1]
        if a == b:
            continue
        od, hd = rec(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b], h0=h0[n:n + 1])
        _close(o[:, a:b], od, rtol=0, what=f"packed slice {n} o")
        _close(ht[n], hd[0], rtol=0, what=f"packed slice {n} ht")
    assert np.all(np.isnan(o[:, 37:])), "rows beyond the terminal offset must stay untouched"


# ---------------------------------------------------------------- P11: extreme decay
def check_extreme_decay(rec):
    """g = -16 per step (the decay magnitude real KDA gates reach): the history is
    scaled by 2^-16 every token, so S_t = beta_t k_t v_t^T + O(2^-16) and
    o_t = scale beta_t (q_t . k_t) v_t to that order; everything stays finite."""
    B, T, H, HV, K, V = 1, 40, 1, 1, 8, 4
    q, k, v, g, beta = _rand_inputs(101, B, T, H, HV, K, V)
    g[:] = -16.0
    h0 = _rng(102).standard_normal((B, HV, K, V))
    o, ht = rec(q, k, v, g, beta, h0=h0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(ht))
    sc = 1.0 / math.sqrt(K)
    for t in range(1, T):
        want = sc * beta[0, t, 0] * float(q[0, t, 0] @ k[0, t, 0]) * v[0, t, 0]
        _close(o[0, t, 0], want, rtol=2e-4, what=f"extreme decay t={t}")



# ---------------------------------------------------------------- a0: L2-norm option
# kernel-fun 0.2.0.dev1 wheel, kda/autograd.py, ChunkKDAFunction.forward
# (use_qk_l2norm) and attention-gym PR #345 commit message "fuse q l2norm": every
# (token, head) row of q and of k is divided by its L2 norm over the K channels;
# the epsilon's value is not printed there (reading: 1e-6 inside the square root).

def _row_scaled_inputs(seed, B, T, H, HV, K, V, lo=1.0, hi=40.0):
    """Rows that are NOT unit norm: q, k ~ N(0,1), each (token, head) row then
    multiplied by its own scale in [lo, hi] (norms well above the epsilon)."""
    q, k, v, g, beta = _rand_inputs(seed, B, T, H, HV, K, V, unit_k=False)
    r = _rng(seed + 1000)
    for x in (q, k):
        n = np.linalg.norm(x, axis=-1, keepdims=True)
        x *= np.maximum(n, 0.5) / n                      # no row shorter than 0.5
        x *= r.uniform(lo, hi, x.shape[:-1] + (1,))
    return q, k, v, g, beta


def check_l2norm_is_scale_invariant_unit_rows(rec):
    """With the option, rows of any length give the result of the plain
    recurrence on the exactly normalised rows q / |q|, k / |k| (to the
    epsilon's relative effect, below 1e-6 here).  Per-row scales differ across
    tokens and heads, so a norm over the wrong extent, a norm applied to q only
    or to k only, or a missing square root changes the result."""
    B, T, H, HV, K, V = 1, 10, 2, 4, 5, 3
    q, k, v, g, beta = _row_scaled_inputs(111, B, T, H, HV, K, V)
    h0 = 0.3 * _rng(112).standard_normal((B, HV, K, V))
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    o1, s1 = rec(q, k, v, g, beta, h0=h0, l2norm=True)
    o2, s2 = rec(unit(q), unit(k), v, g, beta, h0=h0, l2norm=False)
    _close(o1, o2, rtol=1e-5, what="l2norm o vs unit rows")
    _close(s1, s2, rtol=1e-5, what="l2norm ht vs unit rows")
    # the option must matter on such rows: the raw recurrence differs a lot
    o3, _ = rec(q, k, v, g, beta, h0=h0, l2norm=False)
    assert float(np.max(np.abs(o3 - o1))) > 1e-2, "the L2-norm flag had no effect"


def check_l2norm_zero_and_short_rows(rec):
    """A zero q row reads out exactly zero (the epsilon keeps 0 / 0 away); a zero
    k row writes nothing, so the state only decays at that token.  A row of
    length r = 1e-4 (r^2 far below the epsilon) is scaled by 1 / sqrt(r^2 +
    1e-6) to length r / sqrt(r^2 + 1e-6) ~ 0.0995, not to 1: the reading of the
    epsilon, pinned on the one input where it decides the result."""
    B, T, H, HV, K, V = 1, 6, 1, 1, 4, 3
    q, k, v, g, beta = _row_scaled_inputs(121, B, T, H, HV, K, V)
    h0 = _rng(122).standard_normal((B, HV, K, V))
    q[0, 2, 0] = 0.0
    k[0, 4, 0] = 0.0
    o, _ = rec(q, k, v, g, beta, h0=h0, l2norm=True)
    assert np.all(np.isfinite(o)), "zero rows must not produce NaN"
    assert np.all(o[0, 2, 0] == 0.0), "a zero query row must read out zero"
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    # token 4 (k = 0): o_4 = scale * (Diag(2^g_4) S_3)^T q_4 / |q_4|
    _, S3 = rec(q[:, :4], k[:, :4], v[:, :4], g[:, :4], beta[:, :4], h0=h0, l2norm=True)
    S4 = np.exp2(g[0, 4, 0])[:, None] * S3[0, 0]
    _close(o[0, 4, 0], S4.T @ unit(q)[0, 4, 0] / math.sqrt(K), rtol=1e-6,
           what="zero key row writes nothing")  # 1e-6: the epsilon's effect on q_4
    # short rows: q_t = r u with |u| = 1
    r = 1e-4
    qs, ks = q.copy(), k.copy()
    qs[0, 1, 0] = r * unit(q)[0, 1, 0]
    ks[0, 3, 0] = r * unit(k)[0, 3, 0]
    o_s, s_s = rec(qs, ks, v, g, beta, h0=h0, l2norm=True)
    f = r / math.sqrt(r * r + 1e-6)
    unit0 = lambda x: x / np.maximum(np.linalg.norm(x, axis=-1, keepdims=True), 1e-300)
    qe, ke = unit0(qs), unit0(ks)  # the zero rows stay zero
    qe[0, 1, 0] *= f
    ke[0, 3, 0] *= f
    o_e, s_e = rec(qe, ke, v, g, beta, h0=h0, l2norm=False)
    _close(o_s, o_e, rtol=1e-6, what="short rows o")  # 1e-6: epsilon's effect on the long rows
    _close(s_s, s_e, rtol=1e-6, what="short rows ht")


def check_l2norm_rows_are_independent(rec):
    """The norm of a (token, head) row involves that row only: rescaling every
    row of q/k head 1 leaves the value heads of q/k head 0 bit for bit unchanged
    (grouped value heads, HV = 2H) and those of head 1 unchanged to rounding."""
    B, T, H, HV, K, V = 1, 8, 2, 4, 4, 3
    q, k, v, g, beta = _row_scaled_inputs(131, B, T, H, HV, K, V)
    o1, s1 = rec(q, k, v, g, beta, l2norm=True)
    q2, k2 = q.copy(), k.copy()
    q2[:, :, 1] *= 37.0
    k2[:, :, 1] *= 0.03
    o2, s2 = rec(q2, k2, v, g, beta, l2norm=True)
    assert np.array_equal(o1[:, :, :2], o2[:, :, :2]), "head 0 outputs changed"
    assert np.array_equal(s1[:, :2], s2[:, :2]), "head 0 states changed"
    _close(o1[:, :, 2:], o2[:, :, 2:], rtol=1e-5, what="head 1 rescaled rows")


ALL_CHECKS = [
    check_chunked_equals_recurrent,
    check_beta_zero_is_pure_decay,
    check_literal_and_first_order_linear_attention,
    check_linear_in_v,
    check_delta_rule_overwrite,
    check_empty_slots_pass_state_bitwise,
    check_scalar_brute_force,
    check_literal_matrix_update,
    check_gva_equals_repeated_heads,
    check_packed_equals_dense_slices,
    check_extreme_decay,
    check_l2norm_is_scale_invariant_unit_rows,
    check_l2norm_zero_and_short_rows,
    check_l2norm_rows_are_independent,
]


# ---------------------------------------------------------------- P8: gate cumsum
# kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, "Stage 1 -- cumsum": chunk-local
# inclusive prefix sum per channel, times a multiplier.  `cums` has the
# signature of `oracle.gate_cumsum`.

def check_cumsum_is_library_prefix_sum_per_chunk(cums):
    r = _rng(1)
    B, T, HV, K = 2, 150, 3, 5
    g = -r.uniform(0, 1, (B, T, HV, K))
    for chunk in (1, 16, 64):
        got = cums(g, chunk=chunk, g_scale=1.7)
        for s in range(0, T, chunk):
            _close(got[:, s:s + chunk], 1.7 * np.cumsum(g[:, s:s + chunk], axis=1),
                   rtol=1e-13, what=f"cumsum chunk={chunk} s={s}")


def check_cumsum_chunk_one_is_identity(cums):
    g = -_rng(2).uniform(0, 1, (1, 33, 2, 4))
    assert np.array_equal(cums(g, chunk=1), g), "chunk=1 must be the identity"


def check_cumsum_restarts_at_each_sequence_start(cums):
    """All-ones input: a row's value is its 1-based position inside its chunk,
    chunks counted from the sequence's own first row; tail rows stay untouched."""
    T = 100
    g = np.ones((1, T, 1, 1))
    cu = np.array([0, 3, 3, 70, 90], dtype=np.int32)
    got = cums(g, cu_seqlens=cu, chunk=64)[0, :, 0, 0]
    want = np.full(T, np.nan)
    for a, b in zip(cu[:-1], cu[1:]):
        for t in range(a, b):
            want[t] = (t - a) % 64 + 1
    assert np.array_equal(got, want, equal_nan=True), "packed chunk restarts"


CUMSUM_CHECKS = [
    check_cumsum_is_library_prefix_sum_per_chunk,
    check_cumsum_chunk_one_is_identity,
    check_cumsum_restarts_at_each_sequence_start,
]
