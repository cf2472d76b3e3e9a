"""The pins are sharp: each plausible mistake planted in a copy of the oracle
(on the CPU) makes at least one pin fail.

Each mutant is a textual edit of oracle/kda_oracle.c compiled into a temporary
library; the real oracle is never modified.
"""
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

# (name, original text, mutated text)
MUTANTS = [
    ("decay_sign", "exp2(g_scale * gt[d])", "exp2(-g_scale * gt[d])"),
    ("beta_dropped", "delta[j] = bt * (vt[j] - acc)", "delta[j] = (vt[j] - acc)"),
    ("residual_sign", "delta[j] = bt * (vt[j] - acc)", "delta[j] = bt * (vt[j] + acc)"),
    ("readout_uses_key", "acc += S[(size_t)d * V + j] * qt[d];",
     "acc += S[(size_t)d * V + j] * kt[d];"),
    ("readout_transposed", "acc += S[(size_t)d * V + j] * qt[d];",
     "acc += S[(size_t)j * K + d] * qt[d];"),
    ("scale_dropped", "ot[j] = scale * acc;", "ot[j] = acc;"),
    ("head_map_modulo", "const int h = hv / group;", "const int h = hv % H;"),
    ("h0_ignored", "            if (h0)\n                memcpy(S,", "            if (0)\n                memcpy(S,"),
    ("rank1_uses_query", "Srow[j] += kt[d] * delta[j];", "Srow[j] += qt[d] * delta[j];"),
    ("l2norm_no_sqrt", "qn = 1.0 / sqrt(sq + KDA_ORACLE_L2NORM_EPS);",
     "qn = 1.0 / (sq + KDA_ORACLE_L2NORM_EPS);"),
    ("decay_after_write", None, None),  # built below: the decay moved after the rank-1 write
    # the L2-norm option (kernel-fun wheel, kda/autograd.py, use_qk_l2norm)
    ("l2norm_q_only", "kn = 1.0 / sqrt(sk + KDA_ORACLE_L2NORM_EPS);", "kn = 1.0;"),
    ("l2norm_k_takes_q_norm", "kn = 1.0 / sqrt(sk + KDA_ORACLE_L2NORM_EPS);", "kn = qn;"),
    ("l2norm_eps_outside_sqrt", "qn = 1.0 / sqrt(sq + KDA_ORACLE_L2NORM_EPS);\n"
     "                    kn = 1.0 / sqrt(sk + KDA_ORACLE_L2NORM_EPS);",
     "qn = 1.0 / (sqrt(sq) + KDA_ORACLE_L2NORM_EPS);\n"
     "                    kn = 1.0 / (sqrt(sk) + KDA_ORACLE_L2NORM_EPS);"),
    ("l2norm_over_first_head", "sq += qsrc[d] * qsrc[d];\n                        sk += ksrc[d] * ksrc[d];",
     "sq += q[(row * H) * (size_t)K + d] * q[(row * H) * (size_t)K + d];\n"
     "                        sk += k[(row * H) * (size_t)K + d] * k[(row * H) * (size_t)K + d];"),
    ("l2norm_half_the_channels", "                    for (int d = 0; d < K; ++d) {\n                        sq +=",
     "                    for (int d = 0; d < K / 2; ++d) {\n                        sq +="),
]


def _decay_after_write(src: str) -> str:
    decay_start = src.index("                /* S <- Diag(2^{g_t}) S */")
    decay_end = src.index("                /* delta <- beta_t (v_t - S^T k_t) */")
    block = src[decay_start:decay_end]
    src = src[:decay_start] + src[decay_end:]
    anchor = src.index("                /* o_t = scale * S^T q_t */")
    return src[:anchor] + block + src[anchor:]


def _build(text: str, tmp: str, name: str) -> str:
    c = os.path.join(tmp, f"{name}.c")
    so = os.path.join(tmp, f"{name}.so")
    with open(c, "w") as f:
        f.write(text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", c, "-o", so, "-lm"],
                   check=True, capture_output=True)
    return so


@pytest.mark.parametrize("name,orig,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, orig, new):
    src = open(SRC).read()
    if name == "decay_after_write":
        text = _decay_after_write(src)
    else:
        assert src.count(orig) >= 1, f"mutation anchor for {name} not found"
        text = src.replace(orig, new)
    with tempfile.TemporaryDirectory() as tmp:
        L = oracle._bind(_build(text, tmp, name))

        def rec(*a, **kw):
            return oracle.recurrent(*a, _library=L, **kw)

        failed = []
        for check in oracle_pins.ALL_CHECKS:
            try:
                with np.errstate(all="ignore"):
                    check(rec)
            except (AssertionError, ValueError, FloatingPointError):
                failed.append(check.__name__)
        assert failed, f"mutant {name} passed every pin"


CUMSUM_MUTANTS = [
    ("chunks_from_row_zero", "const long start = bos + chunk * ((t - bos) / chunk);",
     "const long start = chunk * (t / chunk);"),
    ("exclusive_sum", "for (long s = start; s <= t; ++s)", "for (long s = start; s < t; ++s)"),
    ("multiplier_dropped", "= g_scale * acc;", "= acc;"),
]


@pytest.mark.parametrize("name,orig,new", CUMSUM_MUTANTS, ids=[m[0] for m in CUMSUM_MUTANTS])
def test_cumsum_mutant_is_caught(name, orig, new):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation anchor for {name} not found"
    with tempfile.TemporaryDirectory() as tmp:
        L = oracle._bind(_build(src.replace(orig, new), tmp, name))
        failed = []
        for check in oracle_pins.CUMSUM_CHECKS:
            try:
                check(lambda *a, **kw: oracle.gate_cumsum(*a, _library=L, **kw))
            except (AssertionError, ValueError):
                failed.append(check.__name__)
        assert failed, f"mutant {name} passed every cumsum pin"


def test_unmutated_copy_passes_every_pin():
    with tempfile.TemporaryDirectory() as tmp:
        L = oracle._bind(_build(open(SRC).read(), tmp, "clean"))
        for check in oracle_pins.ALL_CHECKS:
            check(lambda *a, **kw: oracle.recurrent(*a, _library=L, **kw))
        for check in oracle_pins.CUMSUM_CHECKS:
            check(lambda *a, **kw: oracle.gate_cumsum(*a, _library=L, **kw))
