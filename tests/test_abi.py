"""The C ABI without a GPU: the library loads, exports every symbol include/kda.h
declares, and rejects malformed arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_cumsum_gb300 import build as b

    b.build()
    import gated_delta_rule_cumsum_gb300 as kda

    return kda.load()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("kda_gate_cumsum", "kda_chunk_fwd", "kda_recurrent_fwd",
                 "kda_chunk_workspace_size", "kda_read_device_status", "kda_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in kda.h but not exported"


def test_binding_covers_every_declared_symbol():
    import gated_delta_rule_cumsum_gb300 as kda

    for name in _declared_functions():
        assert hasattr(kda, name), f"binding lacks {name}"


def test_status_strings(lib):
    import gated_delta_rule_cumsum_gb300 as kda

    assert kda.kda_status_string(0) == "KDA_OK"
    assert kda.kda_status_string(3) == "KDA_ERR_BAD_CU_SEQLENS"
    assert kda.kda_version().count(".") == 2


def _shape(**kw):
    import gated_delta_rule_cumsum_gb300 as kda

    d = dict(B=1, T=128, H=2, HV=4, K=64, V=64, num_seqs=1, dtype=1, scale=-1.0, g_scale=1.0,
             flags=0)
    d.update(kw)
    return kda.KdaShape(**d)


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: the host checks fail first


@pytest.mark.parametrize("kw,status", [
    (dict(HV=3), 1),              # HV % H != 0
    (dict(K=0), 1),
    (dict(num_seqs=2), 1),        # dense: num_seqs must equal B
    (dict(dtype=7), 1),
    (dict(flags=1 << 9), 2),      # unknown flag
    (dict(K=96, dtype=0), 2),     # fp32 chunk path: K in {64, 128}
    (dict(K=100), 2),             # bf16: K a multiple of 8 up to 128
    (dict(K=96, V=48), 2),        # bf16 with K outside {64, 128}: V a multiple of 32
    (dict(V=512), 2),
])
def test_chunk_fwd_rejects_on_host(lib, kw, status):
    s = _shape(**kw)
    st = lib.kda_chunk_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, ctypes.byref(s), FAKE, None,
                           FAKE, 1 << 30, None, None)
    assert st == status, lib.kda_last_error_message()
    assert lib.kda_last_error_message()


def test_chunk_fwd_rejects_small_or_misaligned_workspace(lib):
    s = _shape()
    need = lib.kda_chunk_workspace_size(ctypes.byref(s))
    assert need > 0
    st = lib.kda_chunk_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, ctypes.byref(s), FAKE, None,
                           ctypes.c_void_p(0x100000), need - 1, None, None)
    assert st == 1 and b"workspace" in lib.kda_last_error_message()
    st = lib.kda_chunk_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, ctypes.byref(s), FAKE, None,
                           ctypes.c_void_p(0x100010), need + 64, None, None)
    assert st == 1 and b"aligned" in lib.kda_last_error_message()


def test_packed_requires_batch_one(lib):
    s = _shape(B=2, num_seqs=3)
    st = lib.kda_recurrent_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, ctypes.byref(s), FAKE,
                               None, None, None)
    assert st == 1


def test_recurrent_rejects_cumsum_flag_and_large_k(lib):
    s = _shape(flags=2)
    assert lib.kda_recurrent_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, ctypes.byref(s), FAKE,
                                 None, None, None) == 2
    s = _shape(K=300)
    assert lib.kda_recurrent_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, ctypes.byref(s), FAKE,
                                 None, None, None) == 2


def test_null_tensors_rejected(lib):
    s = _shape()
    assert lib.kda_recurrent_fwd(None, FAKE, FAKE, FAKE, FAKE, None, None, ctypes.byref(s), FAKE,
                                 None, None, None) == 1
    assert lib.kda_gate_cumsum(FAKE, FAKE, None, None, 64, None, None) == 1


def test_gate_cumsum_rejects_alias_and_chunk(lib):
    s = _shape()
    assert lib.kda_gate_cumsum(FAKE, FAKE, None, ctypes.byref(s), 64, None, None) == 1
    assert lib.kda_gate_cumsum(FAKE, ctypes.c_void_p(0x2000), None, ctypes.byref(s), 65, None,
                               None) == 2


def test_split_scan_flag_sizes_a_larger_workspace(lib):
    """KDA_FLAG_SPLIT_SCAN on an eligible bf16 shape (few long sequences) adds
    the composition buffers: Q tiles per chunk slot, E0 and E1, P, and E0 as a
    bf16 operand tile; an ineligible shape (fp32) is unchanged."""
    import gated_delta_rule_cumsum_gb300 as kda

    base = dict(B=1, T=2048, H=2, HV=2, K=128, V=128, num_seqs=1, dtype=1)
    plain = lib.kda_chunk_workspace_size(ctypes.byref(_shape(**base)))
    split = lib.kda_chunk_workspace_size(ctypes.byref(_shape(**base, flags=kda.KDA_FLAG_SPLIT_SCAN)))
    slots, nh, K, V = 2048 // 64 + 1, 2, 128, 128
    extra = slots * nh * 64 * K * 2 + nh * (2 * K * V * 4 + K * K * 4 + K * V * 2)
    assert extra <= split - plain <= extra + 5 * 256
    f32 = dict(base, dtype=0)
    assert (lib.kda_chunk_workspace_size(ctypes.byref(_shape(**f32, flags=kda.KDA_FLAG_SPLIT_SCAN)))
            == lib.kda_chunk_workspace_size(ctypes.byref(_shape(**f32))))


@pytest.mark.parametrize("case", ["bias_without_a", "negative_beta_scale", "nan_beta_scale",
                                  "act_with_cumsum_input"])
def test_activation_arguments_rejected_on_host(lib, case):
    import gated_delta_rule_cumsum_gb300 as kda

    act = kda.KdaActivation(FAKE.value, FAKE.value, 0.0)
    flags = 0
    if case == "bias_without_a":
        act.A_log = None
    elif case == "negative_beta_scale":
        act.beta_scale = -1.0
    elif case == "nan_beta_scale":
        act.beta_scale = float("nan")
    else:
        flags = kda.KDA_FLAG_G_IS_CUMSUM
    s = _shape(flags=flags)
    st = lib.kda_chunk_fwd_act(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, ctypes.byref(s),
                               ctypes.byref(act), FAKE, None, FAKE, 1 << 30, None, None)
    assert st == 1, lib.kda_last_error_message()
    if case != "act_with_cumsum_input":
        assert lib.kda_recurrent_fwd_act(FAKE, FAKE, FAKE, FAKE, FAKE, None, None,
                                         ctypes.byref(_shape()), ctypes.byref(act), FAKE, None,
                                         None, None) == 1
        assert lib.kda_gate_cumsum_act(FAKE, ctypes.c_void_p(0x2000), None, ctypes.byref(_shape()),
                                       ctypes.byref(act), 64, None, None) == 1


def test_workspace_size_scales_with_chunks(lib):
    a = lib.kda_chunk_workspace_size(ctypes.byref(_shape(T=64)))
    b = lib.kda_chunk_workspace_size(ctypes.byref(_shape(T=640)))
    assert b > a > 0
    assert lib.kda_chunk_workspace_size(None) == 0


def test_product_never_imports_the_oracle():
    """The product path has no CPU fallback: neither the binding nor the CUDA
    sources mention the oracle."""
    pkg = os.path.join(ROOT, "gated_delta_rule_cumsum_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "kda_oracle" not in text, f


def _bwd(lib, s, grads=True, ws=(FAKE, 1 << 34)):
    g = FAKE if grads else None
    return lib.kda_recurrent_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, ctypes.byref(s), FAKE,
                                 None, g, g, g, g, g, None, ws[0], ws[1], None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(K=160), 2),                  # the backward keeps K <= 128
    (dict(flags=2), 2),                # KDA_FLAG_G_IS_CUMSUM
    (dict(HV=3), 1),
])
def test_recurrent_bwd_rejects_on_host(lib, kw, status):
    st = _bwd(lib, _shape(**kw))
    assert st == status, lib.kda_last_error_message()
    assert lib.kda_last_error_message()


def test_recurrent_bwd_needs_gradients_and_workspace(lib):
    s = _shape()
    assert _bwd(lib, s, grads=False) == 1
    assert b"dq" in lib.kda_last_error_message()
    need = lib.kda_recurrent_bwd_workspace_size(ctypes.byref(s))
    # B=1, T=128, H=2, HV=4, K=V=64: 16 (dense) or 16 + 1 + 1 (packed) checkpoint slots of
    # HV*K*V fp32, one per 8 tokens
    assert need == 18 * 4 * 64 * 64 * 4
    assert _bwd(lib, s, ws=(ctypes.c_void_p(0x100000), need - 1)) == 1
    assert b"workspace" in lib.kda_last_error_message()
    assert _bwd(lib, s, ws=(ctypes.c_void_p(0x100004), need)) == 1
    assert b"aligned" in lib.kda_last_error_message()


@pytest.mark.parametrize("case", ["bias_without_a", "negative_beta_scale", "no_dA_log",
                                  "no_ddt_bias"])
def test_recurrent_bwd_act_rejects_on_host(lib, case):
    import gated_delta_rule_cumsum_gb300 as kda

    act = kda.KdaActivation(FAKE.value, FAKE.value, 0.0)
    dA, ddt = FAKE, FAKE
    if case == "bias_without_a":
        act.A_log = None
    elif case == "negative_beta_scale":
        act.beta_scale = -2.0
    elif case == "no_dA_log":
        dA = None
    else:
        ddt = None
    g = FAKE
    st = lib.kda_recurrent_bwd_act(FAKE, FAKE, FAKE, FAKE, FAKE, None, None,
                                   ctypes.byref(_shape()), ctypes.byref(act), FAKE, None, g, g, g,
                                   g, g, None, dA, ddt, FAKE, 1 << 34, None, None)
    assert st == 1, lib.kda_last_error_message()
    assert lib.kda_last_error_message()
