"""The C ABI library loads, exports every entry point include/fpd.h declares, and rejects bad arguments on the
host with the documented status codes before launching anything.  No GPU needed."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fpd.h")


@pytest.fixture(scope="module")
def fpd():
    import __graft_entry__ as g
    g._compile_all()
    import block_diffusion_speculative_non_gb300 as pkg
    return pkg


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fpd_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(fpd):
    names = header_functions()
    assert len(names) >= 11
    lib = ctypes.CDLL(fpd.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(fpd._EXPORTS)


def _desc(fpd, **kw):
    d = dict(n_layers=5, d_model=512, n_q_heads=8, n_kv_heads=2, head_dim=64, d_ff=1536, vocab=4096, n_feat=3,
             max_pos=256, rms_eps=1e-6, rope_theta=1e6)
    d.update(kw)
    return fpd.ModelDesc(**d)


def _weights(fpd, null=None):
    w = fpd.Weights()
    addr = 1 << 20
    for name in ("embed", "w_fc", "hidden_norm", "final_norm", "lm_head"):
        setattr(w, name, None if name == null else addr)
    for name in ("attn_norm", "wqkv", "q_norm", "k_norm", "wo", "mlp_norm", "w_gate_up", "w_down"):
        arr = getattr(w, name)
        for l in range(8):
            arr[l] = None if name == null else addr
    return w


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), 4), (dict(n_layers=0), 4), (dict(n_layers=9), 4), (dict(d_model=500), 4),
    (dict(n_q_heads=6, n_kv_heads=4), 4), (dict(n_feat=0), 4), (dict(vocab=1), 2), (dict(max_pos=1), 2),
    (dict(rms_eps=0.0), 2), (dict(d_model=16448, d_ff=64), 4),
])
def test_model_create_rejects_bad_shapes(fpd, kw, status):
    h = ctypes.c_void_p()
    st = fpd.lib().fpd_model_create(ctypes.byref(_desc(fpd, **kw)), ctypes.byref(_weights(fpd)), ctypes.byref(h))
    assert st == status, fpd.fpd_last_error()
    assert h.value is None
    assert fpd.fpd_last_error()


@pytest.mark.parametrize("null", ["embed", "lm_head", "wqkv", "w_down"])
def test_model_create_rejects_null_weights(fpd, null):
    h = ctypes.c_void_p()
    st = fpd.lib().fpd_model_create(ctypes.byref(_desc(fpd)), ctypes.byref(_weights(fpd, null)), ctypes.byref(h))
    assert st == 1


def test_model_create_rejects_misaligned_weight(fpd):
    w = _weights(fpd)
    w.lm_head = (1 << 20) + 2
    h = ctypes.c_void_p()
    assert fpd.lib().fpd_model_create(ctypes.byref(_desc(fpd)), ctypes.byref(w), ctypes.byref(h)) == 1


def test_null_model_calls(fpd):
    l = fpd.lib()
    assert l.fpd_draft_block(None, 1, 16, 16, 8, 16, 16, 0, 16, None, 16, 1, None) == 1
    assert l.fpd_constrain_argmax(None, 1, 16, 16, None, 16, None, None, 16, 1, None) == 1
    assert l.fpd_constrain_argmax_noalloc(None, 1, 16, 16, None, 16, None, None) == 1
    arr = (ctypes.c_void_p * 1)(16)
    assert l.fpd_prepare_context(None, 1, 1, 16, None, arr, 16, 8, 16, 1, None) == 1
    assert l.fpd_kv_store_bytes(None, 1, 1) == 0
    assert l.fpd_workspace_bytes(None, 1, 16, 1) == 0


def test_verify_host_validation(fpd):
    l = fpd.lib()
    D, T, A, C = 16, 32, 48, 64     # fake (never dereferenced) device addresses
    assert l.fpd_verify(7, 1, 16, D, T, None, None, -1, A, C, None, None) == 1          # bad mode
    assert l.fpd_verify(0, 0, 16, D, T, None, None, -1, A, C, None, None) == 2          # empty batch
    assert l.fpd_verify(0, 1, 1, D, T, None, None, -1, A, C, None, None) == 2           # L < 2
    assert l.fpd_verify(0, 1, 16, None, T, None, None, -1, A, C, None, None) == 1       # null draft
    assert l.fpd_verify(0, 1, 16, D, None, None, None, -1, A, C, None, None) == 1       # text needs target
    assert l.fpd_verify(1, 1, 16, D, None, None, None, -1, A, C, None, None) == 1       # schema needs layout


def _layout(fpd, off, rng, pos=16):
    return fpd.make_layout(off, rng, pos)


@pytest.mark.parametrize("off,rng,status", [
    ([0, 1], [5, 5], 2),                 # empty range
    ([0, 1], [-1, 5], 2),                # negative id
    ([1, 2], [0, 5], 2),                 # class_off[0] != 0
    ([0, 0], [0, 5], 2),                 # class without a range
    ([0, 2], [10, 20, 5, 8], 2),         # ranges not sorted
    ([0, 2], [10, 20, 15, 30], 2),       # ranges overlap
    ([0, 65], list(range(0, 130)), 3),   # more than FPD_MAX_RANGES ranges
])
def test_layout_validation(fpd, off, rng, status):
    l = fpd.lib()
    lay = _layout(fpd, off, rng)
    st = l.fpd_verify(1, 1, 16, 16, None, ctypes.byref(lay), 32, -1, 48, 64, None, None)
    assert st == status, fpd.fpd_last_error()


def test_layout_too_many_classes(fpd):
    off = list(range(34))
    rng = [v for i in range(33) for v in (2 * i, 2 * i + 1)]
    lay = _layout(fpd, off, rng)
    assert fpd.lib().fpd_verify(1, 1, 16, 16, None, ctypes.byref(lay), 32, -1, 48, 64, None, None) == 3


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    """The product path has no fallback: a missing libfpd.so is an error, not a CPU path."""
    import block_diffusion_speculative_non_gb300 as pkg
    monkeypatch.setattr(pkg, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(pkg, "_lib", None)
    with pytest.raises(RuntimeError):
        pkg.lib()


def test_speculative_step_calls_reject_bad_arguments(fpd):
    """fpd_sd_advance and fpd_prepare_context_rows validate on the host before launching anything."""
    lib = fpd.lib()
    a = 1 << 20
    assert lib.fpd_sd_advance(0, 16, 64, a, a, a, a, a, None) == 2
    assert lib.fpd_sd_advance(1, 1, 64, a, a, a, a, a, None) == 2
    assert lib.fpd_sd_advance(1, 16, 64, None, a, a, a, a, None) == 1
    assert lib.fpd_sd_advance(1, 16, 64, a, a, a, None, a, None) == 1
    feats = (ctypes.c_void_p * 1)(a)
    assert lib.fpd_prepare_context_rows(None, 1, 4, a, a, None, feats, a, 64, a, 1 << 20, None) == 1


def test_fp8_calls_validate_on_the_host(fpd):
    """fpd_model_enable_fp8 and fpd_quantize_fp8 reject bad arguments before touching the device."""
    lib = fpd.lib()
    a = 1 << 20
    assert lib.fpd_model_enable_fp8(None, None) == 1
    assert lib.fpd_model_fp8_enabled(None) == 0
    assert lib.fpd_quantize_fp8(None, 4, 128, 128, a, a, None) == 1
    assert lib.fpd_quantize_fp8(a, 4, 100, 128, a, a, None) == 2      # cols not a multiple of 128
    assert lib.fpd_quantize_fp8(a, 4, 128, 120, a, a, None) == 2      # ld < cols
    assert lib.fpd_quantize_fp8(a, 0, 128, 128, a, a, None) == 2
    assert lib.fpd_quantize_fp8(a + 8, 4, 128, 128, a, a, None) == 1  # misaligned source
