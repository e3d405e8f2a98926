"""fpd_constrain_argmax_noalloc against fpd_constrain_argmax, through the C ABI.

The no-allocation entry point is for callers that cannot call cudaMalloc (a host framework that owns the whole
device heap, or a loop that must not pay cudaMalloc's device synchronisation): it keeps its scratch in a static
device array inside the library instead of a caller-supplied workspace.  Its results must equal those of the
workspace entry point on the same inputs, call after call, because every call reuses that one array.

This file is collected last on purpose, and it must pass both on its own in a fresh process (where the first
call sets the array's address up) and after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from _util import REL_TOL, row_rel_err

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_diffusion_speculative_non_gb300 as p
    p.lib()
    return p


def _call_both(pkg, dr, batch, L, hidden, layout):
    s = dr.shape
    lib = pkg.lib()
    st = torch.cuda.current_stream().cuda_stream
    lay = ctypes.byref(layout) if layout is not None else None
    tok_ref = torch.full((batch, L - 1), -7, dtype=torch.int32, device=DEV)
    tok = torch.full((batch, L - 1), -7, dtype=torch.int32, device=DEV)
    log_ref = torch.full((batch * (L - 1), s.vocab), float("nan"), dtype=torch.float32, device=DEV)
    log = torch.full_like(log_ref, float("nan"))
    assert lib.fpd_constrain_argmax(dr.handle, batch, L, hidden.data_ptr(), lay, tok_ref.data_ptr(),
                                    log_ref.data_ptr(), None, dr.workspace.data_ptr(), dr.ws_bytes, st) == 0, \
        pkg.fpd_last_error()
    assert lib.fpd_constrain_argmax_noalloc(dr.handle, batch, L, hidden.data_ptr(), lay, tok.data_ptr(),
                                            log.data_ptr(), st) == 0, pkg.fpd_last_error()
    torch.cuda.synchronize()
    assert pkg.fpd_device_status() == 0
    t_ref, t = tok_ref.cpu().numpy(), tok.cpu().numpy()
    np.testing.assert_array_equal(t, t_ref)
    assert (t >= 0).all()
    a, b = log.cpu().numpy(), log_ref.cpu().numpy()
    np.testing.assert_array_equal(np.isnan(a), np.isnan(b))          # the same legal columns were computed
    legal = ~np.isnan(b)
    err = row_rel_err(np.where(legal, a, 0.0), np.where(legal, b, 0.0))
    assert err.max() <= REL_TOL, err.max()
    return t


def test_noalloc_matches_workspace_entry_point_twice(pkg):
    s = synth.TINY
    w = synth.make_weights(s, 9001)
    lay_np = synth.layout_special_tokens(s.vocab, n_waypoints=3, coord_lo=2000, n_coord=1001, delim_id=3100,
                                         start_id=3101)
    L2 = lay_np["block_len"]
    dr = pkg.Drafter(s, w, 3, max(16, L2), 64, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(9002)
    # first call: unconstrained vocabulary, 2 requests of 16 positions
    h1 = torch.randn(2 * 16, s.d_model, device=DEV, generator=g).to(torch.bfloat16)
    _call_both(pkg, dr, 2, 16, h1, None)
    # second call in a row: a constrained layout over 3 requests; the array still holds the first call's data
    h2 = torch.randn(3 * L2, s.d_model, device=DEV, generator=g).to(torch.bfloat16)
    lay, _ = pkg.Drafter.layout(lay_np, 3, L2, DEV)
    t = _call_both(pkg, dr, 3, L2, h2, lay)
    coord = (t >= 2000) & (t < 3001)
    assert np.all(coord | (t == 3100))
    dr.close()


def test_noalloc_rejects_sizes_beyond_the_static_array(pkg):
    s = synth.FULL
    desc = pkg.ModelDesc(s.n_layers, s.d_model, s.n_q_heads, s.n_kv_heads, s.head_dim, s.d_ff, s.vocab, s.n_feat,
                         4096, s.rms_eps, s.rope_theta)
    # weights are never read: the call must fail on the host before any launch
    buf = torch.empty(64, dtype=torch.uint8, device=DEV)
    W = pkg.Weights()
    for k in ("embed", "w_fc", "hidden_norm", "final_norm", "lm_head"):
        setattr(W, k, buf.data_ptr())
    for k in ("attn_norm", "wqkv", "q_norm", "k_norm", "wo", "mlp_norm", "w_gate_up", "w_down"):
        arr = getattr(W, k)
        for l in range(s.n_layers):
            arr[l] = buf.data_ptr()
    h = pkg.fpd_model_create(desc, W)
    try:
        st = pkg.lib().fpd_constrain_argmax_noalloc(h, 64, 385, buf.data_ptr(), None, buf.data_ptr(), None,
                                                   torch.cuda.current_stream().cuda_stream)
        assert st == 3                                                        # FPD_ERR_CAPACITY
        assert "bytes" in pkg.fpd_last_error()
    finally:
        pkg.fpd_model_destroy(h)
