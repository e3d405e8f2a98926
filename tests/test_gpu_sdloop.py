"""GPU: the multi-block text speculative loop and failure detection.

The loop (draft -> argmax -> target row -> verify -> advance -> append of the accepted rows' features) runs K steps
inside one captured CUDA graph, which also keeps a copy of the context K/V store at the start of every step; the
oracle then checks every stage of every step on the GPU's own inputs (reading R21): the block pass on the store the
GPU held, the LM head and argmax on the GPU's hidden states (ids exact above the 1e-2 margin), the synthetic target
row, the verification, the context bookkeeping (positions, lengths, next anchors) and the append, i.e. the store
after the step against the oracle's append of the accepted rows to the store before it.
(VFlash blog "Method"; FlashDrive §3.2; VFlash paper (zh) §2.2.)
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from _util import (assert_logits, assert_rows_close, assert_tokens, bits_of, synthetic_target)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_diffusion_speculative_non_gb300 as p
    l = p.lib()
    vp = ctypes.c_void_p
    l.fpd_test_synthetic_target.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, ctypes.c_uint32, vp, vp]
    l.fpd_test_synthetic_target.restype = ctypes.c_int
    l.fpd_test_stream_timeout.argtypes = [vp, ctypes.c_size_t, vp]
    l.fpd_test_stream_timeout.restype = ctypes.c_int
    l.fpd_test_stream_timeout_workspace_bytes.restype = ctypes.c_size_t
    return p


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def _run_loop(pkg, orc, shape, w, ctx0, anchor0, L, K, t_cap, seed):
    B = len(ctx0)
    rng = np.random.default_rng(seed)
    agree = np.minimum(rng.geometric(0.35, size=(K, B)) - 1, L - 1).astype(np.int32)
    salts = rng.integers(1, 2**31, size=K)
    feats = [synth.make_features(shape, B * L, seed + 1 + k) for k in range(K)]
    off0 = np.concatenate([[0], np.cumsum(ctx0)]).astype(np.int32)
    f0 = synth.make_features(shape, int(off0[-1]), seed)

    # ---- GPU: initial context, then K steps captured in one graph and replayed once ----
    dr = pkg.Drafter(shape, w, B, L, t_cap, device=DEV)
    if off0[-1] > 0:
        dr.prepare_context(B, off0, f0)
    st = dr.spec_state(B, L, ctx0, anchor0)
    agree_d = torch.from_numpy(agree).to(DEV)
    feats_d = [[torch.from_numpy(f.view(np.int16)).to(DEV).view(torch.bfloat16) for f in fk] for fk in feats]
    V = shape.vocab
    bufs = {"hid": torch.empty(K, B * L, shape.d_model, dtype=torch.bfloat16, device=DEV),
            "tok": torch.empty(K, B, L - 1, dtype=torch.int32, device=DEV),
            "tgt": torch.empty(K, B, L, dtype=torch.int32, device=DEV),
            "acc": torch.empty(K, B, dtype=torch.int32, device=DEV),
            "com": torch.empty(K, B, L, dtype=torch.int32, device=DEV),
            "ctx": torch.empty(K, B, dtype=torch.int32, device=DEV),
            "anc": torch.empty(K, B, dtype=torch.int32, device=DEV),
            "pos": torch.empty(K, B, dtype=torch.int32, device=DEV),
            "log": torch.empty(K, B * (L - 1), V, dtype=torch.float32, device=DEV),
            "kv": torch.empty((K + 1,) + tuple(dr.kv_view(B).shape), dtype=torch.bfloat16, device=DEV)}
    lib = pkg.lib()
    step = [0]

    def record(s):
        k = step[0]
        bufs["hid"][k].copy_(s.hidden)
        bufs["tok"][k].copy_(s.tokens)
        bufs["tgt"][k].copy_(s.target)
        bufs["acc"][k].copy_(s.accept)
        bufs["com"][k].copy_(s.committed)

    st.hooks.append(record)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        for k in range(K):
            step[0] = k

            def make_target(tok, tgt, k=k):
                assert lib.fpd_test_synthetic_target(B, L, V, tok.data_ptr(), agree_d[k].data_ptr(),
                                                     int(salts[k]), tgt.data_ptr(), cs.cuda_stream) == 0

            bufs["kv"][k].copy_(dr.kv_view(B))
            dr.spec_step(st, feats_d[k], make_target, V - 1, stream=cs, logits_out=bufs["log"][k])
            bufs["ctx"][k].copy_(st.ctx_len)
            bufs["anc"][k].copy_(st.anchor)
            bufs["pos"][k].copy_(st.pos_start)
        bufs["kv"][K].copy_(dr.kv_view(B))
    g.replay()
    torch.cuda.synchronize()
    assert pkg.fpd_device_status() == 0
    H = {k: v.cpu() for k, v in bufs.items()}

    # ---- oracle: every stage of every step on the GPU's inputs ----
    om = orc.Model(shape, w)
    kv0 = orc.prepare_context(om, off0, f0, t_cap, batch=B) if off0[-1] > 0 else \
        np.zeros((shape.n_layers, B, 2, shape.n_kv_heads, t_cap, shape.head_dim), np.uint16)
    g_kv = bits_of(H["kv"])
    for b in range(B):                                   # the initial preparation
        T = int(ctx0[b])
        if T:
            assert_rows_close(g_kv[0][:, b, :, :, :T].reshape(-1, shape.head_dim),
                              kv0[:, b, :, :, :T].reshape(-1, shape.head_dim), f"initial store request {b}")
    ctx, anchor = np.array(ctx0, np.int32), np.array(anchor0, np.int32)
    accepted = []
    for k in range(K):
        kv_k = np.ascontiguousarray(g_kv[k])
        o_hid = orc.draft_block(om, kv_k, t_cap, ctx, anchor, V - 1, L)
        g_hid = bits_of(H["hid"][k])
        assert_rows_close(g_hid, o_hid, f"step {k} hidden (on the GPU's store)")
        o_tok, o_margin, o_log = orc.constrain_argmax(om, g_hid, B, L, want_logits=True)
        tok = H["tok"][k].numpy()
        g_log = H["log"][k].numpy()
        assert_logits(g_log, o_log, f"step {k} logits (on the GPU's hidden)")
        assert_tokens(tok, o_tok, o_margin, f"step {k} ids (on the GPU's hidden)")
        target = synthetic_target(tok, agree[k], int(salts[k]), V)
        np.testing.assert_array_equal(H["tgt"][k].numpy(), target)
        oacc, ocom, _ = orc.verify(0, tok, target)
        np.testing.assert_array_equal(H["acc"][k].numpy(), oacc)
        np.testing.assert_array_equal(H["com"][k].numpy(), ocom)
        pos = ctx.copy()
        ctx = ctx + oacc
        anchor = ocom[np.arange(B), oacc - 1].astype(np.int32)
        np.testing.assert_array_equal(H["pos"][k].numpy(), pos)
        np.testing.assert_array_equal(H["ctx"][k].numpy(), ctx)
        np.testing.assert_array_equal(H["anc"][k].numpy(), anchor)
        # the append: the target's features at the anchor and the accepted drafts join the context
        off = np.concatenate([[0], np.cumsum(oacc)]).astype(np.int32)
        rows = [f[np.concatenate([np.arange(b * L, b * L + oacc[b]) for b in range(B)])] for f in feats[k]]
        want = orc.prepare_context(om, off, rows, t_cap, batch=B, pos_start=pos, kv_store=kv_k.copy())
        got = g_kv[k + 1]
        for b in range(B):
            new_rows = slice(int(pos[b]), int(ctx[b]))
            assert_rows_close(got[:, b, :, :, new_rows].reshape(-1, shape.head_dim),
                              want[:, b, :, :, new_rows].reshape(-1, shape.head_dim), f"step {k} append request {b}")
            np.testing.assert_array_equal(got[:, b, :, :, :int(pos[b])], kv_k[:, b, :, :, :int(pos[b])])
        accepted.append(oacc)
    dr.close()
    return np.array(accepted)


def test_tiny_speculative_loop_in_one_graph(pkg, orc):
    """Tiny drafter, three requests (one starting with an empty context), blocks of 8, six steps in one graph."""
    s = synth.TINY
    w = synth.make_weights(s, 6100)
    acc = _run_loop(pkg, orc, s, w, np.array([40, 0, 97], np.int32), np.array([3, 4000, 77], np.int32), 8, 6, 160,
                    6101)
    assert acc.shape == (6, 3) and acc.min() >= 1 and acc.max() <= 8
    assert (acc > 1).any()   # some steps accept drafted positions, not only the target's token


def test_full_speculative_loop_few_token(pkg, orc, full_weights):
    """4B-shape drafter, one request, context 2048, blocks of 16 (the few-token path), three steps in one graph."""
    _run_loop(pkg, orc, synth.FULL, full_weights, np.array([2048], np.int32), np.array([1234], np.int32), 16, 3,
              2048 + 3 * 16, 6201)


def test_bounded_wait_timeout_is_reported(pkg):
    """A weight stage declared 16 bytes larger than its copy: the MMA warp's bounded wait gives up after 1 s, the
    kernel returns, fpd_device_status reports FPD_CHECK_WAIT_TIMEOUT (2), and the context keeps working."""
    lib = pkg.lib()
    n = int(lib.fpd_test_stream_timeout_workspace_bytes())
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    cs = torch.cuda.current_stream().cuda_stream
    assert lib.fpd_test_stream_timeout(ws.data_ptr(), n, cs) == 0
    torch.cuda.synchronize()
    assert pkg.fpd_device_status() == 2
    assert pkg.fpd_device_status() == 0   # read and cleared
    # the library's next kernel on the same context computes normally
    draft = torch.randint(0, 1000, (4, 15), dtype=torch.int32, device=DEV)
    agree = torch.tensor([0, 3, 15, 7], dtype=torch.int32, device=DEV)
    tgt = torch.empty(4, 16, dtype=torch.int32, device=DEV)
    assert lib.fpd_test_synthetic_target(4, 16, 1000, draft.data_ptr(), agree.data_ptr(), 99, tgt.data_ptr(), cs) == 0
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tgt.cpu().numpy(), synthetic_target(draft.cpu().numpy(), agree.cpu().numpy(), 99, 1000))
    assert pkg.fpd_device_status() == 0
