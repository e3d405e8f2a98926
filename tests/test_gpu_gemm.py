"""Single kernels through the test hooks of include/fpd_testing.h against plain PyTorch fp32 references: the
tcgen05 GEMM (both operand placements, split-K, ragged tiles), the gate/up kernel with its SwiGLU epilogue, and the
two attention kernels (mma.sync 64-row tiles; tcgen05 128-row tiles with the accumulators in tensor memory)."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_diffusion_speculative_non_gb300 as pkg
    l = pkg.lib()
    l.fpd_test_gemm.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    l.fpd_test_gemm.restype = ctypes.c_int
    l.fpd_test_gemm_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    l.fpd_test_gemm_workspace_bytes.restype = ctypes.c_size_t
    l.fpd_test_swiglu.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_void_p, ctypes.c_void_p]
    l.fpd_test_swiglu.restype = ctypes.c_int
    i, vp = ctypes.c_int, ctypes.c_void_p
    l.fpd_test_attention.argtypes = [i, i, i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    l.fpd_test_attention.restype = ctypes.c_int
    l.fpd_test_attention_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
    l.fpd_test_attention_workspace_bytes.restype = ctypes.c_size_t
    return l


def run(lib, placement, M, N, K, seed=0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = (0.02 * torch.randn(N, K, device="cuda", generator=g)).to(torch.bfloat16)
    C = torch.full((M, N), float("nan"), device="cuda")
    wsb = lib.fpd_test_gemm_workspace_bytes(M, N, K)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    st = lib.fpd_test_gemm(placement, M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), ws.data_ptr(), wsb,
                           torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    ref = A.float() @ B.float().T
    err = ((C - ref).abs().max() / ref.abs().max()).item()
    return err


SHAPES = [
    (15, 6144, 2560),    # batch-1 text block QKV: weights on the 128-row operand, split-K
    (16, 300, 256),      # ragged weight tile
    (40, 1000, 640),     # 64-wide token tile, ragged
    (64, 2560, 9728),    # down projection at 64 tokens
    (385, 2560, 2560),   # primitive block: token tiles of 128, ragged tail, 256-wide weight tiles
    (200, 200, 128),     # 128-wide weight tiles, ragged in both
    (1, 128, 64),        # single token, single K block
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_tc_gemm_auto(lib, M, N, K):
    assert run(lib, -1, M, N, K) < 1e-5


@pytest.mark.parametrize("M,N,K,placement", [(15, 384, 512, 0), (300, 256, 512, 1), (100, 1100, 192, 1),
                                             (64, 640, 320, 0)])
def test_tc_gemm_forced_placement(lib, M, N, K, placement):
    assert run(lib, placement, M, N, K, seed=1) < 1e-5


@pytest.mark.parametrize("M,F,K", [(1, 256, 128), (15, 9728, 2560), (32, 320, 256), (64, 1536, 512),
                                   (65, 1536, 512), (385, 1000, 640)])
def test_tc_swiglu(lib, M, F, K):
    """Gate/up projection with the SwiGLU epilogue against silu(x Wg^T) * (x Wu^T) in fp32; the result is
    stored in bf16, so it must agree within a bf16 rounding step of the fp32 reference."""
    g = torch.Generator(device="cuda").manual_seed(M + F)
    X = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    W = (0.05 * torch.randn(2 * F, K, device="cuda", generator=g)).to(torch.bfloat16)
    H = torch.full((M, F), float("nan"), device="cuda", dtype=torch.bfloat16)
    st = lib.fpd_test_swiglu(M, F, K, X.data_ptr(), W.data_ptr(), H.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    gu = X.float() @ W.float().T
    ref = torch.nn.functional.silu(gu[:, :F]) * gu[:, F:]
    err = ((H.float() - ref).abs() / (ref.abs() + 1e-3 * ref.abs().max())).max().item()
    assert err < 1e-2, err


def attention_ref(q, kblk, vblk, store, ctx_len, layer, nkv):
    """softmax(q [K_ctx ; K_blk]^T / sqrt(h)) [V_ctx ; V_blk] in fp32, per request and q head."""
    B, nkv_, L, h = kblk.shape
    nq = q.shape[1]
    grp = nq // nkv
    out = torch.empty(B * L, nq, h, device=q.device)
    for b in range(B):
        T = int(ctx_len[b])
        for i in range(nq):
            g = i // grp
            K = torch.cat([store[layer, b, 0, g, :T], kblk[b, g]]).float()
            V = torch.cat([store[layer, b, 1, g, :T], vblk[b, g]]).float()
            s = q[b * L:(b + 1) * L, i].float() @ K.T / h ** 0.5
            out[b * L:(b + 1) * L, i] = torch.softmax(s, dim=1) @ V
    return out


ATTN_CASES = [
    # B, L, nq, nkv, h, t_cap, ctx lengths
    (1, 385, 32, 8, 128, 4096, [4096]),            # special-token primitive: long context, KV splits
    (2, 381, 32, 8, 128, 700, [537, 0]),           # fixed-width primitive, ragged, one request without context
    (1, 32, 32, 8, 128, 130, [129]),               # one 128-row query tile, context tile of one key
    (3, 40, 8, 2, 128, 300, [300, 1, 77]),         # GQA group 4, partial tiles everywhere
]


def run_attention(lib, impl, B, L, nq, nkv, h, t_cap, ctx, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    layer = 1
    q = torch.randn(B * L, nq, h, device="cuda", generator=g).to(torch.bfloat16)
    kblk = torch.randn(B, nkv, L, h, device="cuda", generator=g).to(torch.bfloat16)
    vblk = torch.randn(B, nkv, L, h, device="cuda", generator=g).to(torch.bfloat16)
    store = torch.randn(layer + 1, B, 2, nkv, t_cap, h, device="cuda", generator=g).to(torch.bfloat16)
    ctx_len = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    out = torch.full((B * L, nq, h), float("nan"), device="cuda", dtype=torch.bfloat16)
    wsb = lib.fpd_test_attention_workspace_bytes(impl, B, L, nq, nkv, h, t_cap)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    st = lib.fpd_test_attention(impl, B, L, nq, nkv, h, t_cap, layer, ctx_len.data_ptr(), q.data_ptr(),
                                kblk.data_ptr(), vblk.data_ptr(), store.data_ptr(), out.data_ptr(), ws.data_ptr(),
                                wsb, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    ref = attention_ref(q, kblk, vblk, store, ctx, layer, nkv)
    return ((out.float() - ref).abs().amax(dim=2) / ref.abs().amax(dim=2)).max().item()


@pytest.mark.parametrize("B,L,nq,nkv,h,t_cap,ctx", ATTN_CASES)
def test_attention_kernels_agree_with_fp32(lib, B, L, nq, nkv, h, t_cap, ctx):
    """Both attention kernels against a plain fp32 softmax attention of the same bf16 inputs.  Each stores bf16
    (half an ulp: 2e-3 of the row's largest value) after a second product on P split into bf16 hi + lo terms, so
    the row error stays within a few bf16 rounding steps; the tcgen05 kernel must be as accurate as the mma.sync
    one."""
    errs = [run_attention(lib, impl, B, L, nq, nkv, h, t_cap, ctx, seed=B * 1000 + L) for impl in (0, 1)]
    print(f"attention row error: mma.sync {errs[0]:.3e}, tcgen05 {errs[1]:.3e}")
    assert errs[0] < 6e-3 and errs[1] < 6e-3, errs
    assert errs[1] < 1.5 * errs[0] + 1e-3, errs


@pytest.mark.parametrize("B,L,nq,nkv,h,t_cap,ctx", [(1, 16, 32, 8, 128, 2048, [2048]), (2, 33, 8, 2, 64, 96, [96, 5])])
def test_attention_mma_sync_small_blocks(lib, B, L, nq, nkv, h, t_cap, ctx):
    assert run_attention(lib, 0, B, L, nq, nkv, h, t_cap, ctx, seed=7) < 6e-3


SHORT_CASES = [
    # few-token blocks: at most 64 query rows per (request, kv head)
    (1, 16, 32, 8, 128, 2048, [2048]),       # the batch-1 text workload
    (1, 16, 32, 8, 128, 16384, [16384]),     # the longest context of the sweep
    (1, 16, 32, 8, 128, 300, [0]),           # no context: block keys only
    (1, 2, 32, 8, 128, 130, [1]),            # two positions, one context key
    (2, 5, 8, 2, 64, 96, [96, 5]),           # tiny drafter shape, ragged
]


@pytest.mark.parametrize("B,L,nq,nkv,h,t_cap,ctx", SHORT_CASES)
def test_attention_short_cluster_kernel(lib, B, L, nq, nkv, h, t_cap, ctx):
    """The few-token cluster kernel against fp32, as accurate as the mma.sync tiles (same per-tile math)."""
    errs = [run_attention(lib, impl, B, L, nq, nkv, h, t_cap, ctx, seed=B * 100 + L) for impl in (0, 2)]
    print(f"short attention row error: mma.sync {errs[0]:.3e}, cluster {errs[1]:.3e}")
    assert errs[1] < 6e-3 and errs[1] < 1.5 * errs[0] + 1e-3, errs


@pytest.mark.parametrize("B,L,nq,nkv,h,t_cap,ctx", SHORT_CASES)
def test_attention_short_covers_every_key_once(lib, B, L, nq, nkv, h, t_cap, ctx):
    test_attention_covers_every_key_once(lib, 2, B, L, nq, nkv, h, t_cap, ctx)


@pytest.mark.parametrize("impl", [0, 1])
@pytest.mark.parametrize("B,L,nq,nkv,h,t_cap,ctx", [(1, 385, 32, 8, 128, 4096, [4096]), (2, 381, 32, 8, 128, 700, [537, 0]),
                                                    (3, 40, 8, 2, 128, 300, [300, 1, 77])])
def test_attention_covers_every_key_once(lib, impl, B, L, nq, nkv, h, t_cap, ctx):
    """K = 0 makes every weight equal (p = 1 exactly, l = T + L exactly), and V[t][d] = 1 when t % h == d, so output
    dimension d counts the keys t (context and block) with t % h == d, divided by T + L.  A key dropped or read twice
    at a tile or split boundary moves one count by 1 (about 3 % here); correct kernels land within bf16 rounding."""
    g = torch.Generator(device="cuda").manual_seed(11)
    layer = 1
    q = torch.randn(B * L, nq, h, device="cuda", generator=g).to(torch.bfloat16)
    kblk = torch.zeros(B, nkv, L, h, device="cuda", dtype=torch.bfloat16)
    onehot = lambda n: (torch.arange(n, device="cuda")[:, None] % h == torch.arange(h, device="cuda")[None, :])
    vblk = onehot(L).to(torch.bfloat16)[None, None].expand(B, nkv, L, h).contiguous()
    store = torch.zeros(layer + 1, B, 2, nkv, t_cap, h, device="cuda", dtype=torch.bfloat16)
    store[:, :, 1] = onehot(t_cap).to(torch.bfloat16)
    ctx_len = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    out = torch.full((B * L, nq, h), float("nan"), device="cuda", dtype=torch.bfloat16)
    wsb = lib.fpd_test_attention_workspace_bytes(impl, B, L, nq, nkv, h, t_cap)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    assert lib.fpd_test_attention(impl, B, L, nq, nkv, h, t_cap, layer, ctx_len.data_ptr(), q.data_ptr(),
                                  kblk.data_ptr(), vblk.data_ptr(), store.data_ptr(), out.data_ptr(), ws.data_ptr(),
                                  wsb, torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    for b in range(B):
        T = ctx[b]
        cnt = onehot(T).float().sum(0) + onehot(L).float().sum(0)
        want = (cnt / (T + L))[None, None, :]
        got = out[b * L:(b + 1) * L].float()
        err = ((got - want).abs().max() / want.abs().max()).item()
        assert err < 5e-3, (b, err)
