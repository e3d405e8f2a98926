"""The tcgen05 GEMM (both operand placements, split-K, ragged tiles) and the CUDA-core tile GEMM against a
plain PyTorch fp32 matrix product of the same bf16 operands."""
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
    l.fpd_test_gemm.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    l.fpd_test_gemm.restype = ctypes.c_int
    l.fpd_test_gemm_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    l.fpd_test_gemm_workspace_bytes.restype = ctypes.c_size_t
    l.fpd_test_swiglu.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_void_p, ctypes.c_void_p]
    l.fpd_test_swiglu.restype = ctypes.c_int
    return l


def run(lib, impl, placement, M, N, K, seed=0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = (0.02 * torch.randn(N, K, device="cuda", generator=g)).to(torch.bfloat16)
    C = torch.full((M, N), float("nan"), device="cuda")
    wsb = lib.fpd_test_gemm_workspace_bytes(M, N, K)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    st = lib.fpd_test_gemm(impl, placement, M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), ws.data_ptr(), wsb,
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
    assert run(lib, 0, -1, M, N, K) < 1e-5


@pytest.mark.parametrize("M,N,K,placement", [(15, 384, 512, 0), (300, 256, 512, 1), (100, 1100, 192, 1),
                                             (64, 640, 320, 0)])
def test_tc_gemm_forced_placement(lib, M, N, K, placement):
    assert run(lib, 0, placement, M, N, K, seed=1) < 1e-5


@pytest.mark.parametrize("M,N,K", [(15, 300, 256), (130, 70, 128)])
def test_simt_gemm(lib, M, N, K):
    assert run(lib, 1, -1, M, N, K, seed=2) < 1e-5


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


@pytest.mark.parametrize("variant", [1, 2, 3, 4])
@pytest.mark.parametrize("M,N,K", [(15, 6144, 2560), (16, 300, 320), (9, 1000, 704)])
def test_tc_gemm_pipeline_variants(lib, variant, M, N, K):
    """The other pipeline shapes of the 16-token weight-tile kernel (several K atoms per stage, tail stages
    with fewer atoms, 1 or 2 CTAs per SM) give the same products."""
    lib.fpd_test_set_variant.argtypes = [ctypes.c_int]
    lib.fpd_test_set_variant(variant)
    try:
        assert run(lib, 0, -1, M, N, K, seed=3) < 1e-5
    finally:
        lib.fpd_test_set_variant(0)
