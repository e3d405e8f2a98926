"""Launch plans (host only, no GPU): the tile widths, K splits and grids the library picks for its GEMMs and
attention, checked for the invariants the kernels rely on over many shapes, and pinned at the shapes whose choice
the design documents (the 385-row QKV on 256-wide tiles, the 2048-row fusion GEMM in 4 K splits, ...)."""
import ctypes
import math

import pytest

KIND_GEMM, KIND_TOK, KIND_SWIGLU, KIND_STREAM = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g._compile_all()
    import block_diffusion_speculative_non_gb300 as pkg
    l = ctypes.CDLL(pkg.LIB_PATH)
    l.fpd_test_plan.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_int32)]
    l.fpd_test_plan.restype = ctypes.c_int
    l.fpd_test_attn_plan.argtypes = [ctypes.c_int] * 7 + [ctypes.POINTER(ctypes.c_int32)] * 2
    l.fpd_test_attn_plan.restype = ctypes.c_int
    return l


def plan(lib, kind, M, N, K, sms=152):
    out = (ctypes.c_int32 * 7)()
    assert lib.fpd_test_plan(kind, M, N, K, sms, out) == 0
    return dict(zip(("swap", "bn", "pt", "qt", "splits", "k_split", "grid"), list(out)))


def attn_plan(lib, impl, B, L, nq, nkv, t_cap, sms=152):
    s, c = ctypes.c_int32(), ctypes.c_int32()
    assert lib.fpd_test_attn_plan(impl, B, L, nq, nkv, t_cap, sms, ctypes.byref(s), ctypes.byref(c)) == 0
    return s.value, c.value


ROWS = [1, 5, 16, 17, 33, 64, 65, 100, 128, 129, 160, 256, 257, 385, 1000, 1024, 1540, 2048, 4096, 12192, 24640]
# (N, K) of the 4B-shape and tiny drafters' projections: QKV, O, down, context fusion, every layer's K/V
GEMMS = [(6144, 2560), (2560, 4096), (2560, 9728), (2560, 12800), (10240, 2560), (768, 512), (512, 512),
         (512, 1536)]


def _check_k(p, K):
    assert p["k_split"] % 64 == 0 and p["k_split"] >= 64
    assert p["splits"] >= 1
    assert p["splits"] * p["k_split"] >= K, "the splits cover K"
    assert (p["splits"] - 1) * p["k_split"] < K, "no split is empty"


@pytest.mark.parametrize("sms", [152, 148, 132])
def test_gemm_plans_are_consistent(lib, sms):
    for M in ROWS:
        for N, K in GEMMS:
            p = plan(lib, KIND_GEMM, M, N, K, sms)
            _check_k(p, K)
            slots = sms * (2 if p["swap"] else 1)
            assert p["swap"] == (M <= 64)
            if p["swap"]:
                assert p["bn"] in (16, 32, 64) and p["bn"] >= min(M, 64)
                assert p["pt"] == math.ceil(N / 128) and p["qt"] == math.ceil(M / p["bn"])
            else:
                assert p["bn"] in (128, 256)
                assert p["pt"] == math.ceil(M / 128) and p["qt"] == math.ceil(N / p["bn"])
            tiles = p["pt"] * p["qt"]
            assert p["grid"] == min(tiles * p["splits"], slots) and p["grid"] >= 1
            if not p["swap"] and 2 * tiles > slots:
                # a split is taken only when it shortens the waves of K work
                nkb = K // 64
                assert math.ceil(tiles * p["splits"] / slots) * math.ceil(nkb / p["splits"]) <= \
                    math.ceil(tiles / slots) * nkb


@pytest.mark.parametrize("sms", [152, 132])
def test_token_tile_plans_are_consistent(lib, sms):
    for M in ROWS:
        for N, K in GEMMS:
            p = plan(lib, KIND_TOK, M, N, K, sms)
            assert p["swap"] == 0 and p["splits"] == 1 and p["k_split"] == K
            assert p["bn"] in (128, 256)
            assert p["pt"] == math.ceil(M / 128) and p["qt"] == math.ceil(N / p["bn"])
            assert p["grid"] == min(p["pt"] * p["qt"], sms)
            # the width with the fewer waves x operand bytes per tile
            w = {bn: math.ceil(p["pt"] * math.ceil(N / bn) / sms) * (128 + bn) for bn in (128, 256)}
            assert w[p["bn"]] == min(w.values())


def test_swiglu_and_stream_plans_are_consistent(lib):
    for M in ROWS:
        for F, K in [(9728, 2560), (1536, 512)]:
            p = plan(lib, KIND_SWIGLU, M, F, K)
            assert p["splits"] == 1 and p["swap"] == (M <= 64) and p["grid"] >= 1
    for tiles, K in [(48, 2560), (20, 4096), (152, 2560), (20, 9728), (6, 512), (4, 1536), (1187, 2560)]:
        p = plan(lib, KIND_STREAM, 16, tiles, K)
        _check_k(p, K)
        assert p["pt"] == tiles and p["grid"] == tiles * p["splits"]
        if tiles < 152:
            assert p["grid"] <= 152
        assert p["k_split"] // 64 <= 48, "the activation slice fits beside the weight ring"


def test_plans_the_design_documents(lib):
    # the 385-row special-token QKV: 96 tiles of 256 features in one wave (not 192 tiles of 128 in two)
    p = plan(lib, KIND_TOK, 385, 6144, 2560)
    assert (p["bn"], p["pt"], p["qt"], p["grid"]) == (256, 4, 24, 96)
    # its O projection: 80 tiles of 128 (40 of 256 would cost the same waves for more bytes per tile)
    assert plan(lib, KIND_TOK, 385, 2560, 4096)["bn"] == 128
    # the context fusion GEMM (K = 5 x 2560) of 2048 and 4096 rows: 160 / 320 tiles, K split 4 ways
    assert plan(lib, KIND_GEMM, 2048, 2560, 12800)["splits"] == 4
    assert plan(lib, KIND_GEMM, 4096, 2560, 12800)["splits"] == 4
    # 256-row blocks on the weight-tile GEMMs fill the SMs with K splits
    p = plan(lib, KIND_GEMM, 256, 2560, 4096)
    assert (p["swap"], p["bn"], p["splits"], p["grid"]) == (0, 256, 7, 140)
    # the batch-1 QKV stream GEMM: 48 tiles x 3 K splits of 14 atoms
    p = plan(lib, KIND_STREAM, 16, 48, 2560)
    assert (p["splits"], p["k_split"], p["grid"]) == (3, 896, 144)


def test_attention_plans(lib):
    for impl, kt in ((0, 64), (1, 128)):
        for B, L, T in [(1, 16, 2048), (1, 385, 4096), (32, 381, 2048), (64, 16, 16384), (4, 5, 1), (1, 2, 1)]:
            if impl == 1 and L * 4 < 128:
                continue
            s, c = attn_plan(lib, impl, B, L, 32, 8, T)
            keys = T + L
            assert c % kt == 0 and 1 <= s <= 128
            assert s * c >= keys and (s - 1) * c < keys
    # the 16-position text block at context 2048: 17 splits of 128 keys (8 kv heads x 17 CTAs)
    assert attn_plan(lib, 0, 1, 16, 32, 8, 2048) == (17, 128)
    # the 385-position special-token block at context 4096: two splits on the tensor-memory kernel
    assert attn_plan(lib, 1, 1, 385, 32, 8, 4096)[0] == 2
