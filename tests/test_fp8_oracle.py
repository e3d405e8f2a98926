"""f2 in the oracle: E4M3 codes, the 128-element group quantisation with power-of-two scales, the FP8 linear
layer and its use in the drafter pass (FlashDrive §3.4 "Quantization"; reading R25).  CPU only.

Pins, each independent of the oracle's own arithmetic:
  - E4M3's defining constants (OCP OFP8 format: bias 7, largest finite 448, smallest normal 2^-6, smallest
    subnormal 2^-9, one NaN code per sign) and PyTorch's float8_e4m3fn conversion (a library routine: round to
    nearest even) on every finite code and on random and tie values;
  - brute force: the nearest of the 253 finite values, ties to the even code;
  - the group exponent against a search over k;
  - groups that are already E4M3 values times 2^k quantise to themselves, so the FP8 linear layer reduces to the
    plain (pinned) bf16 one;
  - the drafter's FP8 switch reads each FP8 copy, and routes by the 16-position rule."""
import numpy as np
import pytest
import torch

import synth

F8 = torch.float8_e4m3fn


def _torch_encode(x):
    return torch.tensor(np.asarray(x, np.float32)).to(F8).view(torch.uint8).numpy()


def _torch_decode(c):
    return torch.tensor(np.asarray(c, np.uint8)).view(F8).to(torch.float64).numpy()


def test_e4m3_defining_constants(oracle_lib):
    o = oracle_lib
    d = lambda c: float(o.e4m3_decode(np.uint8(c)))
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0          # largest finite: exponent 1111, mantissa 110
    assert d(0x08) == 2.0 ** -6                               # smallest normal
    assert d(0x01) == 2.0 ** -9 and d(0x07) == 7 * 2.0 ** -9  # subnormals m/8 * 2^-6
    assert d(0x38) == 1.0 and d(0x40) == 2.0 and d(0x3C) == 1.5 and d(0xB8) == -1.0
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert d(0x00) == 0.0 and d(0x80) == 0.0
    vals = o.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert (np.diff(vals) > 0).all()                          # codes 0..0x7E increase strictly
    np.testing.assert_array_equal(o.e4m3_decode(np.arange(0x80, 0xFF, dtype=np.uint8)), -vals)


def test_e4m3_decode_matches_torch(oracle_lib):
    c = np.array([i for i in range(256) if i not in (0x7F, 0xFF)], np.uint8)
    np.testing.assert_array_equal(oracle_lib.e4m3_decode(c), _torch_decode(c))


def test_e4m3_encode_matches_torch(oracle_lib):
    rng = np.random.default_rng(11)
    finite = oracle_lib.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (finite[1:] + finite[:-1]) / 2                        # every tie between neighbours
    x = np.concatenate([finite, mids, -mids, rng.uniform(-448, 448, 4000),
                        rng.normal(size=4000) * np.exp2(rng.integers(-12, 8, 4000)),
                        mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20)]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    got = oracle_lib.e4m3_encode(x.astype(np.float64))
    want = _torch_encode(x)
    want[(want & 0x7F) == 0] = 0                                  # zero results are the +0 code
    np.testing.assert_array_equal(got, want)
    assert int(oracle_lib.e4m3_encode(1000.0)) == 0x7E and int(oracle_lib.e4m3_encode(-1e30)) == 0xFE


def test_e4m3_encode_brute_force_nearest(oracle_lib):
    codes = np.array([c for c in range(0x7F)], np.uint8)
    vals = oracle_lib.e4m3_decode(codes)
    rng = np.random.default_rng(12)
    mids = (vals[1:] + vals[:-1]) / 2
    xs = np.concatenate([rng.uniform(0, 448, 3000), mids, vals, rng.uniform(0, 2 ** -5, 500)])
    for x in xs:
        dist = np.abs(vals - x)
        best = np.flatnonzero(dist == dist.min())
        if len(best) > 1:                                         # a tie: the even code
            best = best[(codes[best] & 1) == 0]
        want = int(codes[best[0]])
        assert int(oracle_lib.e4m3_encode(x)) == want, x
        assert int(oracle_lib.e4m3_encode(-x)) == (want | 0x80 if want else 0), x


def test_block_exponent_is_the_smallest_fitting_power(oracle_lib):
    rng = np.random.default_rng(13)
    amaxes = np.concatenate([rng.lognormal(0, 6, 2000), [448.0, 449.0, 224.0, 224.5, 1.0, 0.875, 2.0 ** -100,
                                                         3.0e38, 2.0 ** -149]])
    for a in amaxes:
        k = oracle_lib.block_exponent(a)
        want = next(j for j in range(-200, 200) if a * 2.0 ** -j <= 448.0)
        assert k == max(-126, min(127, want)), a
    assert oracle_lib.block_exponent(0.0) == 0


def _representable_rows(rng, n, K):
    """Rows whose 128-groups are E4M3 values times 2^k with one element of magnitude 448 * 2^k (bf16-exact)."""
    ks = rng.integers(-20, 6, size=(n, K // 128))
    codes = rng.integers(0, 0x7F, size=(n, K), dtype=np.uint8) | (rng.integers(0, 2, size=(n, K), dtype=np.uint8) << 7)
    codes[:, ::128] = 0x7E
    return codes, ks.astype(np.int8)


def test_quantise_representable_groups_is_exact(oracle_lib):
    rng = np.random.default_rng(14)
    codes, ks = _representable_rows(rng, 24, 512)
    codes[codes == 0x80] = 0
    x = oracle_lib.dequantize_fp8(codes, ks)
    q, e = oracle_lib.quantize_fp8(x)
    np.testing.assert_array_equal(e, ks)
    np.testing.assert_array_equal(q, codes)
    qb, eb = oracle_lib.quantize_fp8(synth.f32_to_bf16_bits(x.astype(np.float32)))   # bf16 input form
    np.testing.assert_array_equal(qb, codes)
    np.testing.assert_array_equal(eb, ks)


def test_quantise_error_bound_and_range(oracle_lib):
    rng = np.random.default_rng(15)
    x = rng.normal(size=(16, 1024)) * np.exp2(rng.integers(-30, 10, size=(16, 1)))
    x[3, :128] = 0.0
    q, e = oracle_lib.quantize_fp8(x)
    deq = oracle_lib.dequantize_fp8(q, e)
    for n in range(16):
        for g in range(8):
            xs, ds = x[n, g * 128:(g + 1) * 128], deq[n, g * 128:(g + 1) * 128]
            k = int(e[n, g])
            if not np.any(xs):
                assert k == 0 and (q[n, g * 128:(g + 1) * 128] == 0).all()
                continue
            assert 224.0 < np.abs(xs).max() * 2.0 ** -k <= 448.0
            # half a step of E4M3 at the element's binade (subnormal steps 2^-9, scaled)
            step = np.maximum(2.0 ** (np.floor(np.log2(np.maximum(np.abs(xs) * 2.0 ** -k, 2.0 ** -6))) - 3), 2.0 ** -9)
            assert (np.abs(ds - xs) <= step / 2 * 2.0 ** k + 1e-300).all()


def test_fp8_linear_reduces_to_the_bf16_linear(oracle_lib):
    """Weights and activations that quantise to themselves: the FP8 layer equals the plain bf16 layer."""
    rng = np.random.default_rng(16)
    wc, wk = _representable_rows(rng, 40, 384)
    xc, xk = _representable_rows(rng, 7, 384)
    W = oracle_lib.dequantize_fp8(wc, wk)
    X = oracle_lib.dequantize_fp8(xc, xk)
    W_bits = synth.f32_to_bf16_bits(W.astype(np.float32))
    assert (synth.bf16_bits_to_f32(W_bits).astype(np.float64) == W).all()   # bf16-exact
    qw, ew = oracle_lib.quantize_fp8(W_bits)
    got = oracle_lib.linear_fp8(X, qw, ew)
    want = oracle_lib.linear(X, W_bits)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_allclose(got, X @ W.T, rtol=1e-12, atol=0)


def test_fp8_linear_close_to_bf16_linear(oracle_lib):
    """On ordinary inputs the 8-bit layer stays within a few percent of the 16-bit one (E4M3 has 3 mantissa bits)."""
    rng = np.random.default_rng(17)
    W_bits = synth.f32_to_bf16_bits((rng.normal(size=(64, 512)) * 0.02).astype(np.float32))
    X = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(rng.normal(size=(5, 512)).astype(np.float32))).astype(np.float64)
    qw, ew = oracle_lib.quantize_fp8(W_bits)
    got = oracle_lib.linear_fp8(X, qw, ew)
    want = oracle_lib.linear(X, W_bits)
    rel = np.abs(got - want).max() / np.abs(want).max()
    assert 1e-4 < rel < 0.08, rel


def _tiny_case():
    s = synth.TINY
    w = synth.make_weights(s, 4242)
    B, L, T = 1, 16, 40
    off = np.array([0, T], np.int32)
    feats = synth.make_features(s, T, 4243)
    return s, w, B, L, T, off, feats


def test_drafter_fp8_switch_reads_every_copy(oracle_lib):
    """Each FP8 copy feeds the FP8 pass (zeroing its codes changes the hidden states) and none feeds the bf16 pass.
    The FP8 pass is a different model: eight 3-mantissa-bit roundings per layer (four weight, four activation
    operands) leave it about 8 % (RMS) from the bf16 pass after one layer and about 14 % after five on this random
    drafter; the bound below only rules out a gross error."""
    s, w, B, L, T, off, feats = _tiny_case()
    m = oracle_lib.Model(s, w, fp8=True)
    kv = oracle_lib.prepare_context(m, off, feats, T)
    args = (kv, T, np.array([T], np.int32), np.array([7], np.int32), s.vocab - 1, L)
    h8 = synth.bf16_bits_to_f32(oracle_lib.draft_block(m, *args)).astype(np.float64)
    h16 = synth.bf16_bits_to_f32(oracle_lib.draft_block(m, *args, fp8=False)).astype(np.float64)
    rel = np.sqrt(((h8 - h16) ** 2).mean() / (h16 ** 2).mean())
    assert 1e-3 < rel < 0.25, rel
    for name in ("wqkv", "wo", "w_gate_up", "w_down"):
        for layer in (0, s.n_layers - 1):
            codes, _ = m.fp8_copy(name, layer)
            saved = codes.copy()
            codes[:] = 0
            try:
                z8 = synth.bf16_bits_to_f32(oracle_lib.draft_block(m, *args)).astype(np.float64)
                z16 = synth.bf16_bits_to_f32(oracle_lib.draft_block(m, *args, fp8=False)).astype(np.float64)
            finally:
                codes[:] = saved
            assert not np.array_equal(z8, h8), (name, layer)
            np.testing.assert_array_equal(z16, h16)
    # the LM head copy
    hid = oracle_lib.draft_block(m, *args)
    t8, _, lg8 = oracle_lib.constrain_argmax(m, hid, B, L, want_logits=True)
    t16, _, lg16 = oracle_lib.constrain_argmax(m, hid, B, L, want_logits=True, fp8=False)
    assert np.sqrt(((lg8 - lg16) ** 2).mean() / (lg16 ** 2).mean()) < 0.1
    codes, _ = m.fp8_copy("lm_head")
    saved = codes.copy()
    codes[:] = 0
    try:
        _, _, z = oracle_lib.constrain_argmax(m, hid, B, L, want_logits=True)
    finally:
        codes[:] = saved
    assert (z == 0).all()


def test_fp8_routing_rule(oracle_lib):
    """Default routing: FP8 for at most 16 positions (drafter) and for an unconstrained LM head over at most 16
    rows; the bf16 weights otherwise."""
    s, w, B, L, T, off, feats = _tiny_case()
    m = oracle_lib.Model(s, w, fp8=True)
    kv = oracle_lib.prepare_context(m, off, feats, T)
    a1 = (kv, T, np.array([T], np.int32), np.array([7], np.int32), s.vocab - 1)
    np.testing.assert_array_equal(oracle_lib.draft_block(m, *a1, 16), oracle_lib.draft_block(m, *a1, 16, fp8=True))
    np.testing.assert_array_equal(oracle_lib.draft_block(m, *a1, 17), oracle_lib.draft_block(m, *a1, 17, fp8=False))
    hid = oracle_lib.draft_block(m, *a1, 17)
    _, _, d17 = oracle_lib.constrain_argmax(m, hid, 1, 17, want_logits=True)
    _, _, f17 = oracle_lib.constrain_argmax(m, hid, 1, 17, want_logits=True, fp8=True)
    np.testing.assert_array_equal(d17, f17)                    # 16 rows: FP8
    lay = synth.layout_special_tokens(s.vocab, n_waypoints=2, coord_lo=3000, n_coord=101, delim_id=3150,
                                      start_id=3151)
    Lc = lay["block_len"]
    hid = oracle_lib.draft_block(m, *a1, Lc)
    _, _, dl = oracle_lib.constrain_argmax(m, hid, 1, Lc, layout=lay, want_logits=True)
    _, _, bl = oracle_lib.constrain_argmax(m, hid, 1, Lc, layout=lay, want_logits=True, fp8=False)
    np.testing.assert_array_equal(dl, bl)                      # a layout: bf16


def test_layer_range_composes(oracle_lib):
    """Running layers [0, 2) and then [2, n) from that residual equals the whole pass, bf16 and FP8."""
    s, w, B, L, T, off, feats = _tiny_case()
    m = oracle_lib.Model(s, w, fp8=True)
    kv = oracle_lib.prepare_context(m, off, feats, T)
    args = (kv, T, np.array([T], np.int32), np.array([7], np.int32), s.vocab - 1, L)
    for fp8 in (False, True):
        whole, lay = oracle_lib.draft_block(m, *args, want_layers=True, fp8=fp8)
        first = oracle_lib.draft_block(m, *args, fp8=fp8, layers=(0, 2))
        np.testing.assert_array_equal(first, lay[1])
        rest = oracle_lib.draft_block(m, *args, fp8=fp8, layers=(2, s.n_layers), x_in=first)
        np.testing.assert_array_equal(rest, whole)
        one = oracle_lib.draft_block(m, *args, fp8=fp8, layers=(3, 4), x_in=lay[2])
        np.testing.assert_array_equal(one, lay[3])
