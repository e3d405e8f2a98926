"""Pins of the CPU oracle to facts outside itself: closed forms, library routines on special cases,
brute force on tiny inputs, exhaustive enumeration, symmetries and degenerate drafters.  No GPU."""
import itertools
import os

import numpy as np
import pytest
import scipy.special
import torch

import synth

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(x):
    return synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


# ---- bf16 rounding ----------------------------------------------------------------------------------------

def test_round_bf16_known_values(oracle_lib):
    o = oracle_lib
    cases = {
        1.0: 0x3F80, -2.0: 0xC000, 0.0: 0x0000, 3.0: 0x4040,
        1.0 + 2 ** -8: 0x3F80,                 # exact tie -> even (down)
        1.0 + 3 * 2 ** -8: 0x3F82,             # exact tie -> even (up)
        1.0 + 2 ** -8 + 2 ** -30: 0x3F81,      # just above the tie: no double rounding through float
        -(1.0 + 2 ** -8 + 2 ** -30): 0xBF81,
        3.3895313892515355e38: 0x7F7F,         # largest finite bf16
        3.4e38: 0x7F80,                        # rounds past the largest finite -> inf
        2.0 ** -133: 0x0001,                   # smallest bf16 subnormal
        2.0 ** -134: 0x0000,                   # tie between 0 and the smallest subnormal -> even (0)
        1.5 * 2.0 ** -133: 0x0002,             # tie between 1 and 2 subnormal units -> even (2)
    }
    for v, want in cases.items():
        assert int(o.round_bf16(v)) == want, (v, hex(int(o.round_bf16(v))), hex(want))


def test_round_bf16_matches_torch_on_float32_values(oracle_lib):
    """For values exactly representable in float32, fp64->bf16 must equal the library's fp32->bf16."""
    rng = np.random.default_rng(0)
    v = np.concatenate([(rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000)).astype(np.float32),
                        (rng.integers(0, 2 ** 16, 2000).astype(np.uint32) << 16 | 0x8000).view(np.float32)])
    v = v[np.isfinite(v)]
    got = oracle_lib.round_bf16(v.astype(np.float64))
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, want)
    back = oracle_lib.bf16_to_f64(got)
    np.testing.assert_array_equal(back, torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).double().numpy())


# ---- RMSNorm, RoPE, SiLU -------------------------------------------------------------------------------------

def test_rmsnorm_closed_forms(oracle_lib):
    o = oracle_lib
    n = 64
    g = bits(np.linspace(0.5, 1.5, n))
    gv = synth.bf16_bits_to_f32(g).astype(np.float64)
    for c in (0.25, 3.0, -7.5):
        y = o.rmsnorm(np.full(n, c), g, 1e-6)
        np.testing.assert_allclose(y, c / np.sqrt(c * c + 1e-6) * gv, rtol=1e-14)
    y = o.rmsnorm(np.array([3.0, 4.0]), bits([1.0, 1.0]), 0.0)       # mean square 12.5
    np.testing.assert_allclose(y, np.array([3.0, 4.0]) / np.sqrt(12.5), rtol=1e-15)
    x = np.random.default_rng(1).standard_normal(n)
    np.testing.assert_allclose(o.rmsnorm(1000 * x, g, 0.0), o.rmsnorm(x, g, 0.0), rtol=1e-12)  # scale invariant
    assert np.all(o.rmsnorm(np.zeros(n), g, 1e-6) == 0.0)


def test_rope_closed_forms(oracle_lib):
    o = oracle_lib
    # one pair (h = 2): plain rotation by the position, frequency theta^0 = 1
    for p in (0.0, 1.0, 2.5, 1000.0):
        np.testing.assert_allclose(o.rope([1.0, 0.0], p, 1e6), [np.cos(p), np.sin(p)], atol=1e-12)
        np.testing.assert_allclose(o.rope([0.0, 1.0], p, 1e6), [-np.sin(p), np.cos(p)], atol=1e-12)
    # h = 4: pair (1, 3) turns with frequency theta^(-2/4); pairing is rotate-half (i, i + h/2)
    th = 10000.0
    p = 7.0
    y = o.rope([0.0, 1.0, 0.0, 0.0], p, th)
    np.testing.assert_allclose(y, [0.0, np.cos(p * th ** -0.5), 0.0, np.sin(p * th ** -0.5)], atol=1e-12)


def test_rope_invariants(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(2)
    h = 64
    q, k = rng.standard_normal(h), rng.standard_normal(h)
    np.testing.assert_array_equal(o.rope(q, 0.0, 1e6), q)                     # position 0 = identity
    for p in (1.0, 17.0, 4096.0):
        np.testing.assert_allclose(np.linalg.norm(o.rope(q, p, 1e6)), np.linalg.norm(q), rtol=1e-13)
    # <R_m q, R_n k> depends only on m - n
    ref = o.rope(q, 10.0, 1e6) @ o.rope(k, 3.0, 1e6)
    for s in (0.0, 1.0, 500.0, 12345.0):
        np.testing.assert_allclose(o.rope(q, 10.0 + s, 1e6) @ o.rope(k, 3.0 + s, 1e6), ref, rtol=1e-9, atol=1e-9)


def test_silu_closed_form(oracle_lib):
    for v in (-30.0, -2.0, -1e-3, 0.0, 0.5, 3.0, 40.0):
        assert oracle_lib.silu(v) == pytest.approx(v * scipy.special.expit(v), rel=1e-14, abs=1e-300)
    assert oracle_lib.silu(0.0) == 0.0


# ---- linear and attention against library routines / brute force ----------------------------------------------

def test_linear_matches_numpy(oracle_lib):
    rng = np.random.default_rng(3)
    for M, N, K in ((1, 1, 1), (3, 5, 7), (40, 33, 70)):   # 40 rows: spans two row groups of the oracle
        X = rng.standard_normal((M, K))
        Wb = bits(rng.standard_normal((N, K)))
        Y = oracle_lib.linear(X, Wb)
        np.testing.assert_allclose(Y, X @ synth.bf16_bits_to_f32(Wb).astype(np.float64).T, rtol=1e-12, atol=1e-12)


def _attn_bruteforce(q, k, v, scale):
    s = (q @ k.T) * scale
    return scipy.special.softmax(s, axis=1) @ v


def test_attention_bruteforce_tiny(oracle_lib):
    rng = np.random.default_rng(4)
    h = 8
    for n_ctx, n_blk, R in ((0, 1, 1), (1, 1, 2), (5, 3, 4), (8, 4, 4)):
        q = rng.standard_normal((R, h))
        kc, vc = bits(rng.standard_normal((n_ctx, h))), bits(rng.standard_normal((n_ctx, h)))
        kb, vb = rng.standard_normal((n_blk, h)), rng.standard_normal((n_blk, h))
        o = oracle_lib.attention(q, kc, vc, kb, vb, 1 / np.sqrt(h))
        K = np.concatenate([synth.bf16_bits_to_f32(kc).astype(np.float64).reshape(-1, h), kb])
        V = np.concatenate([synth.bf16_bits_to_f32(vc).astype(np.float64).reshape(-1, h), vb])
        np.testing.assert_allclose(o, _attn_bruteforce(q, K, V, 1 / np.sqrt(h)), rtol=1e-12, atol=1e-12)


def test_attention_special_cases(oracle_lib):
    rng = np.random.default_rng(5)
    h = 16
    # all keys equal -> uniform weights -> output is the mean of V
    k = np.tile(rng.standard_normal(h), (6, 1))
    vc = bits(rng.standard_normal((4, h)))
    vb = rng.standard_normal((2, h))
    q = rng.standard_normal((3, h))
    o = oracle_lib.attention(q, bits(k[:4]), vc,
                             synth.bf16_bits_to_f32(bits(k[4:])).astype(np.float64), vb, 0.125)
    V = np.concatenate([synth.bf16_bits_to_f32(vc).astype(np.float64), vb])
    np.testing.assert_allclose(o, np.tile(V.mean(0), (3, 1)), rtol=1e-12)
    # one dominant logit -> that row of V
    kb = np.zeros((3, h))
    kb[1, 0] = 1000.0
    q = np.zeros((1, h))
    q[0, 0] = 1.0
    vb = rng.standard_normal((3, h))
    o = oracle_lib.attention(q, np.zeros((0, h), np.uint16), np.zeros((0, h), np.uint16), kb, vb, 1.0)
    np.testing.assert_allclose(o[0], vb[1], rtol=1e-12)


# ---- whole drafter: degenerate cases and symmetries ---------------------------------------------------------------

def _tiny(seed=11, zero=(), n_layers=None):
    shape = synth.TINY if n_layers is None else synth.ModelShape(**{**synth.TINY.__dict__, "n_layers": n_layers})
    w = synth.make_weights(shape, seed, zero=zero)
    return shape, w


def _ctx(shape, T, seed=12):
    return synth.make_kv_store(shape, 1, T, seed)


def test_identity_layers_give_embedding_argmax(oracle_lib):
    """W_o = W_down = 0: every layer is the identity, so hidden = embedding rows and the token is
    argmax(RMSNorm_final(E[mask]) . W_lm^T) — the logits reduce to one matrix product."""
    o = oracle_lib
    shape, w = _tiny(zero=("wo", "w_down"))
    m = o.Model(shape, w)
    T, L = 9, 6
    kv = _ctx(shape, T)
    anchor = np.array([123], np.int32)
    mask_id = shape.vocab - 1
    hid, layers = o.draft_block(m, kv, T, np.array([T], np.int32), anchor, mask_id, L, want_layers=True)
    E = w["embed"]
    np.testing.assert_array_equal(hid[0], E[123])
    for j in range(1, L):
        np.testing.assert_array_equal(hid[j], E[mask_id])
    for l in range(shape.n_layers):
        np.testing.assert_array_equal(layers[l], hid)
    toks, margin, logits = o.constrain_argmax(m, hid, 1, L, want_logits=True)
    x = synth.bf16_bits_to_f32(E[mask_id]).astype(np.float64)
    g = synth.bf16_bits_to_f32(w["final_norm"]).astype(np.float64)
    z = x / np.sqrt(np.mean(x * x) + shape.rms_eps) * g
    z = synth.bf16_bits_to_f32(o.round_bf16(z)).astype(np.float64)
    lg = synth.bf16_bits_to_f32(w["lm_head"]).astype(np.float64) @ z
    np.testing.assert_allclose(logits[0], lg, rtol=1e-10, atol=1e-10)
    lf = lg.astype(np.float32)
    assert np.all(toks == int(np.argmax(lf)))
    top2 = np.sort(lf)[-2:]
    assert margin[0] == pytest.approx(float(top2[1]) - float(top2[0]), abs=1e-7)


def test_uniform_attention_closed_form(oracle_lib):
    """One layer, W_q = W_k = 0 (uniform attention: output = mean of every value row), W_o = I, MLP off.
    The residual after the layer is then bf16(x0 + bf16(mean of V over [context; block])) per head, with
    q head i reading kv head i // (H_q / H_kv) and block values = bf16(xn . W_v^T)."""
    o = oracle_lib
    shape, w = _tiny(seed=21, zero=("wq_wk", "w_gate_up"), n_layers=1)
    s = shape
    lw = w["layers"][0]
    d, h = s.d_model, s.head_dim
    assert s.n_q_heads * h == d
    lw["wo"][...] = 0
    lw["wo"][np.arange(d), np.arange(d)] = bits(1.0)
    m = o.Model(s, w)
    T, L = 11, 5        # 16 keys: the uniform weight 1/16 is exact, so exact ties round the same on both sides
    kv = _ctx(s, T, seed=22)
    ctx_len = np.array([T], np.int32)
    anchor = np.array([5], np.int32)
    mask_id = s.vocab - 1
    hid = o.draft_block(m, kv, T, ctx_len, anchor, mask_id, L)
    x0 = synth.bf16_bits_to_f32(np.stack([w["embed"][5]] + [w["embed"][mask_id]] * (L - 1))).astype(np.float64)
    gn = synth.bf16_bits_to_f32(lw["attn_norm"]).astype(np.float64)
    xn = x0 / np.sqrt(np.mean(x0 * x0, axis=1, keepdims=True) + s.rms_eps) * gn
    xn = synth.bf16_bits_to_f32(o.round_bf16(xn)).astype(np.float64)
    Wv = synth.bf16_bits_to_f32(lw["wqkv"][(s.n_q_heads + s.n_kv_heads) * h:]).astype(np.float64)
    vblk = synth.bf16_bits_to_f32(o.round_bf16(xn @ Wv.T)).astype(np.float64)      # [L, nkv*h]
    grp = s.n_q_heads // s.n_kv_heads
    want = np.empty_like(x0)
    for i in range(s.n_q_heads):
        g = i // grp
        vctx = synth.bf16_bits_to_f32(kv[0, 0, 1, g, :T]).astype(np.float64)
        mean = np.concatenate([vctx, vblk[:, g * h:(g + 1) * h]]).mean(0)
        ob = synth.bf16_bits_to_f32(o.round_bf16(mean)).astype(np.float64)
        want[:, i * h:(i + 1) * h] = x0[:, i * h:(i + 1) * h] + ob
    want = o.round_bf16(want)
    np.testing.assert_array_equal(hid, want)


def test_mask_rows_identical_under_uniform_attention(oracle_lib):
    """W_q = W_k = 0 removes every position dependence, so the L-1 mask rows stay identical."""
    o = oracle_lib
    shape, w = _tiny(seed=31, zero=("wq_wk",))
    m = o.Model(shape, w)
    T, L = 10, 8
    hid = o.draft_block(m, _ctx(shape, T), T, np.array([T], np.int32), np.array([7], np.int32), shape.vocab - 1, L)
    for j in range(2, L):
        np.testing.assert_array_equal(hid[j], hid[1])
    assert not np.array_equal(hid[0], hid[1])


def test_bidirectional_and_context_dependence(oracle_lib):
    """No causal mask: the anchor row's output changes when a LATER position's token changes.  The context
    K/V matter, and context rows past ctx_len are never read."""
    o = oracle_lib
    shape, w = _tiny(seed=41)
    m = o.Model(shape, w)
    T, L = 12, 4
    kv = _ctx(shape, T)
    a = np.array([9], np.int32)
    h1 = o.draft_block(m, kv, T, np.array([T], np.int32), a, shape.vocab - 1, L)
    h2 = o.draft_block(m, kv, T, np.array([T], np.int32), a, shape.vocab - 2, L)
    assert not np.array_equal(h1[0], h2[0])
    kv2 = kv.copy()
    kv2[:, :, :, :, 3] ^= 0x0100    # perturb context position 3 of every layer
    h3 = o.draft_block(m, kv2, T, np.array([T], np.int32), a, shape.vocab - 1, L)
    assert not np.array_equal(h1, h3)
    h4 = o.draft_block(m, kv2, T, np.array([3], np.int32), a, shape.vocab - 1, L)
    h5 = o.draft_block(m, kv, T, np.array([3], np.int32), a, shape.vocab - 1, L)
    np.testing.assert_array_equal(h4, h5)


def _rel(a, b):
    a = synth.bf16_bits_to_f32(a).astype(np.float64)
    b = synth.bf16_bits_to_f32(b).astype(np.float64)
    return np.max(np.abs(a - b)) / np.max(np.abs(b))


def test_gqa_head_grouping_symmetry(oracle_lib):
    """Swapping two q heads of the same kv group (their W_q rows and W_o columns) leaves the output unchanged;
    swapping q heads of different groups does not.  Pins grouping q head i -> kv head i // (H_q/H_kv)."""
    o = oracle_lib
    shape, w = _tiny(seed=51, n_layers=1)
    s = shape
    h = s.head_dim
    T, L = 6, 4
    kv = _ctx(s, T)
    args = (kv, T, np.array([T], np.int32), np.array([3], np.int32), s.vocab - 1, L)
    base = o.draft_block(o.Model(s, w), *args)

    def swapped(i, j):
        w2 = {**w, "layers": [dict(w["layers"][0])]}
        lw = w2["layers"][0]
        q = lw["wqkv"].copy()
        q[i * h:(i + 1) * h], q[j * h:(j + 1) * h] = lw["wqkv"][j * h:(j + 1) * h], lw["wqkv"][i * h:(i + 1) * h]
        wo = lw["wo"].copy()
        wo[:, i * h:(i + 1) * h], wo[:, j * h:(j + 1) * h] = lw["wo"][:, j * h:(j + 1) * h], lw["wo"][:, i * h:(i + 1) * h]
        lw["wqkv"], lw["wo"] = q, wo
        return o.draft_block(o.Model(s, w2), *args)

    grp = s.n_q_heads // s.n_kv_heads
    assert _rel(swapped(0, 1), base) < 2e-2          # same group (0 // 4 == 1 // 4): equal up to bf16 flips
    assert _rel(swapped(0, grp), base) > 5e-2        # different groups


# ---- context preparation ----------------------------------------------------------------------------------

def test_prepare_context_append_equals_whole(oracle_lib):
    """Writing a context in two appends (pos_start = 0, then T1) gives the same store as one call."""
    o = oracle_lib
    shape, w = _tiny(seed=61)
    m = o.Model(shape, w)
    T1, T2 = 5, 4
    F = synth.make_features(shape, T1 + T2, 62)
    whole = o.prepare_context(m, np.array([0, T1 + T2], np.int32), F, T1 + T2)
    part = o.prepare_context(m, np.array([0, T1], np.int32), [f[:T1] for f in F], T1 + T2)
    part = o.prepare_context(m, np.array([0, T2], np.int32), [f[T1:] for f in F], T1 + T2,
                             pos_start=np.array([T1], np.int32), kv_store=part)
    np.testing.assert_array_equal(part, whole)


def test_prepare_context_ragged_batch_equals_single(oracle_lib):
    o = oracle_lib
    shape, w = _tiny(seed=71)
    m = o.Model(shape, w)
    lens = [3, 0, 5]
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    F = synth.make_features(shape, int(off[-1]), 72)
    tc = 6
    st = o.prepare_context(m, off, F, tc)
    for b, n in enumerate(lens):
        one = o.prepare_context(m, np.array([0, n], np.int32), [f[off[b]:off[b + 1]] for f in F], tc)
        np.testing.assert_array_equal(st[:, b], one[:, 0])


def test_prepare_context_v_is_plain_projection(oracle_lib):
    """hidden_norm gains = 1 and one feature source -> ctx = bf16(RMSNorm(F . W_fc^T)); V = bf16(ctx . W_v^T)
    from numpy's matrix product; K at position 0 has no rotation: bf16(RMSNorm(ctx . W_k^T) * k_norm)."""
    o = oracle_lib
    s = synth.ModelShape(**{**synth.TINY.__dict__, "n_feat": 1, "n_layers": 1})
    w = synth.make_weights(s, 81)
    w["hidden_norm"][...] = bits(1.0)
    m = o.Model(s, w)
    F = synth.make_features(s, 1, 82)
    st = o.prepare_context(m, np.array([0, 1], np.int32), F, 1)
    f64 = lambda b: synth.bf16_bits_to_f32(b).astype(np.float64)
    y = f64(F[0][0]) @ f64(w["w_fc"]).T
    ctx = f64(o.round_bf16(y / np.sqrt(np.mean(y * y) + s.rms_eps)))
    h, nq, nkv = s.head_dim, s.n_q_heads, s.n_kv_heads
    Wk = f64(w["layers"][0]["wqkv"][nq * h:(nq + nkv) * h])
    Wv = f64(w["layers"][0]["wqkv"][(nq + nkv) * h:])
    v = o.round_bf16(ctx @ Wv.T)
    kn = f64(w["layers"][0]["k_norm"])
    for g in range(nkv):
        np.testing.assert_array_equal(st[0, 0, 1, g, 0], v[g * h:(g + 1) * h])
        kr = ctx @ Wk[g * h:(g + 1) * h].T
        np.testing.assert_array_equal(st[0, 0, 0, g, 0], o.round_bf16(kr / np.sqrt(np.mean(kr * kr) + s.rms_eps) * kn))


# ---- constrained argmax -----------------------------------------------------------------------------------

def test_constrained_argmax_invariants(oracle_lib):
    o = oracle_lib
    shape, w = _tiny(seed=91)
    m = o.Model(shape, w)
    V = shape.vocab
    L = 9
    rng = np.random.default_rng(92)
    hid = bits(rng.standard_normal((2 * L, shape.d_model)))
    layout = dict(class_off=np.array([0, 2, 3, 4, 5], np.int32),
                  class_ranges=np.array([10, 20, 100, 105, 4000, 4001, 0, V, 77, 78], np.int32),
                  pos_class=rng.integers(0, 4, (2, L)).astype(np.int16))
    layout["pos_class"][:, 1] = 3
    toks, margin, logits = o.constrain_argmax(m, hid, 2, L, layout=layout, want_logits=True)
    free_toks, _, free_logits = o.constrain_argmax(m, hid, 2, L, want_logits=True)
    legal = {0: set(range(10, 20)) | set(range(100, 105)), 1: {4000}, 2: set(range(V)), 3: {77}}
    for b in range(2):
        for j in range(1, L):
            c = int(layout["pos_class"][b, j])
            r = b * (L - 1) + j - 1
            t = int(toks[b, j - 1])
            assert t in legal[c]
            ids = np.array(sorted(legal[c]))
            lf = free_logits[r, ids].astype(np.float32)
            assert t == ids[np.argmax(lf)]                            # brute force over the legal ids
            assert np.all(np.isnan(np.delete(logits[r], ids)))        # illegal columns never computed
            if c == 2:
                assert t == free_toks[b, j - 1]                       # full-vocab class == unconstrained
            if len(ids) == 1:
                assert t == ids[0] and margin[r] == np.inf            # singleton class returns its id


def test_argmax_tie_takes_lowest_id(oracle_lib):
    o = oracle_lib
    shape, w = _tiny(seed=93)
    w["lm_head"][...] = 0
    w["lm_head"][[20, 50]] = bits(np.ones(shape.d_model))
    m = o.Model(shape, w)
    hid = bits(np.ones((3, shape.d_model)))
    toks, margin, _ = o.constrain_argmax(m, hid, 1, 3)
    assert np.all(toks == 20) and np.all(margin == 0.0)


# ---- acceptance ---------------------------------------------------------------------------------------------

def test_verify_text_geometric_rows(oracle_lib):
    """Target rows built to agree with the draft for exactly g positions give accept = 1 + min(g, L-1)."""
    rng = np.random.default_rng(101)
    for L in (2, 3, 16, 40):
        draft = rng.integers(0, 1000, (300, L - 1)).astype(np.int32)
        target, g = synth.make_target_rows(draft, 1000, 0.25, seed=L)
        acc, com, val = oracle_lib.verify(0, draft, target)
        np.testing.assert_array_equal(acc, 1 + np.minimum(g, L - 1))
        np.testing.assert_array_equal(val, (g >= L - 1).astype(np.int32))


def test_verify_text_exhaustive_binary(oracle_lib):
    """All draft/target pairs over a two-symbol alphabet for L <= 6: accept >= 1, the committed tokens are
    the draft prefix plus the target's own token, and the first unaccepted draft disagrees."""
    for L in range(2, 7):
        drafts = np.array(list(itertools.product([0, 1], repeat=L - 1)), np.int32)
        targets = np.array(list(itertools.product([0, 1], repeat=L)), np.int32)
        D = np.repeat(drafts, len(targets), axis=0)
        T = np.tile(targets, (len(drafts), 1))
        acc, com, val = oracle_lib.verify(0, D, T)
        assert acc.min() >= 1 and acc.max() <= L
        for b in range(len(D)):
            n = acc[b] - 1
            assert np.array_equal(com[b, :n], D[b, :n]) and com[b, n] == T[b, n]
            assert np.all(com[b, n + 1:] == -1)
            assert np.array_equal(D[b, :n], T[b, :n])
            if n < L - 1:
                assert D[b, n] != T[b, n]
        # exactly half of the targets agree with a draft at each next position: counts per accept value
        counts = np.bincount(acc, minlength=L + 1)[1:]
        expect = [len(D) // 2 ** k for k in range(1, L)] + [len(D) // 2 ** (L - 1)]
        np.testing.assert_array_equal(counts, expect)


def _fw_layout():
    # ids: digits 0..9 -> 0..9, '+' 10, '-' 11, pad 12; one field: [sign d d d d d] after the anchor
    lay = dict(class_off=np.array([0, 1, 3], np.int32), class_ranges=np.array([10, 12, 0, 10, 12, 13], np.int32),
               pos_class=np.array([0, 0, 1, 1, 1, 1, 1], np.int16))
    rule = np.array([0, 1, 2, 2, 2, 2, 3], np.int8)
    return lay, rule


def test_schema_exhaustive_single_field(oracle_lib):
    """All 2 * 11^5 sign+digit fields (plus non-member tokens in the sign slot).  A field is valid iff it is
    a sign, k leading pads (0 <= k <= 4), then 5 - k real digits; otherwise the first failing slot is the
    first one whose prefix no valid field shares."""
    lay, rule = _fw_layout()
    syms_sign = [10, 11, 3]
    syms_dig = list(range(10)) + [12]
    fields = np.array([(s,) + d for s in syms_sign for d in itertools.product(syms_dig, repeat=5)], np.int32)
    acc, com, val = oracle_lib.verify(1, fields, layout=lay, rule=rule, pad_id=12)
    valid_set = set()
    prefixes = set()
    for s in (10, 11):
        for k in range(5):
            for digs in itertools.product(range(10), repeat=5 - k):
                f = (s,) + (12,) * k + digs
                valid_set.add(f)
    for f in valid_set:
        for j in range(1, 7):
            prefixes.add(f[:j])
    assert len(valid_set) == 2 * sum(10 ** (5 - k) for k in range(5)) == 222220
    for i, f in enumerate(map(tuple, fields)):
        ok = f in valid_set
        assert val[i] == ok
        if ok:
            assert acc[i] == 6
        else:
            p = next(j for j in range(1, 7) if f[:j] not in prefixes)
            assert acc[i] == p - 1, (f, acc[i], p)


def test_schema_golden_fields(oracle_lib):
    lay, rule = _fw_layout()
    tok = {"+": 10, "-": 11, "P": 12, **{str(i): i for i in range(10)}}
    with open(os.path.join(GOLDEN, "fixed_width_fields.txt")) as fh:
        rows = [ln.split() for ln in fh if ln.strip() and not ln.startswith("#")]
    fields = np.array([[tok[c] for c in r[0]] for r in rows], np.int32)
    acc, com, val = oracle_lib.verify(1, fields, layout=lay, rule=rule, pad_id=12)
    for i, r in enumerate(rows):
        assert val[i] == int(r[1]), r
        first_fail = int(r[2])
        assert acc[i] == (6 if first_fail == 0 else first_fail - 1), r
        if r[1] == "1":
            digits = "".join(c for c in r[0][1:] if c != "P")
            assert int(r[0][0] + digits) == int(r[3])


def test_special_token_layout_always_schema_valid_after_constraints(oracle_lib):
    """Constrained argmax on the dedicated-coordinate-token layout always yields a schema-valid block."""
    o = oracle_lib
    shape, w = _tiny(seed=111)
    V = shape.vocab
    lay = synth.layout_special_tokens(V, n_waypoints=3, coord_lo=2000, n_coord=1001, delim_id=3100, start_id=3101)
    L = lay["block_len"]
    m = o.Model(shape, w)
    hid = bits(np.random.default_rng(112).standard_normal((L, shape.d_model)))
    toks, _, _ = o.constrain_argmax(m, hid, 1, L, layout=lay)
    acc, com, val = o.verify(1, toks, layout=lay, rule=lay["rule"], pad_id=lay["pad_id"])
    assert val[0] == 1 and acc[0] == L - 1
    assert np.all((toks[0] >= 2000) & (toks[0] < 3001) | (toks[0] == 3100))
