"""Pins of how the oracle COMPOSES its pinned building blocks, each against a closed form computed here from
the definition, plus a planted-mistake check: a copy of the oracle source with one plausible mistake (gate and
up swapped, the residual dropped, block RoPE positions not offset by the context length, the fused feature
sources taken in the wrong order) is compiled on the CPU and must fail the same pin.  No GPU.

  - MLP (VFlash blog "Key claims": SwiGLU layer of the five-layer drafter; pre-norm layer form):
    x1 = bf16(x0 + bf16(silu(gate) * up) . W_down^T), gate = rows 0..F-1 of w_gate_up, up = rows F..2F-1.
  - Block positions (VFlash paper (zh) §2.1-§2.2: the block follows the context; RoPE positions of block
    position j are ctx_len + j): with q and k non-zero only on the first rotary pair (frequency theta^0 = 1) a
    score is |q| |k| cos(phi_k - phi_q + pos_k - pos_q).
  - Fusion (VFlash paper (zh) §2.1: features of several target layers are fused): with W_fc selecting source s,
    ctx = bf16(RMSNorm(F_s)).
"""
import contextlib
import os
import subprocess
import tempfile

import numpy as np
import pytest
import scipy.special

import synth

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "fpd_oracle.c")


def bits(x):
    return synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def f64(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


def shape_with(**kw):
    return synth.ModelShape(**{**synth.TINY.__dict__, **kw})


@contextlib.contextmanager
def planted(oracle_lib, old: str, new: str, occurrence: int = 0):
    """Run the oracle from a copy of its source in which the `occurrence`-th appearance of `old` reads `new`."""
    src = open(ORACLE_SRC).read()
    pos = -1
    for _ in range(occurrence + 1):
        pos = src.find(old, pos + 1)
        assert pos >= 0, f"mutation site not found: {old!r}"
    src = src[:pos] + new + src[pos + len(old):]
    with tempfile.TemporaryDirectory() as td:
        c, so = os.path.join(td, "mutant.c"), os.path.join(td, "libmutant.so")
        open(c, "w").write(src)
        subprocess.check_call(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=gnu11", c, "-o", so, "-lm"])
        with oracle_lib.use_library(so):
            yield


# ---- MLP composition -----------------------------------------------------------------------------------------

def _mlp_case():
    """One layer with W_o = 0 (the attention sub-layer adds exactly 0), gate row f = 2 e_{a(f)}, up row
    f = 0.5 e_{b(f)}, W_down row n = 4 e_{sig(n)}: every product has one non-zero term, so the closed form is
    exact up to the declared bf16 storage points."""
    s = shape_with(n_layers=1)
    w = synth.make_weights(s, 301)
    lw = w["layers"][0]
    d, F = s.d_model, s.d_ff
    lw["wo"][...] = 0
    a = np.arange(F) % d
    b = (3 * np.arange(F) + 7) % d
    sig = (5 * np.arange(d) + 2) % F
    gu = np.zeros((2 * F, d), np.float32)
    gu[np.arange(F), a] = 2.0
    gu[F + np.arange(F), b] = 0.5
    lw["w_gate_up"] = bits(gu)
    wd = np.zeros((d, F), np.float32)
    wd[np.arange(d), sig] = 4.0
    lw["w_down"] = bits(wd)
    return s, w, a, b, sig


def _mlp_closed_form(o, s, w, a, b, sig, L, anchor, mask_id, swap=False, residual=True):
    lw = w["layers"][0]
    x0 = f64(np.stack([w["embed"][anchor]] + [w["embed"][mask_id]] * (L - 1)))
    g = f64(lw["mlp_norm"])
    xn = f64(o.round_bf16(x0 / np.sqrt(np.mean(x0 * x0, axis=1, keepdims=True) + s.rms_eps) * g))
    gate, up = 2.0 * xn[:, a], 0.5 * xn[:, b]
    if swap:
        gate, up = up, gate
    hm = f64(o.round_bf16(gate * scipy.special.expit(gate) * up))
    out = 4.0 * hm[:, sig]
    return o.round_bf16(x0 + out if residual else out)


def test_mlp_composition_closed_form(oracle_lib):
    o = oracle_lib
    s, w, a, b, sig = _mlp_case()
    T, L, anchor, mask_id = 7, 5, 11, s.vocab - 1
    kv = synth.make_kv_store(s, 1, T, 302)
    m = o.Model(s, w)
    args = (kv, T, np.array([T], np.int32), np.array([anchor], np.int32), mask_id, L)
    want = _mlp_closed_form(o, s, w, a, b, sig, L, anchor, mask_id)
    np.testing.assert_array_equal(o.draft_block(m, *args), want)
    # the pin separates the plausible mistakes from the definition
    assert not np.array_equal(want, _mlp_closed_form(o, s, w, a, b, sig, L, anchor, mask_id, swap=True))
    assert not np.array_equal(want, _mlp_closed_form(o, s, w, a, b, sig, L, anchor, mask_id, residual=False))
    gate_up = "double gv = dx[(size_t)r * 2 * F + f], uv = dx[(size_t)r * 2 * F + F + f];"
    with planted(o, gate_up, "double uv = dx[(size_t)r * 2 * F + f], gv = dx[(size_t)r * 2 * F + F + f];"):
        assert not np.array_equal(o.draft_block(o.Model(s, w), *args), want)
    with planted(o, "x[e] = rbf(x[e] + dx[e]);", "x[e] = rbf(dx[e]);", occurrence=1):   # drop the MLP residual
        assert not np.array_equal(o.draft_block(o.Model(s, w), *args), want)


# ---- RoPE positions of the block rows ------------------------------------------------------------------------------

def _rope_case(T):
    """One layer; q head 0 and kv head 0 live on the first rotary pair (dims 0 and h/2) only; context key t of kv
    head 0 is R(t) (6, 8) (bf16) and context value t is e_t; block values are 0; W_o = I, MLP off.  The first T
    coordinates of head 0's output are then the softmax weights of the context keys."""
    s = shape_with(n_layers=1)
    w = synth.make_weights(s, 311)
    lw = w["layers"][0]
    d, h, nq, nkv = s.d_model, s.head_dim, s.n_q_heads, s.n_kv_heads
    half = h // 2
    wqkv = np.zeros(((nq + 2 * nkv) * h, d), np.float32)
    wqkv[0, 3], wqkv[half, 40] = 1.0, 1.0                        # q head 0: xn[3], xn[40]
    wqkv[nq * h, 5], wqkv[nq * h + half, 17] = 1.0, -1.0         # k of kv head 0: xn[5], -xn[17]
    lw["wqkv"] = bits(wqkv)
    lw["k_norm"] = bits(np.full(h, 0.25))                       # small block keys: the context dominates
    wo = np.zeros((d, nq * h), np.float32)
    wo[np.arange(d), np.arange(d)] = 1.0
    lw["wo"] = bits(wo)
    lw["w_gate_up"][...] = 0
    kv = np.zeros((1, 1, 2, nkv, T, h), np.uint16)
    t = np.arange(T)
    kv[0, 0, 0, 0, :, 0] = bits(6.0 * np.cos(t) - 8.0 * np.sin(t))
    kv[0, 0, 0, 0, :, half] = bits(8.0 * np.cos(t) + 6.0 * np.sin(t))
    kv[0, 0, 1, 0, t, t] = bits(1.0)
    return s, w, kv


def _rope_closed_form(o, s, w, kv, T, L, anchor, mask_id, offset=True):
    """Context weights of q head 0 for every block row, from |q| |k| cos(phi_k - phi_q + pos_k - pos_q)."""
    lw = w["layers"][0]
    h, nq = s.head_dim, s.n_q_heads
    half = h // 2
    x0 = f64(np.stack([w["embed"][anchor]] + [w["embed"][mask_id]] * (L - 1)))
    xn = f64(o.round_bf16(x0 / np.sqrt(np.mean(x0 * x0, axis=1, keepdims=True) + s.rms_eps) * f64(lw["attn_norm"])))

    def pair(raw, gain):   # per-head RMSNorm over h dims of a vector non-zero only at dims 0 and h/2
        inv = 1.0 / np.sqrt((raw[:, 0] ** 2 + raw[:, 1] ** 2) / h + s.rms_eps)
        return np.stack([raw[:, 0] * inv * gain[0], raw[:, 1] * inv * gain[half]], axis=1)

    q = pair(np.stack([xn[:, 3], xn[:, 40]], 1), f64(lw["q_norm"]))
    kb = pair(np.stack([xn[:, 5], -xn[:, 17]], 1), f64(lw["k_norm"]))
    kc = np.tile([6.0, 8.0], (T, 1))        # stored context key t = R(t) (6, 8): base vector at position t
    pos_q = (T if offset else 0) + np.arange(L)
    pos_kb = (T if offset else 0) + np.arange(L)

    def score(a, pa, b, pb):   # <R(pa) a, R(pb) b> = |a| |b| cos(phi_b - phi_a + pb - pa)
        na, nb = np.hypot(a[:, 0], a[:, 1]), np.hypot(b[:, 0], b[:, 1])
        pha, phb = np.arctan2(a[:, 1], a[:, 0]), np.arctan2(b[:, 1], b[:, 0])
        return na[:, None] * nb[None, :] * np.cos(phb[None, :] - pha[:, None] + pb[None, :] - pa[:, None])

    sc = np.concatenate([score(q, pos_q, kc, np.arange(T)), score(q, pos_q, kb, pos_kb)], axis=1) / np.sqrt(h)
    return scipy.special.softmax(sc, axis=1)[:, :T]


@pytest.mark.parametrize("T", [3, 10])
def test_block_rope_positions_follow_context(oracle_lib, T):
    o = oracle_lib
    L, anchor, mask_id = 4, 21, synth.TINY.vocab - 1
    s, w, kv = _rope_case(T)
    args = (kv, T, np.array([T], np.int32), np.array([anchor], np.int32), mask_id, L)
    x0 = f64(np.stack([w["embed"][anchor]] + [w["embed"][mask_id]] * (L - 1)))[:, :T]
    want = _rope_closed_form(o, s, w, kv, T, L, anchor, mask_id)
    wrong = _rope_closed_form(o, s, w, kv, T, L, anchor, mask_id, offset=False)
    # q, k and the output are stored in bf16, so the weights read back carry ~1e-2 of rounding; the
    # mistaken position convention moves them by far more
    tol = 3e-2
    assert np.max(np.abs(want - wrong)) > 10 * tol
    got = f64(o.draft_block(o.Model(s, w), *args))[:, :T] - x0
    assert np.max(np.abs(got - want)) < tol, np.max(np.abs(got - want))
    with planted(o, "double pos = (double)(ctx_len[b] + j);", "double pos = (double)(j);"):
        bad = f64(o.draft_block(o.Model(s, w), *args))[:, :T] - x0
    assert np.max(np.abs(bad - want)) > 10 * tol
    assert np.max(np.abs(bad - wrong)) < tol


# ---- fusion order of several target-layer features ----------------------------------------------------------

@pytest.mark.parametrize("src", [0, 1, 2])
def test_fusion_selects_feature_source(oracle_lib, src):
    """n_f = 3, W_fc = [0 | I | 0] placed on source `src`, W_v = [I 0] on the first H_kv h dims of ctx:
    V^0(t) = bf16(RMSNorm_hidden(F_src[t])) restricted to those dims, for every context row t."""
    o = oracle_lib
    s = shape_with(n_layers=1, n_feat=3)
    d, h, nq, nkv = s.d_model, s.head_dim, s.n_q_heads, s.n_kv_heads
    w = synth.make_weights(s, 321)
    fc = np.zeros((d, 3 * d), np.float32)
    fc[np.arange(d), src * d + np.arange(d)] = 1.0
    w["w_fc"] = bits(fc)
    wv = np.zeros((nkv * h, d), np.float32)
    wv[np.arange(nkv * h), np.arange(nkv * h)] = 1.0
    w["layers"][0]["wqkv"][(nq + nkv) * h:] = bits(wv)
    T = 4
    feats = synth.make_features(s, T, 322)
    x = f64(feats[src])
    want = o.round_bf16(x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + s.rms_eps) * f64(w["hidden_norm"]))
    want = want[:, :nkv * h].reshape(T, nkv, h).transpose(1, 0, 2)
    run = lambda: o.prepare_context(o.Model(s, w), np.array([0, T], np.int32), feats, T)[0, 0, 1]
    np.testing.assert_array_equal(run(), want)
    if src != 1:   # reversing the concatenation order moves sources 0 and 2
        with planted(o, "bf(feats[s][(size_t)(r0 + r) * d + k])", "bf(feats[nf - 1 - s][(size_t)(r0 + r) * d + k])"):
            assert not np.array_equal(run(), want)
