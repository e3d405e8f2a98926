"""An fp32 restatement of the drafter forward, written from the method's definition in plain numpy.

Test infrastructure only (it is neither the oracle nor the CUDA path, and neither imports it).  It takes the same
steps as the oracle — context K/V given, anchor + mask block, pre-norm layers with per-head q/k RMSNorm and
rotate-half RoPE at positions ctx_len + j, bidirectional softmax attention over [context ; block], SwiGLU MLP,
final RMSNorm and LM head — and rounds to bf16 at the same storage points, but every dot product and reduction
accumulates in float32 (numpy's own summation order) instead of float64.  It answers one question: how far does a
correct implementation that merely accumulates in fp32 land from the fp64 oracle?  (VFlash paper (zh) §2.1-§2.2
for the pass; VFlash blog "Key claims" for the five-layer drafter; readings R1-R5 of this repository.)
"""
import numpy as np

import synth


def _f32(bits):
    return synth.bf16_bits_to_f32(bits)


def _rb(x):
    """float32 -> bf16 storage -> float32 (round to nearest even)."""
    return synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.asarray(x, np.float32)))


def _rmsnorm(x, g, eps):
    ms = np.mean(x * x, axis=-1, keepdims=True, dtype=np.float32)
    return x / np.sqrt(ms + np.float32(eps)) * g


def _rope(x, pos, theta, h):
    half = h // 2
    i = np.arange(half, dtype=np.float64)
    ang = pos[:, None].astype(np.float64) * np.power(float(theta), -2.0 * i / h)[None, :]
    c, s = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    x1, x2 = x[..., :half], x[..., half:]
    c = c.reshape(c.shape[0], *([1] * (x.ndim - 2)), half)
    s = s.reshape(s.shape[0], *([1] * (x.ndim - 2)), half)
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def weights_f32(w):
    """The bf16 weights as float32 arrays (exact), converted once for repeated passes."""
    out = {k: _f32(v) for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: _f32(v) for k, v in lw.items()} for lw in w["layers"]]
    out["_f32"] = True
    return out


def draft_block(shape, w, kv_store, ctx_len, anchor, mask_id, L, want_layers=False):
    """One request (batch 1).  w: bf16-bit weights or weights_f32(w).  kv_store [layers][1][K|V][kv heads][t_cap][h]
    bf16 bits.  Returns the hidden states [L, d] as float32 (bf16 values) and, when asked, every layer's."""
    if not w.get("_f32"):
        w = weights_f32(w)
    s = shape
    d, h, nq, nkv, F = s.d_model, s.head_dim, s.n_q_heads, s.n_kv_heads, s.d_ff
    grp = nq // nkv
    T = int(ctx_len)
    x = np.stack([w["embed"][int(anchor)]] + [w["embed"][int(mask_id)]] * (L - 1))
    pos = np.arange(L) + T
    layers = []
    for l, lw in enumerate(w["layers"]):
        xn = _rb(_rmsnorm(x, lw["attn_norm"], s.rms_eps))
        qkv = xn @ lw["wqkv"].T
        q = qkv[:, :nq * h].reshape(L, nq, h)
        k = qkv[:, nq * h:(nq + nkv) * h].reshape(L, nkv, h)
        v = qkv[:, (nq + nkv) * h:].reshape(L, nkv, h)
        q = _rb(_rope(_rmsnorm(q, lw["q_norm"], s.rms_eps), pos, s.rope_theta, h))
        k = _rb(_rope(_rmsnorm(k, lw["k_norm"], s.rms_eps), pos, s.rope_theta, h))
        v = _rb(v)
        o = np.empty((L, nq, h), np.float32)
        for g in range(nkv):
            K = np.concatenate([_f32(kv_store[l, 0, 0, g, :T]), k[:, g]])
            V = np.concatenate([_f32(kv_store[l, 0, 1, g, :T]), v[:, g]])
            for i in range(g * grp, (g + 1) * grp):
                sc = (q[:, i] @ K.T) * np.float32(1.0 / np.sqrt(h))
                sc = sc - sc.max(axis=1, keepdims=True)
                p = np.exp(sc)
                p /= p.sum(axis=1, keepdims=True, dtype=np.float32)
                o[:, i] = p @ V
        o = _rb(o.reshape(L, nq * h))
        x = _rb(x + o @ lw["wo"].T)
        xn = _rb(_rmsnorm(x, lw["mlp_norm"], s.rms_eps))
        gu = xn @ lw["w_gate_up"].T
        gate, up = gu[:, :F], gu[:, F:]
        hm = _rb(gate / (np.float32(1.0) + np.exp(-gate)) * up)
        x = _rb(x + hm @ lw["w_down"].T)
        layers.append(x)
    return (x, layers) if want_layers else x


def logits(shape, w, hidden, L):
    """Final RMSNorm + unconstrained LM head of block positions 1..L-1, float32."""
    if not w.get("_f32"):
        w = weights_f32(w)
    z = _rb(_rmsnorm(hidden[1:L], w["final_norm"], shape.rms_eps))
    return z @ w["lm_head"].T
