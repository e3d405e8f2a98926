"""CPU oracle of the block-drafter hot path (ctypes wrapper over ``fpd_oracle.c``).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(and its reference arm) may import this package.  The product path (``block_diffusion_speculative_non_gb300``)
never imports it and shares no code with it.

Every function takes the seeded inputs from ``synth`` (bf16 as uint16 bit patterns) and returns numpy
arrays.  Arithmetic is fp64 with bf16 rounding at the storage points documented in ``fpd_oracle.c``.

Parity pins (tests/test_oracle_pins.py) tie each function to something other than itself: closed forms,
exhaustive enumeration, brute force on tiny inputs, numpy's library routines, degenerate cases.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fpd_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_MAX_LAYERS = 8

_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i16p = ctypes.POINTER(ctypes.c_int16)
_i8p = ctypes.POINTER(ctypes.c_int8)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/liboracle.so (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=gnu11", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _OracleModel(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("d", ctypes.c_int32), ("nq", ctypes.c_int32), ("nkv", ctypes.c_int32),
        ("h", ctypes.c_int32), ("F", ctypes.c_int32), ("V", ctypes.c_int32), ("nf", ctypes.c_int32),
        ("eps", ctypes.c_double), ("theta", ctypes.c_double),
        ("embed", _u16p), ("w_fc", _u16p), ("hidden_norm", _u16p), ("final_norm", _u16p), ("lm_head", _u16p),
        ("attn_norm", _u16p * _MAX_LAYERS), ("wqkv", _u16p * _MAX_LAYERS), ("q_norm", _u16p * _MAX_LAYERS),
        ("k_norm", _u16p * _MAX_LAYERS), ("wo", _u16p * _MAX_LAYERS), ("mlp_norm", _u16p * _MAX_LAYERS),
        ("w_gate_up", _u16p * _MAX_LAYERS), ("w_down", _u16p * _MAX_LAYERS),
        ("q_wqkv", _u8p * _MAX_LAYERS), ("q_wo", _u8p * _MAX_LAYERS), ("q_gate_up", _u8p * _MAX_LAYERS),
        ("q_down", _u8p * _MAX_LAYERS), ("q_lm_head", _u8p),
        ("e_wqkv", _i8p * _MAX_LAYERS), ("e_wo", _i8p * _MAX_LAYERS), ("e_gate_up", _i8p * _MAX_LAYERS),
        ("e_down", _i8p * _MAX_LAYERS), ("e_lm_head", _i8p),
    ]


_lib = None


def _configure(l):
    """Declare the ctypes signatures of one build of the oracle."""
    l.oracle_round_bf16.restype = ctypes.c_uint16
    l.oracle_round_bf16.argtypes = [ctypes.c_double]
    l.oracle_bf16_to_double.restype = ctypes.c_double
    l.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    l.oracle_silu.restype = ctypes.c_double
    l.oracle_silu.argtypes = [ctypes.c_double]
    l.oracle_num_threads.restype = ctypes.c_int
    l.oracle_rmsnorm.argtypes = [ctypes.c_int, _f64p, _u16p, ctypes.c_double, _f64p]
    l.oracle_rope.argtypes = [ctypes.c_int, _f64p, ctypes.c_double, ctypes.c_double]
    l.oracle_linear.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _f64p, _u16p, _f64p]
    l.oracle_attention.argtypes = [ctypes.c_int, ctypes.c_int, _f64p, ctypes.c_int, _u16p, _u16p,
                                   ctypes.c_int, _f64p, _f64p, ctypes.c_double, _f64p]
    l.oracle_prepare_context.argtypes = [ctypes.POINTER(_OracleModel), ctypes.c_int, ctypes.c_int, _i32p,
                                         _i32p, ctypes.POINTER(_u16p), _u16p, ctypes.c_int]
    l.oracle_draft_block.argtypes = [ctypes.POINTER(_OracleModel), ctypes.c_int, ctypes.c_int, _u16p,
                                     ctypes.c_int, _i32p, _i32p, ctypes.c_int32, _u16p, _u16p, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, _u16p]
    l.oracle_constrain_argmax.argtypes = [ctypes.POINTER(_OracleModel), ctypes.c_int, ctypes.c_int, _u16p,
                                          ctypes.c_int, _i32p, _i32p, _i16p, _i32p, _f64p, _f64p, ctypes.c_int]
    l.oracle_e4m3_decode.restype = ctypes.c_double
    l.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    l.oracle_e4m3_encode.restype = ctypes.c_uint8
    l.oracle_e4m3_encode.argtypes = [ctypes.c_double]
    l.oracle_block_exponent.restype = ctypes.c_int
    l.oracle_block_exponent.argtypes = [ctypes.c_double]
    l.oracle_quantize_fp8.argtypes = [ctypes.c_int, ctypes.c_int, _f64p, _u8p, _i8p]
    l.oracle_quantize_fp8_bf16.argtypes = [ctypes.c_int, ctypes.c_int, _u16p, _u8p, _i8p]
    l.oracle_linear_fp8.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _f64p, _u8p, _i8p, _f64p]
    l.oracle_verify.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, _i32p, ctypes.c_int, _i32p,
                                _i32p, _i16p, _i8p, ctypes.c_int32, _i32p, _i32p, _i32p]
    return l


def lib():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def use_library(path: str):
    """Route every oracle call through another build of the oracle source (the pin tests use this to run a
    copy with a deliberately planted mistake and check that the pins reject it), then restore the default."""
    global _lib
    saved = lib()
    _lib = _configure(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = saved


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))


def _p(a, t):
    return a.ctypes.data_as(t) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- building blocks (exported for the pins) ------------------------------------------------------------

def round_bf16(x) -> np.ndarray:
    """fp64 -> bf16 bit patterns, round to nearest even."""
    x = np.asarray(x, dtype=np.float64)
    f = lib().oracle_round_bf16
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def bf16_to_f64(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    f = lib().oracle_bf16_to_double
    return np.array([f(int(v)) for v in b.ravel()], dtype=np.float64).reshape(b.shape)


def rmsnorm(x, g_bits, eps) -> np.ndarray:
    x = _c(x, np.float64)
    g = _c(g_bits, np.uint16)
    y = np.empty_like(x)
    lib().oracle_rmsnorm(x.size, _p(x, _f64p), _p(g, _u16p), float(eps), _p(y, _f64p))
    return y


def rope(x, pos, theta) -> np.ndarray:
    y = _c(x, np.float64).copy()
    lib().oracle_rope(y.size, _p(y, _f64p), float(pos), float(theta))
    return y


def silu(v: float) -> float:
    return float(lib().oracle_silu(float(v)))


def linear(X, W_bits) -> np.ndarray:
    X = _c(X, np.float64)
    W = _c(W_bits, np.uint16)
    M, K = X.shape
    N = W.shape[0]
    assert W.shape[1] == K
    Y = np.empty((M, N), dtype=np.float64)
    lib().oracle_linear(M, N, K, _p(X, _f64p), _p(W, _u16p), _p(Y, _f64p))
    return Y


def attention(q, k_ctx_bits, v_ctx_bits, k_blk, v_blk, scale) -> np.ndarray:
    """q [R, h] f64; context keys/values [n_ctx, h] bf16 bits; block keys/values [n_blk, h] f64."""
    q = _c(q, np.float64)
    R, h = q.shape
    kc = _c(k_ctx_bits, np.uint16).reshape(-1, h)
    vc = _c(v_ctx_bits, np.uint16).reshape(-1, h)
    kb = _c(k_blk, np.float64).reshape(-1, h)
    vb = _c(v_blk, np.float64).reshape(-1, h)
    o = np.empty((R, h), dtype=np.float64)
    lib().oracle_attention(h, R, _p(q, _f64p), kc.shape[0], _p(kc, _u16p), _p(vc, _u16p), kb.shape[0],
                           _p(kb, _f64p), _p(vb, _f64p), float(scale), _p(o, _f64p))
    return o


# ---- f2: E4M3 and the 128-element group quantisation (fpd_oracle.c, "f2" section) -------------------------

def e4m3_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8)
    f = lib().oracle_e4m3_decode
    return np.array([f(int(v)) for v in c.ravel()], dtype=np.float64).reshape(c.shape)


def e4m3_encode(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    f = lib().oracle_e4m3_encode
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint8).reshape(x.shape)


def block_exponent(amax: float) -> int:
    return int(lib().oracle_block_exponent(float(amax)))


def quantize_fp8(X) -> tuple:
    """Rows of X (float values, or bf16 bit patterns as uint16) -> (codes [N, K] uint8, exponents [N, K/128] int8)."""
    X = np.asarray(X)
    N, K = X.shape
    assert K % 128 == 0
    codes = np.empty((N, K), dtype=np.uint8)
    exps = np.empty((N, K // 128), dtype=np.int8)
    if X.dtype == np.uint16:
        Xc = _c(X, np.uint16)
        lib().oracle_quantize_fp8_bf16(N, K, _p(Xc, _u16p), _p(codes, _u8p), _p(exps, _i8p))
    else:
        Xc = _c(X, np.float64)
        lib().oracle_quantize_fp8(N, K, _p(Xc, _f64p), _p(codes, _u8p), _p(exps, _i8p))
    return codes, exps


def dequantize_fp8(codes, exps) -> np.ndarray:
    """The values the quantised rows stand for: decode(code) * 2^exponent of its group."""
    codes = np.asarray(codes, dtype=np.uint8)
    v = e4m3_decode(np.arange(256, dtype=np.uint8))[codes]
    return v * np.exp2(np.repeat(np.asarray(exps, dtype=np.float64), 128, axis=1))


def linear_fp8(X, codes, exps) -> np.ndarray:
    """X [M, K] float values (quantised here by rows) against quantised weights [N, K]."""
    X = _c(X, np.float64)
    M, K = X.shape
    q = _c(codes, np.uint8)
    e = _c(exps, np.int8)
    Y = np.empty((M, q.shape[0]), dtype=np.float64)
    lib().oracle_linear_fp8(M, q.shape[0], K, _p(X, _f64p), _p(q, _u8p), _p(e, _i8p), _p(Y, _f64p))
    return Y


# ---- the hot path ---------------------------------------------------------------------------------------

class Model:
    """Holds the weights (bf16 bit patterns from synth.make_weights) and the C struct pointing at them."""

    def __init__(self, shape, weights, fp8=False):
        self.shape = shape
        self.w = weights
        self.fp8 = bool(fp8)
        s = _OracleModel()
        s.n_layers, s.d, s.nq, s.nkv = shape.n_layers, shape.d_model, shape.n_q_heads, shape.n_kv_heads
        s.h, s.F, s.V, s.nf = shape.head_dim, shape.d_ff, shape.vocab, shape.n_feat
        s.eps, s.theta = float(shape.rms_eps), float(shape.rope_theta)
        keep = []

        def ptr(a):
            a = _c(a, np.uint16)
            keep.append(a)
            return a.ctypes.data_as(_u16p)

        s.embed, s.w_fc = ptr(weights["embed"]), ptr(weights["w_fc"])
        s.hidden_norm, s.final_norm = ptr(weights["hidden_norm"]), ptr(weights["final_norm"])
        s.lm_head = ptr(weights["lm_head"])
        for l, lw in enumerate(weights["layers"]):
            for name in ("attn_norm", "wqkv", "q_norm", "k_norm", "wo", "mlp_norm", "w_gate_up", "w_down"):
                getattr(s, name)[l] = ptr(lw[name])
        if fp8:   # the FP8 copies of the streamed matrices, quantised by this oracle from the bf16 weights
            def q(a):
                codes, exps = quantize_fp8(_c(a, np.uint16))
                keep.extend([codes, exps])
                return codes.ctypes.data_as(_u8p), exps.ctypes.data_as(_i8p)

            s.q_lm_head, s.e_lm_head = q(weights["lm_head"])
            for l, lw in enumerate(weights["layers"]):
                for name, qn, en in (("wqkv", "q_wqkv", "e_wqkv"), ("wo", "q_wo", "e_wo"),
                                     ("w_gate_up", "q_gate_up", "e_gate_up"), ("w_down", "q_down", "e_down")):
                    getattr(s, qn)[l], getattr(s, en)[l] = q(lw[name])
        self._keep = keep
        self.c = s

    def fp8_copy(self, name, layer=None):
        """(codes, exponents) numpy views of one FP8 copy: name in wqkv, wo, w_gate_up, w_down, lm_head."""
        assert self.fp8
        sh = self.shape
        d, F, nqkv = sh.d_model, sh.d_ff, (sh.n_q_heads + 2 * sh.n_kv_heads) * sh.head_dim
        rows, K = {"wqkv": (nqkv, d), "wo": (d, sh.n_q_heads * sh.head_dim), "w_gate_up": (2 * F, d),
                   "w_down": (d, F), "lm_head": (sh.vocab, d)}[name]
        qn, en = {"wqkv": ("q_wqkv", "e_wqkv"), "wo": ("q_wo", "e_wo"), "w_gate_up": ("q_gate_up", "e_gate_up"),
                  "w_down": ("q_down", "e_down"), "lm_head": ("q_lm_head", "e_lm_head")}[name]
        qp, ep = getattr(self.c, qn), getattr(self.c, en)
        if layer is not None:
            qp, ep = qp[layer], ep[layer]
        codes = np.ctypeslib.as_array(qp, shape=(rows, K))
        exps = np.ctypeslib.as_array(ep, shape=(rows, K // 128))
        return codes, exps


def prepare_context(model: Model, row_off, feats, t_cap, batch=None, pos_start=None, kv_store=None):
    """Returns the KV store [layer][b][K|V][kv_head][t_cap][h] (bf16 bits); rows not written stay as given
    (zero for a new store)."""
    sh = model.shape
    row_off = _c(row_off, np.int32)
    B = len(row_off) - 1 if batch is None else batch
    total = int(row_off[-1])
    if kv_store is None:
        kv_store = np.zeros((sh.n_layers, B, 2, sh.n_kv_heads, t_cap, sh.head_dim), dtype=np.uint16)
    fs = [_c(f, np.uint16) for f in feats]
    arr = (_u16p * len(fs))(*[f.ctypes.data_as(_u16p) for f in fs])
    ps = None if pos_start is None else _c(pos_start, np.int32)
    rc = lib().oracle_prepare_context(ctypes.byref(model.c), B, total, _p(row_off, _i32p), _p(ps, _i32p), arr,
                                      _p(kv_store, _u16p), int(t_cap))
    if rc:
        raise ValueError("oracle_prepare_context: bad sizes")
    return kv_store


FEW_TOKENS = 16   # calls with at most this many positions run the weight-streaming (FP8-capable) path


def draft_block(model: Model, kv_store, t_cap, ctx_len, anchor, mask_id, block_len, want_layers=False, fp8=None,
                layers=None, x_in=None):
    """Returns hidden [B*L, d] (bf16 bits) and, when asked, the per-layer residual [n_layers, B*L, d].
    fp8 None: the FP8 projections exactly when the model has FP8 copies and the call has at most 16 positions.
    layers (l0, l1) with x_in [B*L, d] bf16 bits: only layers l0..l1-1, starting from the residual x_in."""
    sh = model.shape
    ctx_len = _c(ctx_len, np.int32)
    anchor = _c(anchor, np.int32)
    B = len(anchor)
    kv = _c(kv_store, np.uint16)
    hidden = np.empty((B * block_len, sh.d_model), dtype=np.uint16)
    lay = np.zeros((sh.n_layers, B * block_len, sh.d_model), dtype=np.uint16) if want_layers else None
    if fp8 is None:
        fp8 = model.fp8 and B * block_len <= FEW_TOKENS
    assert not fp8 or model.fp8
    l0, l1 = (0, sh.n_layers) if layers is None else layers
    xi = None if x_in is None else _c(x_in, np.uint16).reshape(B * block_len, sh.d_model)
    rc = lib().oracle_draft_block(ctypes.byref(model.c), B, block_len, _p(kv, _u16p), int(t_cap),
                                  _p(ctx_len, _i32p), _p(anchor, _i32p), int(mask_id), _p(hidden, _u16p),
                                  _p(lay, _u16p), int(bool(fp8)), int(l0), int(l1), _p(xi, _u16p))
    if rc:
        raise ValueError("oracle_draft_block: bad arguments")
    return (hidden, lay) if want_layers else hidden


def constrain_argmax(model: Model, hidden, batch, block_len, layout=None, want_logits=False, fp8=None):
    """Returns (tokens [B, L-1] int32, margin [B*(L-1)] f64, logits [B*(L-1), V] f64 or None).  Logits of
    illegal columns are NaN.  fp8 None: the FP8 LM head exactly when the model has FP8 copies, there is no
    layout and at most 16 positions."""
    sh = model.shape
    hid = _c(hidden, np.uint16)
    P = block_len - 1
    tokens = np.empty((batch, P), dtype=np.int32)
    margin = np.empty(batch * P, dtype=np.float64)
    logits = np.full((batch * P, sh.vocab), np.nan, dtype=np.float64) if want_logits else None
    if layout is None:
        n_class, co, cr, pc = 0, None, None, None
    else:
        n_class = len(layout["class_off"]) - 1
        co = _c(layout["class_off"], np.int32)
        cr = _c(layout["class_ranges"], np.int32)
        pc = _c(np.broadcast_to(layout["pos_class"], (batch, block_len)) if layout["pos_class"].ndim == 1
                else layout["pos_class"], np.int16)
    if fp8 is None:
        fp8 = model.fp8 and layout is None and batch * P <= FEW_TOKENS
    assert not fp8 or model.fp8
    rc = lib().oracle_constrain_argmax(ctypes.byref(model.c), batch, block_len, _p(hid, _u16p), n_class,
                                       _p(co, _i32p), _p(cr, _i32p), _p(pc, _i16p), _p(tokens, _i32p),
                                       _p(logits, _f64p), _p(margin, _f64p), int(bool(fp8)))
    if rc:
        raise ValueError("oracle_constrain_argmax: bad layout")
    if layout is not None and len(layout.get("pairs", ())) and logits is None:
        return constrain_argmax(model, hidden, batch, block_len, layout, want_logits=True, fp8=fp8)[:2] + (None,)
    if layout is not None and len(layout.get("pairs", ())):
        _pair_offscreen(tokens, margin, logits, block_len, layout["pairs"], int(layout["off_id"]))
    return tokens, margin, logits


def _pair_offscreen(tokens, margin, logits, block_len, pairs, off_id):
    """VFlash paper (zh) §2.5, the cross-position rule on the computed logits: the two positions of a pair take the
    off-screen id together or not at all.  The decision compares o_p + o_q with a_p + a_q (a = the best legal logit
    other than off_id, o = off_id's logit), taken like the argmax in fp32 (reading R16); ties stay on screen."""
    P = block_len - 1
    f32 = np.float32
    for b in range(tokens.shape[0]):
        for p, q in np.asarray(pairs).reshape(-1, 2):
            rows = (b * P + int(p) - 1, b * P + int(q) - 1)
            best, offl = [], []
            for r in rows:
                lg = logits[r].astype(np.float32)          # fp32 decision values; illegal ids are NaN
                o = lg[off_id]
                lg = lg.copy()
                lg[off_id] = np.nan
                if np.all(np.isnan(lg)):
                    best = None
                    break
                i = int(np.nanargmax(lg))                  # the lowest id among equal maxima
                best.append((i, lg[i]))
                offl.append(o)
            if best is None:
                continue
            on = f32(f32(best[0][1]) + f32(best[1][1]))
            off = f32(f32(offl[0]) + f32(offl[1]))
            take_off = bool(off > on)
            for k, r in enumerate(rows):
                tokens.reshape(-1)[r] = off_id if take_off else best[k][0]
                margin[r] = min(margin[r], abs(float(off) - float(on)))


def verify(mode, draft, target=None, layout=None, rule=None, pad_id=-1, margin=None, tau=None):
    """mode 0 = text, 1 = schema, 2 = schema + confidence (prefix-k).  Returns (accept_len [B], committed [B, L],
    valid [B])."""
    if mode == 2:
        return _verify_prefix(draft, layout, rule, pad_id, margin, tau)
    draft = _c(draft, np.int32)
    B, P = draft.shape
    L = P + 1
    acc = np.empty(B, dtype=np.int32)
    com = np.empty((B, L), dtype=np.int32)
    val = np.empty(B, dtype=np.int32)
    tg = _c(target, np.int32) if target is not None else None
    if mode == 1:
        n_class = len(layout["class_off"]) - 1
        co = _c(layout["class_off"], np.int32)
        cr = _c(layout["class_ranges"], np.int32)
        pc = _c(np.broadcast_to(layout["pos_class"], (B, L)) if np.asarray(layout["pos_class"]).ndim == 1
                else layout["pos_class"], np.int16)
        rl = _c(np.broadcast_to(rule, (B, L)) if np.asarray(rule).ndim == 1 else rule, np.int8)
    else:
        n_class, co, cr, pc, rl = 0, None, None, None, None
    rc = lib().oracle_verify(int(mode), B, L, _p(draft, _i32p), _p(tg, _i32p), n_class, _p(co, _i32p),
                             _p(cr, _i32p), _p(pc, _i16p), _p(rl, _i8p), int(pad_id), _p(acc, _i32p),
                             _p(com, _i32p), _p(val, _i32p))
    if rc:
        raise ValueError("oracle_verify: bad arguments")
    return acc, com, val


def grid_field_value(tokens, digit_ids, plus_id, minus_id, pad_id):
    """VFlash paper (zh) §2.3: one fixed-width field [sign][d_1..d_w] -> its integer value, or None when the field
    is not a well-formed numeral (sign not + or -, a pad after a real digit, a pad or non-digit in the last slot).
    Unused HIGH digits hold the pad (mask) token, so the digits read most significant first."""
    sign, digits = int(tokens[0]), [int(t) for t in tokens[1:]]
    if sign not in (plus_id, minus_id):
        return None
    value, seen_real = 0, False
    for i, t in enumerate(digits):
        if t == pad_id:
            if seen_real or i == len(digits) - 1:
                return None
            continue
        if t not in digit_ids:
            return None
        seen_real = True
        value = 10 * value + digit_ids.index(t)
    return -value if sign == minus_id else value


def grid_to_text(committed, accept, digit_ids, plus_id, minus_id, pad_id, n_axes=3, width=5, axis_sep=",",
                 point_sep=";"):
    """VFlash paper (zh) §2.3: the fixed-width grid converted back to the target's text format.  committed[b][i]
    holds block position i + 1 (position 0 is the start token); waypoint w starts at block position
    1 + w * (n_axes * (1 + width) + 1) with n_axes fields and one separator.  Request b's text lists its complete
    waypoints inside the accepted positions 1..accept[b], stopping at the first malformed field."""
    digit_ids = [int(t) for t in digit_ids]
    per_wp = n_axes * (1 + width) + 1
    texts = []
    for row, acc in zip(np.asarray(committed), np.asarray(accept)):
        L = len(row) + 0
        acc = max(0, min(int(acc), L - 1))
        points = []
        w = 0
        while True:
            first = 1 + w * per_wp
            if first + n_axes * (1 + width) - 1 > acc:
                break
            vals = []
            for a in range(n_axes):
                p0 = first + a * (1 + width)
                v = grid_field_value(row[p0 - 1:p0 - 1 + 1 + width], digit_ids, plus_id, minus_id, pad_id)
                if v is None:
                    break
                vals.append(str(v))
            if len(vals) < n_axes:
                break
            points.append(axis_sep.join(vals))
            w += 1
        texts.append(point_sep.join(points))
    return texts


def _verify_prefix(draft, layout, rule, pad_id, margin, tau):
    """VFlash paper (zh) §2.5: the first k draft positions are kept; for bounding boxes k stops before the first
    uncertain coordinate.  Reading: a position whose rule is 4 (confident) is uncertain when the drafter's top-2
    margin there is below tau.  The first failing position p is the earlier of the schema's (mode 1) and the first
    uncertain one; k = p - 1."""
    draft = _c(draft, np.int32)
    B, P = draft.shape
    L = P + 1
    rl = np.broadcast_to(rule, (B, L)) if np.asarray(rule).ndim == 1 else np.asarray(rule)
    acc, com, val = verify(1, draft, layout=layout, rule=rl, pad_id=pad_id)
    mg = np.asarray(margin, dtype=np.float64).reshape(B, P)
    for b in range(B):
        p = int(acc[b]) + 1                       # the schema's first failing position (L when none)
        for j in range(1, p):
            if rl[b, j] == 4 and not (mg[b, j - 1] >= tau):
                p = j
                break
        acc[b] = p - 1
        com[b, :p - 1] = draft[b, :p - 1]
        com[b, p - 1:] = -1
        val[b] = int(p == L)
    return acc, com, val
