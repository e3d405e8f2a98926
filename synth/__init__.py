"""Seeded synthetic inputs for the block-drafter hot path.

This module only draws random numbers and lays them out; it contains none of the method's arithmetic.
Both the CPU oracle (``oracle/``) and the CUDA path (``block_diffusion_speculative_non_gb300``) are fed
from here, so that the two sides see bit-identical inputs.

Shapes and distributions follow the workloads the pages describe (no dataset or trained weights are
available, so seeded synthetic data stands in):

* drafter shape: five non-causal layers (VFlash blog, "Key claims"); a 4B-class target shape for the
  full-size configurations; a tiny shape for CPU-speed checks;
* weights N(0, 0.02) in bf16; RMSNorm gains 1 + N(0, 0.02) so activations keep unit scale;
* target-layer features N(0, 1) in bf16;
* 16-position text blocks (VFlash blog, "Method");
* a primitive of 64 waypoints x (2 image + 3 metric coordinates + 1 delimiter) on a contiguous
  1001-token coordinate slice (VFlash paper (zh), §2.3);
* fixed-width numerals: one sign slot {+,-} and five digit slots {0-9, pad} per axis, three axes and a
  separator per waypoint, 20 waypoints (VFlash paper (zh), §2.3);
* target rows whose agreement prefix with the draft is Geometric(p).

All bf16 data is carried as numpy uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = [
    "ModelShape", "CONFIGS", "f32_to_bf16_bits", "bf16_bits_to_f32", "make_weights", "make_features",
    "make_kv_store", "layout_special_tokens", "layout_fixed_width", "layout_bbox", "make_target_rows", "Workload",
    "make_workload",
]


@dataclasses.dataclass(frozen=True)
class ModelShape:
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    vocab: int
    n_feat: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim


TINY = ModelShape(n_layers=5, d_model=512, n_q_heads=8, n_kv_heads=2, head_dim=64, d_ff=1536, vocab=4096,
                  n_feat=3)
FULL = ModelShape(n_layers=5, d_model=2560, n_q_heads=32, n_kv_heads=8, head_dim=128, d_ff=9728,
                  vocab=151936, n_feat=5)

# The five workloads: shape, batch, context lengths, block length, vocabulary layout, acceptance mode.
CONFIGS = {
    "tiny_text_b1": dict(shape=TINY, batch=1, t_ctx=128, block_len=16, layout=None, geo_p=0.3, seed=1000),
    "text_4b_b1": dict(shape=FULL, batch=1, t_ctx=2048, block_len=16, layout=None, geo_p=0.25, seed=2000),
    "primitive_special_b1": dict(shape=FULL, batch=1, t_ctx=4096, block_len=385, layout="special",
                                 geo_p=None, seed=3000),
    "primitive_fixedwidth_b32": dict(shape=FULL, batch=32, t_ctx=(512, 2048), block_len=381,
                                     layout="fixed_width", geo_p=None, seed=4000),
}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(seed_seq: np.random.SeedSequence, shape, std: float, mean: float = 0.0) -> np.ndarray:
    """N(mean, std^2) rounded to bf16; large tensors are filled in parallel chunks of fixed size so the
    values depend only on the seed, never on the thread count."""
    n = int(np.prod(shape))
    chunk = 1 << 22
    n_chunks = (n + chunk - 1) // chunk
    children = seed_seq.spawn(n_chunks)
    out = np.empty(n, dtype=np.uint16)

    def fill(i):
        lo, hi = i * chunk, min(n, (i + 1) * chunk)
        g = np.random.default_rng(children[i])
        v = g.standard_normal(hi - lo, dtype=np.float32)
        v *= np.float32(std)
        if mean:
            v += np.float32(mean)
        out[lo:hi] = f32_to_bf16_bits(v)

    if n_chunks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(max_workers=8) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.reshape(shape)


def make_weights(shape: ModelShape, seed: int, zero: tuple = ()) -> dict:
    """Drafter weights as bf16 bit patterns.  Matrices and embeddings ~ N(0, 0.02); RMSNorm gains
    ~ 1 + N(0, 0.02).  ``zero`` names weight families to set to exactly zero (degenerate-case tests),
    e.g. ("wo", "w_down")."""
    s = shape
    root = np.random.SeedSequence(seed)
    kids = iter(root.spawn(8 + 8 * s.n_layers))
    std = 0.02

    def mat(name, rows, cols):
        t = _normal_bf16(next(kids), (rows, cols), std)
        if name in zero:
            t[...] = 0
        return t

    def gain(name, n):
        t = _normal_bf16(next(kids), (n,), std, mean=1.0)
        if name in zero:
            t[...] = 0
        return t

    w = {
        "embed": mat("embed", s.vocab, s.d_model),
        "w_fc": mat("w_fc", s.d_model, s.n_feat * s.d_model),
        "hidden_norm": gain("hidden_norm", s.d_model),
        "final_norm": gain("final_norm", s.d_model),
        "lm_head": mat("lm_head", s.vocab, s.d_model),
        "layers": [],
    }
    for _ in range(s.n_layers):
        w["layers"].append({
            "attn_norm": gain("attn_norm", s.d_model),
            "wqkv": mat("wqkv", s.qkv_rows, s.d_model),
            "q_norm": gain("q_norm", s.head_dim),
            "k_norm": gain("k_norm", s.head_dim),
            "wo": mat("wo", s.d_model, s.n_q_heads * s.head_dim),
            "mlp_norm": gain("mlp_norm", s.d_model),
            "w_gate_up": mat("w_gate_up", 2 * s.d_ff, s.d_model),
            "w_down": mat("w_down", s.d_model, s.d_ff),
        })
    if "wq_wk" in zero:   # zero the q and k rows of every wqkv (uniform-attention degenerate case)
        for lw in w["layers"]:
            lw["wqkv"][: (s.n_q_heads + s.n_kv_heads) * s.head_dim] = 0
    return w


def make_features(shape: ModelShape, total_rows: int, seed: int) -> list:
    """n_feat target-layer feature matrices [total_rows, d] ~ N(0, 1) (bf16 bits)."""
    kids = np.random.SeedSequence(seed).spawn(shape.n_feat)
    return [_normal_bf16(k, (total_rows, shape.d_model), 1.0) for k in kids]


def make_kv_store(shape: ModelShape, batch: int, t_cap: int, seed: int) -> np.ndarray:
    """A random context KV store [layer][b][K|V][kv_head][t_cap][h] ~ N(0, 1) (bf16 bits).  Used to feed
    block-pass checks at long contexts without running the context preparation first."""
    return _normal_bf16(np.random.SeedSequence(seed),
                        (shape.n_layers, batch, 2, shape.n_kv_heads, t_cap, shape.head_dim), 1.0)


def layout_special_tokens(vocab: int, n_waypoints: int = 64, coord_lo: int = 150000, n_coord: int = 1001,
                          delim_id: int = 151100, start_id: int = 151101, off_id: int | None = None) -> dict:
    """Primitive block with dedicated coordinate tokens: start token, then per waypoint
    [u, v (image), X, Y, Z (metric), delimiter].  All five coordinates share one contiguous slice of
    n_coord ids; the delimiter slot admits one id.  Class 0 = coordinate slice, class 1 = delimiter,
    class 2 = full vocabulary (unused here, kept so tables always carry an unconstrained class)."""
    assert coord_lo + n_coord <= vocab and delim_id < vocab and start_id < vocab
    L = 1 + 6 * n_waypoints
    pos_class = np.zeros(L, dtype=np.int16)
    rule = np.zeros(L, dtype=np.int8)
    for w in range(n_waypoints):
        base = 1 + 6 * w
        pos_class[base:base + 5] = 0
        pos_class[base + 5] = 1
        rule[base:base + 6] = 1
    pos_class[0] = 2
    class_off = np.array([0, 1, 2, 3], dtype=np.int32)
    class_ranges = np.array([coord_lo, coord_lo + n_coord, delim_id, delim_id + 1, 0, vocab], dtype=np.int32)
    lay = dict(block_len=L, pos_class=pos_class, rule=rule, class_off=class_off, class_ranges=class_ranges,
               pad_id=-1, start_id=start_id)
    if off_id is not None:
        # the image coordinates (u, v) of every waypoint may also be off screen, together (class 3 = slice + off)
        assert off_id >= coord_lo + n_coord
        for w in range(n_waypoints):
            pos_class[1 + 6 * w:3 + 6 * w] = 3
        lay["class_off"] = np.array([0, 1, 2, 3, 5], dtype=np.int32)
        lay["class_ranges"] = np.concatenate([class_ranges, [coord_lo, coord_lo + n_coord, off_id, off_id + 1]]
                                             ).astype(np.int32)
        lay["pairs"] = np.array([(1 + 6 * w, 2 + 6 * w) for w in range(n_waypoints)], dtype=np.int16)
        lay["off_id"] = int(off_id)
    return lay


def layout_bbox(vocab: int, n_boxes: int = 16, coord_lo: int = 150000, n_coord: int = 1001, delim_id: int = 151100,
                start_id: int = 151101) -> dict:
    """Bounding-box primitive: start token, then per box [x1, y1, x2, y2, delimiter], coordinates from the
    n_coord-id slice.  Coordinates carry the confidence rule (4): prefix acceptance stops before the first
    coordinate the drafter is unsure of; delimiters must be members."""
    L = 1 + 5 * n_boxes
    pos_class = np.zeros(L, dtype=np.int16)
    rule = np.zeros(L, dtype=np.int8)
    for k in range(n_boxes):
        base = 1 + 5 * k
        pos_class[base:base + 4] = 0
        rule[base:base + 4] = 4
        pos_class[base + 4] = 1
        rule[base + 4] = 1
    pos_class[0] = 2
    class_off = np.array([0, 1, 2, 3], dtype=np.int32)
    class_ranges = np.array([coord_lo, coord_lo + n_coord, delim_id, delim_id + 1, 0, vocab], dtype=np.int32)
    return dict(block_len=L, pos_class=pos_class, rule=rule, class_off=class_off, class_ranges=class_ranges,
                pad_id=-1, start_id=start_id)


def layout_fixed_width(vocab: int, n_waypoints: int = 20, n_axes: int = 3, digit_lo: int = 1000,
                       plus_id: int = 1010, minus_id: int = 1011, sep_id: int = 1012, start_id: int = 1013,
                       pad_id: int | None = None) -> dict:
    """Fixed-width numeral block: start token, then per waypoint and axis [sign d d d d d] and one
    separator per waypoint (19 slots per waypoint for three axes).  Classes: 0 = sign {+,-},
    1 = digit {0..9, pad}, 2 = separator, 3 = full vocabulary.  The pad (mask) id defaults to V-1."""
    pad = vocab - 1 if pad_id is None else pad_id
    per_wp = n_axes * 6 + 1
    L = 1 + per_wp * n_waypoints
    pos_class = np.full(L, 3, dtype=np.int16)
    rule = np.zeros(L, dtype=np.int8)
    for w in range(n_waypoints):
        base = 1 + per_wp * w
        for a in range(n_axes):
            f = base + 6 * a
            pos_class[f] = 0
            rule[f] = 1
            pos_class[f + 1:f + 6] = 1
            rule[f + 1:f + 5] = 2
            rule[f + 5] = 3
        pos_class[base + per_wp - 1] = 2
        rule[base + per_wp - 1] = 1
    assert sorted([plus_id, minus_id]) == [plus_id, plus_id + 1]
    class_off = np.array([0, 1, 3, 4, 5], dtype=np.int32)
    digit_ranges = [digit_lo, digit_lo + 10, pad, pad + 1] if pad > digit_lo + 10 else None
    assert digit_ranges is not None, "pad id must lie above the digit ids"
    class_ranges = np.array([plus_id, plus_id + 2, *digit_ranges, sep_id, sep_id + 1, 0, vocab], dtype=np.int32)
    return dict(block_len=L, pos_class=pos_class, rule=rule, class_off=class_off, class_ranges=class_ranges,
                pad_id=pad, start_id=start_id)


def make_target_rows(draft: np.ndarray, vocab: int, p: float, seed: int) -> tuple:
    """Target rows t_1..t_L for text-mode verification.  For request b the agreement length
    g ~ Geometric(p) on {0, 1, ...} (P(g = k) = (1-p)^k p); t_i = d_i for i <= min(g, L-1); at
    i = g+1 <= L-1 the target differs from the draft; every other entry is uniform.
    draft: [B, L-1] int32.  Returns (target [B, L] int32, g [B])."""
    B, Lm1 = draft.shape
    L = Lm1 + 1
    rng = np.random.default_rng(seed)
    g = rng.geometric(p, size=B) - 1            # numpy's geometric counts trials, starting at 1
    target = rng.integers(0, vocab, size=(B, L), dtype=np.int64)
    r = rng.integers(0, vocab - 1, size=B)
    for b in range(B):
        n = min(int(g[b]), Lm1)
        target[b, :n] = draft[b, :n]
        if n < Lm1:
            target[b, n] = (int(draft[b, n]) + 1 + int(r[b])) % vocab
    return target.astype(np.int32), g


@dataclasses.dataclass
class Workload:
    name: str
    shape: ModelShape
    batch: int
    block_len: int
    ctx_len: np.ndarray          # [B] int32
    row_off: np.ndarray          # [B+1] int32
    t_cap: int
    anchor: np.ndarray           # [B] int32
    mask_id: int
    layout: dict | None
    geo_p: float | None
    seed: int


def make_workload(name: str, batch: int | None = None, t_ctx=None, block_len: int | None = None,
                  seed: int | None = None) -> Workload:
    """Sizes, context lengths, anchors and layout of one of CONFIGS (overrides allowed)."""
    c = dict(CONFIGS[name])
    if batch is not None:
        c["batch"] = batch
    if t_ctx is not None:
        c["t_ctx"] = t_ctx
    if seed is not None:
        c["seed"] = seed
    s = c["shape"]
    rng = np.random.default_rng(c["seed"] + 7)
    B = c["batch"]
    if isinstance(c["t_ctx"], tuple):
        ctx_len = rng.integers(c["t_ctx"][0], c["t_ctx"][1] + 1, size=B).astype(np.int32)
    else:
        ctx_len = np.full(B, int(c["t_ctx"]), dtype=np.int32)
    layout = None
    L = c["block_len"]
    if c["layout"] == "special":
        layout = layout_special_tokens(s.vocab)
    elif c["layout"] == "fixed_width":
        layout = layout_fixed_width(s.vocab)
    if layout is not None:
        L = layout["block_len"]
    if block_len is not None:
        if layout is not None:
            raise ValueError("block length is fixed by the layout")
        L = block_len
    if layout is not None:
        anchor = np.full(B, layout["start_id"], dtype=np.int32)
    else:
        anchor = rng.integers(0, s.vocab - 1, size=B).astype(np.int32)
    row_off = np.zeros(B + 1, dtype=np.int32)
    row_off[1:] = np.cumsum(ctx_len)
    return Workload(name=name, shape=s, batch=B, block_len=L, ctx_len=ctx_len, row_off=row_off,
                    t_cap=int(ctx_len.max()), anchor=anchor, mask_id=s.vocab - 1, layout=layout,
                    geo_p=c["geo_p"], seed=c["seed"])
