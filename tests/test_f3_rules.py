"""f3 in the oracle: the cross-position rule (off-screen coordinates in pairs) and prefix acceptance up to the first
uncertain coordinate (VFlash paper (zh) §2.5; readings R23, R24).  CPU only.

The pair rule is pinned to a brute-force search over every joint assignment the rule allows; prefix acceptance to
blocks built with a known first failing position."""
import numpy as np

import synth

F32 = np.float32


def _brute_pair(lg_p, lg_q, legal_p, legal_q, off):
    """Best joint assignment over all (i, j) that are both on screen or both off_id, scored as the fp32 sum of the
    fp32 logits; on a tie the on-screen assignment wins, and among on-screen ones the lowest ids."""
    best, pick = None, None
    for i in legal_p:
        if i == off:
            continue
        for j in legal_q:
            if j == off:
                continue
            v = F32(F32(lg_p[i]) + F32(lg_q[j]))
            if best is None or v > best:
                best, pick = v, (i, j)
    v = F32(F32(lg_p[off]) + F32(lg_q[off]))
    if v > best:
        pick = (off, off)
    return pick, abs(float(v) - float(best))


def test_pair_rule_equals_brute_force(oracle_lib):
    rng = np.random.default_rng(31)
    V, P = 40, 7                       # 7 drafted positions, ids 0..39; off-screen id 39
    off = 39
    legal = [list(range(10, 20)) + [off], list(range(10, 20)) + [off], list(range(20, 25))]
    for trial in range(300):
        logits = np.full((P, V), np.nan)
        cls = [0, 1, 2, 0, 1, 2, 2]
        for r in range(P):
            ids = legal[cls[r]]
            logits[r, ids] = rng.normal(size=len(ids)) * (3.0 if trial % 3 == 0 else 1.0)
            if trial % 5 == 0:         # exact ties among on-screen ids
                logits[r, ids[1]] = logits[r, ids[0]]
        tokens = np.array([[int(np.nanargmax(logits[r].astype(np.float32))) for r in range(P)]], np.int32)
        margin = np.full(P, np.inf)
        pairs = np.array([[1, 2], [4, 5]], np.int16)          # block positions -> rows 0/1 and 3/4
        oracle_lib._pair_offscreen(tokens, margin, logits, P + 1, pairs, off)
        for p, q in pairs:
            (i, j), gap = _brute_pair(logits[p - 1], logits[q - 1], legal[cls[p - 1]], legal[cls[q - 1]], off)
            assert (tokens[0, p - 1], tokens[0, q - 1]) == (i, j), trial
            assert (tokens[0, p - 1] == off) == (tokens[0, q - 1] == off)
            assert margin[p - 1] <= gap + 1e-12 and margin[q - 1] <= gap + 1e-12
        assert tokens[0, 2] == int(np.nanargmax(logits[2].astype(np.float32)))   # unpaired rows untouched


def pair_case(s, seed, n_waypoints=12, B=4):
    """Weights whose off-screen LM-head row is four times the others' scale, and random final hidden rows (bf16),
    so that the pair decision goes both ways; the special-token layout in the tiny vocabulary."""
    w = synth.make_weights(s, seed)
    off = 3200
    w["lm_head"] = w["lm_head"].copy()
    w["lm_head"][off] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(w["lm_head"][off]) * 4.0)
    lay = synth.layout_special_tokens(s.vocab, n_waypoints=n_waypoints, coord_lo=3000, n_coord=101, delim_id=3150,
                                      start_id=3151, off_id=off)
    L = lay["block_len"]
    rng = np.random.default_rng(seed + 1)
    hid = synth.f32_to_bf16_bits(rng.normal(size=(B * L, s.d_model)).astype(np.float32))
    return w, lay, hid


def test_pair_rule_through_the_oracle_lm_head(oracle_lib):
    """The oracle's constrained argmax with the rule: every pair ends both on or both off screen, and every
    decision matches the brute force on the oracle's own logits."""
    s = synth.TINY
    w, lay, hid = pair_case(s, 901)
    off, L, B = lay["off_id"], lay["block_len"], 4
    m = oracle_lib.Model(s, w)
    tok, margin, logits = oracle_lib.constrain_argmax(m, hid, B, L, layout=lay, want_logits=True)
    ids = list(range(3000, 3101)) + [off]
    n_off = 0
    for b in range(B):
        for p, q in lay["pairs"]:
            rp, rq = b * (L - 1) + p - 1, b * (L - 1) + q - 1
            a, c = tok[b, p - 1], tok[b, q - 1]
            assert (a == off) == (c == off)
            (i, j), _ = _brute_pair(logits[rp], logits[rq], ids, ids, off)
            assert (a, c) == (i, j)
            n_off += int(a == off)
    assert 0 < n_off < B * len(lay["pairs"])     # both branches occur


def _bbox_rows(rng, n_boxes, B):
    lay = synth.layout_bbox(4096, n_boxes=n_boxes, coord_lo=3000, n_coord=101, delim_id=3150, start_id=3151)
    L = lay["block_len"]
    draft = np.empty((B, L - 1), np.int32)
    for b in range(B):
        for j in range(1, L):
            draft[b, j - 1] = 3150 if lay["pos_class"][j] == 1 else int(rng.integers(3000, 3101))
    return lay, draft


def test_prefix_acceptance_stops_at_the_first_uncertain_coordinate(oracle_lib):
    rng = np.random.default_rng(77)
    lay, draft = _bbox_rows(rng, 4, 64)
    L = lay["block_len"]
    tau = 0.5
    margin = rng.uniform(0.6, 3.0, size=(64, L - 1))
    want = np.full(64, L - 1)
    for b in range(64):                      # plant the first uncertain coordinate at a chosen position
        if b % 4 == 0:
            continue                         # none: the whole block is kept
        coords = [j for j in range(1, L) if lay["rule"][j] == 4]
        j = coords[int(rng.integers(0, len(coords)))]
        margin[b, j - 1] = rng.uniform(0.0, 0.49) if b % 4 != 3 else np.nan
        later = [k for k in coords if k > j]
        for k in later[:2]:
            margin[b, k - 1] = 0.1           # later uncertain coordinates do not matter
        want[b] = j - 1
    acc, com, val = oracle_lib.verify(2, draft, layout=lay, rule=lay["rule"], pad_id=-1, margin=margin, tau=tau)
    np.testing.assert_array_equal(acc, want)
    np.testing.assert_array_equal(val, (want == L - 1).astype(np.int32))
    for b in range(64):
        np.testing.assert_array_equal(com[b, :want[b]], draft[b, :want[b]])
        assert (com[b, want[b]:] == -1).all()


def test_prefix_acceptance_reduces_to_the_schema_rule(oracle_lib):
    """tau = 0 with finite non-negative margins: exactly the schema mode; a schema failure before the first
    uncertain coordinate decides."""
    rng = np.random.default_rng(78)
    lay, draft = _bbox_rows(rng, 4, 32)
    L = lay["block_len"]
    draft[::3, 6] = 17                     # an illegal id at block position 7 (a coordinate)
    margin = rng.uniform(0.0, 2.0, size=(32, L - 1))
    a2, c2, v2 = oracle_lib.verify(2, draft, layout=lay, rule=lay["rule"], pad_id=-1, margin=margin, tau=0.0)
    a1, c1, v1 = oracle_lib.verify(1, draft, layout=lay, rule=lay["rule"], pad_id=-1)
    np.testing.assert_array_equal(a2, a1)
    np.testing.assert_array_equal(c2, c1)
    np.testing.assert_array_equal(v2, v1)
    assert (a1[::3] == 6).all()
