"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the same seeded inputs.

Sizes: the tiny drafter end to end (the oracle finishes in seconds) with ragged batches, appends, and the
degenerate cases; the 4B-shape drafter at the full text size (context 2048, block 16) and at the full primitive
sizes, checked per request (requests are independent) and, for the context preparation, on sampled rows.
"""
import numpy as np
import pytest
import torch

import synth
from _util import (assert_logits, assert_margin, assert_rows_close, assert_tokens, assert_tokens_chain, bits_of,
                   dev_i32, f64)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_diffusion_speculative_non_gb300 as p
    p.lib()
    return p


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def _prepare_both(pkg, orc, shape, w, row_off, t_cap, max_block_len, batch, feats_seed, pos_start=None):
    feats = synth.make_features(shape, int(row_off[-1]), feats_seed)
    dr = pkg.Drafter(shape, w, batch, max_block_len, t_cap, device=DEV)
    dr.prepare_context(batch, row_off, feats, pos_start=pos_start)
    om = orc.Model(shape, w)
    kv = orc.prepare_context(om, row_off, feats, t_cap, batch=batch, pos_start=pos_start)
    return dr, om, kv, feats


def _compare_store(dr, kv_ref, ctx_len, batch):
    got = bits_of(dr.kv_view(batch))
    n = 0
    for b in range(batch):
        T = int(ctx_len[b])
        if T == 0:
            continue
        g = got[:, b, :, :, :T].reshape(-1, got.shape[-1])
        r = kv_ref[:, b, :, :, :T].reshape(-1, got.shape[-1])
        assert_rows_close(g, r, f"KV store request {b}")
        n += 1
    return n


def _stagewise(dr, kv_ref, ctx_len, batch):
    """Reading R21: the store the GPU prepared is checked against the oracle's preparation, and the block pass is
    then compared with the oracle run on the GPU's store (each call given the same inputs)."""
    _compare_store(dr, kv_ref, ctx_len, batch)
    return bits_of(dr.kv_view(batch))


def _draft_and_compare(pkg, orc, dr, om, kv_ref, t_cap, ctx_len, anchor, mask_id, L, batch, layout=None,
                       requests=None):
    """GPU draft + argmax over the whole batch; oracle on `requests` (default all); returns gpu tokens.  kv_ref is
    the oracle's store [layer][b][...] or a function b -> that request's store [layer][1][...]."""
    s = dr.shape
    lh = torch.empty(s.n_layers, batch * L, s.d_model, dtype=torch.bfloat16, device=DEV)
    hid = dr.draft_block(batch, L, dev_i32(ctx_len), dev_i32(anchor), mask_id, layer_hidden=lh)
    lay_d = None
    if layout is not None:
        lay_d, _ = pkg.Drafter.layout(layout, batch, L, DEV)
    logits = torch.full((batch * (L - 1), s.vocab), float("nan"), dtype=torch.float32, device=DEV)
    toks = dr.constrain_argmax(batch, L, hid, layout=lay_d, logits_out=logits)
    torch.cuda.synchronize()
    assert pkg.fpd_device_status() == 0
    g_tok = toks.cpu().numpy()
    reqs = range(batch) if requests is None else requests
    for b in reqs:
        sl = slice(b * L, (b + 1) * L)
        g_hid_b, g_lh_b = bits_of(hid[sl]), bits_of(lh[:, sl])   # only the checked requests leave the GPU
        kv_b = kv_ref(b) if callable(kv_ref) else (kv_ref[:, b:b + 1] if kv_ref.shape[1] > 1 else kv_ref)
        o_hid, o_lh = orc.draft_block(om, kv_b, t_cap, ctx_len[b:b + 1], anchor[b:b + 1], mask_id, L,
                                      want_layers=True)
        for l in range(s.n_layers):
            assert_rows_close(g_lh_b[l], o_lh[l], f"request {b} layer {l} hidden")
        assert_rows_close(g_hid_b, o_hid, f"request {b} hidden")
        lay_b = None
        if layout is not None:
            lay_b = dict(layout)
            pc = np.asarray(layout["pos_class"])
            lay_b["pos_class"] = pc if pc.ndim == 1 else pc[b]
        o_tok, o_margin, o_log = orc.constrain_argmax(om, o_hid, 1, L, layout=lay_b, want_logits=True)
        g_log_b = logits[b * (L - 1):(b + 1) * (L - 1)].cpu().numpy()
        assert_logits(g_log_b, o_log, f"request {b} logits")
        assert_tokens_chain(g_tok[b], o_tok[0], o_margin, g_log_b, o_log, f"request {b} tokens")
        # the LM head + argmax stage alone, given the oracle's hidden states: the strict id rule
        hid_o = torch.from_numpy(o_hid.view(np.int16)).to(DEV).view(torch.bfloat16)
        lay_1 = None
        if layout is not None:
            lay_1, _ = pkg.Drafter.layout(lay_b, 1, L, DEV)
        lg1 = torch.full((L - 1, s.vocab), float("nan"), dtype=torch.float32, device=DEV)
        mg1 = torch.full((L - 1,), float("nan"), dtype=torch.float32, device=DEV)
        t1 = dr.constrain_argmax(1, L, hid_o, layout=lay_1, logits_out=lg1, margin_out=mg1)
        torch.cuda.synchronize()
        assert_logits(lg1.cpu().numpy(), o_log, f"request {b} logits from oracle hidden")
        assert_tokens(t1.cpu().numpy()[0], o_tok[0], o_margin, f"request {b} tokens from oracle hidden")
        assert_margin(mg1.cpu().numpy(), lg1.cpu().numpy(), o_margin, o_log, f"request {b} margin")
    return g_tok, hid


# ---- tiny drafter, end to end --------------------------------------------------------------------------------------

def test_tiny_text_end_to_end(pkg, orc):
    wl = synth.make_workload("tiny_text_b1")
    s = wl.shape
    w = synth.make_weights(s, wl.seed)
    dr, om, kv, _ = _prepare_both(pkg, orc, s, w, wl.row_off, wl.t_cap, wl.block_len, wl.batch, wl.seed + 1)
    assert _compare_store(dr, kv, wl.ctx_len, wl.batch) == 1
    kv_g = _stagewise(dr, kv, wl.ctx_len, wl.batch)
    toks, _ = _draft_and_compare(pkg, orc, dr, om, kv_g, wl.t_cap, wl.ctx_len, wl.anchor, wl.mask_id, wl.block_len,
                                 wl.batch)
    # verify against geometric target rows built from the GPU ids; bit-exact given the ids
    target, g = synth.make_target_rows(toks, s.vocab, wl.geo_p, wl.seed + 2)
    acc, com, val = dr.verify_text(wl.batch, wl.block_len, dev_i32(toks), dev_i32(target))
    oacc, ocom, oval = orc.verify(0, toks, target)
    np.testing.assert_array_equal(acc.cpu().numpy(), oacc)
    np.testing.assert_array_equal(com.cpu().numpy(), ocom)
    np.testing.assert_array_equal(val.cpu().numpy(), oval)
    np.testing.assert_array_equal(oacc, 1 + np.minimum(g, wl.block_len - 1))
    dr.close()


def test_tiny_ragged_batch_with_append(pkg, orc):
    """Ragged contexts (one of length 1, one empty), written in two appends, blocks of 5."""
    s = synth.TINY
    w = synth.make_weights(s, 1234)
    lens1 = np.array([1, 0, 37, 64], np.int32)
    lens2 = np.array([0, 3, 33, 1], np.int32)
    ctx_len = lens1 + lens2
    t_cap = int(ctx_len.max())
    B, L = 4, 5
    off1 = np.concatenate([[0], np.cumsum(lens1)]).astype(np.int32)
    off2 = np.concatenate([[0], np.cumsum(lens2)]).astype(np.int32)
    dr, om, kv, _ = _prepare_both(pkg, orc, s, w, off1, t_cap, L, B, 77)
    f2 = synth.make_features(s, int(off2[-1]), 78)
    dr.prepare_context(B, off2, f2, pos_start=lens1)
    kv = orc.prepare_context(om, off2, f2, t_cap, batch=B, pos_start=lens1, kv_store=kv)
    _compare_store(dr, kv, ctx_len, B)
    anchor = np.array([5, 6, 7, 4000], np.int32)
    kv_g = _stagewise(dr, kv, ctx_len, B)
    _draft_and_compare(pkg, orc, dr, om, kv_g, t_cap, ctx_len, anchor, s.vocab - 1, L, B)
    dr.close()


def test_tiny_few_token_batch_ragged(pkg, orc):
    """Three requests of 5 positions (15 block positions in all: the few-token path), ragged contexts."""
    s = synth.TINY
    w = synth.make_weights(s, 4242)
    ctx_len = np.array([40, 0, 97], np.int32)
    off = np.concatenate([[0], np.cumsum(ctx_len)]).astype(np.int32)
    B, L = 3, 5
    dr, om, kv, _ = _prepare_both(pkg, orc, s, w, off, int(ctx_len.max()), L, B, 4243)
    kv_g = _stagewise(dr, kv, ctx_len, B)
    _draft_and_compare(pkg, orc, dr, om, kv_g, int(ctx_len.max()), ctx_len, np.array([3, 4000, 77], np.int32),
                       s.vocab - 1, L, B)
    dr.close()


def test_tiny_medium_batch_weight_tiles(pkg, orc):
    """Eight requests of 20 positions (160 block rows: below the token-tile threshold, the weight-tile GEMMs with K
    split over the SMs and the row kernels' reductions), ragged contexts including an empty one."""
    s = synth.TINY
    w = synth.make_weights(s, 4343)
    ctx_len = np.array([40, 0, 97, 1, 128, 64, 5, 77], np.int32)
    off = np.concatenate([[0], np.cumsum(ctx_len)]).astype(np.int32)
    B, L = 8, 20
    dr, om, kv, _ = _prepare_both(pkg, orc, s, w, off, int(ctx_len.max()), L, B, 4344)
    kv_g = _stagewise(dr, kv, ctx_len, B)
    _draft_and_compare(pkg, orc, dr, om, kv_g, int(ctx_len.max()), ctx_len, (np.arange(B, dtype=np.int32) * 411 + 3) % s.vocab,
                       s.vocab - 1, L, B)
    dr.close()


@pytest.mark.parametrize("L,ctx", [(2, 0), (2, 1), (16, 0), (33, 96)])
def test_tiny_degenerate_blocks(pkg, orc, L, ctx):
    """Shortest block (one proposal), no context at all, and a context filling the store."""
    s = synth.TINY
    w = synth.make_weights(s, 99)
    t_cap = max(ctx, 1)
    off = np.array([0, ctx], np.int32)
    dr, om, kv, _ = _prepare_both(pkg, orc, s, w, off, t_cap, L, 1, 98)
    kv_g = _stagewise(dr, kv, np.array([ctx], np.int32), 1)
    _draft_and_compare(pkg, orc, dr, om, kv_g, t_cap, np.array([ctx], np.int32), np.array([17], np.int32),
                       s.vocab - 1, L, 1)
    dr.close()


def test_tiny_special_token_primitive(pkg, orc):
    """Block of a 64-waypoint primitive with dedicated coordinate tokens (L = 385) on the tiny drafter:
    1001-id coordinate slice + singleton delimiter; every block is schema-valid."""
    s = synth.TINY
    w = synth.make_weights(s, 555)
    lay = synth.layout_special_tokens(s.vocab, 64, coord_lo=2000, n_coord=1001, delim_id=3100, start_id=3101)
    L = lay["block_len"]
    T = 200
    dr, om, kv, _ = _prepare_both(pkg, orc, s, w, np.array([0, T], np.int32), T, L, 1, 556)
    kv_g = _stagewise(dr, kv, np.array([T], np.int32), 1)
    toks, _ = _draft_and_compare(pkg, orc, dr, om, kv_g, T, np.array([T], np.int32), np.array([3101], np.int32),
                                 s.vocab - 1, L, 1, layout=lay)
    lay_d, rule_d = pkg.Drafter.layout(lay, 1, L, DEV)
    acc, com, val = dr.verify_schema(1, L, dev_i32(toks), lay_d, rule_d, -1)
    assert int(acc.item()) == L - 1 and int(val.item()) == 1
    dr.close()


def test_tiny_fixed_width_primitive_batch(pkg, orc):
    """Fixed-width numerals (sign + 5 digit slots, pad = mask id), L = 381, ragged batch of 4."""
    s = synth.TINY
    w = synth.make_weights(s, 777)
    lay = synth.layout_fixed_width(s.vocab)
    L = lay["block_len"]
    ctx_len = np.array([50, 120, 77, 1], np.int32)
    off = np.concatenate([[0], np.cumsum(ctx_len)]).astype(np.int32)
    B = 4
    dr, om, kv, _ = _prepare_both(pkg, orc, s, w, off, int(ctx_len.max()), L, B, 778)
    anchor = np.full(B, lay["start_id"], np.int32)
    kv_g = _stagewise(dr, kv, ctx_len, B)
    toks, _ = _draft_and_compare(pkg, orc, dr, om, kv_g, int(ctx_len.max()), ctx_len, anchor, s.vocab - 1, L, B,
                                 layout=lay)
    lay_d, rule_d = pkg.Drafter.layout(lay, B, L, DEV)
    acc, com, val = dr.verify_schema(B, L, dev_i32(toks), lay_d, rule_d, lay["pad_id"])
    oacc, ocom, oval = orc.verify(1, toks, layout=lay, rule=lay["rule"], pad_id=lay["pad_id"])
    np.testing.assert_array_equal(acc.cpu().numpy(), oacc)
    np.testing.assert_array_equal(com.cpu().numpy(), ocom)
    np.testing.assert_array_equal(val.cpu().numpy(), oval)
    dr.close()


def test_repeat_runs_bit_identical(pkg, orc):
    """Fixed split/merge orders and order-independent argmax: two runs agree bit for bit."""
    wl = synth.make_workload("tiny_text_b1")
    s = wl.shape
    w = synth.make_weights(s, 4321)
    feats = synth.make_features(s, int(wl.row_off[-1]), 4322)
    dr = pkg.Drafter(s, w, 1, wl.block_len, wl.t_cap, device=DEV)
    dr.prepare_context(1, wl.row_off, feats)
    outs = []
    for _ in range(2):
        hid = dr.draft_block(1, wl.block_len, dev_i32(wl.ctx_len), dev_i32(wl.anchor), wl.mask_id)
        toks = dr.constrain_argmax(1, wl.block_len, hid)
        outs.append((bits_of(hid), toks.cpu().numpy(), bits_of(dr.kv_view(1))))
    for a, b in zip(outs[0], outs[1]):
        np.testing.assert_array_equal(a, b)
    dr.close()


def test_bad_anchor_reported_by_device_check(pkg):
    s = synth.TINY
    w = synth.make_weights(s, 1)
    dr = pkg.Drafter(s, w, 1, 4, 8, device=DEV)
    dr.draft_block(1, 4, dev_i32([0]), dev_i32([s.vocab + 5]), s.vocab - 1)
    torch.cuda.synchronize()
    assert pkg.fpd_device_status() == 1          # kCheckBadToken, no fault
    assert pkg.fpd_device_status() == 0          # cleared by the read
    dr.close()


# ---- verify kernel: exhaustive cases -------------------------------------------------------------------------------

def test_verify_text_exhaustive_binary(pkg, orc):
    import itertools
    for L in (2, 5, 8, 33, 40):
        if L <= 8:
            drafts = np.array(list(itertools.product([0, 1], repeat=L - 1)), np.int32)
            targets = np.array(list(itertools.product([0, 1], repeat=L)), np.int32)
            D = np.repeat(drafts, len(targets), axis=0)
            T = np.tile(targets, (len(drafts), 1))
        else:
            rng = np.random.default_rng(L)
            D = rng.integers(0, 2, (5000, L - 1)).astype(np.int32)
            T = D.copy()
            T = np.concatenate([T, rng.integers(0, 2, (5000, 1))], axis=1).astype(np.int32)
            cut = rng.integers(0, L, 5000)
            for i, c in enumerate(cut):
                if c < L - 1:
                    T[i, c] = 1 - T[i, c]
        B = len(D)
        acc = torch.empty(B, dtype=torch.int32, device=DEV)
        com = torch.empty(B, L, dtype=torch.int32, device=DEV)
        val = torch.empty(B, dtype=torch.int32, device=DEV)
        pkg.fpd_verify(0, B, L, dev_i32(D), dev_i32(T), None, None, -1, acc, com, val)
        oacc, ocom, oval = orc.verify(0, D, T)
        np.testing.assert_array_equal(acc.cpu().numpy(), oacc)
        np.testing.assert_array_equal(com.cpu().numpy(), ocom)
        np.testing.assert_array_equal(val.cpu().numpy(), oval)


def test_verify_schema_exhaustive_field(pkg, orc):
    import itertools
    lay = dict(class_off=np.array([0, 1, 3], np.int32), class_ranges=np.array([10, 12, 0, 10, 12, 13], np.int32),
               pos_class=np.array([0, 0, 1, 1, 1, 1, 1], np.int16))
    rule = np.array([0, 1, 2, 2, 2, 2, 3], np.int8)
    syms = list(range(10)) + [12]
    fields = np.array([(sg,) + dd for sg in (10, 11, 3) for dd in itertools.product(syms, repeat=5)], np.int32)
    B, L = len(fields), 7
    lay_d, rule_d = pkg.Drafter.layout(dict(lay, rule=rule), B, L, DEV)
    acc = torch.empty(B, dtype=torch.int32, device=DEV)
    com = torch.empty(B, L, dtype=torch.int32, device=DEV)
    val = torch.empty(B, dtype=torch.int32, device=DEV)
    pkg.fpd_verify(1, B, L, dev_i32(fields), None, lay_d, rule_d, 12, acc, com, val)
    oacc, ocom, oval = orc.verify(1, fields, layout=lay, rule=rule, pad_id=12)
    np.testing.assert_array_equal(acc.cpu().numpy(), oacc)
    np.testing.assert_array_equal(com.cpu().numpy(), ocom)
    np.testing.assert_array_equal(val.cpu().numpy(), oval)


# ---- 4B-shape drafter at full sizes ------------------------------------------------------------------------------

def test_full_text_block(pkg, orc, full_weights):
    """Text mode at the 4B shape: context 2048 (random context K/V), block 16, unconstrained vocabulary."""
    wl = synth.make_workload("text_4b_b1")
    s = wl.shape
    kv = synth.make_kv_store(s, 1, wl.t_cap, 2001)
    dr = pkg.Drafter(s, full_weights, 1, wl.block_len, wl.t_cap, device=DEV)
    dr.kv_view(1).copy_(torch.from_numpy(kv.view(np.int16)).view(torch.bfloat16))
    om = orc.Model(s, full_weights)
    toks, _ = _draft_and_compare(pkg, orc, dr, om, kv, wl.t_cap, wl.ctx_len, wl.anchor, wl.mask_id, wl.block_len, 1)
    target, g = synth.make_target_rows(toks, s.vocab, wl.geo_p, 2002)
    acc, com, val = dr.verify_text(1, wl.block_len, dev_i32(toks), dev_i32(target))
    assert int(acc.item()) == 1 + min(int(g[0]), wl.block_len - 1)
    dr.close()


def test_full_prepare_context_sampled_rows(pkg, orc, full_weights):
    """Context fusion + per-layer K/V at the 4B shape, 2048 rows on the GPU; the oracle recomputes a head, a
    middle and a tail slice of rows at their own positions (rows are independent)."""
    s = synth.FULL
    T = 2048
    feats = synth.make_features(s, T, 2003)
    dr = pkg.Drafter(s, full_weights, 1, 16, T, device=DEV)
    dr.prepare_context(1, np.array([0, T], np.int32), feats)
    got = bits_of(dr.kv_view(1))
    om = orc.Model(s, full_weights)
    for lo, hi in ((0, 3), (1000, 1002), (T - 3, T)):
        ref = orc.prepare_context(om, np.array([0, hi - lo], np.int32), [f[lo:hi] for f in feats], T,
                                  pos_start=np.array([lo], np.int32))
        g = got[:, 0, :, :, lo:hi].reshape(-1, s.head_dim)
        r = ref[:, 0, :, :, lo:hi].reshape(-1, s.head_dim)
        assert_rows_close(g, r, f"context rows {lo}..{hi}")
    dr.close()


def test_full_special_token_primitive(pkg, orc, full_weights):
    """Primitive with dedicated coordinate tokens at full size: context 4096, L = 385, one request."""
    wl = synth.make_workload("primitive_special_b1")
    s = wl.shape
    kv = synth.make_kv_store(s, 1, wl.t_cap, 3001)
    dr = pkg.Drafter(s, full_weights, 1, wl.block_len, wl.t_cap, device=DEV)
    dr.kv_view(1).copy_(torch.from_numpy(kv.view(np.int16)).view(torch.bfloat16))
    om = orc.Model(s, full_weights)
    toks, _ = _draft_and_compare(pkg, orc, dr, om, kv, wl.t_cap, wl.ctx_len, wl.anchor, wl.mask_id, wl.block_len, 1,
                                 layout=wl.layout)
    lay_d, rule_d = pkg.Drafter.layout(wl.layout, 1, wl.block_len, DEV)
    acc, com, val = dr.verify_schema(1, wl.block_len, dev_i32(toks), lay_d, rule_d, -1)
    assert int(val.item()) == 1 and int(acc.item()) == wl.block_len - 1
    dr.close()


def test_full_fixed_width_batch_sampled_requests(pkg, orc, full_weights):
    """Fixed-width numerals at full size: 32 requests, ragged contexts U[512, 2048], L = 381; the oracle checks
    the first and last request."""
    wl = synth.make_workload("primitive_fixedwidth_b32")
    s = wl.shape
    kv = synth.make_kv_store(s, wl.batch, wl.t_cap, 4001)
    dr = pkg.Drafter(s, full_weights, wl.batch, wl.block_len, wl.t_cap, device=DEV)
    dr.kv_view(wl.batch).copy_(torch.from_numpy(kv.view(np.int16)).view(torch.bfloat16))
    om = orc.Model(s, full_weights)
    toks, _ = _draft_and_compare(pkg, orc, dr, om, kv, wl.t_cap, wl.ctx_len, wl.anchor, wl.mask_id, wl.block_len,
                                 wl.batch, layout=wl.layout, requests=[0, wl.batch - 1])
    lay = wl.layout
    lay_d, rule_d = pkg.Drafter.layout(lay, wl.batch, wl.block_len, DEV)
    acc, com, val = dr.verify_schema(wl.batch, wl.block_len, dev_i32(toks), lay_d, rule_d, lay["pad_id"])
    oacc, ocom, oval = orc.verify(1, toks, layout=lay, rule=lay["rule"], pad_id=lay["pad_id"])
    np.testing.assert_array_equal(acc.cpu().numpy(), oacc)
    np.testing.assert_array_equal(com.cpu().numpy(), ocom)
    dr.close()


# ---- 4B shape: the context preparation chained into the block pass ----------------------------------------------

def test_full_prepare_then_draft_ragged_append(pkg, orc, full_weights):
    """Context preparation chained into the block pass at the 4B shape: four requests with ragged contexts (one
    empty before its append, one receiving nothing in the second), written in two appends, then one 16-position
    text block per request (64 block rows: the weight-tile path).  Each stage is checked against the oracle given
    the same input: the store against the oracle's preparation from the same features, the block pass (every
    request) against the oracle run on the GPU's store, then the greedy verification."""
    s = synth.FULL
    lens1 = np.array([200, 0, 500, 13], np.int32)
    lens2 = np.array([56, 40, 0, 3], np.int32)
    ctx_len = lens1 + lens2
    t_cap = int(ctx_len.max())
    B, L = 4, 16
    off1 = np.concatenate([[0], np.cumsum(lens1)]).astype(np.int32)
    off2 = np.concatenate([[0], np.cumsum(lens2)]).astype(np.int32)
    dr, om, kv, _ = _prepare_both(pkg, orc, s, full_weights, off1, t_cap, L, B, 3101)
    f2 = synth.make_features(s, int(off2[-1]), 3102)
    dr.prepare_context(B, off2, f2, pos_start=lens1)
    kv = orc.prepare_context(om, off2, f2, t_cap, batch=B, pos_start=lens1, kv_store=kv)
    assert _compare_store(dr, kv, ctx_len, B) == 4
    anchor = np.array([11, 150000, 77777, 151934], np.int32)
    # stage by stage (reading R21): the block pass against the oracle run on the store the GPU prepared
    toks, _ = _draft_and_compare(pkg, orc, dr, om, bits_of(dr.kv_view(B)), t_cap, ctx_len, anchor, s.vocab - 1, L, B)
    target, g = synth.make_target_rows(toks, s.vocab, 0.25, 3103)
    acc, com, val = dr.verify_text(B, L, dev_i32(toks), dev_i32(target))
    oacc, ocom, oval = orc.verify(0, toks, target)
    np.testing.assert_array_equal(acc.cpu().numpy(), oacc)
    np.testing.assert_array_equal(com.cpu().numpy(), ocom)
    np.testing.assert_array_equal(oacc, 1 + np.minimum(g, L - 1))
    dr.close()


def test_full_prepare_then_draft_few_token(pkg, orc, full_weights):
    """The batch-1 text workload with a prepared context instead of a random store: 2048 rows written in two
    appends (1500 + 548), then one 16-position block on the few-token path (stream GEMMs, cluster attention)."""
    s = synth.FULL
    lens1, lens2 = np.array([1500], np.int32), np.array([548], np.int32)
    T = 2048
    dr, om, kv, _ = _prepare_both(pkg, orc, s, full_weights, np.array([0, 1500], np.int32), T, 16, 1, 3201)
    f2 = synth.make_features(s, 548, 3202)
    dr.prepare_context(1, np.array([0, 548], np.int32), f2, pos_start=lens1)
    kv = orc.prepare_context(om, np.array([0, 548], np.int32), f2, T, batch=1, pos_start=lens1, kv_store=kv)
    ctx_len = lens1 + lens2
    assert _compare_store(dr, kv, ctx_len, 1) == 1
    _draft_and_compare(pkg, orc, dr, om, bits_of(dr.kv_view(1)), T, ctx_len, np.array([4242], np.int32),
                       s.vocab - 1, 16, 1)
    dr.close()


# ---- 4B shape: corner points of the throughput sweep --------------------------------------------------------------

@pytest.mark.parametrize("B,T,L", [(1, 512, 16), (64, 16384, 16), (64, 16384, 385), (16, 512, 16)])
def test_sweep_corner(pkg, orc, full_weights, B, T, L):
    """Corners of the sweep (batch {1, 64} x context {512, 16384} x block {16 text, 385 special-token}) at full
    size, and B 16 x L 16 (256 block rows: the token-tile GEMMs split K three ways, reduced by the last CTA).  Requests 0 and B - 1 take their context K/V from the seeded host generator and are checked end to end
    by the oracle (requests are independent); the others are drawn on the device and only run."""
    base = "text_4b_b1" if L == 16 else "primitive_special_b1"
    wl = synth.make_workload(base, batch=B, t_ctx=T, seed=5100 + B + L)
    s = wl.shape
    dr = pkg.Drafter(s, full_weights, B, wl.block_len, T, device=DEV)
    kv_dev = dr.kv_view(B)
    gen = torch.Generator(device=DEV).manual_seed(5200 + B + L)
    for layer in range(s.n_layers):
        kv_dev[layer].normal_(generator=gen)
    host = {}
    for b in sorted({0, B - 1}):
        kvb = synth.make_kv_store(s, 1, T, 5300 + b)
        kv_dev[:, b:b + 1].copy_(torch.from_numpy(kvb.view(np.int16)).view(torch.bfloat16))
        host[b] = kvb
    om = orc.Model(s, full_weights)
    toks, _ = _draft_and_compare(pkg, orc, dr, om, lambda b: host[b], T, wl.ctx_len, wl.anchor, wl.mask_id,
                                 wl.block_len, B, layout=wl.layout, requests=sorted(host))
    if wl.layout is None:
        target, _ = synth.make_target_rows(toks, s.vocab, 0.25, 5400)
        acc, com, val = dr.verify_text(B, wl.block_len, dev_i32(toks), dev_i32(target))
        oacc, ocom, oval = orc.verify(0, toks, target)
    else:
        lay = wl.layout
        lay_d, rule_d = pkg.Drafter.layout(lay, B, wl.block_len, DEV)
        acc, com, val = dr.verify_schema(B, wl.block_len, dev_i32(toks), lay_d, rule_d, lay["pad_id"])
        oacc, ocom, oval = orc.verify(1, toks, layout=lay, rule=lay["rule"], pad_id=lay["pad_id"])
    np.testing.assert_array_equal(acc.cpu().numpy(), oacc)
    np.testing.assert_array_equal(com.cpu().numpy(), ocom)
    np.testing.assert_array_equal(val.cpu().numpy(), oval)
    dr.close()
