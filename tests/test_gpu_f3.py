"""GPU: f3 — off-screen coordinates in pairs inside the constrained argmax, and prefix acceptance up to the first
uncertain coordinate, against the oracle (VFlash paper (zh) §2.5; readings R23, R24)."""
import numpy as np
import pytest
import torch

import synth
from _util import assert_logits, assert_tokens, bits_of, dev_i32
from test_f3_rules import pair_case

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_diffusion_speculative_non_gb300 as p
    p.lib()
    return p


def _lm_stage(pkg, orc, s, w, lay, hid, B):
    """GPU constrained argmax with the pair rule on given hidden rows against the oracle's (strict stage rule)."""
    L = lay["block_len"]
    dr = pkg.Drafter(s, w, B, L, 16, device=DEV)
    lay_d, _ = pkg.Drafter.layout(lay, B, L, DEV)
    h = torch.from_numpy(hid.view(np.int16)).to(DEV).view(torch.bfloat16)
    lg = torch.full((B * (L - 1), s.vocab), float("nan"), dtype=torch.float32, device=DEV)
    mg = torch.empty(B * (L - 1), dtype=torch.float32, device=DEV)
    tok = dr.constrain_argmax(B, L, h, layout=lay_d, logits_out=lg, margin_out=mg)
    torch.cuda.synchronize()
    assert pkg.fpd_device_status() == 0
    om = orc.Model(s, w)
    otok, omargin, olog = orc.constrain_argmax(om, hid, B, L, layout=lay, want_logits=True)
    assert_logits(lg.cpu().numpy(), olog, "logits")
    gt = tok.cpu().numpy()
    flips = assert_tokens(gt, otok, omargin, "tokens")
    off = lay["off_id"]
    n_off = 0
    for b in range(B):
        for p, q in lay["pairs"]:
            assert (gt[b, p - 1] == off) == (gt[b, q - 1] == off), (b, p, q)
            n_off += int(gt[b, p - 1] == off)
    dr.close()
    return n_off, flips


def test_pair_rule_tiny(pkg, oracle_lib):
    s = synth.TINY
    w, lay, hid = pair_case(s, 901)
    n_off, flips = _lm_stage(pkg, oracle_lib, s, w, lay, hid, 4)
    print(f"pairs off screen: {n_off}, ids differing at exempt margins: {flips}")
    assert 0 < n_off < 4 * len(lay["pairs"])


def test_pair_rule_full_size(pkg, oracle_lib, full_weights):
    """The 4B shape's 151936-id LM head, the 64-waypoint special-token layout with off-screen pairs (off id
    151102, its LM-head row scaled by four), random final hidden rows of two requests."""
    s = synth.FULL
    w = dict(full_weights)
    w["lm_head"] = full_weights["lm_head"].copy()
    off = 151102
    w["lm_head"][off] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(w["lm_head"][off]) * 4.0)
    lay = synth.layout_special_tokens(s.vocab, off_id=off)
    B, L = 2, lay["block_len"]
    hid = synth.f32_to_bf16_bits(np.random.default_rng(7).normal(size=(B * L, s.d_model)).astype(np.float32))
    n_off, flips = _lm_stage(pkg, oracle_lib, s, w, lay, hid, B)
    print(f"pairs off screen: {n_off} of {B * 64}, ids differing at exempt margins: {flips}")
    assert 0 < n_off < B * 64


@pytest.mark.parametrize("tau", [0.0, 0.25, 1.0])
def test_prefix_verification_matches_oracle(pkg, oracle_lib, tau):
    rng = np.random.default_rng(int(tau * 100) + 5)
    lay = synth.layout_bbox(151936, n_boxes=16)
    L, B = lay["block_len"], 256
    draft = np.empty((B, L - 1), np.int32)
    for j in range(1, L):
        draft[:, j - 1] = 151100 if lay["pos_class"][j] == 1 else rng.integers(150000, 151001, size=B)
    bad = rng.random((B, L - 1)) < 0.01                      # a few illegal ids
    draft[bad] = rng.integers(0, 150000, size=int(bad.sum()))
    margin = rng.exponential(2.0, size=(B, L - 1)).astype(np.float32)
    margin[rng.random((B, L - 1)) < 0.002] = np.nan          # NaN margins count as uncertain
    lay_d, rule_d = pkg.Drafter.layout(lay, B, L, DEV)
    dr_margin = torch.from_numpy(margin).to(DEV)
    acc = torch.empty(B, dtype=torch.int32, device=DEV)       # verification needs no model
    com = torch.empty(B, L, dtype=torch.int32, device=DEV)
    val = torch.empty(B, dtype=torch.int32, device=DEV)
    pkg.fpd_verify_prefix(B, L, dev_i32(draft), dr_margin, tau, lay_d, rule_d, -1, acc, com, val)
    torch.cuda.synchronize()
    oacc, ocom, oval = oracle_lib.verify(2, draft, layout=lay, rule=lay["rule"], pad_id=-1, margin=margin, tau=tau)
    np.testing.assert_array_equal(acc.cpu().numpy(), oacc)
    np.testing.assert_array_equal(com.cpu().numpy(), ocom)
    np.testing.assert_array_equal(val.cpu().numpy(), oval)
    assert len(set(oacc.tolist())) > 5
