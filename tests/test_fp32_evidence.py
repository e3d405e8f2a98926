"""Evidence for the end-to-end token rule: what a correct implementation that merely accumulates in fp32 does.

tests/fp32_restatement.py restates the drafter from the method's definition in numpy float32, with the oracle's
bf16 storage points and exact softmax.  It is neither the oracle nor the CUDA path.  These CPU tests show
  - that it is a correct implementation: its hidden states meet the 2e-2 row tolerance against the oracle;
  - that through the five layers and the 151936-id LM head of the 4B shape it flips ids at oracle top-2 margins
    above 1e-2, while every flip stays below MARGIN_CHAIN and its logits stay within about 5e-2 of the oracle's.
So "ids bit-exact except where the oracle's top-2 margin is below 1e-2" can hold for the LM-head stage given the
oracle's hidden states (tests/test_gpu_parity.py, assert_tokens) but not through the whole chain of any fp32
implementation; the chain rule of tests/_util.py (assert_tokens_chain) uses the fixed MARGIN_CHAIN instead.
Where exactly the flips fall depends on float32 summation order (the BLAS), so the search covers 24 requests.
"""
import numpy as np
import pytest

import synth
import fp32_restatement as fr
from _util import MARGIN_CHAIN, MARGIN_EXEMPT, REL_TOL, f64, row_rel_err


def test_restatement_meets_hidden_tolerance_tiny(oracle_lib):
    o = oracle_lib
    s = synth.TINY
    w = synth.make_weights(s, 1000)
    T, L = 128, 16
    feats = synth.make_features(s, T, 1001)
    m = o.Model(s, w)
    kv = o.prepare_context(m, np.array([0, T], np.int32), feats, T)
    oh, ol = o.draft_block(m, kv, T, np.array([T], np.int32), np.array([5], np.int32), s.vocab - 1, L,
                           want_layers=True)
    fh, fl = fr.draft_block(s, w, kv, T, 5, s.vocab - 1, L, want_layers=True)
    for l in range(s.n_layers):
        e = row_rel_err(fl[l].astype(np.float64), f64(ol[l]))
        assert e.max() <= REL_TOL, (l, e.max())
    # and it is not the oracle: fp32 accumulation moves some bf16 values by an ulp
    assert not np.array_equal(synth.f32_to_bf16_bits(fh), oh)


@pytest.mark.slow
def test_fp32_restatement_flips_ids_above_the_stage_margin_at_4b_shape(oracle_lib):
    o = oracle_lib
    s = synth.FULL
    w = synth.make_weights(s, 2000)
    wf = fr.weights_f32(w)
    m = o.Model(s, w)
    T, L = 2048, 16
    flip_margins, worst_err = [], 0.0
    for req in range(24):
        kv = synth.make_kv_store(s, 1, T, 5000 + req)
        anchor = 1000 + 37 * req
        oh = o.draft_block(m, kv, T, np.array([T], np.int32), np.array([anchor], np.int32), s.vocab - 1, L)
        ot, om, ol = o.constrain_argmax(m, oh, 1, L, want_logits=True)
        fl = fr.logits(s, wf, fr.draft_block(s, wf, kv, T, anchor, s.vocab - 1, L), L)
        worst_err = max(worst_err, float(np.abs(fl.astype(np.float64) - ol).max()))
        ft = np.argmax(fl, axis=1)
        flip_margins += [float(om[i]) for i in np.nonzero(ft != ot[0])[0]]
    print(f"fp32 restatement: {len(flip_margins)} flips in {24 * (L - 1)} positions at oracle margins "
          f"{sorted(round(x, 4) for x in flip_margins)}; largest logit error {worst_err:.3e}")
    assert max(flip_margins) > MARGIN_EXEMPT          # the stage rule cannot hold through the chain
    assert max(flip_margins) < MARGIN_CHAIN           # the chain rule's fixed bound covers it
    assert worst_err < 2 * MARGIN_CHAIN
