"""Pins for three readings of the oracle that the decode invariants alone do
not fix:

* the [M] rows of the draft window use the single added mask-token embedding
  row and nothing else (GravityOCR review, §3.1 "AR-to-Diffusion Conversion":
  one learnable mask embedding, shared backbone); the boundary row never
  reads it (review §3.2: the boundary position is causal);
* the first output token is the argmax of the prefill's last row (the
  shift-by-one convention of review §3.1 applied to the prompt's last
  position), checked against a torch library composition of the decoder;
* the top-two margin of a row is the log-ratio of its two largest softmax
  probabilities (review Appendix B.3 measures first divergences by it).
"""
import math

import numpy as np
import scipy.special

import oracle
import test_oracle_components as comp
from self_speculative_block_gb300 import synth


def _cfg():
    return synth.ModelConfig(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16,
                             ffn=96, vocab=97, dtype=synth.F32)


def _state(W, cfg, prefix, n_ar=2):
    m = oracle.Model(W, cfg)
    st = oracle.prefill(m, prefix)
    for _ in range(n_ar):
        oracle.ar_step(m, st)
    return m, st


def test_mask_rows_read_the_mask_embedding_only():
    cfg = _cfg()
    W = synth.make_weights(cfg, seed=21, std=0.3)
    prefix = synth.make_prefix(cfg, 9, seed=4).astype(np.float64)
    B = 5
    m, st = _state(W, cfg, prefix)
    assert st.x0 != cfg.vocab - 1
    base, _, _ = oracle.draft_forward(m, st, B)

    # a different [M] row changes every [M] row's logits and not the boundary row's
    W2 = dict(W)
    W2["mask_embed"] = W["mask_embed"] + np.float32(0.5)
    m2, st2 = _state(W2, cfg, prefix)
    lg2, _, _ = oracle.draft_forward(m2, st2, B)
    np.testing.assert_array_equal(lg2[0], base[0])
    for r in range(1, B + 1):
        assert np.abs(lg2[r] - base[r]).max() > 1e-6

    # the last vocabulary row (a plausible stand-in for a mask id) is not read
    W3 = dict(W)
    E = W["embed"].copy()
    E[-1] += np.float32(0.5)
    W3["embed"] = E
    m3, st3 = _state(W3, cfg, prefix)
    assert st3.out == st.out
    lg3, _, _ = oracle.draft_forward(m3, st3, B)
    np.testing.assert_array_equal(lg3, base)

    # and the boundary row reads the boundary token's own embedding row
    W4 = dict(W)
    E = W["embed"].copy()
    E[st.x0] += np.float32(0.5)
    W4["embed"] = E
    m4 = oracle.Model(W4, cfg)
    lg4, _, _ = oracle.draft_forward(m4, st, B)
    assert np.abs(lg4[0] - base[0]).max() > 1e-6


def test_prefill_token_is_the_argmax_of_the_last_prefix_row():
    cfg = _cfg()
    W = synth.make_weights(cfg, seed=23, std=0.3)
    for P in (1, 6, 13):
        prefix = synth.make_prefix(cfg, P, seed=P).astype(np.float64)
        st = oracle.prefill(oracle.Model(W, cfg), prefix)
        lg, _, _ = oracle.prefill_cache(oracle.Model(W, cfg), prefix)
        ref = comp._torch_forward(W, cfg, prefix, np.arange(P, dtype=np.float64))
        assert st.out == [int(np.argmax(ref[-1]))] == [int(np.argmax(lg[-1]))]
        assert st.x0 == st.out[0] and st.p == P


def test_top2_margin_closed_forms():
    assert oracle.top2_margin(np.array([0.0, -1.0, 2.0])) == 2.0
    assert oracle.top2_margin(np.array([1.0, 3.5, 2.25, 3.5])) == 0.0
    assert oracle.top2_margin(np.array([-7.0, -7.5])) == 0.5
    rng = np.random.default_rng(5)
    for _ in range(20):
        lg = rng.standard_normal(40) * 2
        p = np.sort(scipy.special.softmax(lg))
        assert abs(oracle.top2_margin(lg) - math.log(p[-1] / p[-2])) < 1e-12
