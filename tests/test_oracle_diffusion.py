"""Pins for the oracle's block-diffusion paths against what the pages and the
mathematics fix (never against a retyped copy of the same code):

* confidence is the largest softmax probability (blog, threshold paragraph):
  scipy's softmax and closed forms;
* the threshold rule of one denoising step (GravityOCR review, Appendix B.1):
  a set-based construction written from the rule text;
* block size 1 is AR greedy decoding (the block's only slot is predicted by
  the causal boundary row);
* the first slot of every block is the AR prediction at the block's state;
* after every block's cache-write forward the cache equals a fresh causal
  prefill of the committed prefix (the cache holds causal state only);
* threshold 0 fixes a whole block in one step, equal to the one-shot
  self-speculative draft at the same state; a threshold above 1 fixes one
  slot per step, always the most confident one;
* EOS cut and max_new truncation (review Appendix B.1);
* the pages' direct-diffusion TPF figures lie under the bound B/2 that
  counting the cache-write forward implies (tests/golden/);
* a refined draft (review Appendix D) keeps the output equal to AR greedy,
  and one step is the one-shot round.
"""
import json
import os

import numpy as np
import pytest
import scipy.special

import oracle
from self_speculative_block_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def small_cfg(vocab=97):
    return synth.ModelConfig(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16,
                             ffn=96, vocab=vocab, dtype=synth.F32)


@pytest.fixture(scope="module")
def model():
    cfg = small_cfg()
    return oracle.Model(synth.make_weights(cfg, seed=11, std=0.3), cfg)


@pytest.fixture(scope="module")
def prefix(model):
    return synth.make_prefix(model.cfg, 12, seed=2).astype(np.float64)


@pytest.fixture(scope="module")
def ar_out(model, prefix):
    return oracle.ar_decode(model, prefix, 40)


# ---------------------------------------------------------------- confidence and the step rule

def test_confidence_is_the_softmax_maximum():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((6, 50)) * 3
    tok, conf = oracle.confidence(lg)
    p = scipy.special.softmax(lg, axis=-1)
    np.testing.assert_allclose(conf, p.max(-1), rtol=1e-13)
    np.testing.assert_array_equal(tok, p.argmax(-1))


def test_confidence_closed_forms():
    V = 64
    _, c = oracle.confidence(np.zeros((1, V)))          # uniform: 1 / V
    assert abs(c[0] - 1.0 / V) < 1e-15
    lg = np.full((1, V), -1e4)
    lg[0, 5] = lg[0, 9] = 2.0                            # two equal maxima, the rest ~0 mass
    tok, c = oracle.confidence(lg)
    assert tok[0] == 5 and abs(c[0] - 0.5) < 1e-12
    lg = np.array([[np.log(3.0), 0.0]])                  # p = (3/4, 1/4)
    assert abs(oracle.confidence(lg)[1][0] - 0.75) < 1e-15


def _rule_from_text(conf, masked, tau):
    """Fix every masked slot at or over the threshold; if none, the one most
    confident masked slot (lowest index among equals)."""
    over = {s for s in masked if conf[s] >= tau}
    if over:
        return over
    top = max(conf[s] for s in masked)
    return {min(s for s in masked if conf[s] == top)}


def test_choose_slots_matches_the_rule_text():
    rng = np.random.default_rng(8)
    for trial in range(400):
        B = int(rng.integers(1, 12))
        conf = np.round(rng.uniform(0, 1, B), 1)  # rounding makes ties and exact-threshold hits
        masked = sorted(rng.choice(B, size=int(rng.integers(1, B + 1)), replace=False).tolist())
        tau = float(np.round(rng.uniform(0, 1.1), 1))
        assert set(oracle.choose_slots(conf, masked, tau)) == _rule_from_text(conf, masked, tau)
    assert oracle.choose_slots([0.5, 0.5, 0.2], [0, 1, 2], 0.9) == [0]
    assert oracle.choose_slots([0.5, 0.9, 0.9], [1, 2], 0.9) == [1, 2]
    assert oracle.choose_slots([0.1], [], 0.5) == []


# ---------------------------------------------------------------- direct block diffusion

def test_block_size_one_is_ar_greedy(model, prefix, ar_out):
    for tau in (0.0, 0.5, 2.0):
        out, logs = oracle.diffusion_decode(model, prefix, 1, tau, 40)
        assert out == ar_out
        assert all(len(g.steps) == 1 for g in logs)


@pytest.mark.parametrize("tau", [0.0, 0.4, 0.8, 1.5])
def test_first_slot_of_each_block_is_the_ar_prediction(model, prefix, tau):
    st = oracle.prefill(model, prefix)
    for _ in range(4):
        lg_ar, _, _ = oracle.ar_forward(model, st)
        want = int(oracle.argmax_lowest(lg_ar)[0])
        g = oracle.diffusion_block(model, st, 6, tau, 10 ** 6)
        assert g.block[0] == want


@pytest.mark.parametrize("tau", [0.0, 0.5, 1.5])
def test_cache_after_each_block_equals_causal_prefill(model, prefix, tau):
    st = oracle.prefill(model, prefix)
    P = prefix.shape[0]
    for _ in range(4):
        g = oracle.diffusion_block(model, st, 5, tau, 10 ** 6)
        assert g.cache_write
        c = len(st.out)
        assert st.p == P + c - 1 and st.x0 == st.out[-1] == g.block[-1]
        _, k, v = oracle.prefill_cache(model, prefix, st.out[:-1])
        for l in range(model.cfg.n_layers):
            np.testing.assert_allclose(st.cache_k[l], k[l], rtol=0, atol=1e-10)
            np.testing.assert_allclose(st.cache_v[l], v[l], rtol=0, atol=1e-10)


def test_threshold_zero_is_the_one_shot_draft(model, prefix):
    B = 7
    st = oracle.prefill(model, prefix)
    for _ in range(3):
        lg, _, _ = oracle.draft_forward(model, st, B)
        want = [int(t) for t in oracle.argmax_lowest(lg)[:B]]  # a0, d_1..d_{B-1}
        g = oracle.diffusion_block(model, st, B, 0.0, 10 ** 6)
        assert len(g.steps) == 1 and g.block == want


def test_threshold_above_one_fixes_the_most_confident_slot_each_step(model, prefix):
    B = 6
    out, logs = oracle.diffusion_decode(model, prefix, B, 1.01, 25)
    fed_back = False
    for g in logs:
        assert len(g.steps) == B
        masked = list(range(B))
        for i, s in enumerate(g.steps):
            assert len(s.fixed) == 1
            top = max(s.conf[m] for m in masked)
            assert s.fixed[0] == min(m for m in masked if s.conf[m] == top)
            assert g.block[s.fixed[0]] == s.tokens[s.fixed[0]]
            masked.remove(s.fixed[0])
            if i and s.tokens != g.steps[i - 1].tokens:
                fed_back = True
    # the fixed tokens are fed back into the window: later steps predict differently
    assert fed_back


def test_eos_cut_and_max_new(model, prefix):
    out, logs = oracle.diffusion_decode(model, prefix, 5, 0.5, 40)
    assert len(out) == 40
    # an EOS token that first appears inside a block's middle
    first = {}
    for i, t in enumerate(out[1:], start=1):
        first.setdefault(t, i)
    cand = [t for t, i in first.items() if (i - 1) % 5 not in (0, 4) and i < 30]
    eos = cand[0]
    out_e, logs_e = oracle.diffusion_decode(model, prefix, 5, 0.5, 40, eos_id=eos)
    assert out_e == out[: first[eos] + 1]
    assert not logs_e[-1].cache_write and logs_e[-1].committed[-1] == eos


def test_pages_direct_diffusion_tpf_under_the_cache_write_bound():
    with open(os.path.join(HERE, "golden", "direct_diffusion_pages.json")) as f:
        g = json.load(f)
    B = g["block"]
    bound = B / 2.0  # one denoising step plus one cache-write forward per block at best
    for row in g["rows"]:
        assert 0 < row["tpf"] <= bound, row
    # and the oracle meets the bound exactly with one step per block
    cfg = small_cfg()
    m = oracle.Model(synth.make_weights(cfg, seed=11, std=0.3), cfg)
    pre = synth.make_prefix(cfg, 12, seed=2).astype(np.float64)
    Bs = 4
    _, logs = oracle.diffusion_decode(m, pre, Bs, 0.0, 1 + 3 * Bs + 1)
    full = [g for g in logs if g.cache_write]
    s = oracle.diffusion_stats(full)
    assert s["tpf"] == Bs / 2.0


# ---------------------------------------------------------------- refined drafts

@pytest.mark.parametrize("n_steps", [1, 2, 4])
@pytest.mark.parametrize("tau_d", [0.0, 0.5, 2.0])
def test_refined_drafts_keep_ar_output(model, prefix, ar_out, n_steps, tau_d):
    out, logs = oracle.refined_decode(model, prefix, 6, tau_d, n_steps, 40)
    assert out == ar_out
    for g in logs:
        assert 1 <= len(g.steps) <= n_steps
        if tau_d > 1.0:
            assert len(g.steps) == min(n_steps, 6)
    for g in logs[:-1]:
        assert 2 <= len(g.committed) <= 6 + 2


def test_one_refinement_step_is_the_one_shot_round(model, prefix):
    for tau_d in (0.0, 0.7, 2.0):
        st1 = oracle.prefill(model, prefix)
        st2 = oracle.prefill(model, prefix)
        for _ in range(5):
            a = oracle.selfspec_round(model, st1, 6, 10 ** 6)
            b = oracle.refined_round(model, st2, 6, tau_d, 1, 10 ** 6)
            assert (a.a0, a.drafts, a.verify, a.A, a.committed) == (b.a0, b.drafts, b.verify, b.A, b.committed)


def test_refined_fixed_slots_survive_to_verify(model, prefix):
    st = oracle.prefill(model, prefix)
    for _ in range(4):
        g = oracle.refined_round(model, st, 6, 2.0, 3, 10 ** 6)
        window = [g.a0] + g.drafts
        for s in g.steps:
            for f in s.fixed:
                assert window[f] == s.tokens[f]
        assert g.a0 == g.steps[0].tokens[0]
