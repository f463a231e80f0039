"""Pins for the oracle's decoding loops against what the pages fix:

* exact-arithmetic self-speculative output equals AR greedy output, whatever
  the drafts are (GravityOCR review, Appendix B.3; velog review, inference);
* every round commits between 2 and B + 2 tokens unless truncated (review §3.2);
* after every round the cache holds only causal state, i.e. equals a fresh
  causal prefill of the committed prefix (review, Appendix B.2);
* the boundary row is causal, so a0 is the AR prediction (review §3.2);
* TPF (eq. 5) from accepted drafts per round matches the pages' tables.
"""
import json
import os

import numpy as np
import pytest

import oracle
from self_speculative_block_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def small_cfg(vocab=97):
    return synth.ModelConfig(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16,
                             ffn=96, vocab=vocab, dtype=synth.F32)


@pytest.fixture(scope="module")
def model():
    cfg = small_cfg()
    # large init so that the random decoder has clear argmax margins
    return oracle.Model(synth.make_weights(cfg, seed=11, std=0.3), cfg)


@pytest.fixture(scope="module")
def prefix(model):
    return synth.make_prefix(model.cfg, 12, seed=2).astype(np.float64)


@pytest.fixture(scope="module")
def ar_out(model, prefix):
    return oracle.ar_decode(model, prefix, 40)


@pytest.mark.parametrize("B", [1, 2, 4, 8])
def test_selfspec_equals_ar_natural_drafts(model, prefix, ar_out, B):
    out, logs = oracle.selfspec_decode(model, prefix, B, 40)
    assert out == ar_out
    for g in logs[:-1]:
        assert 2 <= len(g.committed) <= B + 2
    assert 1 <= len(logs[-1].committed) <= B + 2


@pytest.mark.parametrize("B", [2, 4, 8])
def test_selfspec_equals_ar_random_drafts(model, prefix, ar_out, B):
    rng = np.random.default_rng(B)
    ov = lambda r, c, d: [int(x) for x in rng.integers(0, model.cfg.vocab, size=len(d))]
    out, _ = oracle.selfspec_decode(model, prefix, B, 40, override=ov)
    assert out == ar_out


@pytest.mark.parametrize("B", [2, 4, 8])
def test_forced_correct_drafts_commit_B_plus_2(model, prefix, ar_out, B):
    ov = oracle.forced_override(ar_out, [10 ** 6] * 100, model.cfg.vocab)
    out, logs = oracle.selfspec_decode(model, prefix, B, 40, override=ov)
    assert out == ar_out
    for g in logs[:-1]:
        assert g.A == B and len(g.committed) == B + 2


@pytest.mark.parametrize("B", [1, 4, 8])
def test_always_wrong_drafts_equal_two_ar_steps(model, prefix, ar_out, B):
    ov = oracle.forced_override(ar_out, [0] * 100, model.cfg.vocab)
    out, logs = oracle.selfspec_decode(model, prefix, B, 40, override=ov)
    assert out == ar_out
    for g in logs[:-1]:
        assert g.A == 0 and len(g.committed) == 2


def test_forced_schedule_gives_scheduled_acceptance(model, prefix, ar_out):
    B = 8
    sched = synth.accept_schedule(3.0, 100, seed=4)
    ov = oracle.forced_override(ar_out, sched, model.cfg.vocab)
    out, logs = oracle.selfspec_decode(model, prefix, B, 40, override=ov)
    assert out == ar_out
    for r, g in enumerate(logs[:-1]):
        assert g.A == min(int(sched[r]), B)


def test_cache_after_each_round_equals_causal_prefill(model, prefix):
    B = 4
    st = oracle.prefill(model, prefix)
    P = prefix.shape[0]
    for r in range(6):
        oracle.selfspec_round(model, st, B, 10 ** 6)
        c = len(st.out)
        assert st.p == P + c - 1  # the boundary token is not in the cache
        _, k, v = oracle.prefill_cache(model, prefix, st.out[:-1])
        for l in range(model.cfg.n_layers):
            np.testing.assert_allclose(st.cache_k[l], k[l], rtol=0, atol=1e-10)
            np.testing.assert_allclose(st.cache_v[l], v[l], rtol=0, atol=1e-10)
        assert st.x0 == st.out[-1]


def test_boundary_row_is_the_ar_prediction(model, prefix):
    st = oracle.prefill(model, prefix)
    for _ in range(3):
        oracle.ar_step(model, st)
    lg_ar, _, _ = oracle.ar_forward(model, st)
    lg_d, _, _ = oracle.draft_forward(model, st, 8)
    np.testing.assert_allclose(lg_d[0], lg_ar[0], rtol=0, atol=1e-10)
    # and the [M] rows do read the window: their logits differ from row 0
    assert np.abs(lg_d[1] - lg_d[0]).max() > 1e-6


def test_verify_row_j_equals_ar_at_that_position(model, prefix, ar_out):
    # Verify rows are causal: with the AR continuation as drafts, row j's
    # logits equal the AR forward at position p+1+j.
    st = oracle.prefill(model, prefix)
    B = 4
    lg_d, kd, vd = oracle.draft_forward(model, st, B)
    a0 = int(oracle.argmax_lowest(lg_d[:1])[0])
    st.append([k[:1] for k in kd], [v[:1] for v in vd])
    drafts = ar_out[2:2 + B]
    lg_v, _, _ = oracle.verify_forward(model, st, a0, drafts)
    st2 = oracle.prefill(model, prefix)
    for j in range(B + 1):
        oracle.ar_step(model, st2)
        lg_a, _, _ = oracle.ar_forward(model, st2)
        np.testing.assert_allclose(lg_v[j], lg_a[0], rtol=0, atol=1e-10)


def test_eos_truncation(model, prefix, ar_out):
    eos = ar_out[9]
    first = ar_out.index(eos)
    want = ar_out[: first + 1]
    assert oracle.ar_decode(model, prefix, 40, eos_id=eos) == want
    for B in (2, 8):
        out, logs = oracle.selfspec_decode(model, prefix, B, 40, eos_id=eos)
        assert out == want


def test_max_new_truncation_and_minimum(model, prefix, ar_out):
    for max_new in (1, 2, 3, 7):
        out, logs = oracle.selfspec_decode(model, prefix, 8, max_new)
        assert out == ar_out[:max_new]


def test_accept_length_definition():
    assert oracle.accept_length([1, 2, 3], [1, 2, 3, 9]) == 3
    assert oracle.accept_length([1, 5, 3], [1, 2, 3, 9]) == 1
    assert oracle.accept_length([4, 2, 3], [1, 2, 3, 9]) == 0
    assert oracle.accept_length([], [7]) == 0


def test_tpf_matches_pages_tables():
    g = json.load(open(os.path.join(HERE, "golden", "tpf_pages.json")))
    for row in g["rows"]:
        a = row["accepted_per_round"]
        # rounds with A accepted drafts commit A + 2 tokens in two forwards
        rounds = 1000
        tpf = oracle.tokens_per_forward(rounds * (a + 2), 2 * rounds)
        assert abs(tpf - row["tpf"]) <= 0.051, row
    rb = g["round_bounds"]
    B = rb["B"]
    assert oracle.accept_length(list(range(B)), list(range(B + 1))) + 2 == rb["max_commit"]
    assert oracle.accept_length([1] * B, [0] * (B + 1)) + 2 == rb["min_commit"]


def test_round_stats_ar_has_tpf_one_shape(model, prefix):
    out, logs = oracle.selfspec_decode(model, prefix, 4, 30)
    s = oracle.round_stats(logs)
    assert s["committed"] == len(out) - 1
    assert s["forwards"] == 2 * s["rounds"]
    assert s["committed"] == s["accepted_drafts"] + 2 * s["rounds"] - (
        (2 + logs[-1].A) - len(logs[-1].committed))
