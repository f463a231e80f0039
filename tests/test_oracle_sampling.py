"""Pins for the sampling oracle (oracle/sampling.py):

* Philox4x32-10 against its published known-answer vectors (tests/golden/);
  its uniforms pass a Kolmogorov-Smirnov test;
* a Gumbel-max draw has the target categorical distribution (counting);
* the acceptance-rejection rule returns the target distribution: exactly, in
  closed form, and by counting through the oracle's own functions;
* self-speculative sampling commits tokens distributed as AR sampling
  (counting over seeds; review §2 "Speculative Decoding", blog AR-equivalence
  paragraph); a0 is pathwise the AR sample; a near-zero temperature gives the
  greedy output; every round commits 2 .. B + 2 tokens.
"""
import json
import os

import numpy as np
import pytest
import scipy.stats

import oracle
from oracle import sampling as smp
from self_speculative_block_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def test_philox_known_answers():
    with open(os.path.join(HERE, "golden", "philox4x32_10_kat.json")) as f:
        kat = json.load(f)["vectors"]
    for v in kat:
        ctr = np.array([[int(x, 16) for x in v["ctr"]]], np.uint64)
        out = smp.philox4x32_10(ctr, [int(x, 16) for x in v["key"]])[0]
        assert [int(x) for x in out] == [int(x, 16) for x in v["out"]]


def test_uniforms_are_uniform_and_distinct_per_stream():
    u = smp.uniforms(seed=123, req=0, pos=7, purpose=0, n=200_000)
    assert u.min() > 0 and u.max() < 1
    assert scipy.stats.kstest(u, "uniform").pvalue > 1e-3
    v = smp.uniforms(seed=123, req=0, pos=8, purpose=0, n=1000)
    w = smp.uniforms(seed=123, req=1, pos=7, purpose=0, n=1000)
    assert not np.array_equal(u[:1000], v) and not np.array_equal(u[:1000], w)
    assert np.array_equal(u[:1000], smp.uniforms(seed=123, req=0, pos=7, purpose=0, n=1000))


def _chisq_p(counts, probs):
    m = probs * counts.sum() >= 5
    exp = probs[m] * counts.sum()
    obs = counts[m]
    obs = np.append(obs, counts[~m].sum())
    exp = np.append(exp, probs[~m].sum() * counts.sum())
    keep = exp > 0
    return scipy.stats.chisquare(obs[keep], exp[keep] * obs[keep].sum() / exp[keep].sum()).pvalue


def test_gumbel_argmax_draws_the_categorical():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal(12) * 1.5
    p = smp.probs(logits, 1.0)
    draws = [smp.gumbel_argmax(logits, smp.uniforms(9, 0, pos, 0, 12)) for pos in range(20000)]
    assert _chisq_p(np.bincount(draws, minlength=12), p) > 1e-3


def test_acceptance_rejection_preserves_the_target_closed_form():
    rng = np.random.default_rng(5)
    for _ in range(50):
        V = int(rng.integers(2, 30))
        p = rng.dirichlet(np.ones(V) * 0.5)
        q = rng.dirichlet(np.ones(V) * 0.5)
        acc = q * np.minimum(1.0, p / q)
        resid = np.maximum(0.0, p - q)
        out = acc + (1.0 - acc.sum()) * (resid / resid.sum() if resid.sum() > 0 else 0.0)
        np.testing.assert_allclose(out, p, atol=1e-12)


def test_acceptance_rejection_by_counting_through_the_oracle():
    rng = np.random.default_rng(6)
    V = 8
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    lq = np.log(q)
    out = []
    for pos in range(40000):
        d = smp.gumbel_argmax(lq, smp.uniforms(1, 0, pos, smp.PURPOSE_DRAFT, V))
        u = smp.uniforms(1, 0, pos, smp.PURPOSE_ACCEPT, 1)[0]
        A, _ = smp.accept_reject([d], q[None], p[None], [u])
        out.append(d if A == 1 else smp.residual_sample(p, q, smp.uniforms(1, 0, pos, smp.PURPOSE_RESIDUAL, V)))
    assert _chisq_p(np.bincount(out, minlength=V), p) > 1e-3


@pytest.fixture(scope="module")
def tiny():
    cfg = synth.ModelConfig(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16, ffn=96, vocab=97,
                            dtype=synth.F32)
    m = oracle.Model(synth.make_weights(cfg, seed=11, std=0.3), cfg)
    return m, synth.make_prefix(cfg, 12, seed=2).astype(np.float64)


def test_selfspec_sampling_matches_ar_sampling_by_counting(tiny):
    m, prefix = tiny
    T, B, n = 1.0, 4, 6
    ar, ss = [], []
    for seed in range(1500):
        a = smp.ar_sample_decode(m, prefix, n, T, seed)
        s, logs = smp.selfspec_sample_decode(m, prefix, B, n, T, seed + 100_000)
        ar.append(a)
        ss.append(s)
        assert s[1] == smp.selfspec_sample_decode(m, prefix, B, 2, T, seed + 100_000)[0][1]
        for g in logs[:-1]:
            assert 2 <= len(g.committed) <= B + 2
    ar, ss = np.array(ar), np.array(ss)
    assert (ar[:, 0] == ss[:, 0]).all()  # the greedy prefill token
    for pos in (1, 2, 3, 5):
        V = m.cfg.vocab
        ca, cs = np.bincount(ar[:, pos], minlength=V), np.bincount(ss[:, pos], minlength=V)
        keep = (ca + cs) > 0
        assert scipy.stats.chi2_contingency(np.stack([ca[keep], cs[keep]])).pvalue > 1e-3, pos


def test_a0_is_pathwise_the_ar_sample(tiny):
    m, prefix = tiny
    for seed in range(20):
        a = smp.ar_sample_decode(m, prefix, 2, 1.0, seed)
        s, _ = smp.selfspec_sample_decode(m, prefix, 4, 2, 1.0, seed)
        assert a == s


def test_near_zero_temperature_is_greedy(tiny):
    m, prefix = tiny
    greedy = oracle.ar_decode(m, prefix, 30)
    assert smp.ar_sample_decode(m, prefix, 30, 1e-4, 3) == greedy
    out, logs = smp.selfspec_sample_decode(m, prefix, 4, 30, 1e-4, 3)
    assert out == greedy
