"""Sampling decodes through the C ABI (gocr_decode_ex with a temperature)
against the sampling oracle (oracle/sampling.py), which draws the same
Philox4x32-10 uniforms.

Sources: GravityOCR review §2 "Speculative Decoding" (the standard
acceptance-rejection rule); the Trillion Labs blog (the rule preserves the AR
distribution).

* fp32 decoder: the GPU's AR-sampling and self-speculative-sampling token
  streams equal the oracle's, up to the first draw or acceptance decided
  closer than fp32 arithmetic can resolve (top-two perturbed-score gap
  1e-3, acceptance uniform within 1e-3 of its threshold);
* by counting over seeds, self-speculative sampling on the GPU gives the
  token distribution of AR sampling on the GPU;
* a0 is the AR sample of its position (the same uniforms, bit-identical
  logits); a near-zero temperature reproduces the greedy decodes.
"""
import numpy as np
import pytest
import scipy.stats

import oracle
from oracle import sampling as smp

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GAP = 1e-3


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("gpu tests need a CUDA device")
    from self_speculative_block_gb300 import build, gocr, synth
    build.build()
    return gocr, synth


@pytest.fixture(scope="module")
def tiny(lib):
    g, synth = lib
    cfg = synth.TINY
    W = synth.make_weights(cfg, seed=0, std=0.3)
    prefix = synth.make_prefix(cfg, 16, seed=1)
    return cfg, W, prefix, oracle.Model(W, cfg)


@pytest.mark.parametrize("T", [0.7, 1.0])
def test_ar_sampling_matches_oracle(lib, tiny, T):
    g, synth = lib
    cfg, W, prefix, model = tiny
    max_new = 30
    dec = g.Decoder(cfg, W, max_ctx=16 + max_new + 8, max_block=4)
    try:
        compared = 0
        for seed in (1, 2, 3, 4):
            dec.prefill(0, prefix)
            outs, _ = dec.decode_ex([0], g.MODE_AR, 0, [max_new], temperature=T, seed=seed)
            diag = []
            ref = smp.ar_sample_decode(model, prefix.astype(np.float64), max_new, T, seed, diag=diag)
            k = next((i for i, d in enumerate(diag) if d <= GAP), len(diag))
            assert list(outs[0][:k + 1]) == ref[:k + 1], (seed, k)
            compared += k
        assert compared >= 60
    finally:
        dec.close()


@pytest.mark.parametrize("B", [4, 8])
def test_selfspec_sampling_matches_oracle(lib, tiny, B):
    g, synth = lib
    cfg, W, prefix, model = tiny
    max_new, T = 40, 1.0
    dec = g.Decoder(cfg, W, max_ctx=16 + max_new + B + 8, max_block=B)
    try:
        rounds_cmp = 0
        for seed in (5, 6, 7):
            dec.prefill(0, prefix)
            outs, sts = dec.decode_ex([0], g.MODE_SELFSPEC, B, [max_new], temperature=T, seed=seed)
            ref, logs = smp.selfspec_sample_decode(model, prefix.astype(np.float64), B, max_new, T, seed)
            k = next((i for i, lg in enumerate(logs) if lg.margin <= GAP or lg.accept_gap <= GAP), len(logs))
            n = 1 + sum(len(lg.committed) for lg in logs[:k])
            assert list(outs[0][:n]) == ref[:n], (seed, k)
            if k == len(logs):
                st = sts[0]
                assert st["rounds"] == len(logs) and st["accepted_drafts"] == sum(lg.A for lg in logs)
            rounds_cmp += k
        assert rounds_cmp >= 10
    finally:
        dec.close()


def test_selfspec_sampling_distribution_equals_ar_sampling(lib, tiny):
    """Counting over seeds and request slots: tokens at the first decode
    positions after a0 are distributed alike under AR sampling and under
    self-speculative sampling with the rejection rule (GPU against GPU)."""
    g, synth = lib
    cfg, W, prefix, _ = tiny
    n_req, calls, max_new, B = 32, 48, 5, 4
    dec = g.Decoder(cfg, W, max_ctx=16 + max_new + B + 8, max_block=B, max_requests=n_req)
    try:
        samples = {g.MODE_AR: [], g.MODE_SELFSPEC: []}
        for mode in samples:
            for c in range(calls):
                for r in range(n_req):
                    dec.prefill(r, prefix)
                outs, _ = dec.decode_ex(list(range(n_req)), mode, B if mode == g.MODE_SELFSPEC else 0,
                                        [max_new] * n_req, temperature=1.0, seed=1000 * c + (7 if mode else 0))
                samples[mode] += [list(o) for o in outs]
    finally:
        dec.close()
    a = np.array(samples[g.MODE_AR])
    s = np.array(samples[g.MODE_SELFSPEC])
    for pos in (2, 3, 4):
        ca = np.bincount(a[:, pos], minlength=cfg.vocab)
        cs = np.bincount(s[:, pos], minlength=cfg.vocab)
        common = (ca + cs) >= 10  # rare tokens pooled into one cell
        table = np.stack([np.append(ca[common], ca[~common].sum()), np.append(cs[common], cs[~common].sum())])
        table = table[:, table.sum(0) > 0]
        assert table.shape[1] >= 3, pos
        assert scipy.stats.chi2_contingency(table).pvalue > 1e-4, pos


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_a0_is_the_ar_sample_and_cold_limit_is_greedy(lib, dt):
    g, synth = lib
    if dt == "f32":
        cfg = synth.TINY
        W = synth.make_weights(cfg, seed=0, std=0.3)
    else:
        cfg = synth.ModelConfig(n_layers=2, hidden=512, n_q_heads=6, n_kv_heads=2, head_dim=128, ffn=1024,
                                vocab=2048, dtype=synth.BF16)
        W = synth.make_weights(cfg, seed=21, std=0.1)
    prefix = synth.make_prefix(cfg, 24, seed=22)
    max_new, B = 24, 8
    dec = g.Decoder(cfg, W, max_ctx=24 + max_new + B + 8, max_block=B)
    try:
        for seed in range(6):
            dec.prefill(0, prefix)
            ar, _ = dec.decode_ex([0], g.MODE_AR, 0, [2], temperature=1.0, seed=seed)
            dec.prefill(0, prefix)
            ss, st = dec.decode_ex([0], g.MODE_SELFSPEC, B, [max_new], temperature=1.0, seed=seed)
            assert list(ss[0][:2]) == list(ar[0])
            assert st[0]["committed"] == max_new - 1
        dec.prefill(0, prefix)
        greedy, _ = dec.decode(0, g.MODE_AR, 0, max_new)
        for mode in (g.MODE_AR, g.MODE_SELFSPEC):
            dec.prefill(0, prefix)
            cold, _ = dec.decode_ex([0], mode, B if mode else 0, [max_new], temperature=1e-4, seed=9)
            assert list(cold[0]) == list(greedy), mode
        with pytest.raises(g.GocrError):
            dec.decode_ex([0], g.MODE_DIFFUSION, B, [max_new], tau=0.5, temperature=1.0)
    finally:
        dec.close()
