"""bf16 decode path (tcgen05 GEMMs + tensor-core split-KV attention) through the C ABI.

* a small bf16 decoder with the 0.5B model's head geometry (GQA 3:1, head_dim
  128): draft / verify / AR logits vs the oracle within max-abs 3e-2 /
  relative 2e-2, replayed AR tokens, KV cache vs an oracle prefill;
* the GPU's self-speculative output equals its own AR output bit for bit for
  every block size up to 64, natural and forced drafts, single and batched;
* the 0.5B-class decoder at the text-region and table-region sizes: bit
  exactness against the GPU AR path, and sampled logits against the oracle.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ATOL, RTOL = 3e-2, 2e-2


def close(got, ref):
    err = np.abs(got - ref)
    return bool(np.all(err <= ATOL + RTOL * np.abs(ref))), float(err.max())


@pytest.fixture(scope="module")
def small():
    if not torch.cuda.is_available():
        pytest.fail("gpu tests need a CUDA device")
    from self_speculative_block_gb300 import build, gocr, synth
    build.build()
    cfg = synth.ModelConfig(n_layers=2, hidden=512, n_q_heads=6, n_kv_heads=2, head_dim=128, ffn=1024,
                            vocab=2048, dtype=synth.BF16)
    W = synth.make_weights(cfg, seed=21)
    prefix = synth.make_prefix(cfg, 100, seed=22)
    dec = gocr.Decoder(cfg, W, max_ctx=100 + 200 + 64 + 8, max_block=64, max_requests=4)
    yield dict(g=gocr, synth=synth, cfg=cfg, W=W, prefix=prefix, dec=dec, model=oracle.Model(W, cfg))
    dec.close()


@pytest.fixture(scope="module")
def small_ar(small):
    dec, g = small["dec"], small["g"]
    dec.prefill(0, small["prefix"])
    out, _ = dec.decode(0, g.MODE_AR, 0, 200)
    return out


@pytest.mark.parametrize("B", [1, 8, 32, 64])
def test_small_draft_verify_logits(small, B):
    dec, g, model = small["dec"], small["g"], small["model"]
    prefix = small["prefix"].astype(np.float64)
    dec.prefill(0, small["prefix"])
    cl, x0 = dec.state(0)
    lg_d = dec.debug_forward(0, g.FWD_DRAFT, [x0] + [0] * B)
    st = oracle.prefill(model, prefix)
    ref_d, kd, vd = oracle.draft_forward(model, st, B)
    ok, err = close(lg_d, ref_d)
    assert ok, err
    a0 = int(np.argmax(lg_d[0]))
    drafts = [int(t) for t in np.random.default_rng(B).integers(0, small["cfg"].vocab, B)]
    lg_v = dec.debug_forward(0, g.FWD_VERIFY, [a0] + drafts)
    st.append([k[:1] for k in kd], [v[:1] for v in vd])
    ref_v, _, _ = oracle.verify_forward(model, st, a0, drafts)
    ok, err = close(lg_v, ref_v)
    assert ok, err


def test_small_ar_replay_and_kv(small, small_ar):
    dec, g, model = small["dec"], small["g"], small["model"]
    prefix = small["prefix"].astype(np.float64)
    out = list(small_ar)
    logits, K, V = oracle.prefill_cache(model, prefix, out[:-1])
    P = prefix.shape[0]
    agree = 0
    for i, t in enumerate(out):
        row = logits[P - 1 + i]
        assert row[t] >= row.max() - 2 * ATOL, (i, t, row.max() - row[t])
        agree += int(np.argmax(row) == t)
    print(f"bf16 GPU AR vs oracle argmax agreement: {agree}/{len(out)}")
    dec.prefill(0, small["prefix"])
    dec.decode(0, g.MODE_AR, 0, 200)
    for l in range(small["cfg"].n_layers):
        k, v = dec.read_kv(0, l, 0, P + 199)
        ok, err = close(k, K[l])
        assert ok, err
        ok, err = close(v, V[l])
        assert ok, err


@pytest.mark.parametrize("B", [1, 2, 8, 32, 64])
def test_small_selfspec_bit_exact(small, small_ar, B):
    dec, g = small["dec"], small["g"]
    dec.prefill(0, small["prefix"])
    out, st = dec.decode(0, g.MODE_SELFSPEC, B, 200)
    assert list(out) == list(small_ar)
    kv_ss = dec.read_kv(0, 1, 0, 100 + 199)
    dec.prefill(0, small["prefix"])
    dec.decode(0, g.MODE_AR, 0, 200)
    kv_ar = dec.read_kv(0, 1, 0, 100 + 199)
    assert np.array_equal(kv_ss[0], kv_ar[0]) and np.array_equal(kv_ss[1], kv_ar[1])


@pytest.mark.parametrize("B,mean", [(8, 4.0), (32, 9.0), (64, 19.0)])
def test_small_forced_acceptance_bit_exact(small, small_ar, B, mean):
    dec, g, synth = small["dec"], small["g"], small["synth"]
    sched = synth.accept_schedule(mean, 200, seed=synth.SCHEDULE_SEED)
    dec.prefill(0, small["prefix"])
    dec.set_draft_override(0, small_ar, sched)
    try:
        out, st = dec.decode(0, g.MODE_SELFSPEC, B, 200)
    finally:
        dec.clear_draft_override(0)
    assert list(out) == list(small_ar)
    want = np.bincount([min(int(x), B) for x in sched[: st["rounds"] - 1]], minlength=65)
    got = np.array(st["accept_hist"])
    assert np.all(got >= want) and (got - want).sum() == 1


def test_small_batched_ragged_equals_single_ar(small):
    dec, g, synth, cfg = small["dec"], small["g"], small["synth"], small["cfg"]
    lens = [37, 100, 64, 129]
    news = [40, 120, 7, 90]
    prefixes = [synth.make_prefix(cfg, n, seed=1000 + r) for r, n in enumerate(lens)]
    refs = []
    for r in range(4):
        dec.prefill(r, prefixes[r])
        out, _ = dec.decode(r, g.MODE_AR, 0, news[r])
        refs.append(list(out))
    # B = 64: 4 x 65 = 260 rows, past two 128-token slices, so the batched
    # forwards run the many-slice GEMM; on this batching handle the O and down
    # projections (4 weight tiles, 8 chunks) sum in two groups on two-CTA
    # clusters, which must reproduce the clustered kernel's bits for AR
    for mode, B in ((g.MODE_SELFSPEC, 8), (g.MODE_AR, 0), (g.MODE_SELFSPEC, 32), (g.MODE_SELFSPEC, 64)):
        for r in range(4):
            dec.prefill(r, prefixes[r])
        outs, sts = dec.decode_batch([0, 1, 2, 3], mode, B, news)
        for r in range(4):
            assert list(outs[r]) == refs[r], (mode, B, r)
            assert sts[r]["committed"] == news[r] - 1


def test_small_tcgen05_attention_handle(small, monkeypatch):
    """A handle with the tcgen05 attention: draft and verify logits against the
    oracle, and its self-speculative output (single and batched) equal to its
    own AR-greedy output bit for bit."""
    g, synth, cfg, model = small["g"], small["synth"], small["cfg"], small["model"]
    monkeypatch.setenv("GOCR_ATTN", "tc")
    dec = g.Decoder(cfg, small["W"], max_ctx=100 + 200 + 64 + 8, max_block=64, max_requests=4)
    monkeypatch.delenv("GOCR_ATTN")
    try:
        assert dec.attention_kind() == g.ATTN_TCGEN05
        prefix = small["prefix"].astype(np.float64)
        for B in (1, 32, 64):
            dec.prefill(0, small["prefix"])
            cl, x0 = dec.state(0)
            lg_d = dec.debug_forward(0, g.FWD_DRAFT, [x0] + [0] * B)
            st = oracle.prefill(model, prefix)
            ref_d, kd, vd = oracle.draft_forward(model, st, B)
            ok, err = close(lg_d, ref_d)
            assert ok, (B, err)
            a0 = int(np.argmax(lg_d[0]))
            drafts = [int(t) for t in np.random.default_rng(B).integers(0, cfg.vocab, B)]
            lg_v = dec.debug_forward(0, g.FWD_VERIFY, [a0] + drafts)
            st.append([k[:1] for k in kd], [v[:1] for v in vd])
            ref_v, _, _ = oracle.verify_forward(model, st, a0, drafts)
            ok, err = close(lg_v, ref_v)
            assert ok, (B, err)
        dec.prefill(0, small["prefix"])
        ar, _ = dec.decode(0, g.MODE_AR, 0, 200)
        for B in (8, 32, 64):
            dec.prefill(0, small["prefix"])
            ss, _ = dec.decode(0, g.MODE_SELFSPEC, B, 200)
            assert list(ss) == list(ar), B
        lens, news = [37, 100, 64, 129], [40, 120, 7, 90]
        prefixes = [synth.make_prefix(cfg, n, seed=1000 + r) for r, n in enumerate(lens)]
        refs = []
        for r in range(4):
            dec.prefill(r, prefixes[r])
            refs.append(list(dec.decode(r, g.MODE_AR, 0, news[r])[0]))
        for r in range(4):
            dec.prefill(r, prefixes[r])
        outs, _ = dec.decode_batch([0, 1, 2, 3], g.MODE_SELFSPEC, 32, news)
        assert [list(o) for o in outs] == refs
    finally:
        dec.close()


# ------------------------------------------------------------------ 0.5B-class decoder

@pytest.fixture(scope="module")
def base():
    if not torch.cuda.is_available():
        pytest.fail("gpu tests need a CUDA device")
    from self_speculative_block_gb300 import build, gocr, synth
    build.build()
    cfg = synth.BASE
    W = synth.make_weights(cfg)
    dec = gocr.Decoder(cfg, W, max_ctx=2048 + 872 + 64 + 8, max_block=64, max_requests=1)
    yield dict(g=gocr, synth=synth, cfg=cfg, W=W, dec=dec)
    dec.close()


def test_base_text_region_selfspec_equals_ar(base):
    dec, g, synth = base["dec"], base["g"], base["synth"]
    wl = synth.WORKLOADS["text"]
    prefix = synth.make_prefix(wl.model, wl.prefix_len)
    dec.prefill(0, prefix)
    ar, _ = dec.decode(0, g.MODE_AR, 0, wl.max_new)
    dec.prefill(0, prefix)
    ss, st = dec.decode(0, g.MODE_SELFSPEC, wl.block, wl.max_new)
    assert list(ss) == list(ar)
    assert st["committed"] == wl.max_new - 1


def test_base_table_region_forced_selfspec_equals_ar(base):
    dec, g, synth = base["dec"], base["g"], base["synth"]
    wl = synth.WORKLOADS["table"]
    prefix = synth.make_prefix(wl.model, wl.prefix_len)
    dec.prefill(0, prefix)
    ar, _ = dec.decode(0, g.MODE_AR, 0, wl.max_new)
    sched = synth.accept_schedule(wl.forced_mean, wl.max_new)
    dec.prefill(0, prefix)
    dec.set_draft_override(0, ar, sched)
    try:
        ss, st = dec.decode(0, g.MODE_SELFSPEC, wl.block, wl.max_new)
    finally:
        dec.clear_draft_override(0)
    assert list(ss) == list(ar)
    tpf = st["committed"] / st["forwards"]
    # forced mean 9 accepted drafts: about (9 + 2) / 2 tokens per forward
    assert 4.0 < tpf < 7.0, tpf


def test_base_sampled_logits_vs_oracle(base):
    """Full-size model, text-region prefix: draft and verify logits of one round
    against the fp64 oracle on sampled rows (all B + 1 rows, a vocab sample)."""
    dec, g, synth, cfg = base["dec"], base["g"], base["synth"], base["cfg"]
    wl = synth.WORKLOADS["text"]
    prefix = synth.make_prefix(cfg, wl.prefix_len)
    dec.prefill(0, prefix)
    cl, x0 = dec.state(0)
    B = wl.block
    lg_d = dec.debug_forward(0, g.FWD_DRAFT, [x0] + [0] * B)
    model = oracle.Model(base["W"], cfg)
    st = oracle.prefill(model, prefix.astype(np.float64))
    st.x0 = x0  # the window starts from the GPU's boundary token
    ref_d, kd, vd = oracle.draft_forward(model, st, B)
    ok, err = close(lg_d, ref_d)
    assert ok, err
    drafts = [int(t) for t in np.argmax(lg_d[1:], axis=-1)]
    a0 = int(np.argmax(lg_d[0]))
    lg_v = dec.debug_forward(0, g.FWD_VERIFY, [a0] + drafts)
    st.append([k[:1] for k in kd], [v[:1] for v in vd])
    ref_v, _, _ = oracle.verify_forward(model, st, a0, drafts)
    ok, err = close(lg_v, ref_v)
    assert ok, err
    agree = float(np.mean(np.argmax(lg_v, -1) == np.argmax(ref_v, -1)))
    print(f"0.5B verify-row argmax agreement with the oracle: {agree:.3f}")
