"""Batched rounds and the full-size block sweep and page batch through the C ABI.

* one batched draft and one batched verify forward over ragged request caches
  (more than 256 rows: the many-slice GEMM and the batching handle's
  two-group split-K sums run) against the oracle's draft and verify forwards
  of every request, within max-abs 3e-2 / relative 2e-2 (velog review,
  "Throughput Scaling with Batch Size"; GravityOCR review Appendix C, page
  concurrency);
* the block-size sweep on the 0.5B-class decoder (prefix 2048, 512 tokens):
  forced acceptance of mean 4 at B = 8 and of mean 19 at B = 64, output equal
  to the GPU's own AR greedy output bit for bit (review Appendix B.3);
* the 16-request ragged page batch on the 0.5B-class decoder: every request's
  batched self-speculative output equals its single-request AR output on the
  same handle, and one request's batched draft logits match the oracle.
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
def lib():
    if not torch.cuda.is_available():
        pytest.fail("gpu tests need a CUDA device")
    from self_speculative_block_gb300 import build, gocr, synth
    build.build()
    return gocr, synth


def test_small_batched_forwards_match_oracle(lib):
    g, synth = lib
    cfg = synth.ModelConfig(n_layers=2, hidden=512, n_q_heads=6, n_kv_heads=2, head_dim=128, ffn=1024,
                            vocab=2048, dtype=synth.BF16)
    W = synth.make_weights(cfg, seed=21)
    model = oracle.Model(W, cfg)
    lens = [37, 100, 64, 129]
    prefixes = [synth.make_prefix(cfg, n, seed=1000 + r) for r, n in enumerate(lens)]
    dec = g.Decoder(cfg, W, max_ctx=129 + 2 * 65 + 8, max_block=64, max_requests=4)
    try:
        for B in (64, 8):  # 4 x 65 = 260 rows (many-slice GEMM) and 4 x 9 = 36 rows (clustered GEMM)
            states = []
            x0s = []
            for r in range(4):
                dec.prefill(r, prefixes[r])
                states.append(oracle.prefill(model, prefixes[r].astype(np.float64)))
                x0s.append(dec.state(r)[1])
                states[-1].x0 = x0s[-1]  # the window starts from the GPU's boundary token
            toks = np.array([[x0s[r]] + [0] * B for r in range(4)], np.int32)
            lg_d = dec.debug_forward_batch([0, 1, 2, 3], g.FWD_DRAFT, toks)
            rng = np.random.default_rng(B)
            vt = []
            for r in range(4):
                ref_d, kd, vd = oracle.draft_forward(model, states[r], B)
                ok, err = close(lg_d[r], ref_d)
                assert ok, (B, r, err)
                states[r].append([k[:1] for k in kd], [v[:1] for v in vd])
                a0 = int(np.argmax(lg_d[r, 0]))
                vt.append([a0] + [int(t) for t in rng.integers(0, cfg.vocab, B)])
            lg_v = dec.debug_forward_batch([0, 1, 2, 3], g.FWD_VERIFY, np.array(vt, np.int32))
            for r in range(4):
                ref_v, _, _ = oracle.verify_forward(model, states[r], vt[r][0], vt[r][1:])
                ok, err = close(lg_v[r], ref_v)
                assert ok, (B, r, err)
            # a request's rows do not depend on the other requests in the launch
            lg_1 = dec.debug_forward_batch([2], g.FWD_VERIFY, np.array(vt[2:3], np.int32))
            assert np.array_equal(lg_1[0].view(np.uint32), lg_v[2].view(np.uint32))
    finally:
        dec.close()


@pytest.fixture(scope="module")
def base(lib):
    g, synth = lib
    cfg = synth.BASE
    W = synth.make_weights(cfg)
    return dict(g=g, synth=synth, cfg=cfg, W=W)


@pytest.mark.parametrize("B,mean", [(8, 4.0), (64, 19.0)])
def test_base_block_sweep_forced_selfspec_equals_ar(base, B, mean):
    g, synth, cfg = base["g"], base["synth"], base["cfg"]
    wl = synth.WORKLOADS["sweep"]
    prefix = synth.make_prefix(cfg, wl.prefix_len)
    dec = g.Decoder(cfg, base["W"], max_ctx=wl.prefix_len + wl.max_new + max(synth.SWEEP_BLOCKS) + 8,
                    max_block=max(synth.SWEEP_BLOCKS))
    try:
        dec.prefill(0, prefix)
        ar, _ = dec.decode(0, g.MODE_AR, 0, wl.max_new)
        sched = synth.accept_schedule(mean, wl.max_new)
        dec.prefill(0, prefix)
        dec.set_draft_override(0, ar, sched)
        ss, st = dec.decode(0, g.MODE_SELFSPEC, B, wl.max_new)
        dec.clear_draft_override(0)
        assert list(ss) == list(ar)
        assert st["committed"] == wl.max_new - 1
        # every round but the last accepts min(G_r, B) drafts
        want = np.bincount([min(int(x), B) for x in sched[: st["rounds"] - 1]], minlength=65)
        got = np.array(st["accept_hist"])
        assert np.all(got >= want) and (got - want).sum() == 1
    finally:
        dec.close()


def test_base_page_batch(base):
    g, synth, cfg = base["g"], base["synth"], base["cfg"]
    wl = synth.WORKLOADS["batch"]
    n = wl.n_requests
    plens, news = synth.batch_lengths(n)
    B = wl.block
    dec = g.Decoder(cfg, base["W"], max_ctx=max(plens) + max(news) + B + 8, max_block=B, max_requests=n)
    try:
        prefixes = [synth.make_prefix(cfg, plens[r], seed=synth.REQUEST_PREFIX_SEED0 + r) for r in range(n)]
        refs = []
        for r in range(n):
            dec.prefill(r, prefixes[r])
            out, _ = dec.decode(r, g.MODE_AR, 0, news[r])
            refs.append(list(out))
        for r in range(n):
            dec.prefill(r, prefixes[r])
            dec.set_draft_override(r, refs[r], synth.accept_schedule(wl.forced_mean, news[r],
                                                                     seed=synth.SCHEDULE_SEED + r))
        outs, sts = dec.decode_batch(list(range(n)), g.MODE_SELFSPEC, B, news)
        for r in range(n):
            dec.clear_draft_override(r)
        for r in range(n):
            assert list(outs[r]) == refs[r], r
            assert sts[r]["committed"] == news[r] - 1
        # one batched draft forward (16 x 33 = 528 rows) at the post-prefill
        # states; the request with the shortest prefix against the oracle
        x0s = []
        for r in range(n):
            dec.prefill(r, prefixes[r])
            x0s.append(dec.state(r)[1])
        lg = dec.debug_forward_batch(list(range(n)), g.FWD_DRAFT,
                                     np.array([[x0s[r]] + [0] * B for r in range(n)], np.int32))
        r = int(np.argmin(plens))
        model = oracle.Model(base["W"], cfg)
        st = oracle.prefill(model, prefixes[r].astype(np.float64))
        st.x0 = x0s[r]  # the window starts from the GPU's boundary token
        ref, _, _ = oracle.draft_forward(model, st, B)
        ok, err = close(lg[r], ref)
        assert ok, err
    finally:
        dec.close()
