"""Direct block-diffusion decoding and refined-draft rounds through the C ABI
(gocr_decode_ex), against the oracle (oracle/diffusion.py) and the GPU's own
AR path.

Sources: GravityOCR review §2 "Block Diffusion" and Appendix B.1 "Direct
Block-Diffusion Decoding" (threshold rule, cache-write forward, EOS cut);
Appendix D "Draft Schedule" (refined drafts); Appendix B.3 (the verify step
keeps the output equal to AR greedy).

A threshold decision and an argmax are floating-point decisions of integers:
the GPU and the oracle agree on them wherever the oracle's own margin exceeds
what the arithmetic can move (fp32: 2e-4 in a logit, 1e-3 relative in a
confidence).  fp32 token streams are compared up to the first block whose
decisions are closer than that (the thresholds here decide every fp32 stream
with margin); the bf16 stream is replayed in the oracle slot by slot.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

FP32_TOL = dict(logit=2e-4, conf=1e-3)


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("gpu tests need a CUDA device")
    from self_speculative_block_gb300 import build, gocr, synth
    build.build()
    return gocr, synth


def first_ambiguous_block(logs, tau, tol):
    """Index of the first block with a decision within tol of flipping, or len(logs)."""
    for b, g in enumerate(logs):
        B = len(g.block)
        masked = list(range(B))
        for s in g.steps:
            conf = s.conf
            for r in masked:
                if s.margin[r] <= tol["logit"]:
                    return b
                if abs(conf[r] - tau) <= tol["conf"] * max(tau, conf[r]):
                    return b
            if not any(conf[r] >= tau for r in masked) and len(masked) > 1:
                top = sorted((conf[r] for r in masked), reverse=True)
                if top[0] - top[1] <= tol["conf"] * top[0]:
                    return b
            masked = [r for r in masked if r not in s.fixed]
    return len(logs)


def tiny_sharp(synth):
    """The tiny fp32 decoder with a larger init, so that confidences spread
    over (0, 1) and a threshold near 0.5 both passes and fails slots."""
    cfg = synth.TINY
    return cfg, synth.make_weights(cfg, seed=0, std=0.3)


def _stats_from_logs(logs):
    steps = [len(g.steps) for g in logs]
    hist = np.bincount(steps, minlength=65)
    return dict(rounds=len(logs), forwards=sum(steps) + sum(1 for g in logs if g.cache_write),
                committed=sum(len(g.committed) for g in logs), hist=hist)


@pytest.mark.parametrize("B", [4, 8])
@pytest.mark.parametrize("tau", [0.0, 0.35, 0.6, 0.9, 2.0])
def test_diffusion_matches_oracle_fp32(lib, B, tau):
    g, synth = lib
    cfg, W = tiny_sharp(synth)
    prefix = synth.make_prefix(cfg, 16, seed=1)
    max_new = 41
    ref, logs = oracle.diffusion_decode(oracle.Model(W, cfg), prefix.astype(np.float64), B, tau, max_new)
    k = first_ambiguous_block(logs, tau, FP32_TOL)
    dec = g.Decoder(cfg, W, max_ctx=16 + max_new + 2 * B + 8, max_block=B)
    try:
        dec.prefill(0, prefix)
        outs, sts = dec.decode_ex([0], g.MODE_DIFFUSION, B, [max_new], tau=tau)
    finally:
        dec.close()
    got = list(outs[0])
    n_cmp = 1 + sum(len(g_.committed) for g_ in logs[:k])
    assert got[:n_cmp] == ref[:n_cmp], (k, len(logs))
    if k == len(logs):
        want = _stats_from_logs(logs)
        st = sts[0]
        assert (st["rounds"], st["forwards"], st["committed"]) == (want["rounds"], want["forwards"],
                                                                   want["committed"])
        assert np.array_equal(np.array(st["accept_hist"]), want["hist"])
    # thresholds 0 and 2 decide by argmax and confidence order only: the whole stream must be unambiguous
    if tau in (0.0, 2.0):
        assert k == len(logs), (tau, k)


def test_diffusion_threshold_mixes_passes_and_fallbacks(lib):
    """At least one fp32 case above fixes several slots in one step and also
    falls back to a single slot in another, with the whole stream decided."""
    g, synth = lib
    cfg, W = tiny_sharp(synth)
    prefix = synth.make_prefix(cfg, 16, seed=1)
    model = oracle.Model(W, cfg)
    seen = False
    for tau in (0.35, 0.6, 0.9):
        _, logs = oracle.diffusion_decode(model, prefix.astype(np.float64), 8, tau, 41)
        if first_ambiguous_block(logs, tau, FP32_TOL) < len(logs):
            continue
        multi = any(len(s.fixed) > 1 for g_ in logs for s in g_.steps)
        single = any(len(s.fixed) == 1 and max(s.conf[r] for r in s.fixed) < tau for g_ in logs for s in g_.steps)
        seen |= multi and single
    assert seen


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_diffusion_block_one_is_ar_and_threshold_zero_is_one_shot(lib, dt):
    g, synth = lib
    if dt == "f32":
        cfg, W = synth.TINY, synth.make_weights(synth.TINY, seed=0)
    else:
        cfg = synth.ModelConfig(n_layers=2, hidden=512, n_q_heads=6, n_kv_heads=2, head_dim=128, ffn=1024,
                                vocab=2048, dtype=synth.BF16)
        W = synth.make_weights(cfg, seed=21)
    prefix = synth.make_prefix(cfg, 40, seed=22)
    max_new, B = 33, 8
    dec = g.Decoder(cfg, W, max_ctx=40 + max_new + 2 * B + 8, max_block=B)
    try:
        dec.prefill(0, prefix)
        ar, _ = dec.decode(0, g.MODE_AR, 0, max_new)
        for tau in (0.0, 0.5, 2.0):
            dec.prefill(0, prefix)
            outs, sts = dec.decode_ex([0], g.MODE_DIFFUSION, 1, [max_new], tau=tau)
            assert list(outs[0]) == list(ar), tau
            assert sts[0]["forwards"] == 2 * sts[0]["rounds"] - 1
        # threshold 0: one denoising step per block; the first block is the
        # one-shot draft forward's rows 0..B-1
        dec.prefill(0, prefix)
        x0 = dec.state(0)[1]
        lg = dec.debug_forward(0, g.FWD_DRAFT, [x0] + [0] * B)
        dec.prefill(0, prefix)
        outs, sts = dec.decode_ex([0], g.MODE_DIFFUSION, B, [max_new], tau=0.0)
        assert list(outs[0][1:1 + B]) == [int(t) for t in np.argmax(lg[:B], axis=-1)]
        assert sts[0]["accept_hist"][1] == sts[0]["rounds"]
        # a threshold no confidence reaches: one slot per step, B steps per block
        dec.prefill(0, prefix)
        outs, sts = dec.decode_ex([0], g.MODE_DIFFUSION, B, [max_new], tau=2.0)
        assert sts[0]["accept_hist"][B] == sts[0]["rounds"] == 4
        assert sts[0]["forwards"] == 4 * B + 3
    finally:
        dec.close()


def test_diffusion_bf16_against_oracle(lib):
    """bf16, threshold 0 (one denoising step per block, so only argmaxes
    decide): the GPU's blocks are replayed in the oracle, which takes the GPU's
    committed tokens as its state (cache write included); every slot whose
    oracle top-two margin exceeds twice the logit tolerance must carry the
    oracle's argmax, and most slots must be that clear."""
    g, synth = lib
    cfg = synth.ModelConfig(n_layers=2, hidden=512, n_q_heads=6, n_kv_heads=2, head_dim=128, ffn=1024,
                            vocab=2048, dtype=synth.BF16)
    W = synth.make_weights(cfg, seed=21, std=0.1)
    prefix = synth.make_prefix(cfg, 40, seed=22)
    max_new, B = 49, 8
    dec = g.Decoder(cfg, W, max_ctx=40 + max_new + 2 * B + 8, max_block=B)
    try:
        dec.prefill(0, prefix)
        x0 = dec.state(0)[1]
        outs, sts = dec.decode_ex([0], g.MODE_DIFFUSION, B, [max_new], tau=0.0)
    finally:
        dec.close()
    got = [int(t) for t in outs[0]]
    assert got[0] == x0 and sts[0]["accept_hist"][1] == sts[0]["rounds"]
    model = oracle.Model(W, cfg)
    st = oracle.prefill(model, prefix.astype(np.float64))
    st.x0, st.out = x0, [x0]
    checked = clear = 0
    pos = 1
    while pos < len(got):
        blk = got[pos:pos + B]
        lg, _, _ = oracle.window_forward(model, st, [-1] * B)
        for r, t in enumerate(blk):
            checked += 1
            tol = 2 * (3e-2 + 2e-2 * float(np.abs(lg[r]).max()))
            if oracle.top2_margin(lg[r]) > tol:
                clear += 1
                assert int(np.argmax(lg[r])) == t, (pos + r, int(np.argmax(lg[r])), t)
        if len(blk) < B:
            break
        p = st.p
        rows = oracle.token_rows(model, [st.x0] + blk)
        ps = np.arange(p, p + B + 1)
        _, k, v = oracle.forward(model, rows, ps, st.cache_k, st.cache_v, oracle.causal_mask(ps, p + B + 1))
        st.append(k, v)
        st.truncate(p + B)
        st.x0 = blk[-1]
        pos += B
    assert checked == max_new - 1 and clear >= checked // 2, (clear, checked)
    print(f"bf16 direct diffusion: {clear} of {checked} slots decided with margin, all equal to the oracle")


def test_diffusion_eos_cut(lib):
    g, synth = lib
    cfg, W = tiny_sharp(synth)
    prefix = synth.make_prefix(cfg, 16, seed=1)
    B, tau, max_new = 4, 2.0, 41
    ref, logs = oracle.diffusion_decode(oracle.Model(W, cfg), prefix.astype(np.float64), B, tau, max_new)
    # an EOS token whose first appearance sits inside a block
    first = {}
    for i, t in enumerate(ref[1:], start=1):
        first.setdefault(t, i)
    eos = next(t for t, i in sorted(first.items(), key=lambda x: x[1]) if (i - 1) % B not in (B - 1,) and i > B)
    ref_e, _ = oracle.diffusion_decode(oracle.Model(W, cfg), prefix.astype(np.float64), B, tau, max_new, eos_id=eos)
    dec = g.Decoder(cfg, W, max_ctx=16 + max_new + 2 * B + 8, max_block=B, eos_id=eos)
    try:
        dec.prefill(0, prefix)
        outs, sts = dec.decode_ex([0], g.MODE_DIFFUSION, B, [max_new], tau=tau)
    finally:
        dec.close()
    n = len(ref_e)
    assert ref_e[-1] == eos and n < max_new
    assert list(outs[0][:n]) == ref_e
    assert sts[0]["committed"] == n - 1


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_refined_rounds_equal_ar(lib, dt):
    g, synth = lib
    if dt == "f32":
        cfg, W = tiny_sharp(synth)
    else:
        cfg = synth.ModelConfig(n_layers=2, hidden=512, n_q_heads=6, n_kv_heads=2, head_dim=128, ffn=1024,
                                vocab=2048, dtype=synth.BF16)
        W = synth.make_weights(cfg, seed=21)
    prefix = synth.make_prefix(cfg, 40, seed=22)
    max_new, B = 60, 8
    dec = g.Decoder(cfg, W, max_ctx=40 + max_new + B + 8, max_block=B)
    try:
        dec.prefill(0, prefix)
        ar, _ = dec.decode(0, g.MODE_AR, 0, max_new)
        dec.prefill(0, prefix)
        ss, st_ss = dec.decode(0, g.MODE_SELFSPEC, B, max_new)
        for tau, steps in ((0.5, 1), (2.0, 1), (0.5, 2), (2.0, 4), (0.0, 3), (0.9, 8)):
            dec.prefill(0, prefix)
            outs, sts = dec.decode_ex([0], g.MODE_REFINED, B, [max_new], tau=tau, draft_steps=steps)
            assert list(outs[0]) == list(ar), (tau, steps)
            st = sts[0]
            assert st["committed"] == max_new - 1
            if steps == 1:  # the one-shot round, stats included
                for key in ("rounds", "forwards", "committed", "accepted_drafts", "accept_hist"):
                    assert st[key] == st_ss[key], key
            if tau > 1.0:  # one slot per draft step: every round runs all its steps
                assert st["forwards"] == (min(steps, B) + 1) * st["rounds"]
    finally:
        dec.close()


def test_refined_rounds_match_oracle_fp32(lib):
    """Accepted drafts per round of the fp32 GPU path equal the oracle's
    refined rounds (the rounds are decided with margin)."""
    g, synth = lib
    cfg, W = tiny_sharp(synth)
    prefix = synth.make_prefix(cfg, 16, seed=1)
    B, max_new = 6, 40
    model = oracle.Model(W, cfg)
    dec = g.Decoder(cfg, W, max_ctx=16 + max_new + B + 8, max_block=B)
    try:
        compared = 0
        for tau, steps in ((0.6, 2), (2.0, 3), (0.35, 4)):
            out, logs = oracle.refined_decode(model, prefix.astype(np.float64), B, tau, steps, max_new)
            ok = True
            for lg in logs:
                for s in lg.steps:
                    if min(s.margin) <= FP32_TOL["logit"]:
                        ok = False
                    masked_conf = s.conf
                    if any(abs(c - tau) <= FP32_TOL["conf"] * max(c, tau) for c in masked_conf):
                        ok = False
            dec.prefill(0, prefix)
            outs, sts = dec.decode_ex([0], g.MODE_REFINED, B, [max_new], tau=tau, draft_steps=steps)
            assert list(outs[0]) == out
            if ok:
                want = oracle.refined_stats(logs)
                assert (sts[0]["rounds"], sts[0]["forwards"], sts[0]["accepted_drafts"]) == (
                    want["rounds"], want["forwards"], want["accepted_drafts"]), (tau, steps)
                compared += 1
        assert compared >= 1
    finally:
        dec.close()


def test_diffusion_batched_equals_single(lib):
    g, synth = lib
    cfg = synth.ModelConfig(n_layers=2, hidden=512, n_q_heads=6, n_kv_heads=2, head_dim=128, ffn=1024,
                            vocab=2048, dtype=synth.BF16)
    W = synth.make_weights(cfg, seed=21)
    lens, news = [30, 71, 52], [25, 40, 17]
    B = 8
    dec = g.Decoder(cfg, W, max_ctx=71 + 40 + 2 * B + 8, max_block=B, max_requests=3)
    try:
        prefixes = [synth.make_prefix(cfg, n, seed=1000 + r) for r, n in enumerate(lens)]
        for mode, tau, steps in ((g.MODE_DIFFUSION, 0.0, 1), (g.MODE_DIFFUSION, 2.0, 1), (g.MODE_REFINED, 2.0, 3)):
            single = []
            for r in range(3):
                dec.prefill(r, prefixes[r])
                o, _ = dec.decode_ex([r], mode, B, [news[r]], tau=tau, draft_steps=steps)
                single.append(list(o[0]))
            for r in range(3):
                dec.prefill(r, prefixes[r])
            outs, _ = dec.decode_ex([0, 1, 2], mode, B, news, tau=tau, draft_steps=steps)
            assert [list(o) for o in outs] == single, (mode, tau)
    finally:
        dec.close()
