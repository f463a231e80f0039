"""Decode-level parity of the CUDA path through the C ABI.

* tiny fp32 decoder (2 layers, hidden 256, 4q/2kv heads, vocab 1024, prefix 64):
  logits of AR, draft and verify forwards vs the oracle within 1e-4; AR tokens
  vs the oracle by teacher-forced replay; the KV cache after decoding vs an
  oracle causal prefill of the committed prefix;
* the GPU's self-speculative output equals its own AR-greedy output bit for bit,
  for natural, random-forced and scheduled-forced drafts, and so do the caches;
* host and device error paths (capacity, call order, bad block size).
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.fail("gpu tests need a CUDA device")
    from self_speculative_block_gb300 import build, gocr, synth
    build.build()
    cfg = synth.TINY
    W = synth.make_weights(cfg, seed=synth.WEIGHT_SEED)
    prefix = synth.make_prefix(cfg, 64, seed=synth.PREFIX_SEED)
    dec = gocr.Decoder(cfg, W, max_ctx=64 + 128 + 64 + 8, max_block=64, max_requests=2)
    model = oracle.Model(W, cfg)
    yield dict(g=gocr, synth=synth, cfg=cfg, W=W, prefix=prefix, dec=dec, model=model)
    dec.close()


@pytest.fixture(scope="module")
def ar128(env):
    dec, g = env["dec"], env["g"]
    dec.prefill(0, env["prefix"])
    out, st = dec.decode(0, g.MODE_AR, 0, 128)
    return out, st


def test_prefill_token_and_state(env):
    dec = env["dec"]
    dec.prefill(1, env["prefix"])
    cl, x0 = dec.state(1)
    st = oracle.prefill(env["model"], env["prefix"].astype(np.float64))
    assert cl == 64 and x0 == st.x0


def test_ar_logits_and_kv_match_oracle(env):
    dec, g, model = env["dec"], env["g"], env["model"]
    prefix = env["prefix"].astype(np.float64)
    dec.prefill(0, env["prefix"])
    cl, x0 = dec.state(0)
    lg = dec.debug_forward(0, g.FWD_AR, [x0])
    st = oracle.prefill(model, prefix)
    ref, _, _ = oracle.ar_forward(model, st)
    np.testing.assert_allclose(lg, ref, rtol=0, atol=1e-4)
    k, v = dec.read_kv(0, 1, 0, 64)
    np.testing.assert_allclose(k, st.cache_k[1], rtol=0, atol=1e-4)
    np.testing.assert_allclose(v, st.cache_v[1], rtol=0, atol=1e-4)


@pytest.mark.parametrize("B", [1, 8, 64])
def test_draft_and_verify_logits_match_oracle(env, B):
    dec, g, model = env["dec"], env["g"], env["model"]
    prefix = env["prefix"].astype(np.float64)
    dec.prefill(0, env["prefix"])
    cl, x0 = dec.state(0)
    lg_d = dec.debug_forward(0, g.FWD_DRAFT, [x0] + [0] * B)
    st = oracle.prefill(model, prefix)
    ref_d, kd, vd = oracle.draft_forward(model, st, B)
    np.testing.assert_allclose(lg_d, ref_d, rtol=0, atol=1e-4)
    a0 = int(np.argmax(ref_d[0]))
    drafts = [int(t) for t in np.random.default_rng(B).integers(0, env["cfg"].vocab, B)]
    lg_v = dec.debug_forward(0, g.FWD_VERIFY, [a0] + drafts)
    st.append([k[:1] for k in kd], [v[:1] for v in vd])
    ref_v, _, _ = oracle.verify_forward(model, st, a0, drafts)
    np.testing.assert_allclose(lg_v, ref_v, rtol=0, atol=1e-4)


def test_ar_tokens_match_oracle_by_replay(env, ar128):
    out, st = ar128
    model = env["model"]
    prefix = env["prefix"].astype(np.float64)
    assert st["committed"] == 127 and st["forwards"] == 127 and st["tpf"] == 1.0
    logits, _, _ = oracle.prefill_cache(model, prefix, out[:-1])
    P = prefix.shape[0]
    agree = 0
    for i, t in enumerate(out):
        row = logits[P - 1 + i]
        # the GPU's choice is the oracle's argmax up to the fp32 tolerance
        assert row[t] >= row.max() - 2e-4, (i, t)
        agree += int(np.argmax(row) == t)
    assert agree >= 0.95 * len(out)


@pytest.mark.parametrize("B", [1, 2, 8, 32, 64])
def test_selfspec_equals_gpu_ar_bit_exact(env, ar128, B):
    dec, g = env["dec"], env["g"]
    ar, _ = ar128
    dec.prefill(0, env["prefix"])
    ss, st = dec.decode(0, g.MODE_SELFSPEC, B, 128)
    assert list(ss) == list(ar)
    assert st["committed"] == 127 and st["forwards"] == 2 * st["rounds"]
    hist = st["accept_hist"]
    assert sum(hist) == st["rounds"] and st["accepted_drafts"] == sum(a * n for a, n in enumerate(hist))


def test_kv_after_selfspec_equals_ar_and_oracle_prefill(env, ar128):
    dec, g, model = env["dec"], env["g"], env["model"]
    ar, _ = ar128
    dec.prefill(0, env["prefix"])
    dec.decode(0, g.MODE_AR, 0, 128)
    kv_ar = [dec.read_kv(0, l, 0, 64 + 127) for l in range(env["cfg"].n_layers)]
    dec.prefill(0, env["prefix"])
    dec.decode(0, g.MODE_SELFSPEC, 8, 128)
    cl, x0 = dec.state(0)
    assert cl == 64 + 127 and x0 == ar[-1]
    _, K, V = oracle.prefill_cache(model, env["prefix"].astype(np.float64), ar[:-1])
    for l in range(env["cfg"].n_layers):
        k, v = dec.read_kv(0, l, 0, 64 + 127)
        assert np.array_equal(k, kv_ar[l][0]) and np.array_equal(v, kv_ar[l][1])
        np.testing.assert_allclose(k, K[l], rtol=0, atol=1e-4)
        np.testing.assert_allclose(v, V[l], rtol=0, atol=1e-4)


@pytest.mark.parametrize("B,mean", [(8, 3.0), (32, 9.0), (64, 19.0)])
def test_forced_acceptance_follows_schedule(env, ar128, B, mean):
    dec, g, synth = env["dec"], env["g"], env["synth"]
    ar, _ = ar128
    sched = synth.accept_schedule(mean, 128, seed=synth.SCHEDULE_SEED)
    dec.prefill(0, env["prefix"])
    dec.set_draft_override(0, ar, sched)
    try:
        ss, st = dec.decode(0, g.MODE_SELFSPEC, B, 128)
    finally:
        dec.clear_draft_override(0)
    assert list(ss) == list(ar)
    # every round but the last accepts exactly min(G_r, B) drafts
    want = np.bincount([min(int(x), B) for x in sched[: st["rounds"] - 1]], minlength=65)
    got = np.array(st["accept_hist"])
    assert np.all(got >= want) and (got - want).sum() == 1


def test_always_wrong_drafts_commit_two_per_round(env, ar128):
    dec, g = env["dec"], env["g"]
    ar, _ = ar128
    dec.prefill(0, env["prefix"])
    dec.set_draft_override(0, ar, [0] * 128)
    try:
        ss, st = dec.decode(0, g.MODE_SELFSPEC, 8, 128)
    finally:
        dec.clear_draft_override(0)
    assert list(ss) == list(ar)
    assert st["rounds"] == 64 and st["accept_hist"][0] >= st["rounds"] - 1


def test_max_new_truncation(env, ar128):
    dec, g = env["dec"], env["g"]
    ar, _ = ar128
    for n in (2, 3, 11):
        dec.prefill(0, env["prefix"])
        ss, st = dec.decode(0, g.MODE_SELFSPEC, 8, n)
        assert list(ss) == list(ar[:n])


def test_capacity_and_call_order_errors(env):
    dec, g = env["dec"], env["g"]
    dec.prefill(0, env["prefix"])
    cap = dec.max_ctx
    # exactly at capacity works: P + max_new + B + 2 == cap
    max_new = cap - 64 - 8 - 2
    out, _ = dec.decode(0, g.MODE_SELFSPEC, 8, max_new)
    dec.prefill(0, env["prefix"])
    with pytest.raises(g.GocrError) as e:
        dec.decode(0, g.MODE_SELFSPEC, 8, max_new + 1)
    assert e.value.code == -2
    with pytest.raises(g.GocrError) as e:
        dec.decode(0, g.MODE_SELFSPEC, 65, 10)
    assert e.value.code == -2
    with pytest.raises(g.GocrError) as e:
        dec.prefill(0, np.zeros((cap, env["cfg"].hidden), np.float32))
    assert e.value.code == -2


def test_decode_before_prefill_is_a_state_error(env):
    from self_speculative_block_gb300 import gocr
    d2 = gocr.Decoder(env["cfg"], env["W"], max_ctx=128, max_block=8)
    try:
        with pytest.raises(gocr.GocrError) as e:
            d2.decode(0, gocr.MODE_AR, 0, 4)
        assert e.value.code == -7
    finally:
        d2.close()


def test_eos_truncation(env, ar128):
    from self_speculative_block_gb300 import gocr
    ar, _ = ar128
    eos = int(ar[20])
    want = list(ar[: list(ar).index(eos) + 1])
    d2 = gocr.Decoder(env["cfg"], env["W"], max_ctx=256, max_block=8, eos_id=eos)
    try:
        for mode, B in ((gocr.MODE_AR, 0), (gocr.MODE_SELFSPEC, 8)):
            d2.prefill(0, env["prefix"])
            out, st = d2.decode(0, mode, B, 128)
            assert list(out[: len(want)]) == want
    finally:
        d2.close()
