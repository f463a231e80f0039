"""The persistent decode forward (one kernel per forward, one CTA per SM)
against the per-operation forward (one kernel per GEMM and attention), on a
handle with the mma.sync attention, whose tile code the persistent kernel
shares.

Both run the same reductions in the same order, so every result must be
bit-identical: draft, verify and AR logits, the KV cache rows the forward
writes, AR and self-speculative token streams, forced acceptance and the
batched ragged round.  The per-operation forward is itself checked against
the fp64 oracle in test_gpu_bf16 and test_gpu_ops.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def small():
    if not torch.cuda.is_available():
        pytest.fail("gpu tests need a CUDA device")
    import os
    from self_speculative_block_gb300 import build, gocr, synth
    build.build()
    cfg = synth.ModelConfig(n_layers=2, hidden=512, n_q_heads=6, n_kv_heads=2, head_dim=128, ffn=1024,
                            vocab=2048, dtype=synth.BF16)
    W = synth.make_weights(cfg, seed=31)
    prefix = synth.make_prefix(cfg, 150, seed=32)
    # the persistent forward shares the mma.sync attention's tile code (the default)
    assert os.environ.get("GOCR_ATTN") is None
    dec = gocr.Decoder(cfg, W, max_ctx=150 + 200 + 64 + 8, max_block=64, max_requests=4)
    assert dec.attention_kind() == gocr.ATTN_MMA_SYNC
    assert dec.forward_path() == gocr.FORWARD_OPS
    yield dict(g=gocr, synth=synth, cfg=cfg, prefix=prefix, dec=dec)
    dec.close()


def both_paths(dec, g, fn):
    """fn() under the per-operation forward, then under the persistent one;
    checks that the persistent kernel ran (and only in the second call)."""
    dec.set_forward_path(g.FORWARD_OPS)
    a = fn()
    assert dec.persistent_forwards() == 0
    dec.set_forward_path(g.FORWARD_PERSISTENT)
    try:
        b = fn()
        assert dec.persistent_forwards() > 0
    finally:
        dec.set_forward_path(g.FORWARD_OPS)
    return a, b


def bits(x):
    return np.ascontiguousarray(x).view(np.uint32)


@pytest.mark.parametrize("B", [1, 7, 32, 64])
def test_debug_forwards_bit_identical(small, B):
    dec, g, cfg = small["dec"], small["g"], small["cfg"]

    def run():
        dec.prefill(0, small["prefix"])
        cl, x0 = dec.state(0)
        lg_d = dec.debug_forward(0, g.FWD_DRAFT, [x0] + [0] * B)
        kd, vd = dec.read_kv(0, cfg.n_layers - 1, cl, B + 1)
        a0 = int(np.argmax(lg_d[0]))
        drafts = [int(t) for t in np.argmax(lg_d[1:], -1)]
        lg_v = dec.debug_forward(0, g.FWD_VERIFY, [a0] + drafts)
        kv, vv = dec.read_kv(0, 0, cl + 1, B + 1)
        lg_a = dec.debug_forward(0, g.FWD_AR, [x0])
        n_pers = dec.persistent_forwards()
        assert n_pers == (1 if dec.forward_path() == g.FORWARD_PERSISTENT else 0)
        return lg_d, kd, vd, lg_v, kv, vv, lg_a

    ops, pers = both_paths(dec, g, run)
    for name, a, b in zip(("draft", "draft K", "draft V", "verify", "verify K", "verify V", "ar"), ops, pers):
        assert np.array_equal(bits(a), bits(b)), name


def test_decode_streams_bit_identical(small):
    dec, g = small["dec"], small["g"]

    def run():
        dec.prefill(0, small["prefix"])
        ar, _ = dec.decode(0, g.MODE_AR, 0, 150)
        dec.prefill(0, small["prefix"])
        ss, st = dec.decode(0, g.MODE_SELFSPEC, 16, 150)
        if dec.forward_path() == g.FORWARD_PERSISTENT:
            assert dec.persistent_forwards() == st["forwards"] == 2 * st["rounds"]
        k, v = dec.read_kv(0, 1, 0, 150 + 149)
        return list(ar), list(ss), k, v, st["rounds"]

    ops, pers = both_paths(dec, g, run)
    assert ops[0] == pers[0]
    assert ops[1] == pers[1] == pers[0]
    assert np.array_equal(bits(ops[2]), bits(pers[2]))
    assert np.array_equal(bits(ops[3]), bits(pers[3]))
    assert ops[4] == pers[4]


def test_forced_acceptance_bit_identical(small):
    dec, g, synth = small["dec"], small["g"], small["synth"]
    dec.prefill(0, small["prefix"])
    ref, _ = dec.decode(0, g.MODE_AR, 0, 180)
    sched = synth.accept_schedule(9, 180, seed=7)

    def run():
        dec.prefill(0, small["prefix"])
        dec.set_draft_override(0, ref, sched)
        try:
            out, st = dec.decode(0, g.MODE_SELFSPEC, 32, 180)
        finally:
            dec.clear_draft_override(0)
        return list(out), st["rounds"], st["accepted_drafts"]

    ops, pers = both_paths(dec, g, run)
    assert ops == pers
    assert pers[0] == list(ref)


def test_batched_ragged_bit_identical(small):
    dec, g, synth, cfg = small["dec"], small["g"], small["synth"], small["cfg"]
    lens = [40, 150, 77]
    news = [60, 35, 100]
    prefixes = [synth.make_prefix(cfg, n, seed=2000 + r) for r, n in enumerate(lens)]

    def run():
        res = []
        for mode, B in ((g.MODE_SELFSPEC, 8), (g.MODE_AR, 0), (g.MODE_SELFSPEC, 32)):
            for r in range(3):
                dec.prefill(r, prefixes[r])
            outs, _ = dec.decode_batch([0, 1, 2], mode, B, news)
            res.append([list(o) for o in outs])
        return res

    ops, pers = both_paths(dec, g, run)
    assert ops == pers
    assert pers[0] == pers[1] == pers[2]


def test_persistent_forward_needs_the_mma_sync_attention(small, monkeypatch):
    g, synth, cfg = small["g"], small["synth"], small["cfg"]
    W = synth.make_weights(cfg, seed=31)
    monkeypatch.setenv("GOCR_ATTN", "tc")
    dec = g.Decoder(cfg, W, max_ctx=256, max_block=8)
    monkeypatch.delenv("GOCR_ATTN")
    try:
        assert dec.attention_kind() == g.ATTN_TCGEN05
        with pytest.raises(g.GocrError):
            dec.set_forward_path(g.FORWARD_PERSISTENT)
        assert dec.forward_path() == g.FORWARD_OPS
    finally:
        dec.close()


def test_attention_kernel_follows_chunks_per_rank(small, monkeypatch):
    """A handle whose ranks average at least four chunks at full capacity
    (here 16 requests: 8 ranks over 64 chunks) takes the tcgen05 attention;
    GOCR_ATTN=mma overrides, and one request at the same capacity (48 ranks)
    keeps mma.sync."""
    g, synth, cfg = small["g"], small["synth"], small["cfg"]
    W = synth.make_weights(cfg, seed=31)
    monkeypatch.delenv("GOCR_ATTN", raising=False)
    for env, n_req, want in ((None, 16, g.ATTN_TCGEN05), ("mma", 16, g.ATTN_MMA_SYNC), (None, 1, g.ATTN_MMA_SYNC)):
        if env:
            monkeypatch.setenv("GOCR_ATTN", env)
        dec = g.Decoder(cfg, W, max_ctx=2048, max_block=8, max_requests=n_req)
        monkeypatch.delenv("GOCR_ATTN", raising=False)
        try:
            assert dec.attention_kind() == want, (env, n_req)
        finally:
            dec.close()


def test_option_round_trip(small):
    dec, g = small["dec"], small["g"]
    dec.set_forward_path(g.FORWARD_PERSISTENT)
    assert dec.forward_path() == g.FORWARD_PERSISTENT
    dec.set_forward_path(g.FORWARD_OPS)
    assert dec.forward_path() == g.FORWARD_OPS
    with pytest.raises(g.GocrError):
        dec.set_forward_path(7)
