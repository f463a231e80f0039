"""The LM-head argmax's tie-break and the NaN error path on the GPU.

* Lowest index on ties: an LM head with two identical rows gives two bitwise
  equal logits; when they are the row maximum, the committed token is the
  lower index (the argmax reading shared with the oracle).  Checked for the
  GEMM paths (bf16 tcgen05: the streaming LM-head kernel of decode shapes and,
  with GOCR_LM_WAVES=1, the tile-CTA kernel that larger forwards use; fp32 CUDA
  cores), with the tied rows in one 128-row weight tile and in two tiles.
* NaN logits are a device error: a NaN placed in a weight on the host comes
  back as GOCR_EDEVICE from the call whose forward met it, with no fault, and
  other handles keep working.
"""
import copy

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("gpu tests need a CUDA device")
    from self_speculative_block_gb300 import build, gocr, synth
    build.build()
    return gocr, synth


def _cfg(synth, dt):
    if dt.startswith("bf16"):
        # 160 LM-head tiles: the split rule gives the LM head one K split, so at
        # decode shapes it runs on the streaming kernel (GOCR_LM_WAVES=1: tile CTAs)
        return synth.ModelConfig(n_layers=2, hidden=512, n_q_heads=6, n_kv_heads=2, head_dim=128, ffn=1024,
                                 vocab=20480, dtype=synth.BF16)
    return synth.TINY


def _first_token(g, cfg, W, prefix):
    dec = g.Decoder(cfg, W, max_ctx=prefix.shape[0] + 16, max_block=4)
    try:
        dec.prefill(0, prefix)
        t0 = dec.state(0)[1]
        out, _ = dec.decode(0, g.MODE_AR, 0, 3)
        lg = dec.debug_forward(0, g.FWD_AR, [int(out[-1])])
        return t0, list(out), lg[0]
    finally:
        dec.close()


def _lm_kernel(monkeypatch, dt):
    if dt == "bf16-waves":
        monkeypatch.setenv("GOCR_LM_WAVES", "1")
    else:
        monkeypatch.delenv("GOCR_LM_WAVES", raising=False)


@pytest.mark.parametrize("dt", ["bf16", "bf16-waves", "f32"])
def test_argmax_ties_go_to_the_lowest_index(lib, monkeypatch, dt):
    g, synth = lib
    _lm_kernel(monkeypatch, dt)
    cfg = _cfg(synth, dt)
    W = synth.make_weights(cfg, seed=31)
    for seed in range(40, 60):
        prefix = synth.make_prefix(cfg, 24, seed=seed)
        t0, _, _ = _first_token(g, cfg, W, prefix)
        if t0 >= 129 and t0 % 128 != 0:
            break
    else:
        pytest.fail("no prefix gave a first token past the first weight tile")
    # j1 in the same 128-row tile as t0, j2 in another tile, both lower indices
    for j in (t0 - 1, t0 % 128):
        W2 = copy.copy(W)
        W2["lm_head"] = W["lm_head"].copy()
        W2["lm_head"][j] = W["lm_head"][t0]
        t0b, outb, lgb = _first_token(g, cfg, W2, prefix)
        assert t0b == j, (dt, j, t0, t0b)
        # identical weight rows give bitwise equal logits in every forward
        assert lgb[j].view(np.uint32) == lgb[t0].view(np.uint32)


@pytest.mark.parametrize("dt", ["bf16", "bf16-waves", "f32"])
@pytest.mark.parametrize("where", ["lm_head", "wo"])
def test_nan_weight_is_a_device_error(lib, monkeypatch, dt, where):
    g, synth = lib
    _lm_kernel(monkeypatch, dt)
    cfg = _cfg(synth, dt)
    W = synth.make_weights(cfg, seed=33)
    prefix = synth.make_prefix(cfg, 24, seed=3)
    Wn = copy.copy(W)
    if where == "lm_head":
        Wn["lm_head"] = W["lm_head"].copy()
        Wn["lm_head"][5, 7] = np.nan
    else:
        Wn["layers"] = [dict(lw) for lw in W["layers"]]
        Wn["layers"][1]["wo"] = W["layers"][1]["wo"].copy()
        Wn["layers"][1]["wo"][3, 11] = np.nan
    dec = g.Decoder(cfg, Wn, max_ctx=64, max_block=4)
    try:
        with pytest.raises(g.GocrError) as ei:
            dec.prefill(0, prefix)
        assert ei.value.code == -4 and "NaN" in str(ei.value)
        # the failed prefill leaves the slot unprefilled: decode is a call-order error
        with pytest.raises(g.GocrError) as ei:
            dec.decode(0, g.MODE_AR, 0, 4)
        assert ei.value.code == -7
    finally:
        dec.close()
    # the context is intact: a clean handle decodes
    t0, out, _ = _first_token(g, cfg, W, prefix)
    assert len(out) == 3 and out[0] == t0


def test_streaming_lm_head_above_64_rows_equals_tile_ctas(lib, monkeypatch):
    """A 65-row draft forward (B = 64) runs its LM head on the streaming kernel
    with one CTA per SM (above 64 rows); its logits and committed argmax are
    bitwise those of the tile-CTA kernel (GOCR_LM_WAVES=1)."""
    g, synth = lib
    cfg = _cfg(synth, "bf16")
    W = synth.make_weights(cfg, seed=35)
    prefix = synth.make_prefix(cfg, 40, seed=5)
    res = {}
    for kind in ("bf16", "bf16-waves"):
        _lm_kernel(monkeypatch, kind)
        dec = g.Decoder(cfg, W, max_ctx=prefix.shape[0] + 160, max_block=64)
        try:
            dec.prefill(0, prefix)
            x0 = dec.state(0)[1]
            lg = dec.debug_forward(0, g.FWD_DRAFT, [x0] + [0] * 64)
            out, _ = dec.decode(0, g.MODE_SELFSPEC, 64, 70)
            res[kind] = (lg, list(out))
        finally:
            dec.close()
    assert res["bf16"][0].shape == (65, cfg.vocab)
    assert np.array_equal(res["bf16"][0].view(np.uint32), res["bf16-waves"][0].view(np.uint32))
    assert res["bf16"][1] == res["bf16-waves"][1]
