"""Pins for the oracle's components against closed forms, library routines and
brute-force constructions (never against a retyped copy of the same formula).
"""
import math

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

import oracle
from self_speculative_block_gb300 import synth

RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_constant_vector_closed_form():
    # x = c * ones: mean(x^2) = c^2, so y = c / sqrt(c^2 + eps) * g
    for c in (-3.0, -0.5, 0.25, 7.0):
        x = np.full((1, 64), c)
        g = RNG.uniform(0.5, 2.0, size=64)
        eps = 1e-6
        y = oracle.rmsnorm(x, g, eps)
        np.testing.assert_allclose(y[0], c / math.sqrt(c * c + eps) * g, rtol=0, atol=1e-15)


def test_rmsnorm_matches_torch_library():
    x = RNG.standard_normal((7, 96))
    g = RNG.uniform(0.5, 1.5, size=96)
    ref = F.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.rmsnorm(x, g, 1e-6), ref, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- RoPE

def _rope_complex(x, pos, theta):
    """Independent statement: pair (x_i, x_{i+d/2}) as the complex number
    x_i + 1j x_{i+d/2} and multiply by exp(1j * pos * theta^(-2i/d))."""
    n, H, d = x.shape
    half = d // 2
    z = x[..., :half] + 1j * x[..., half:]
    w = np.array([theta ** (-2.0 * i / d) for i in range(half)])
    rot = np.exp(1j * np.outer(pos, w))[:, None, :]
    zr = z * rot
    return np.concatenate([zr.real, zr.imag], axis=-1)


def test_rope_equals_complex_rotation():
    x = RNG.standard_normal((5, 3, 16))
    pos = np.array([0, 1, 7, 100, 4095])
    np.testing.assert_allclose(oracle.rope(x, pos, 10000.0), _rope_complex(x, pos, 10000.0),
                               rtol=0, atol=1e-12)


def test_rope_position_zero_is_identity_and_norm_preserving():
    x = RNG.standard_normal((4, 2, 32))
    np.testing.assert_array_equal(oracle.rope(x, np.zeros(4, int), 1e4), x)
    y = oracle.rope(x, np.array([3, 17, 250, 2049]), 1e4)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_scores_depend_only_on_relative_position():
    q = RNG.standard_normal((1, 1, 64))
    k = RNG.standard_normal((1, 1, 64))
    base = None
    for shift in (0, 5, 300, 2000):
        m, n = 40 + shift, 13 + shift
        s = float(np.sum(oracle.rope(q, np.array([m]), 1e4) * oracle.rope(k, np.array([n]), 1e4)))
        if base is None:
            base = s
        assert abs(s - base) < 1e-10


def test_rope_two_dims_is_a_plane_rotation():
    # d = 2: one pair, frequency 1, angle = pos
    x = np.array([[[1.0, 0.0]]])
    for p in (1, 2, 5):
        y = oracle.rope(x, np.array([p]), 1e4)[0, 0]
        np.testing.assert_allclose(y, [math.cos(p), math.sin(p)], atol=1e-15)


# ---------------------------------------------------------------- SiLU, softmax, argmax

def test_silu_matches_logistic():
    z = np.linspace(-30, 30, 301)
    np.testing.assert_allclose(oracle.silu(z), z * scipy.special.expit(z), rtol=1e-13, atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0


def test_softmax_masked_rows_sum_to_one_and_zero_masked():
    s = RNG.standard_normal((6, 9))
    allowed = RNG.uniform(size=(6, 9)) < 0.6
    allowed[:, 0] = True
    p = oracle.softmax_masked(s, allowed)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-15)
    assert np.all(p[~allowed] == 0)
    full = oracle.softmax_masked(s, np.ones_like(allowed))
    np.testing.assert_allclose(full, scipy.special.softmax(s, axis=-1), rtol=1e-13)


def test_argmax_lowest_index_on_ties_and_nan_error():
    assert list(oracle.argmax_lowest(np.array([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 5.0, 5.0]]))) == [1, 0]
    with pytest.raises(FloatingPointError):
        oracle.argmax_lowest(np.array([[1.0, np.nan]]))


# ---------------------------------------------------------------- masks (brute force)

def _allowed_set_draft(p, B):
    """From the rule text: the boundary row at position p reads the cache and
    itself; each [M] row reads the cache, x0 and every [M] of the window."""
    s = set()
    for r in range(B + 1):
        for key in range(p + B + 1):
            if r == 0:
                if key <= p:
                    s.add((r, key))
            else:
                s.add((r, key))
    return s


def _allowed_set_causal(positions, n_keys):
    return {(r, key) for r, t in enumerate(positions) for key in range(n_keys) if key <= t}


@pytest.mark.parametrize("p", [0, 1, 5])
@pytest.mark.parametrize("B", [1, 2, 4])
def test_masks_brute_force(p, B):
    dm = oracle.draft_mask(p, B)
    assert {tuple(ix) for ix in np.argwhere(dm)} == _allowed_set_draft(p, B)
    vm = oracle.verify_mask(p, B)
    pos = list(range(p + 1, p + B + 2))
    assert {tuple(ix) for ix in np.argwhere(vm)} == _allowed_set_causal(pos, p + B + 2)
    cm = oracle.causal_mask([p], p + 1)
    assert cm.all()


# ---------------------------------------------------------------- attention vs library

@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (6, 2), (12, 4)])
def test_attention_matches_torch_sdpa(Hq, Hkv):
    n, nk, d = 9, 23, 16
    q = RNG.standard_normal((n, Hq, d))
    k = RNG.standard_normal((nk, Hkv, d))
    v = RNG.standard_normal((nk, Hkv, d))
    allowed = oracle.causal_mask(np.arange(nk - n, nk), nk)
    allowed[2, :] = oracle.draft_mask(nk - n, n - 1)[1, :]
    o = oracle.attention(q, k, v, allowed)
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)[None]
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(allowed))
    np.testing.assert_allclose(o, ref[0].permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- whole forward vs library composition

def _tiny_cfg():
    return synth.ModelConfig(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16,
                             ffn=96, vocab=50, dtype=synth.F32)


def _torch_forward(W, cfg, x, pos):
    """A causal prefill built from torch library calls (rms_norm, linear,
    scaled_dot_product_attention with its own GQA, silu) and complex-number RoPE."""
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    x = t(x)
    n = x.shape[0]
    Hq, Hkv, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    half = d // 2
    w = torch.tensor([cfg.rope_theta ** (-2.0 * i / d) for i in range(half)], dtype=torch.float64)
    rot = torch.polar(torch.ones(n, half, dtype=torch.float64), torch.outer(t(pos), w))

    def rope_c(a):  # a [n, H, d]
        z = torch.complex(a[..., :half], a[..., half:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], dim=-1)

    for lw in W["layers"]:
        xn = F.rms_norm(x, (cfg.hidden,), t(lw["g_attn"]), eps=cfg.rms_eps)
        q = rope_c(F.linear(xn, t(lw["wq"])).view(n, Hq, d))
        k = rope_c(F.linear(xn, t(lw["wk"])).view(n, Hkv, d))
        v = F.linear(xn, t(lw["wv"])).view(n, Hkv, d)
        o = F.scaled_dot_product_attention(q.transpose(0, 1)[None], k.transpose(0, 1)[None],
                                           v.transpose(0, 1)[None], is_causal=True,
                                           enable_gqa=True)[0].transpose(0, 1).reshape(n, Hq * d)
        x = x + F.linear(o, t(lw["wo"]))
        xn = F.rms_norm(x, (cfg.hidden,), t(lw["g_mlp"]), eps=cfg.rms_eps)
        x = x + F.linear(F.silu(F.linear(xn, t(lw["wg"]))) * F.linear(xn, t(lw["wu"])), t(lw["wd"]))
    return F.linear(F.rms_norm(x, (cfg.hidden,), t(W["g_final"]), eps=cfg.rms_eps),
                    t(W["lm_head"])).numpy()


def test_forward_matches_torch_library_composition():
    cfg = _tiny_cfg()
    W = synth.make_weights(cfg, seed=7, std=0.2)
    # non-trivial gains so a dropped gain fails
    for lw in W["layers"]:
        lw["g_attn"] = RNG.uniform(0.5, 1.5, cfg.hidden).astype(np.float32)
        lw["g_mlp"] = RNG.uniform(0.5, 1.5, cfg.hidden).astype(np.float32)
    W["g_final"] = RNG.uniform(0.5, 1.5, cfg.hidden).astype(np.float32)
    m = oracle.Model(W, cfg)
    x = RNG.standard_normal((11, cfg.hidden))
    logits, _, _ = oracle.prefill_cache(m, x)
    ref = _torch_forward(W, cfg, x, np.arange(11, dtype=np.float64))
    np.testing.assert_allclose(logits, ref, rtol=1e-11, atol=1e-11)


def test_incremental_cache_equals_one_pass_prefill():
    cfg = _tiny_cfg()
    m = oracle.Model(synth.make_weights(cfg, seed=3, std=0.2), cfg)
    x = RNG.standard_normal((10, cfg.hidden))
    full, fk, fv = oracle.prefill_cache(m, x)
    ck, cv = oracle.prefill_cache(m, x[:6])[1:]
    for i in range(6, 10):
        lg, k, v = oracle.forward(m, x[i:i + 1], [i], ck, cv, oracle.causal_mask([i], i + 1))
        np.testing.assert_allclose(lg[0], full[i], rtol=0, atol=1e-12)
        ck = [np.concatenate([a, b]) for a, b in zip(ck, k)]
        cv = [np.concatenate([a, b]) for a, b in zip(cv, v)]
    for l in range(cfg.n_layers):
        np.testing.assert_allclose(ck[l], fk[l], atol=1e-12)
        np.testing.assert_allclose(cv[l], fv[l], atol=1e-12)


def test_forward_respects_mask_a_masked_key_changes_nothing():
    # Changing a key the mask hides must leave the row's output unchanged.
    cfg = _tiny_cfg()
    m = oracle.Model(synth.make_weights(cfg, seed=5, std=0.2), cfg)
    x = RNG.standard_normal((8, cfg.hidden))
    lg1, _, _ = oracle.prefill_cache(m, x)
    x2 = x.copy()
    x2[7] += 1.0
    lg2, _, _ = oracle.prefill_cache(m, x2)
    np.testing.assert_array_equal(lg1[:7], lg2[:7])
    assert np.abs(lg1[7] - lg2[7]).max() > 1e-6


def test_bf16_rounding_is_round_to_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38, 1e-40], np.float32)
    got = synth.bf16_to_f32(synth.bf16_bits(vals))
    ref = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(got, ref)
