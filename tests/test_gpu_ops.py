"""Kernel-level parity of the CUDA path against the oracle's definitions, through
the C ABI's single-kernel entry points: the split-K GEMM, RMSNorm and the
masked GQA attention, at sizes that span several tiles with ragged tails.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.fail("gpu tests need a CUDA device")
    from self_speculative_block_gb300 import build, gocr
    build.build()
    gocr.load()
    return gocr


def _dev(a, dt):
    from self_speculative_block_gb300 import synth
    return torch.from_numpy(np.ascontiguousarray(synth.bf16_bits(a)).view(np.int16)).cuda().view(
        torch.bfloat16) if dt == "bf16" else torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def _rounded(a, dt):
    from self_speculative_block_gb300 import synth
    return synth.round_to_storage(a, dt).astype(np.float64)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("T,N,K", [(1, 128, 64), (33, 300, 200), (70, 2560, 1536), (33, 1536, 4096),
                                   (5, 1024, 256), (129, 384, 704)])
def test_linear_matches_oracle_matmul(g, dt, T, N, K):
    rng = np.random.default_rng(T * 7 + N + K)
    x = _rounded(rng.standard_normal((T, K)).astype(np.float32), dt)
    w = _rounded((0.02 * rng.standard_normal((N, K))).astype(np.float32), dt)
    y = g.op_linear(_dev(x, dt), _dev(w, dt)).cpu().numpy()
    ref = x @ w.T  # fp64 on the same (rounded) inputs
    np.testing.assert_allclose(y, ref, rtol=1e-4, atol=2e-5 * np.sqrt(K / 64))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_linear_row_bits_do_not_depend_on_row_count(g, dt):
    rng = np.random.default_rng(5)
    N, K = 2560, 1536
    x = _dev(rng.standard_normal((528, K)).astype(np.float32), dt)
    w = _dev((0.02 * rng.standard_normal((N, K))).astype(np.float32), dt)
    full = g.op_linear(x, w)
    for T in (1, 33, 65, 200):
        part = g.op_linear(x[:T].contiguous(), w)
        assert torch.equal(part, full[:T]), T


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_rmsnorm_matches_oracle(g, dt):
    rng = np.random.default_rng(9)
    x = rng.standard_normal((37, 1536)).astype(np.float32) * 3
    gain = rng.uniform(0.5, 1.5, 1536).astype(np.float32)
    y = g.op_rmsnorm(torch.from_numpy(x).cuda(), torch.from_numpy(gain).cuda(), 1e-6,
                     torch.bfloat16 if dt == "bf16" else torch.float32)
    ref = oracle.rmsnorm(x.astype(np.float64), gain.astype(np.float64), 1e-6)
    tol = 8e-3 if dt == "bf16" else 2e-6
    np.testing.assert_allclose(y.float().cpu().numpy(), ref, rtol=tol, atol=tol)


def _attn_case(rng, T, Hq, Hkv, d, cap, lims, dt):
    q = _rounded(rng.standard_normal((T, Hq, d)).astype(np.float32), dt)
    k = _rounded(rng.standard_normal((Hkv, cap, d)).astype(np.float32), dt)
    v = _rounded(rng.standard_normal((Hkv, cap, d)).astype(np.float32), dt)
    lim = np.asarray(lims, np.int32)
    allowed = np.arange(cap)[None, :] <= lim[:, None]
    ref = oracle.attention(q, k.transpose(1, 0, 2), v.transpose(1, 0, 2), allowed)
    o = g_op_attention(q, k, v, lim, dt)
    return o, ref


def g_op_attention(q, k, v, lim, dt):
    from self_speculative_block_gb300 import gocr
    o = gocr.op_attention(_dev(q, dt), _dev(k, dt), _dev(v, dt), torch.from_numpy(lim).cuda())
    return o.float().cpu().numpy()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("Hq,Hkv,d", [(4, 2, 64), (12, 4, 128)])
@pytest.mark.parametrize("p,B", [(0, 1), (5, 4), (130, 8), (1000, 32)])
def test_attention_draft_and_verify_masks(g, dt, Hq, Hkv, d, p, B):
    rng = np.random.default_rng(p + B + d)
    cap = p + B + 3
    tol = 2e-2 if dt == "bf16" else 2e-5
    # draft: boundary row causal (lim p), [M] rows see the window (lim p+B)
    o, ref = _attn_case(rng, B + 1, Hq, Hkv, d, cap, [p] + [p + B] * B, dt)
    np.testing.assert_allclose(o, ref, rtol=tol, atol=tol)
    # verify: row j at p+1+j, token-causal
    o, ref = _attn_case(rng, B + 1, Hq, Hkv, d, cap, list(range(p + 1, p + B + 2)), dt)
    np.testing.assert_allclose(o, ref, rtol=tol, atol=tol)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_attention_row_bits_do_not_depend_on_other_rows(g, dt):
    from self_speculative_block_gb300 import gocr
    rng = np.random.default_rng(3)
    Hq, Hkv, d, cap = 12, 4, 128, 700
    q = _dev(rng.standard_normal((65, Hq, d)).astype(np.float32), dt)
    k = _dev(rng.standard_normal((Hkv, cap, d)).astype(np.float32), dt)
    v = _dev(rng.standard_normal((Hkv, cap, d)).astype(np.float32), dt)
    lim = torch.arange(600, 665, dtype=torch.int32, device="cuda")
    full = gocr.op_attention(q, k, v, lim)
    for j in (0, 1, 31, 64):
        one = gocr.op_attention(q[j:j + 1].contiguous(), k, v, lim[j:j + 1].contiguous())
        assert torch.equal(one[0], full[j]), j
