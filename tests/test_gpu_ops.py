"""Kernel-level parity of the CUDA path against the oracle's definitions, through
the C ABI's single-kernel entry points: the split-K GEMM and the masked GQA
attention, at sizes that span several tiles with ragged tails.
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


def _bf16_planes_of(a):
    """fp32 array -> (hi, lo) bf16 tensors with a = hi + lo, and hi + lo in fp64."""
    from self_speculative_block_gb300 import synth
    hi = synth.bf16_bits(a)
    lo = synth.bf16_bits(a.astype(np.float32) - synth.bf16_to_f32(hi))
    t = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).cuda().view(torch.bfloat16)
    return t(hi), t(lo), synth.bf16_to_f32(hi).astype(np.float64) + synth.bf16_to_f32(lo).astype(np.float64)


# up to two 128-row slices: K chunks over a cluster; three or more: one CTA
# runs every K chunk (ragged last slices: 300 = 2 x 128 + 44, 528 = 4 x 128 + 16)
@pytest.mark.parametrize("T,N,K", [(1, 128, 64), (33, 2560, 1536), (256, 384, 704), (300, 384, 704),
                                   (528, 1536, 4096), (1000, 256, 1536)])
def test_linear_planes_matches_oracle_matmul(g, T, N, K):
    from self_speculative_block_gb300 import synth
    rng = np.random.default_rng(T * 11 + N + K)
    xh, xl, x = _bf16_planes_of(rng.standard_normal((T, K)).astype(np.float32))
    w = _rounded((0.02 * rng.standard_normal((N, K))).astype(np.float32), "bf16")
    y = g.op_linear_planes(xh, xl, _dev(w, "bf16")).cpu().numpy()
    ref = x @ w.T  # fp64 on the kernel's exact operands
    np.testing.assert_allclose(y, ref, rtol=1e-4, atol=2e-5 * np.sqrt(K / 64))


def test_linear_planes_row_bits_do_not_depend_on_row_count_or_kernel(g):
    rng = np.random.default_rng(9)
    N, K = 1536, 4096
    xh, xl, _ = _bf16_planes_of(rng.standard_normal((528, K)).astype(np.float32))
    w = _dev((0.02 * rng.standard_normal((N, K))).astype(np.float32), "bf16")
    full = g.op_linear_planes(xh, xl, w)  # five slices: one CTA per (tile, slice)
    for T in (1, 33, 65, 200, 256, 300):  # T <= 256: the clustered kernel
        part = g.op_linear_planes(xh[:T].contiguous(), xl[:T].contiguous(), w)
        assert torch.equal(part, full[:T]), T


def _planes(a, dtype):
    """fp32 array -> the kernel's operand: fp32 tensor, or (hi, lo) bf16 tensors with a = hi + lo."""
    from self_speculative_block_gb300 import gocr, synth
    if dtype == gocr.DTYPE_F32:
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    hi = synth.bf16_bits(a)
    lo = synth.bf16_bits(a.astype(np.float32) - synth.bf16_to_f32(hi))
    t = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).cuda().view(torch.bfloat16)
    return (t(hi), t(lo))


def _attn_case(rng, T, Hq, Hkv, d, cap, lims, dtype):
    from self_speculative_block_gb300 import gocr
    q = rng.standard_normal((T, Hq, d)).astype(np.float32)
    k = rng.standard_normal((Hkv, cap, d)).astype(np.float32)
    v = rng.standard_normal((Hkv, cap, d)).astype(np.float32)
    lim = np.asarray(lims, np.int32)
    allowed = np.arange(cap)[None, :] <= lim[:, None]
    ref = oracle.attention(q.astype(np.float64), k.transpose(1, 0, 2).astype(np.float64),
                           v.transpose(1, 0, 2).astype(np.float64), allowed)
    o = gocr.op_attention(_planes(q, dtype), _planes(k, dtype), _planes(v, dtype),
                          torch.from_numpy(lim).cuda(), dtype).cpu().numpy()
    return o, ref


def _attn_kind(monkeypatch, dt):
    """bf16: the mma.sync kernel (default); bf16-tc: the tcgen05 kernel."""
    if dt == "bf16-tc":
        monkeypatch.setenv("GOCR_ATTN", "tc")
    else:
        monkeypatch.delenv("GOCR_ATTN", raising=False)


@pytest.mark.parametrize("dt", ["f32", "bf16", "bf16-tc"])
@pytest.mark.parametrize("Hq,Hkv,d", [(4, 2, 64), (12, 4, 128)])
@pytest.mark.parametrize("p,B", [(0, 1), (5, 4), (130, 8), (1000, 32), (300, 64)])
def test_attention_draft_and_verify_masks(g, monkeypatch, dt, Hq, Hkv, d, p, B):
    _attn_kind(monkeypatch, dt)
    rng = np.random.default_rng(p + B + d)
    cap = p + B + 3
    dtype = g.DTYPE_F32 if dt == "f32" else g.DTYPE_BF16
    # the bf16 kernel takes hi/lo bf16 planes of the fp32 inputs and bf16 probabilities
    tol = 2e-5 if dt == "f32" else 5e-3
    # draft: boundary row causal (lim p), [M] rows see the window (lim p+B)
    o, ref = _attn_case(rng, B + 1, Hq, Hkv, d, cap, [p] + [p + B] * B, dtype)
    np.testing.assert_allclose(o, ref, rtol=tol, atol=tol)
    # verify: row j at p+1+j, token-causal
    o, ref = _attn_case(rng, B + 1, Hq, Hkv, d, cap, list(range(p + 1, p + B + 2)), dtype)
    np.testing.assert_allclose(o, ref, rtol=tol, atol=tol)


@pytest.mark.parametrize("dt", ["f32", "bf16", "bf16-tc"])
def test_attention_row_bits_do_not_depend_on_other_rows(g, monkeypatch, dt):
    _attn_kind(monkeypatch, dt)
    rng = np.random.default_rng(3)
    dtype = g.DTYPE_F32 if dt == "f32" else g.DTYPE_BF16
    Hq, Hkv, d, cap = 12, 4, 128, 700
    qn = rng.standard_normal((65, Hq, d)).astype(np.float32)
    k = _planes(rng.standard_normal((Hkv, cap, d)).astype(np.float32), dtype)
    v = _planes(rng.standard_normal((Hkv, cap, d)).astype(np.float32), dtype)
    lim = torch.arange(600, 665, dtype=torch.int32, device="cuda")
    full = g.op_attention(_planes(qn, dtype), k, v, lim, dtype)
    for j in (0, 1, 31, 64):
        one = g.op_attention(_planes(qn[j:j + 1], dtype), k, v, lim[j:j + 1].contiguous(), dtype)
        assert torch.equal(one[0], full[j]), j


@pytest.mark.parametrize("dt", ["f32", "bf16-mma", "bf16-tc"])
@pytest.mark.parametrize("P,N,B,Hq,Hkv,d", [(5, 24, 8, 4, 2, 64), (40, 90, 32, 12, 4, 128), (0, 33, 7, 12, 4, 128),
                                            (130, 200, 32, 6, 2, 128), (300, 160, 16, 12, 4, 128)])
def test_attention_three_stream_training_mask(g, monkeypatch, dt, P, N, B, Hq, Hkv, d):
    """The joint-training mask (review §3.1; blog three-stream figure) as a
    second key interval per row, against the oracle's mask built from the
    rule text, over the packed [prefix, clean, corrupted 1, corrupted 2]; bf16
    on the mma.sync and on the tcgen05 kernel (both skip the key chunks masked
    for a whole row tile)."""
    if dt != "f32":
        monkeypatch.setenv("GOCR_ATTN", dt.split("-")[1])
    rng = np.random.default_rng(P + N + B + d)
    L = P + 3 * N
    dtype = g.DTYPE_F32 if dt == "f32" else g.DTYPE_BF16
    tol = 2e-5 if dt == "f32" else 5e-3
    lim, lo2, hi2, _ = g.three_stream_ranges(P, N, B)
    q = rng.standard_normal((L, Hq, d)).astype(np.float32)
    k = rng.standard_normal((Hkv, L, d)).astype(np.float32)
    v = rng.standard_normal((Hkv, L, d)).astype(np.float32)
    ref = oracle.attention(q.astype(np.float64), k.transpose(1, 0, 2).astype(np.float64),
                           v.transpose(1, 0, 2).astype(np.float64), oracle.three_stream_mask(P, N, B))
    dev = lambda a: torch.from_numpy(a).cuda()
    o = g.op_attention(_planes(q, dtype), _planes(k, dtype), _planes(v, dtype), dev(lim), dtype,
                       lo2=dev(lo2), hi2=dev(hi2)).cpu().numpy()
    np.testing.assert_allclose(o, ref, rtol=tol, atol=tol)


@pytest.mark.parametrize("kind", [None, "mma"])
def test_attention_three_stream_full_size_sampled(g, monkeypatch, kind):
    """The training-mask call at the size bench.py times (prefix 1024, three
    512-token streams, blocks of 32, 12 q / 4 kv heads, d 128: 2,560 rows)
    with the call's own kernel and rank choice (and on the mma.sync kernel),
    against the oracle on sampled rows: the first and last rows of every
    stream and block edge, plus seeded random rows, every head."""
    if kind:
        monkeypatch.setenv("GOCR_ATTN", kind)
    P, N, B, Hq, Hkv, d = 1024, 512, 32, 12, 4, 128
    L = P + 3 * N
    rng = np.random.default_rng(2560)
    lim, lo2, hi2, _ = g.three_stream_ranges(P, N, B)
    q = rng.standard_normal((L, Hq, d)).astype(np.float32)
    k = rng.standard_normal((Hkv, L, d)).astype(np.float32)
    v = rng.standard_normal((Hkv, L, d)).astype(np.float32)
    dev = lambda a: torch.from_numpy(a).cuda()
    o = g.op_attention(_planes(q, g.DTYPE_BF16), _planes(k, g.DTYPE_BF16), _planes(v, g.DTYPE_BF16), dev(lim),
                       g.DTYPE_BF16, lo2=dev(lo2), hi2=dev(hi2)).cpu().numpy()
    edges = [0, 1, 31, 32, P - 1]
    for s0 in (P, P + N, P + 2 * N):
        edges += [s0, s0 + 1, s0 + B - 1, s0 + B, s0 + N // 2, s0 + N - B, s0 + N - 1]
    rows = np.unique(np.concatenate([edges, rng.integers(0, L, 24)]))
    mask = oracle.three_stream_mask(P, N, B)[rows]
    ref = oracle.attention(q[rows].astype(np.float64), k.transpose(1, 0, 2).astype(np.float64),
                           v.transpose(1, 0, 2).astype(np.float64), mask)
    np.testing.assert_allclose(o[rows], ref, rtol=5e-3, atol=5e-3)


@pytest.mark.parametrize("kind", ["mma", "tc"])
@pytest.mark.parametrize("ranks", [1, 3, 7])
def test_attention_three_stream_few_ranks(g, monkeypatch, kind, ranks):
    """The training mask with few key-chunk ranks, so that each rank walks
    many chunks across the span it skips (past the clean limit, before the
    corrupted block) on both bf16 kernels, against the oracle."""
    monkeypatch.setenv("GOCR_ATTN", kind)
    monkeypatch.setenv("GOCR_ATTN_RANKS", str(ranks))
    P, N, B, Hq, Hkv, d = 200, 256, 32, 12, 4, 128
    rng = np.random.default_rng(ranks)
    L = P + 3 * N
    lim, lo2, hi2, _ = g.three_stream_ranges(P, N, B)
    q = rng.standard_normal((L, Hq, d)).astype(np.float32)
    k = rng.standard_normal((Hkv, L, d)).astype(np.float32)
    v = rng.standard_normal((Hkv, L, d)).astype(np.float32)
    ref = oracle.attention(q.astype(np.float64), k.transpose(1, 0, 2).astype(np.float64),
                           v.transpose(1, 0, 2).astype(np.float64), oracle.three_stream_mask(P, N, B))
    dev = lambda a: torch.from_numpy(a).cuda()
    o = g.op_attention(_planes(q, g.DTYPE_BF16), _planes(k, g.DTYPE_BF16), _planes(v, g.DTYPE_BF16), dev(lim),
                       g.DTYPE_BF16, lo2=dev(lo2), hi2=dev(hi2)).cpu().numpy()
    np.testing.assert_allclose(o, ref, rtol=5e-3, atol=5e-3)
