"""The allocation-free GEMM entry point, gocr_op_linear_static.

It serves callers that cannot allocate device memory (a plug-in inside a host
application that owns every allocation, a real-time loop that must not enter
the allocator, a sandbox without cudaMalloc): instead of a caller-provided
workspace it uses the library's fixed-size static device scratch array.  Its
results must match the workspace version, gocr_op_linear, on the same inputs,
on consecutive calls that reuse the shared array.  This file is collected last
so that a run stopping at the first failure has run every other test first.
"""
import ctypes

import numpy as np
import pytest

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
    if dt == "bf16":
        return torch.from_numpy(np.ascontiguousarray(synth.bf16_bits(a)).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_static_scratch_matches_workspace_version_twice(g, dt):
    """Same kernel, same split rule: the results equal the workspace version's
    bit for bit, on consecutive calls that reuse the shared array.  The fp32
    path reduces its split-K partials through the array; its smaller second
    call follows a larger first one, so leftover partial sums or counters of
    the first call would show in the second."""
    rng = np.random.default_rng(17)
    shapes = ((65, 2560, 1536), (33, 1536, 4096)) if dt == "f32" else ((33, 1536, 4096), (65, 2560, 1536))
    if dt == "f32":
        lib = g.load()
        assert lib.gocr_op_linear_workspace(*shapes[0]) > lib.gocr_op_linear_workspace(*shapes[1])
    for T, N, K in shapes:
        x = _dev(rng.standard_normal((T, K)).astype(np.float32), dt)
        w = _dev((0.02 * rng.standard_normal((N, K))).astype(np.float32), dt)
        ref = g.op_linear(x, w).cpu().numpy()
        got = g.op_linear_static(x, w).cpu().numpy()
        np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_static_scratch_rejects_oversized_shapes(g):
    lib = g.load()
    T, N, K = 4096, 8192, 4096  # needs far more than the static array holds
    assert lib.gocr_op_linear_workspace(T, N, K) > 16 << 20
    rc = lib.gocr_op_linear_static(0, ctypes.c_void_p(1), ctypes.c_void_p(1), ctypes.c_void_p(1), T, N, K, None)
    assert rc == -2
    assert "static array" in g.last_error(None)
