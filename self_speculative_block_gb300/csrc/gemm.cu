// Weight-streaming GEMM Y[T, N] = X[T, K] W[N, K]^T with a fixed split-K
// reduction and fused epilogues (RoPE + KV write, SwiGLU, residual add,
// LM-head argmax).
//
// Reduction order is independent of T: the K range is cut into `splits`
// chunks that depend on (N, K) only; each CTA accumulates its chunk with a
// sequential fused multiply-add chain per output, writes fp32 partials, and
// the last CTA of a (tile, token slice) sums the partials in split order.  A
// row's result is therefore bit-identical whether the forward carries 1 row
// (AR), B+1 rows (draft / verify) or a batch, which is what makes the GPU's
// self-speculative output equal its own AR-greedy output token for token.
//
// This file holds the split rule and the CUDA-core kernel of the fp32 models;
// bf16 models run the tcgen05 kernel of gemm_tc.cu with the same reduction.
#include "epilogue.cuh"

namespace gocr {

namespace {
constexpr int KC = 32;       // K elements staged per step
constexpr int TZ = 64;       // tokens per CTA (grid z slices)
constexpr int THREADS = 256;
constexpr int SM_COUNT = 152;  // fixed so the split rule is the same on every device
constexpr int YS_LD = NTILE + 1;

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }
}  // namespace

int gemm_kchunk(int N, int K) {
  const int tiles = cdiv(N, NTILE);
  const int kb = cdiv(K, 64);
  int want = (2 * SM_COUNT) / tiles;  // at most two CTAs per SM in one wave
  int s = want < kb ? want : kb;
  if (s < 1) s = 1;
  return cdiv(kb, s) * 64;
}

int gemm_splits(int N, int K) { return cdiv(K, gemm_kchunk(N, K)); }

size_t gemm_ws_floats(int T, int N, int K, bool single_split) {
  int s = single_split ? 1 : gemm_splits(N, K);
  return (size_t)s * T * N;
}

int gemm_counter_ints(int T, int N) { return cdiv(T, TZ) * cdiv(N, NTILE) + 1; }

template <typename T>
__global__ void __launch_bounds__(THREADS) gemm_simt_kernel(GemmArgs a) {
  extern __shared__ float sm[];
  float* Ws = sm;                          // [NTILE][KC + 1]
  float* Xs = Ws + NTILE * (KC + 1);       // [TZ][KC]
  float* Ys = Xs + TZ * KC;                // [TZ][YS_LD]
  __shared__ int s_last;

  const int tile = blockIdx.x, split = blockIdx.y, z = blockIdx.z;
  const int n_tiles = gridDim.x;
  const int n0 = tile * NTILE;
  const int t0 = z * TZ;
  const int tn = min(TZ, a.T - t0);
  const int k0 = split * a.kchunk;
  const int k1 = min(a.K, k0 + a.kchunk);
  const T* X = reinterpret_cast<const T*>(a.x);
  const T* W = reinterpret_cast<const T*>(a.w);
  const int tid = threadIdx.x;
  const int nl = tid & (NTILE - 1);
  const int tg = tid >> 7;  // 0..1: tokens tg*32 .. tg*32+31 of the slice

  float acc[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) acc[j] = 0.f;

  for (int kb = k0; kb < k1; kb += KC) {
    const int kc = min(KC, k1 - kb);
    for (int i = tid; i < NTILE * KC; i += THREADS) {
      int r = i / KC, c = i % KC, n = n0 + r;
      Ws[r * (KC + 1) + c] = (n < a.N && c < kc) ? to_f32<T>(W[(size_t)n * a.K + kb + c]) : 0.f;
    }
    for (int i = tid; i < TZ * KC; i += THREADS) {
      int r = i / KC, c = i % KC;
      Xs[r * KC + c] = (r < tn && c < kc) ? to_f32<T>(X[(size_t)(t0 + r) * a.ldx + kb + c]) : 0.f;
    }
    __syncthreads();
    for (int c = 0; c < kc; ++c) {
      const float w = Ws[nl * (KC + 1) + c];
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = fmaf(Xs[(tg * 32 + j) * KC + c], w, acc[j]);
    }
    __syncthreads();
  }

  // partials -> workspace
  const int n = n0 + nl;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    int tl = tg * 32 + j;
    if (tl < tn && n < a.N) a.ws[((size_t)split * a.T + t0 + tl) * a.N + n] = acc[j];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    int* ctr = a.counters + z * n_tiles + tile;
    int prev = atomicAdd(ctr, 1);
    s_last = (prev == a.splits - 1);
    if (s_last) *ctr = 0;  // ready for the next launch
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // fixed-order reduction over splits
#pragma unroll 4
  for (int j = 0; j < 32; ++j) {
    int tl = tg * 32 + j;
    if (tl < tn && n < a.N) {
      size_t base = (size_t)(t0 + tl) * a.N + n;
      float v = __ldcg(a.ws + base);
      for (int s = 1; s < a.splits; ++s) v += __ldcg(a.ws + (size_t)s * a.T * a.N + base);
      Ys[tl * YS_LD + nl] = v;
    } else if (tl < TZ) {
      Ys[tl * YS_LD + nl] = 0.f;
    }
  }
  __syncthreads();
  apply_epilogue<T>(a, Ys, YS_LD, tile, t0, tn);

  if (a.epi == EPI_ARGMAX) {
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      int* gc = a.counters + gridDim.z * n_tiles;
      int prev = atomicAdd(gc, 1);
      s_last = (prev == n_tiles * (int)gridDim.z - 1);
      if (s_last) *gc = 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    argmax_finish(a);
  }
}

bool launch_gemm(int dtype, const GemmArgs& a, cudaStream_t s) {
  if (dtype == 1) return launch_gemm_tc(a, s);
  dim3 grid(cdiv(a.N, NTILE), a.splits, cdiv(a.T, TZ));
  size_t smem = sizeof(float) * (NTILE * (KC + 1) + TZ * KC + TZ * YS_LD);
  {
    static bool init = false;
    if (!init) {
      cudaFuncSetAttribute(gemm_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      init = true;
    }
    gemm_simt_kernel<float><<<grid, THREADS, smem, s>>>(a);
  }
  return true;
}

}  // namespace gocr
