// Weight-streaming GEMM Y[T, N] = X[T, K] W[N, K]^T: the split rule shared by
// both implementations, and the CUDA-core kernel that fp32 models run.
//
// Reduction order is independent of T: the K range is cut into `splits`
// chunks that depend on (N, K) only; each chunk accumulates in a fixed order
// and the partial sums of a tile are added in split order.  A row's result is
// therefore bit-identical whether the forward carries 1 row (AR), B+1 rows
// (draft / verify) or a batch, which is what makes the GPU's self-speculative
// output equal its own AR-greedy output token for token.
#include "epilogue.cuh"

#include <cstdlib>
#include <cstring>

namespace gocr {

namespace {
constexpr int KC = 32;       // K elements staged per step
constexpr int TZ = 64;       // tokens per CTA (grid z slices)
constexpr int THREADS = 256;
constexpr int MAX_SPLITS = 12;  // split-K partials are reduced inside one cluster (non-portable size)
constexpr int YS_LD = NTILE + 1;

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }
}  // namespace

// Split rule, fixed for the process (GOCR_SPLIT_K: "wave", the default, or
// the largest K chunk in elements).
//   wave:  enough splits to fill two CTAs per SM in one wave (at most 12), so
//          that every SM streams an equal share of a matrix's weights: one
//          SM's TMA ring sustains only about 1/150 of HBM bandwidth.
//   chunk: K is cut into ceil(K / chunk) equal splits (fewer reductions,
//          fewer SMs per matrix).
static int split_chunk_limit() {
  static int lim = -1;
  if (lim < 0) {
    const char* v = getenv("GOCR_SPLIT_K");
    lim = 0;
    if (v && strncmp(v, "wave", 4) != 0 && atoi(v) >= 64) lim = atoi(v) / 64 * 64;
  }
  return lim;
}

// CTAs per SM the wave rule fills and its split cap
// (GOCR_SPLIT_K=wave<ctas per SM>[:<max splits>], default wave2:12).
static void wave_params(int* ctas, int* cap) {
  static int w = 0, c = 0;
  if (!w) {
    w = 2;
    c = MAX_SPLITS;
    const char* v = getenv("GOCR_SPLIT_K");
    if (v && strncmp(v, "wave", 4) == 0) {
      if (v[4] >= '1' && v[4] <= '4') w = v[4] - '0';
      const char* colon = strchr(v, ':');
      if (colon && atoi(colon + 1) >= 1 && atoi(colon + 1) <= 16) c = atoi(colon + 1);
    }
  }
  *ctas = w;
  *cap = c;
}

int gemm_kchunk(int N, int K) {
  const int tiles = cdiv(N, NTILE);
  const int kb = cdiv(K, 64);
  const int lim = split_chunk_limit();
  int s;
  if (lim > 0) {
    s = cdiv(kb, lim / 64);
  } else {
    int w, cap;
    wave_params(&w, &cap);
    s = (w * SM_COUNT) / tiles;  // CTAs per SM in one wave
    if (s > cap) s = cap;
  }
  if (s > kb) s = kb;
  if (s < 1) s = 1;
  return cdiv(kb, s) * 64;
}

int gemm_splits(int N, int K) { return cdiv(K, gemm_kchunk(N, K)); }

// Chunks per reduction group.  A tile's split-K sum is taken as group sums
// (the group's chunk sums added in chunk order) added in group order.  With
// two_groups (handles that batch requests), narrow matrices (at most 16
// weight tiles) with four or more chunks use two groups, so that the
// many-slice GEMM can give each group a CTA of its own; otherwise one group,
// the plain chunk-order sum.  A handle fixes the choice, so its results
// depend on (N, K) only.  The kernels take at most two groups.
int gemm_kgroup(int N, int K, bool two_groups) {
  const int S = gemm_splits(N, K);
  if (two_groups && cdiv(N, NTILE) <= 16 && S >= 4) return cdiv(S, 2);
  return S;
}

size_t gemm_ws_floats(int T, int N, int K) { return (size_t)gemm_splits(N, K) * T * N; }

int gemm_counter_ints(int T, int N) { return cdiv(T, TZ) * cdiv(N, NTILE) + 1; }

__global__ void __launch_bounds__(THREADS) gemm_simt_kernel(GemmArgs a) {
  extern __shared__ float sm[];
  float* Ws = sm;                          // [NTILE][KC + 1]
  float* Xs = Ws + NTILE * (KC + 1);       // [TZ][KC]
  float* Ys = Xs + TZ * KC;                // [TZ][YS_LD]
  float* scratch = Ys + TZ * YS_LD;        // epilogue scratch
  __shared__ int s_last;

  const int tile = blockIdx.x, split = blockIdx.y, z = blockIdx.z;
  const int n_tiles = gridDim.x;
  const int n0 = tile * NTILE;
  const int t0 = z * TZ;
  const int tn = min(TZ, a.T - t0);
  const int k0 = split * a.kchunk;
  const int k1 = min(a.K, k0 + a.kchunk);
  const float* X = reinterpret_cast<const float*>(a.x);
  const float* W = reinterpret_cast<const float*>(a.w);
  const int tid = threadIdx.x;
  const int nl = tid & (NTILE - 1);
  const int tg = tid >> 7;  // 0..1: tokens tg*32 .. tg*32+31 of the slice

  asm volatile("griddepcontrol.wait;" ::: "memory");
  float acc[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) acc[j] = 0.f;

  for (int kb = k0; kb < k1; kb += KC) {
    const int kc = min(KC, k1 - kb);
    for (int i = tid; i < NTILE * KC; i += THREADS) {
      int r = i / KC, c = i % KC, n = n0 + r;
      Ws[r * (KC + 1) + c] = (n < a.N && c < kc) ? W[(size_t)n * a.K + kb + c] : 0.f;
    }
    for (int i = tid; i < TZ * KC; i += THREADS) {
      int r = i / KC, c = i % KC;
      Xs[r * KC + c] = (r < tn && c < kc) ? X[(size_t)(t0 + r) * a.ldx + kb + c] : 0.f;
    }
    __syncthreads();
    for (int c = 0; c < kc; ++c) {
      const float w = Ws[nl * (KC + 1) + c];
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = fmaf(Xs[(tg * 32 + j) * KC + c], w, acc[j]);
    }
    __syncthreads();
  }

  // partials -> workspace; the last CTA of the (tile, token slice) reduces in split order
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
  if (s_last) {
    __threadfence();
#pragma unroll 4
    for (int j = 0; j < 32; ++j) {
      int tl = tg * 32 + j;
      float v = 0.f;
      if (tl < tn && n < a.N) {
        size_t base = (size_t)(t0 + tl) * a.N + n;
        v = __ldcg(a.ws + base);
        for (int s = 1; s < a.splits; ++s) v += __ldcg(a.ws + (size_t)s * a.T * a.N + base);
      }
      Ys[tl * YS_LD + nl] = v;
    }
    __syncthreads();
    apply_epilogue(a, Ys, YS_LD, tile, t0, tn, scratch);
  }
  if (a.epi == EPI_ARGMAX && s_last) {
    // every (tile, slice) contributes once; the grid counter expects tiles * slices
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const int total = n_tiles * (int)gridDim.z;
      const int prev = atomicAdd(a.e.grid_ctr, 1);
      s_last = (prev == total - 1);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      for (int t = tid; t < a.T; t += THREADS) {
        const unsigned long long k = atomicExch(a.e.amax + t, 0ull);
        a.e.am_out[t] = k ? (int)(0xFFFFFFFFu - (unsigned)(k & 0xFFFFFFFFull)) : 0;
      }
      if (tid == 0) *a.e.grid_ctr = 0;
    }
  }
}

bool launch_gemm(int dtype, const GemmArgs& a, cudaStream_t s, bool pdl) {
  if (dtype == 1) return launch_gemm_tc(a, s, pdl);
  dim3 grid(cdiv(a.N, NTILE), a.splits, cdiv(a.T, TZ));
  size_t smem = sizeof(float) * (NTILE * (KC + 1) + TZ * KC + TZ * YS_LD + EPI_SCRATCH_FLOATS);
  if (!kernel_smem_at_least(reinterpret_cast<const void*>(gemm_simt_kernel), smem)) return false;
  return launch_k(gemm_simt_kernel, grid, dim3(THREADS), smem, s, pdl, a) == cudaSuccess;
}

}  // namespace gocr
