// bf16 weight-streaming GEMM on the 5th-generation tensor cores.
//
// Y[T, N] = X[T, K] W[N, K]^T with the weights as the 128-row MMA operand
// ("swap AB"): one CTA owns a 128-row tile of W and one K chunk, so a decode
// forward with T = B + 1 tokens is an M = 128, N = 16..256 tcgen05.mma with an
// fp32 accumulator in tensor memory.  TMA streams W tiles (128 x 64, 128-byte
// swizzle) and the matching X tiles (16-row boxes) through a ring of shared
// memory stages; one thread issues the TMA loads, one thread issues the MMAs,
// and the four warps read the accumulator back with tcgen05.ld.
//
// The K chunking (split count) depends on (N, K) only and partial sums are
// added in split order by the last CTA of a tile, exactly as in the CUDA-core
// path, so a row's bits do not depend on how many rows share the launch.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <map>
#include <mutex>
#include <tuple>

#include "epilogue.cuh"
#include "tc.cuh"

namespace gocr {

namespace {
constexpr int TC_THREADS = 128;
constexpr int TZ_TC = 256;       // tokens per CTA (MMA N <= 256)
constexpr int EG = 32;           // tokens per epilogue group
constexpr int YS_LD_TC = NTILE + 1;
constexpr int A_BYTES = NTILE * 64 * 2;  // 128 x 64 bf16
constexpr int SMEM_BUDGET = 200 * 1024;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_mu;
std::map<std::tuple<const void*, int, int, int>, CUtensorMap> g_maps;

bool encoder() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// Row-major bf16 matrix [rows, cols] (cols contiguous), box = 64 cols x box_rows.
bool tmap_2d(CUtensorMap* out, const void* ptr, int rows, int cols, int box_rows) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_tuple(ptr, rows, cols, box_rows);
  auto it = g_maps.find(key);
  if (it != g_maps.end()) { *out = it->second; return true; }
  if (!encoder()) return false;
  CUtensorMap m;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (g_maps.size() > 4096) g_maps.clear();
  g_maps[key] = m;
  *out = m;
  return true;
}

__host__ __device__ inline int cdiv_i(int a, int b) { return (a + b - 1) / b; }
}  // namespace

__global__ void __launch_bounds__(TC_THREADS) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmw,
                                                            const __grid_constant__ CUtensorMap tmx,
                                                            GemmArgs a, int nt, int stages) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int b_bytes = nt * 128;
  uint8_t* sA = smem;
  uint8_t* sB = sA + stages * A_BYTES;
  float* Ys = reinterpret_cast<float*>(sB + stages * b_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(Ys + EG * YS_LD_TC);
  uint64_t* empty = full + stages;
  uint64_t* done = empty + stages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done + 1);
  __shared__ int s_last;
  __shared__ int s_fail;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, split = blockIdx.y, z = blockIdx.z;
  const int n_tiles = gridDim.x;
  const int n0 = tile * NTILE;
  const int t0 = z * TZ_TC;
  const int tn = min(TZ_TC, a.T - t0);
  const int k0 = split * a.kchunk;
  const int k1 = min(a.K, k0 + a.kchunk);
  const int nkb = cdiv_i(k1 - k0, 64);
  const uint32_t ncols = nt <= 32 ? 32 : (nt <= 64 ? 64 : (nt <= 128 ? 128 : 256));

  if (tid == 0) {
    tc::prefetch_tmap(&tmw);
    tc::prefetch_tmap(&tmx);
    for (int s = 0; s < stages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(done, 1);
    tc::fence_mbar_init();
    s_fail = 0;
  }
  __syncwarp();
  if (warp == 0) tc::tmem_alloc(tmem_holder, ncols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_holder;

  if (tid == 0) {
    // TMA producer
    const uint64_t pol = tc::policy_evict_first();
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % stages;
      const int use = kb / stages;
      if (use > 0 && !tc::mbar_wait(&empty[s], (use - 1) & 1)) { s_fail = 1; break; }
      tc::mbar_expect_tx(&full[s], A_BYTES + b_bytes);
      const int kx = k0 + kb * 64;
      tc::tma_load_2d_hint(sA + s * A_BYTES, &tmw, kx, n0, &full[s], pol);
      for (int g = 0; g < nt / 16; ++g) tc::tma_load_2d(sB + s * b_bytes + g * 2048, &tmx, kx, t0 + 16 * g, &full[s]);
    }
  } else if (tid == 32) {
    // MMA issuer
    const uint32_t idesc = tc::idesc_bf16(NTILE, nt);
    bool ok = true;
    for (int kb = 0; kb < nkb && ok; ++kb) {
      const int s = kb % stages;
      const int use = kb / stages;
      if (!tc::mbar_wait(&full[s], use & 1)) { ok = false; s_fail = 1; break; }
      tc::fence_after_sync();
      const uint32_t a_base = tc::smem_u32(sA + s * A_BYTES);
      const uint32_t b_base = tc::smem_u32(sB + s * b_bytes);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_bf16(tmem, tc::sdesc_sw128(a_base + kk * 32), tc::sdesc_sw128(b_base + kk * 32), idesc,
                     (kb > 0 || kk > 0) ? 1u : 0u);
      tc::mma_commit(&empty[s]);
    }
    tc::mma_commit(done);
  }
  __syncwarp();
  const bool ok_done = tc::mbar_wait(done, 0);
  tc::fence_after_sync();
  __syncthreads();
  const bool failed = !ok_done || s_fail;
  if (failed) {
    if (tid == 0) set_err(a.e.err, DERR_TIMEOUT);
  } else {
    const int row = warp * 32 + lane;
    const int n = n0 + row;
    const int n_groups = cdiv_i(tn, EG);
    if (a.splits == 1) {
      for (int g = 0; g < n_groups; ++g) {
        float v[32];
        tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + g * EG, v);
        const int gn = min(EG, tn - g * EG);
#pragma unroll
        for (int j = 0; j < 32; ++j) Ys[j * YS_LD_TC + row] = j < gn ? v[j] : 0.f;
        __syncthreads();
        apply_epilogue<bf16>(a, Ys, YS_LD_TC, tile, t0 + g * EG, gn);
        __syncthreads();
      }
    } else {
      for (int g = 0; g < n_groups; ++g) {
        float v[32];
        tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + g * EG, v);
        const int gn = min(EG, tn - g * EG);
        if (n < a.N) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < gn) a.ws[((size_t)split * a.T + t0 + g * EG + j) * a.N + n] = v[j];
        }
      }
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        int* ctr = a.counters + z * n_tiles + tile;
        int prev = atomicAdd(ctr, 1);
        s_last = (prev == a.splits - 1);
        if (s_last) *ctr = 0;
      }
      __syncthreads();
      if (s_last) {
        __threadfence();
        for (int g = 0; g < n_groups; ++g) {
          const int gn = min(EG, tn - g * EG);
          for (int j = 0; j < EG; ++j) {
            float acc = 0.f;
            if (j < gn && n < a.N) {
              const size_t base = (size_t)(t0 + g * EG + j) * a.N + n;
              acc = __ldcg(a.ws + base);
              for (int s = 1; s < a.splits; ++s) acc += __ldcg(a.ws + (size_t)s * a.T * a.N + base);
            }
            Ys[j * YS_LD_TC + row] = acc;
          }
          __syncthreads();
          apply_epilogue<bf16>(a, Ys, YS_LD_TC, tile, t0 + g * EG, gn);
          __syncthreads();
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, ncols);
  if (failed) return;

  if (a.epi == EPI_ARGMAX && (a.splits == 1 || s_last)) {
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

bool launch_gemm_tc(const GemmArgs& a, cudaStream_t s) {
  CUtensorMap tmw, tmx;
  if (!tmap_2d(&tmw, a.w, a.N, a.K, NTILE)) return false;
  if (!tmap_2d(&tmx, a.x, a.T, a.K, 16)) return false;
  const int nt = ((a.T < TZ_TC ? a.T : TZ_TC) + 15) / 16 * 16;
  const int nkb = cdiv_i(a.kchunk, 64);
  const int stage_bytes = A_BYTES + nt * 128;
  const int fixed = 1024 + EG * YS_LD_TC * 4 + 64;
  int stages = (SMEM_BUDGET - fixed) / stage_bytes;
  if (stages > 6) stages = 6;
  if (stages > nkb) stages = nkb;
  if (stages < 1) stages = 1;
  const size_t smem = fixed + (size_t)stages * stage_bytes + (2 * stages + 2) * 8;
  static size_t configured = 0;
  if (smem > configured) {
    if (cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return false;
    configured = smem;
  }
  dim3 grid(cdiv_i(a.N, NTILE), a.splits, cdiv_i(a.T, TZ_TC));
  gemm_tc_kernel<<<grid, TC_THREADS, smem, s>>>(tmw, tmx, a, nt, stages);
  return true;
}

}  // namespace gocr
