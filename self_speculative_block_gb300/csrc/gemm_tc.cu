// bf16 weight-streaming GEMM on the 5th-generation tensor cores.
//
// Y[T, N] = X[T, K] W[N, K]^T with the weights as the 128-row MMA operand
// ("swap AB"): one CTA owns a 128-row tile of W and one K chunk.  The token
// side carries both planes of the activation: rows [0, nt) of the B tile are
// the hi plane and rows [nt, 2 nt) the lo plane of the same tokens, so one
// M = 128, N = 2 nt tcgen05.mma accumulates W x_hi and W x_lo side by side in
// tensor memory and the epilogue adds the two columns of each token.
//
// TMA streams W tiles (128 x 64, 128-byte swizzle, evict-first) and X tiles
// (16-row boxes per plane) through a ring of shared-memory stages; one thread
// issues the loads, one thread the MMAs.  Under programmatic dependent launch
// the weight loads of the first stages are issued before griddepcontrol.wait,
// so they overlap the tail of the kernel that produces X.
//
// The K chunks of a tile run on the CTAs of one thread-block cluster (at most
// 16).  Each CTA parks its fp32 partial tile in shared memory and sends the
// rows of each peer's token range to that peer by a bulk shared-to-cluster
// copy; CTA r adds the partials of its token range in rank order and runs the
// epilogue.  At decode shapes the receive buffers sit past the operand ring
// and are armed at the kernel's start ("early exchange"), so a CTA sends as
// soon as its own accumulator is drained instead of after a cluster barrier
// that waits for every peer's mainloop.  The split count depends on (N, K)
// only, so a row's bits do not depend on how many rows share the launch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cooperative_groups.h>

#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "epilogue.cuh"
#include "tc.cuh"

namespace gocr {

namespace {
constexpr int TC_THREADS = 128;
constexpr int TZ_TC = 128;       // tokens per CTA (two planes: MMA N <= 256)
constexpr int EG = 32;           // tokens per cluster-reduce group
constexpr int YLD = NTILE + 4;   // fp32 row stride of the partial tiles (16-byte multiple)
constexpr int A_BYTES = NTILE * 64 * 2;  // 128 x 64 bf16
constexpr int SMEM_CAP = 200 * 1024;
constexpr int DECODE_STAGE_CAP = 3;      // decode shapes: keep two CTAs per SM
// outside the ring: row scales of the z-slice; the first epilogue group's
// residual rows (RESID) or RoPE rows (QKV); the tile's next-norm gains; the
// first group's positions and requests; barriers; TMEM holder
constexpr int TAIL_BYTES = TZ_TC * 4 + EG * NTILE * 4 + NTILE * 4 + 2 * EG * 4 + 16 * 8 + 64;
constexpr int L2_PREFETCH_BLOCKS = 8;    // weight tiles a CTA brings into L2 ahead of its ring
constexpr int MAX_CLUSTER = 16;          // split-K ranks of one tile
constexpr size_t TWO_CTA_SMEM = 113 * 1024;  // dynamic shared memory of each of two CTAs on one SM

// Layout over the ring after the mainloop (gemm_tc_kernel):
// the partial tile [nt], the peers' rows [S x per] and, after them, the
// reduced rows [EG] and the epilogue scratch.  The compact layout (one
// epilogue pass: per <= EG; or S = 1) keeps [min(per, EG)] reduced rows and
// puts the scratch over the peers' rows, which are dead by then.  It is taken
// only where it is what lets two CTAs share an SM: measured at 33 tokens, the
// smaller footprint alone made the decode round slower (its CTAs and the next
// kernel's share SMs differently under programmatic dependent launch).
struct YLayout {
  int ys, scratch, floats;  // offsets of the reduced rows and the scratch; total fp32 words
};
inline YLayout gemm_y_layout(int nt, int S, int per, bool compact) {
  const int rx = S * per * YLD;
  if (!compact) return {nt * YLD + rx, nt * YLD + rx + EG * YLD, nt * YLD + rx + EG * YLD + EPI_SCRATCH_FLOATS};
  if (S == 1) return {nt * YLD, nt * YLD, nt * YLD + EPI_SCRATCH_FLOATS};
  const int ys = nt * YLD + (rx > EPI_SCRATCH_FLOATS ? rx : EPI_SCRATCH_FLOATS);
  return {ys, nt * YLD, ys + per * YLD};
}

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

// An environment switch (1 = set).
bool getenv_flag(const char* name) {
  const char* v = getenv(name);
  return v && v[0] == '1';
}
}  // namespace

bool encode_tmap_bf16(void* out, const void* ptr, int rows, int cols, int box_rows) {
  return tmap_2d(reinterpret_cast<CUtensorMap*>(out), ptr, rows, cols, box_rows);
}

// Shared memory: the ring (>= stages * (A tile + B tile), and, after the
// mainloop, the partial tile, the reduced rows and the epilogue scratch at
// the offsets of gemm_y_layout), in the early exchange layout the peers'
// partial rows past it (rx_off, in floats), then the tail at tail_off bytes.
// EPI: the fused epilogue (a.epi), one instantiation per kind.  TRACE: the
// instantiation that records the launch timeline (a.trace), launched only
// when a record is attached, so that the other carries no trace code.
template <int EPI, bool TRACE, bool TWO>
__global__ void __launch_bounds__(TC_THREADS) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmw,
                                                            const __grid_constant__ CUtensorMap tmx_hi,
                                                            const __grid_constant__ CUtensorMap tmx_lo,
                                                            GemmArgs a, int nt, int two, int stages,
                                                            int tail_off, int per, int ys_off, int scr_off,
                                                            int rx_off, int pre_rows) {
  namespace cg = cooperative_groups;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte-swizzled tiles, by pointer arithmetic
  // on the shared array so that the compiler keeps shared-memory addressing
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int b_bytes = (two ? 2 : 1) * nt * 128;
  uint8_t* sA = smem;
  uint8_t* sB = sA + stages * A_BYTES;
  // after the MMAs the ring is free: the partial tile, the partial rows the
  // cluster peers send, the reduced rows and the epilogue scratch live there
  // at the offsets of gemm_y_layout
  // the peers' partial rows: in the ring (rx_off < 0), or, in the early
  // exchange layout, in a region of their own past the ring that peers may
  // fill while this CTA's mainloop still uses the ring
  float* Yp = reinterpret_cast<float*>(smem);             // [nt][YLD]
  float* RX = rx_off >= 0 ? Yp + rx_off : Yp + nt * YLD;   // [S][per][YLD] peers' partial rows
  float* Ys = Yp + ys_off;                                 // reduced rows (unused when S = 1)
  float* scratch = Yp + scr_off;                           // epilogue scratch
  uint8_t* tail = smem + tail_off;
  float* rs_all = reinterpret_cast<float*>(tail);          // [TZ_TC] rstd of the slice's tokens
  float* rr_pre = rs_all + TZ_TC;                          // [pre_rows][NTILE] residual rows, or
  float2* rope_pre = reinterpret_cast<float2*>(rr_pre);    //   [pre_rows][head_dim / 2] RoPE rows
  float* gn_pre = rr_pre + pre_rows * NTILE;               // [NTILE] next-norm gains
  int* pos_pre = reinterpret_cast<int*>(gn_pre + NTILE);   // [EG] row positions
  int* req_pre = pos_pre + EG;                             // [EG] row requests
  uint64_t* full = reinterpret_cast<uint64_t*>(req_pre + EG);
  uint64_t* empty = full + stages;
  uint64_t* done = empty + stages;
  uint64_t* rxbar = done + 1;   // peers' partial rows landed
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(rxbar + 1);
  __shared__ int s_fail;
  __shared__ int s_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, split = blockIdx.y, z = blockIdx.z;
  const int S = gridDim.y;  // the cluster spans the splits of one tile
  const int n0 = tile * NTILE;
  const int t0 = z * TZ_TC;
  const int tn = min(TZ_TC, a.T - t0);
  const int k0 = split * a.kchunk;
  const int k1 = min(a.K, k0 + a.kchunk);
  const int nkb = cdiv_i(k1 - k0, 64);
  const int nmma = (two ? 2 : 1) * nt;
  const uint32_t ncols = nmma <= 32 ? 32 : (nmma <= 64 ? 64 : (nmma <= 128 ? 128 : 256));
  // early exchange: every CTA arms its receive barrier and arrives on the
  // cluster barrier at its start, so that after the mainloop a peer only has
  // to wait for that barrier (long complete by then), not for every peer's
  // mainloop, before sending its partial rows
  const bool early = S > 1 && rx_off >= 0;

  if (tid == 0) {
    if (TRACE) trace_at(a, 0);
    tc::prefetch_tmap(&tmw);
    tc::prefetch_tmap(&tmx_hi);
    if (two) tc::prefetch_tmap(&tmx_lo);
    for (int s = 0; s < stages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(done, 1);
    tc::mbar_init(rxbar, 1);
    if (early) {
      const int ta = min(tn, split * per), tb = min(tn, ta + per);
      tc::mbar_expect_tx(rxbar, (uint32_t)((S - 1) * (tb - ta) * YLD * 4));
    }
    tc::fence_mbar_init();
    s_fail = 0;
    tc::grid_dep_launch();
  }
  if (tid == 96 && a.pf_next) {
    // this CTA's share of the next GEMM's weights into L2, in 32 KB pieces
    const unsigned n_cta = gridDim.x * gridDim.y * gridDim.z;
    const unsigned cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    const size_t piece = 32768, pieces = (a.pf_bytes + piece - 1) / piece;
    for (size_t i = cta; i < pieces; i += n_cta) {
      const size_t off = i * piece;
      const size_t len = a.pf_bytes - off < piece ? a.pf_bytes - off : piece;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"((const char*)a.pf_next + off),
                   "r"((unsigned)(len & ~(size_t)15))
                   : "memory");
    }
  }
  __syncwarp();
  if (warp == 0) tc::tmem_alloc(tmem_holder, ncols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_holder;
  if (early) tc::cluster_arrive_release();  // this CTA's receive barrier is armed

  if (tid == 0) {
    // TMA producer.  Weights do not depend on the previous kernel: the first
    // stages' weight tiles go out before the grid dependency wait.
    const uint64_t pol = tc::policy_evict_first();
    const int pre = nkb < stages ? nkb : stages;
    for (int kb = 0; kb < pre; ++kb) {
      tc::mbar_expect_tx(&full[kb], A_BYTES + b_bytes);
      tc::tma_load_2d_hint(sA + kb * A_BYTES, &tmw, k0 + kb * 64, n0, &full[kb], pol);
    }
    // the rest of this CTA's weight tiles go to L2 now, so the ring refills
    // after the dependency wait do not pay a DRAM round trip
    for (int kb = pre; kb < nkb && kb < pre + L2_PREFETCH_BLOCKS; ++kb) tc::tma_prefetch_2d(&tmw, k0 + kb * 64, n0);
    tc::grid_dep_wait();
    if (TRACE) trace_at(a, 1);
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % stages;
      const int use = kb / stages;
      const int kx = k0 + kb * 64;
      if (kb >= pre) {
        if (!tc::mbar_wait(&empty[s], (use - 1) & 1)) { s_fail = 1; break; }
        tc::mbar_expect_tx(&full[s], A_BYTES + b_bytes);
        tc::tma_load_2d_hint(sA + s * A_BYTES, &tmw, kx, n0, &full[s], pol);
      }
      uint8_t* b = sB + s * b_bytes;
      tc::tma_load_2d(b, &tmx_hi, kx, t0, &full[s]);
      if (two) tc::tma_load_2d(b + nt * 128, &tmx_lo, kx, t0, &full[s]);
    }
  } else if (tid == 32) {
    // MMA issuer
    const uint32_t idesc = tc::idesc_bf16(NTILE, nmma);
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % stages;
      const int use = kb / stages;
      if (!tc::mbar_wait(&full[s], use & 1)) { s_fail = 1; break; }
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
  // the norm gains are weights: fetched before the dependency wait
  if (EPI == EPI_RESID && warp >= 2)
    for (int c = tid - 64; c < NTILE; c += 64) gn_pre[c] = n0 + c < a.e.H ? a.e.g_next[n0 + c] : 0.f;
  tc::grid_dep_wait();  // the epilogue reads and writes what earlier kernels touch
  // epilogue token range of this CTA: the whole slice, or its share of the cluster
  const int ea = S == 1 ? 0 : min(tn, split * per);
  const int eb = S == 1 ? tn : min(tn, ea + per);
  const int pre_n = min(EG, eb - ea);
  const bool pre_rope = EPI == EPI_QKV && a.e.head_dim <= NTILE;  // [EG][head_dim / 2] float2 fits rr_pre
  if (warp >= 2) {
    // warps 2 and 3 have no mainloop role: fetch the epilogue's inputs now
    // (the residual rows as one batch of loads, issued with the norm partials)
    const int it = tid - 64;
    // QKV: the rows' positions and slots go out with the norm partials
    int pos_l = 0, slot_l = 0;
    if (EPI == EPI_QKV && it < pre_n) {
      pos_l = a.e.row_pos[t0 + ea + it];
      slot_l = a.e.row_slot[t0 + ea + it];
    }
    constexpr int RR4 = EG * NTILE / 4 / 64;  // residual float4 per thread
    float4 rr[EPI == EPI_RESID ? RR4 : 1];
    const int n4 = pre_n * (NTILE / 4);
    if (EPI == EPI_RESID) {
#pragma unroll
      for (int u = 0; u < RR4; ++u) {
        const int x = it + 64 * u;
        if (x < n4)
          rr[u] = *reinterpret_cast<const float4*>(a.e.resid + (size_t)(t0 + ea + x / (NTILE / 4)) * a.e.H + n0 +
                                                   (x % (NTILE / 4)) * 4);
      }
    }
    if (a.e.ssq_in)
      for (int tl = it; tl < tn; tl += 64)
        rs_all[tl] = row_rstd(a.e, a.e.in_rows ? a.e.in_rows[t0 + tl] : t0 + tl);
    if (EPI == EPI_RESID) {
#pragma unroll
      for (int u = 0; u < RR4; ++u) {
        const int x = it + 64 * u;
        if (x < n4) reinterpret_cast<float4*>(rr_pre)[x] = rr[u];
      }
    }
    if (EPI == EPI_QKV) {
      if (it < pre_n) {
        pos_pre[it] = pos_l;
        req_pre[it] = a.e.plan->slot_req[slot_l];
      }
      asm volatile("bar.sync 1, 64;" ::: "memory");  // warps 2 and 3 only
      if (pre_rope) {
        const int half = a.e.head_dim / 2;
        for (int x = it; x < pre_n * half; x += 64) {
          const int tl = x / half;
          const int pc = min(max(pos_pre[tl], 0), a.e.cap - 1);  // a bad position is flagged by the epilogue
          rope_pre[x] = a.e.rope[(size_t)pc * half + x % half];
        }
      }
    }
  }
  const bool ok_done = tc::mbar_wait(done, 0);
  if (TRACE && tid == 0) trace_at(a, 4);
  tc::fence_after_sync();
  __syncthreads();
  const bool failed = !ok_done || s_fail;
  if (failed && tid == 0) set_err(a.e.err, DERR_TIMEOUT);

  // accumulator -> partial tile Yp[token][row]: hi column + lo column of each token
  const int row = warp * 32 + lane;
  for (int g = 0; g < nt / 16; ++g) {
    float vh[16], vl[16];
    tc::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + g * 16, vh);
    if (two) {
      tc::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + nt + g * 16, vl);
#pragma unroll
      for (int j = 0; j < 16; ++j) vh[j] += vl[j];
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) Yp[(g * 16 + j) * YLD + row] = failed ? 0.f : vh[j];
  }
  if (early) tc::fence_proxy_async_smem();  // the partial tile is read by bulk copies
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, ncols);
  if (TRACE && tid == 0) trace_at(a, 7);

  if (S == 1) {
    if (!failed) {
      for (int g0 = 0; g0 < tn; g0 += EG) {
        const int cnt = min(EG, tn - g0);
        EpiPre pre;
        pre.rs = a.e.ssq_in ? rs_all + g0 : nullptr;
        if (EPI == EPI_RESID) pre.gn = gn_pre;
        if (g0 == 0) {
          if (EPI == EPI_RESID) pre.rr = rr_pre;
          if (EPI == EPI_QKV) {
            pre.pos = pos_pre;
            pre.req = req_pre;
            if (pre_rope) pre.rope = rope_pre;
          }
        }
        apply_epilogue_k<EPI>(a, Yp + g0 * YLD, YLD, tile, t0 + g0, cnt, scratch, pre, Grp::block());
      }
    }
  } else {
    // split-K reduction: every CTA sends the rows of each peer's token range
    // to that peer with one bulk shared-memory copy; the owner adds the
    // partials in rank order
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int ta = min(tn, rank * per), tb = min(tn, ta + per);
    if (early) {
      tc::cluster_wait_acquire();  // every peer's receive barrier is armed (at its start)
    } else {
      if (tid == 0) tc::mbar_expect_tx(rxbar, (uint32_t)((S - 1) * (tb - ta) * YLD * 4));
      tc::fence_proxy_async_smem();
      cluster.sync();  // every partial tile is written and every receive barrier armed
    }
    if (TRACE && tid == 0) trace_at(a, 6);
    if (tid == 0) {
      for (int r = 0; r < S; ++r) {
        const int ra = min(tn, r * per), rb = min(tn, ra + per);
        if (r == rank || rb <= ra) continue;
        tc::bulk_s2s(tc::mapa(tc::smem_u32(RX + (size_t)rank * per * YLD), r), Yp + (size_t)ra * YLD,
                     (uint32_t)((rb - ra) * YLD * 4), tc::mapa(tc::smem_u32(rxbar), r));
      }
      tc::bulk_commit();
    }
    const bool rx_ok = tc::mbar_wait(rxbar, 0);
    if (TRACE && tid == 0) trace_at(a, 5);
    if (!rx_ok && tid == 0) set_err(a.e.err, DERR_TIMEOUT);
    for (int g0 = ta; g0 < tb; g0 += EG) {
      const int cnt = min(EG, tb - g0);
      // thread x: token x / 32, columns 4 (x % 32) .. +3; every partial is
      // loaded first, then they are added in rank (chunk) order within each
      // reduction group of kgroup ranks, and the group sums in group order
      const int gs = TWO ? a.kgroup : S;
      for (int x = tid; x < cnt * (NTILE / 4); x += TC_THREADS) {
        const int j = x / (NTILE / 4), c4 = (x % (NTILE / 4)) * 4;
        float4 v[MAX_CLUSTER];
#pragma unroll
        for (int sp = 0; sp < MAX_CLUSTER; ++sp)
          if (sp < S) {
            const float* src = sp == rank ? Yp + (size_t)(g0 + j) * YLD : RX + ((size_t)sp * per + (g0 - ta) + j) * YLD;
            v[sp] = *reinterpret_cast<const float4*>(src + c4);
          }
        float4 acc = v[0];
        if (!TWO) {
#pragma unroll
          for (int sp = 1; sp < MAX_CLUSTER; ++sp)
            if (sp < S) {
              acc.x += v[sp].x;
              acc.y += v[sp].y;
              acc.z += v[sp].z;
              acc.w += v[sp].w;
            }
        } else {
          // two groups (gemm_kgroup): ranks [0, gs) and [gs, S)
          float4 g1 = v[0];
#pragma unroll
          for (int sp = 1; sp < MAX_CLUSTER; ++sp)
            if (sp < S) {
              if (sp < gs) {
                acc.x += v[sp].x;
                acc.y += v[sp].y;
                acc.z += v[sp].z;
                acc.w += v[sp].w;
              } else if (sp == gs) {
                g1 = v[sp];
              } else {
                g1.x += v[sp].x;
                g1.y += v[sp].y;
                g1.z += v[sp].z;
                g1.w += v[sp].w;
              }
            }
          acc.x += g1.x;
          acc.y += g1.y;
          acc.z += g1.z;
          acc.w += g1.w;
        }
        *reinterpret_cast<float4*>(Ys + (size_t)j * YLD + c4) = acc;
      }
      __syncthreads();
      if (TRACE && tid == 0 && g0 == ta) trace_at(a, 2);
      if (!failed && rx_ok) {
        EpiPre pre;
        pre.rs = a.e.ssq_in ? rs_all + g0 : nullptr;
        if (EPI == EPI_RESID) pre.gn = gn_pre;
        if (g0 == ta) {
          if (EPI == EPI_RESID) pre.rr = rr_pre;
          if (EPI == EPI_QKV) {
            pre.pos = pos_pre;
            pre.req = req_pre;
            if (pre_rope) pre.rope = rope_pre;
          }
        }
        apply_epilogue_k<EPI>(a, Ys, YLD, tile, t0 + g0, cnt, scratch, pre, Grp::block());
      }
    }
    if (tid == 0) tc::bulk_wait_read();  // the copies have read this CTA's partial tile
  }
  if (EPI == EPI_ARGMAX && !failed) argmax_grid_finish(a, &s_flag);
  if (TRACE && tid == 0) trace_at(a, 3);
}

// Streaming variant for wide matrices without split K at decode shapes (the
// LM head: 512 weight tiles, at most 128 tokens): the CTAs (two per SM up to
// 64 tokens, one above) walk the tiles tile0, tile0 + gridDim.x, ... with one
// TMA ring that runs across tile boundaries, so the weight stream does not
// stop between tiles or waves.
// Warp 0 lane 0 loads, warp 1 lane 0 issues the MMAs into one of two tensor
// memory accumulators (tile i uses buffer i % 2), warps 2..5 drain an
// accumulator into shared memory and run the epilogue while the next tile's
// MMAs run.  The MMAs, the drain (hi + lo columns) and the epilogue are those
// of gemm_tc_kernel, so the results are the same bits.
constexpr int STREAM_THREADS = 192;
template <int EPI, bool TRACE>
__global__ void __launch_bounds__(STREAM_THREADS, 2)
    gemm_tc_stream_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx_hi,
                          const __grid_constant__ CUtensorMap tmx_lo, GemmArgs a, int nt, int stages) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int b_bytes = 2 * nt * 128;
  uint8_t* sA = smem;
  uint8_t* sB = sA + stages * A_BYTES;
  float* Yp = reinterpret_cast<float*>(sB + stages * b_bytes);  // [nt][YLD] drained accumulator
  float* rs_all = Yp + nt * YLD;                                 // [TZ_TC] rstd of the tokens
  uint64_t* full = reinterpret_cast<uint64_t*>(rs_all + TZ_TC);
  uint64_t* empty = full + stages;
  uint64_t* tfull = empty + stages;   // [2] accumulator written
  uint64_t* tempty = tfull + 2;       // [2] accumulator drained
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + 2);
  __shared__ int s_fail;
  __shared__ int s_efail;  // written by the epilogue warps only, read by them after their barrier
  __shared__ int s_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = cdiv_i(a.N, NTILE);
  const int my_tiles = n_tiles > (int)blockIdx.x ? cdiv_i(n_tiles - (int)blockIdx.x, (int)gridDim.x) : 0;
  const int nkb = cdiv_i(a.K, 64);
  const int total = my_tiles * nkb;  // k-blocks this CTA streams
  const int tn = min(TZ_TC, a.T);
  const int nmma = 2 * nt;
  // per accumulator: 2 x ncols columns of tensor memory, 256 per CTA up to 64
  // tokens (two CTAs per SM), 512 above (one CTA per SM)
  const uint32_t ncols = nmma <= 32 ? 32 : (nmma <= 64 ? 64 : (nmma <= 128 ? 128 : 256));

  if (tid == 0) {
    if (TRACE) trace_at(a, 0);
    tc::prefetch_tmap(&tmw);
    tc::prefetch_tmap(&tmx_hi);
    tc::prefetch_tmap(&tmx_lo);
    for (int s = 0; s < stages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], 128);
    }
    tc::fence_mbar_init();
    s_fail = 0;
    s_efail = 0;
    tc::grid_dep_launch();
  }
  if (warp == 1) tc::tmem_alloc(tmem_holder, 2 * ncols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_holder;

  if (tid == 0) {
    // TMA producer: the weight tiles of the first stages go out before the
    // grid dependency wait, the token planes after it
    const uint64_t pol = tc::policy_evict_first();
    const int pre = total < stages ? total : stages;
    for (int it = 0; it < pre; ++it) {
      const int tile = blockIdx.x + (it / nkb) * gridDim.x, kb = it % nkb;
      tc::mbar_expect_tx(&full[it], A_BYTES + b_bytes);
      tc::tma_load_2d_hint(sA + it * A_BYTES, &tmw, kb * 64, tile * NTILE, &full[it], pol);
    }
    tc::grid_dep_wait();
    if (TRACE) trace_at(a, 1);
    for (int it = 0; it < total; ++it) {
      const int s = it % stages, use = it / stages;
      const int tile = blockIdx.x + (it / nkb) * gridDim.x, kb = it % nkb;
      if (it >= pre) {
        if (!tc::mbar_wait(&empty[s], (use - 1) & 1)) { s_fail = 1; break; }
        tc::mbar_expect_tx(&full[s], A_BYTES + b_bytes);
        tc::tma_load_2d_hint(sA + s * A_BYTES, &tmw, kb * 64, tile * NTILE, &full[s], pol);
      }
      uint8_t* b = sB + s * b_bytes;
      tc::tma_load_2d(b, &tmx_hi, kb * 64, 0, &full[s]);
      tc::tma_load_2d(b + nt * 128, &tmx_lo, kb * 64, 0, &full[s]);
    }
  } else if (tid == 32) {
    // MMA issuer: tile i accumulates in buffer i % 2 once the epilogue has
    // drained that buffer's previous tile
    const uint32_t idesc = tc::idesc_bf16(NTILE, nmma);
    int it = 0;
    for (int li = 0; li < my_tiles && !s_fail; ++li) {
      const int buf = li & 1;
      if (li >= 2 && !tc::mbar_wait(&tempty[buf], ((li >> 1) - 1) & 1)) { s_fail = 1; break; }
      tc::fence_after_sync();
      const uint32_t acc = tmem + (uint32_t)buf * ncols;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int s = it % stages, use = it / stages;
        if (!tc::mbar_wait(&full[s], use & 1)) { s_fail = 1; break; }
        tc::fence_after_sync();
        const uint32_t a_base = tc::smem_u32(sA + s * A_BYTES);
        const uint32_t b_base = tc::smem_u32(sB + s * b_bytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(acc, tc::sdesc_sw128(a_base + kk * 32), tc::sdesc_sw128(b_base + kk * 32), idesc,
                       (kb > 0 || kk > 0) ? 1u : 0u);
        tc::mma_commit(&empty[s]);
      }
      tc::mma_commit(&tfull[buf]);
    }
  } else if (warp >= 2) {
    // epilogue warps: warp w drains tensor-memory lanes 32 (w % 4) .. +31
    const Grp eg{tid - 64, 128, 1};
    const int q = warp & 3, row = q * 32 + lane;
    tc::grid_dep_wait();  // the norm partials are written by the previous kernel
    if (a.e.ssq_in)
      for (int tl = eg.tid; tl < tn; tl += 128)
        rs_all[tl] = row_rstd(a.e, a.e.in_rows ? a.e.in_rows[tl] : tl);
    eg.sync();
    for (int li = 0; li < my_tiles; ++li) {
      const int buf = li & 1, tile = blockIdx.x + li * gridDim.x;
      const bool ok = tc::mbar_wait(&tfull[buf], (li >> 1) & 1);
      tc::fence_after_sync();
      const uint32_t acc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)buf * ncols;
      for (int g = 0; g < nt / 16; ++g) {
        float vh[16], vl[16];
        tc::tmem_ld16(acc + g * 16, vh);
        tc::tmem_ld16(acc + nt + g * 16, vl);
#pragma unroll
        for (int j = 0; j < 16; ++j) Yp[(g * 16 + j) * YLD + row] = ok ? vh[j] + vl[j] : 0.f;
      }
      tc::fence_before_sync();
      tc::mbar_arrive(&tempty[buf]);  // this lane's accumulator columns are read
      if (!ok) s_efail = 1;
      eg.sync();
      if (s_efail) break;  // the same decision in every epilogue thread
      // the row scales come prefetched, so the epilogue needs no scratch
      for (int g0 = 0; g0 < tn; g0 += EG) {
        EpiPre pre;
        pre.rs = a.e.ssq_in ? rs_all + g0 : nullptr;
        apply_epilogue_k<EPI>(a, Yp + g0 * YLD, YLD, tile, g0, min(EG, tn - g0), nullptr, pre, eg);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  const bool failed = s_fail || s_efail;
  if (failed && tid == 0) set_err(a.e.err, DERR_TIMEOUT);
  if (warp == 1) tc::tmem_dealloc(tmem, 2 * ncols);
  if (EPI == EPI_ARGMAX && !failed) argmax_grid_finish(a, &s_flag);
  if (TRACE && tid == 0) trace_at(a, 3);
}

// Many-slice variant (more than two 128-token slices, e.g. prefill and the
// batched round): one CTA per (128-row weight tile, NT-token slice) runs the S
// K chunks of the split rule one after another.  Each chunk's MMAs start a
// fresh accumulator (two in TMEM, so the next chunk's MMAs overlap this
// chunk's drain), and four drain warps add the chunk sums into running sums
// held in registers (thread = weight row, one register per token), in chunk
// order: p0 + p1 + ... + p(S-1), the clustered kernel's reduction, so a
// token's bits do not depend on which kernel ran it.  After the last chunk
// the sums go to shared memory over the then idle operand ring, where all
// eight warps run the epilogue.  Warp 0: TMA producer; warp 1: MMA issuer;
// warps 4-7: drain.  Inputs are bf16 hi + lo planes (single-plane launches
// take the clustered kernel).
// NT = 128: one CTA per SM, four 48 KB stages.  NT = 64: two CTAs per SM,
// three 32 KB stages, twice the work units, so that narrow matrices (few
// weight tiles) still occupy every SM.  A matrix with several reduction
// groups (gemm_kgroup) gives each group a CTA of a cluster: CTA g sums its
// group's chunks in order, then each CTA adds the group sums in group order
// for its share of the slice's tokens (read from the peers' shared memory)
// and runs their epilogue; the clustered kernel adds its ranks' partials in
// the same two levels.
constexpr int SEQ_THREADS = 256;

template <int EPI, bool TRACE, int NT>
__global__ void __launch_bounds__(SEQ_THREADS, NT == 64 ? 2 : 1)
    gemm_tc_seq_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx_hi,
                       const __grid_constant__ CUtensorMap tmx_lo, GemmArgs a, int stages) {
  static_assert(NT == 64 || NT == 128, "token slice of 64 or 128");
  constexpr int nt = NT;
  constexpr int two = 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int b_bytes = (two ? 2 : 1) * nt * 128;
  uint8_t* sA = smem;
  uint8_t* sB = sA + stages * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + stages * b_bytes);
  uint64_t* empty = full + stages;
  uint64_t* accf = empty + stages;  // [2] chunk accumulator ready
  uint64_t* acce = accf + 2;        // [2] chunk accumulator drained
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acce + 2);
  __shared__ int s_fail;
  __shared__ int s_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // reduction groups of the tile: CTA grp of a cluster of P takes chunks
  // [grp * gs, (grp + 1) * gs)
  const int S = a.splits, kpc = a.kchunk / 64, nkb_all = cdiv_i(a.K, 64);
  const int gs = a.kgroup > 0 ? a.kgroup : S;
  const int P = cdiv_i(S, gs);
  const int unit = blockIdx.x / P, grp = blockIdx.x % P;
  const int c_beg = grp * gs, c_end = min(S, c_beg + gs);
  const int kb_beg = min(nkb_all, c_beg * kpc), kb_end = min(nkb_all, c_end * kpc);
  const int nkb = kb_end - kb_beg;
  // after the mainloop, over the ring: the group sum [nt], the reduced rows of
  // this CTA's tokens [per] (clusters only) and the epilogue scratch
  const int per = cdiv_i(NT, P);
  float* Ysum = reinterpret_cast<float*>(smem);                   // [nt][YLD]
  float* Yred = Ysum + (size_t)nt * YLD;                          // [per][YLD]
  float* scratch = P > 1 ? Yred + (size_t)per * YLD : Yred;
  // the slices of one weight tile are adjacent in launch order, so the tile
  // comes from HBM once and from L2 for the other slices
  const int nz = cdiv_i(a.T, NT);
  const int tile = unit / nz, z = unit % nz;
  const int n0 = tile * NTILE;
  const int t0 = z * NT;
  const int tn = min(NT, a.T - t0);
  const int nmma = (two ? 2 : 1) * nt;
  constexpr uint32_t bufcols = 2 * NT;

  if (tid == 0) {
    if (TRACE) trace_at(a, 0);
    tc::prefetch_tmap(&tmw);
    tc::prefetch_tmap(&tmx_hi);
    if (two) tc::prefetch_tmap(&tmx_lo);
    for (int st = 0; st < stages; ++st) {
      tc::mbar_init(&full[st], 1);
      tc::mbar_init(&empty[st], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accf[b], 1);
      tc::mbar_init(&acce[b], 4);  // one arrival per drain warp
    }
    tc::fence_mbar_init();
    s_fail = 0;
    tc::grid_dep_launch();
  }
  __syncwarp();
  if (warp == 0) tc::tmem_alloc(tmem_holder, 2 * bufcols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_holder;

  const int nc = c_end - c_beg;  // this CTA's chunks
  if (tid == 0) {
    // TMA producer: every k block of the CTA's chunks, chunk after chunk; the
    // first stages' weight tiles go out before the grid dependency wait
    const uint64_t pol = tc::policy_evict_first();
    const int pre = nkb < stages ? nkb : stages;
    for (int kb = 0; kb < pre; ++kb) {
      tc::mbar_expect_tx(&full[kb], A_BYTES + b_bytes);
      tc::tma_load_2d_hint(sA + kb * A_BYTES, &tmw, (kb_beg + kb) * 64, n0, &full[kb], pol);
    }
    for (int kb = pre; kb < nkb && kb < pre + L2_PREFETCH_BLOCKS; ++kb)
      tc::tma_prefetch_2d(&tmw, (kb_beg + kb) * 64, n0);
    tc::grid_dep_wait();
    if (TRACE) trace_at(a, 1);
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb % stages;
      const int use = kb / stages;
      const int kx = (kb_beg + kb) * 64;
      if (kb >= pre) {
        if (!tc::mbar_wait(&empty[st], (use - 1) & 1)) { s_fail = 1; break; }
        tc::mbar_expect_tx(&full[st], A_BYTES + b_bytes);
        tc::tma_load_2d_hint(sA + st * A_BYTES, &tmw, kx, n0, &full[st], pol);
        if (kb + L2_PREFETCH_BLOCKS < nkb) tc::tma_prefetch_2d(&tmw, kx + L2_PREFETCH_BLOCKS * 64, n0);
      }
      uint8_t* b = sB + st * b_bytes;
      tc::tma_load_2d(b, &tmx_hi, kx, t0, &full[st]);
      if (two) tc::tma_load_2d(b + nt * 128, &tmx_lo, kx, t0, &full[st]);
    }
  } else if (tid == 32) {
    // MMA issuer: the CTA's lc-th chunk accumulates into TMEM buffer lc & 1
    const uint32_t idesc = tc::idesc_bf16(NTILE, nmma);
    int kb = 0;
    for (int lc = 0; lc < nc && !s_fail; ++lc) {
      const int b = lc & 1;
      if (lc >= 2 && !tc::mbar_wait(&acce[b], ((lc >> 1) - 1) & 1)) { s_fail = 1; break; }
      tc::fence_after_sync();
      const uint32_t d = tmem + (uint32_t)b * bufcols;
      const int kend = min(nkb_all, (c_beg + lc + 1) * kpc) - kb_beg;
      for (int k0 = kb; kb < kend; ++kb) {
        const int st = kb % stages;
        if (!tc::mbar_wait(&full[st], (kb / stages) & 1)) { s_fail = 1; break; }
        tc::fence_after_sync();
        const uint32_t a_base = tc::smem_u32(sA + st * A_BYTES);
        const uint32_t b_base = tc::smem_u32(sB + st * b_bytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(d, tc::sdesc_sw128(a_base + kk * 32), tc::sdesc_sw128(b_base + kk * 32), idesc,
                       (kb > k0 || kk > 0) ? 1u : 0u);
        tc::mma_commit(&empty[st]);
      }
      tc::mma_commit(&accf[b]);
    }
  }
  float acc[nt];  // drain warps: running sums of weight row q*32 + lane, one per token
  if (warp >= 4) {
    // drain: chunk sums (hi + lo products) added to the running sums in chunk order
    const int q = warp & 3;
    for (int c = 0; c < nc; ++c) {
      const int b = c & 1;
      if (!tc::mbar_wait(&accf[b], (c >> 1) & 1)) {
        s_fail = 1;
        break;
      }
      tc::fence_after_sync();
      const uint32_t taddr = tmem + (uint32_t)b * bufcols + ((uint32_t)(q * 32) << 16);
#pragma unroll
      for (int g = 0; g < nt / 16; ++g) {
        float vh[16], vl[16];
        tc::tmem_ld16x2(taddr + g * 16, taddr + nt + g * 16, vh, vl);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float v = vh[j] + vl[j];
          acc[g * 16 + j] = c == 0 ? v : acc[g * 16 + j] + v;
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acce[b]);
    }
  }
  __syncwarp();
  tc::grid_dep_wait();  // the epilogue reads and writes what earlier kernels touch
  tc::fence_before_sync();
  __syncthreads();  // every chunk drained: the MMAs, and so the ring's TMA writes, are complete
  if (TRACE && tid == 0) trace_at(a, 4);
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 2 * bufcols);
  }
  const bool failed = s_fail != 0;
  if (failed && tid == 0) set_err(a.e.err, DERR_TIMEOUT);
  if (P == 1) {
    if (failed) return;
    if (warp >= 4) {
      const int row = (warp & 3) * 32 + lane;
#pragma unroll
      for (int t = 0; t < nt; ++t) Ysum[(size_t)t * YLD + row] = acc[t];
    }
    __syncthreads();
    for (int g0 = 0; g0 < tn; g0 += EG) {
      const int cnt = min(EG, tn - g0);
      apply_epilogue_k<EPI>(a, Ysum + (size_t)g0 * YLD, YLD, tile, t0 + g0, cnt, scratch, EpiPre(), Grp::block());
    }
    if (EPI == EPI_ARGMAX) argmax_grid_finish(a, &s_flag);
  } else {
    // every CTA of the cluster passes both cluster barriers, failed or not
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    if (warp >= 4) {
      const int row = (warp & 3) * 32 + lane;
#pragma unroll
      for (int t = 0; t < nt; ++t) Ysum[(size_t)t * YLD + row] = acc[t];
    }
    cluster.sync();  // every group sum of the slice is in its CTA's shared memory
    // this CTA's tokens: the group sums added in group order
    const int ta = min(tn, grp * per), tb = min(tn, ta + per);
    for (int x = tid; x < (tb - ta) * (NTILE / 4); x += SEQ_THREADS) {
      const int j = x / (NTILE / 4), c4 = (x % (NTILE / 4)) * 4;
      const size_t off = (size_t)(ta + j) * YLD + c4;
      float4 r = *reinterpret_cast<const float4*>(cluster.map_shared_rank(Ysum, 0) + off);
      for (int g = 1; g < P; ++g) {
        const float4 v = *reinterpret_cast<const float4*>(cluster.map_shared_rank(Ysum, g) + off);
        r.x += v.x;
        r.y += v.y;
        r.z += v.z;
        r.w += v.w;
      }
      *reinterpret_cast<float4*>(Yred + (size_t)j * YLD + c4) = r;
    }
    __syncthreads();
    if (!failed)
      for (int g0 = ta; g0 < tb; g0 += EG) {
        const int cnt = min(EG, tb - g0);
        apply_epilogue_k<EPI>(a, Yred + (size_t)(g0 - ta) * YLD, YLD, tile, t0 + g0, cnt, scratch, EpiPre(),
                              Grp::block());
      }
    if (EPI == EPI_ARGMAX) argmax_grid_finish(a, &s_flag);  // every CTA of the grid counts itself
    cluster.sync();  // the peers have read this CTA's group sums
  }
  if (TRACE && tid == 0) trace_at(a, 3);
}

template <int EPI, bool TRACE, int NT>
static bool launch_gemm_tc_seq(const GemmArgs& a, cudaStream_t s, bool pdl) {
  CUtensorMap tmw, tmh, tml;
  if (!tmap_2d(&tmw, a.w, a.N, a.K, NTILE)) return false;
  const int nt = NT;
  if (!a.x_lo || !tmap_2d(&tmh, a.x, a.T, a.K, nt) || !tmap_2d(&tml, a.x_lo, a.T, a.K, nt)) return false;
  const int stage_bytes = A_BYTES + 2 * nt * 128;
  // 64-token slices: three stages keep two CTAs per SM; a grid that fits one
  // CTA per SM (narrow matrices) takes a six-stage ring instead, since each
  // CTA's k loop is bound by the stages it has in flight
  static int n_sm = 0;
  if (!n_sm) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n_sm = 1;
  }
  const int ctas = cdiv_i(a.N, NTILE) * cdiv_i(a.T, NT) * cdiv_i(a.splits, a.kgroup > 0 ? a.kgroup : a.splits);
  const int stages = NT == 128 ? 4 : (ctas <= n_sm ? 6 : 3);
  const int gsz = a.kgroup > 0 ? a.kgroup : a.splits;
  const int P = cdiv_i(a.splits, gsz);  // reduction groups: CTAs per cluster
  if (P > 8) return false;
  const size_t ring = (size_t)stages * stage_bytes;
  // aliases the ring after the mainloop: group sum, reduced rows, scratch
  const size_t epi = ((size_t)(nt + (P > 1 ? cdiv_i(nt, P) : 0)) * YLD + EPI_SCRATCH_FLOATS) * 4;
  if (epi > ring) return false;
  const size_t smem = 1024 + ring + (2 * stages + 4) * 8 + 16;
  if (smem > 227 * 1024) return false;
  if (!kernel_smem_at_least(reinterpret_cast<const void*>(gemm_tc_seq_kernel<EPI, TRACE, NT>), smem)) return false;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(cdiv_i(a.N, NTILE) * cdiv_i(a.T, NT) * P);
  cfg.blockDim = dim3(SEQ_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  int na = 0;
  if (P > 1) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = P;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemm_tc_seq_kernel<EPI, TRACE, NT>, tmw, tmh, tml, a, stages) == cudaSuccess;
}

template <int EPI, bool TRACE, bool TWO>
static bool launch_gemm_tc_kt(const GemmArgs& a, cudaStream_t s, bool pdl) {
  if (a.splits < 1 || a.splits > MAX_CLUSTER) return false;
  CUtensorMap tmw, tmh, tml;
  if (!tmap_2d(&tmw, a.w, a.N, a.K, NTILE)) return false;
  const int nt = ((a.T < TZ_TC ? a.T : TZ_TC) + 15) / 16 * 16;
  if (!tmap_2d(&tmh, a.x, a.T, a.K, nt)) return false;
  const int two = a.x_lo != nullptr;
  if (two) {
    if (!tmap_2d(&tml, a.x_lo, a.T, a.K, nt)) return false;
  } else {
    tml = tmh;
  }
  const int nkb = cdiv_i(a.kchunk, 64);
  const int stage_bytes = A_BYTES + (two ? 2 : 1) * nt * 128;
  const int per = cdiv_i(a.T < TZ_TC ? a.T : TZ_TC, a.splits);  // tokens each cluster rank reduces
  bool compact = false;
  auto smem_of = [&](int st) {
    int ring = st * stage_bytes;
    const int y_bytes = gemm_y_layout(nt, a.splits, per, compact).floats * 4;
    if (ring < y_bytes) ring = y_bytes;
    ring = (ring + 1023) / 1024 * 1024;
    return std::make_pair((size_t)1024 + ring + TAIL_BYTES, ring);
  };
  // early exchange layout (decode shapes with split K): the peers' partial
  // rows in a region past the ring, the epilogue scratch in the ring after
  // the partial tile and this CTA's reduced rows, and the tail's prefetch
  // rows sized to the tokens this CTA reduces
  const int pre_rows_e = per < EG ? per : EG;
  const int rx_bytes = a.splits * per * YLD * 4;
  const int tail_e = TZ_TC * 4 + pre_rows_e * NTILE * 4 + NTILE * 4 + 2 * EG * 4 + 16 * 8 + 64;
  auto early_of = [&](int st) {  // (total bytes, ring bytes)
    int ring = st * stage_bytes;
    const int y_bytes = ((nt + per) * YLD + EPI_SCRATCH_FLOATS) * 4;
    if (ring < y_bytes) ring = y_bytes;
    ring = (ring + 1023) / 1024 * 1024;
    return std::make_pair((size_t)1024 + ring + rx_bytes + tail_e, ring);
  };
  if (a.splits > 1 && a.T <= 2 * 64 + 1 && !getenv_flag("GOCR_LATE_EXCHANGE")) {
    int st = DECODE_STAGE_CAP < nkb ? DECODE_STAGE_CAP : nkb;
    while (st > 2 && early_of(st).first > TWO_CTA_SMEM) --st;
    if (st < 1) st = 1;
    if (early_of(st).first <= TWO_CTA_SMEM) {
      const int ring = early_of(st).second;
      const size_t smem = early_of(st).first;
      if (!kernel_smem_at_least(reinterpret_cast<const void*>(gemm_tc_kernel<EPI, TRACE, TWO>), smem, true))
        return false;
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(cdiv_i(a.N, NTILE), a.splits, cdiv_i(a.T, TZ_TC));
      cfg.blockDim = dim3(TC_THREADS);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = s;
      cudaLaunchAttribute at[2];
      int na = 0;
      at[na].id = cudaLaunchAttributeClusterDimension;
      at[na].val.clusterDim.x = 1;
      at[na].val.clusterDim.y = a.splits;
      at[na].val.clusterDim.z = 1;
      ++na;
      if (pdl) {
        at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
      }
      cfg.attrs = at;
      cfg.numAttrs = na;
      const int ys = nt * YLD, scr = (nt + per) * YLD, rx = ring / 4;
      return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<EPI, TRACE, TWO>, tmw, tmh, tml, a, nt, two, st,
                                ring + rx_bytes, per, ys, scr, rx, pre_rows_e) == cudaSuccess;
    }
  }
  int stages = (SMEM_CAP - 1024 - TAIL_BYTES) / stage_bytes;
  if (stages > 6) stages = 6;
  if (a.T <= 2 * 64 + 1) {
    // decode shapes: the deepest ring (at most DECODE_STAGE_CAP, at least
    // two stages) that keeps two CTAs per SM, in the compact layout if the
    // regular one does not allow that
    if (stages > DECODE_STAGE_CAP) stages = DECODE_STAGE_CAP;
    if (stages > nkb) stages = nkb;
    while (stages > 2 && smem_of(stages).first > TWO_CTA_SMEM) --stages;
    if (smem_of(stages).first > TWO_CTA_SMEM && (a.splits == 1 || per <= EG)) {
      compact = true;
      stages = DECODE_STAGE_CAP;
      while (stages > 2 && smem_of(stages).first > TWO_CTA_SMEM) --stages;
    }
  }
  if (stages > nkb) stages = nkb;
  if (stages < 1) stages = 1;
  const int ring = smem_of(stages).second;
  const size_t smem = smem_of(stages).first;
  const YLayout yl = gemm_y_layout(nt, a.splits, per, compact);
  if (smem > 227 * 1024) return false;
  if (!kernel_smem_at_least(reinterpret_cast<const void*>(gemm_tc_kernel<EPI, TRACE, TWO>), smem, true)) return false;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(cdiv_i(a.N, NTILE), a.splits, cdiv_i(a.T, TZ_TC));
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  int na = 0;
  at[na].id = cudaLaunchAttributeClusterDimension;
  at[na].val.clusterDim.x = 1;
  at[na].val.clusterDim.y = a.splits;
  at[na].val.clusterDim.z = 1;
  ++na;
  if (pdl) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<EPI, TRACE, TWO>, tmw, tmh, tml, a, nt, two, stages, ring, per,
                            yl.ys, yl.scratch, -1, EG) == cudaSuccess;
}

// Up to 64 tokens two CTAs per SM, above one (at most the tile count), with
// the deepest ring that fits their shared memory; at most 128 tokens.
template <int EPI, bool TRACE>
static bool launch_gemm_tc_stream(const GemmArgs& a, cudaStream_t s, bool pdl) {
  CUtensorMap tmw, tmh, tml;
  if (a.T < 1 || a.T > 128) return false;
  const int nt = (a.T + 15) / 16 * 16;
  const int per_sm = nt <= 64 ? 2 : 1;
  const size_t budget = per_sm == 2 ? TWO_CTA_SMEM : (size_t)227 * 1024;
  if (!tmap_2d(&tmw, a.w, a.N, a.K, NTILE) || !tmap_2d(&tmh, a.x, a.T, a.K, nt) ||
      !tmap_2d(&tml, a.x_lo, a.T, a.K, nt))
    return false;
  const int stage_bytes = A_BYTES + 2 * nt * 128;
  const size_t fixed = 1024 + (size_t)nt * YLD * 4 + TZ_TC * 4 + 64 + 16;
  int stages = (int)((budget - fixed) / (stage_bytes + 16));
  if (stages > 8) stages = 8;
  if (stages < 2) return false;
  const size_t smem = fixed + (size_t)stages * (stage_bytes + 16);
  if (!kernel_smem_at_least(reinterpret_cast<const void*>(gemm_tc_stream_kernel<EPI, TRACE>), smem)) return false;
  const int n_tiles = cdiv_i(a.N, NTILE);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(n_tiles < per_sm * SM_COUNT ? n_tiles : per_sm * SM_COUNT);
  cfg.blockDim = dim3(STREAM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemm_tc_stream_kernel<EPI, TRACE>, tmw, tmh, tml, a, nt, stages) == cudaSuccess;
}

// Launches of more than two 128-token slices of hi + lo planes run the K
// chunks in one CTA (gemm_tc_seq_kernel); the others split them over a
// cluster.  Both add the chunk sums in chunk order.
static int seq_slice_tokens() {
  static int nt = 0;
  if (!nt) {
    const char* v = getenv("GOCR_SEQ_NT");
    nt = v && atoi(v) == 128 ? 128 : 64;
  }
  return nt;
}

template <int EPI>
static bool launch_gemm_tc_k(const GemmArgs& a, cudaStream_t s, bool pdl) {
  // the LM head at decode shapes (up to 128 tokens): streaming CTAs instead of waves of tile CTAs
  if constexpr (EPI == EPI_ARGMAX) {
    if (a.splits == 1 && a.T <= 128 && a.x_lo && !getenv_flag("GOCR_LM_WAVES"))
      return a.trace ? launch_gemm_tc_stream<EPI, true>(a, s, pdl) : launch_gemm_tc_stream<EPI, false>(a, s, pdl);
  }
  if (cdiv_i(a.T, TZ_TC) > 2 && a.x_lo) {
    if (seq_slice_tokens() == 128)
      return a.trace ? launch_gemm_tc_seq<EPI, true, 128>(a, s, pdl) : launch_gemm_tc_seq<EPI, false, 128>(a, s, pdl);
    return a.trace ? launch_gemm_tc_seq<EPI, true, 64>(a, s, pdl) : launch_gemm_tc_seq<EPI, false, 64>(a, s, pdl);
  }
  // a separate instantiation for two reduction groups, so that the common
  // one-group kernel keeps its code (its timing under programmatic dependent
  // launch is sensitive to register allocation)
  if (a.kgroup > 0 && a.kgroup < a.splits) {
    if (2 * a.kgroup < a.splits) return false;  // at most two groups
    return a.trace ? launch_gemm_tc_kt<EPI, true, true>(a, s, pdl) : launch_gemm_tc_kt<EPI, false, true>(a, s, pdl);
  }
  return a.trace ? launch_gemm_tc_kt<EPI, true, false>(a, s, pdl) : launch_gemm_tc_kt<EPI, false, false>(a, s, pdl);
}

bool launch_gemm_tc(const GemmArgs& a, cudaStream_t s, bool pdl) {
  switch (a.epi) {
    case EPI_STORE: return launch_gemm_tc_k<EPI_STORE>(a, s, pdl);
    case EPI_RESID: return launch_gemm_tc_k<EPI_RESID>(a, s, pdl);
    case EPI_QKV: return launch_gemm_tc_k<EPI_QKV>(a, s, pdl);
    case EPI_SWIGLU: return launch_gemm_tc_k<EPI_SWIGLU>(a, s, pdl);
    case EPI_ARGMAX: return launch_gemm_tc_k<EPI_ARGMAX>(a, s, pdl);
  }
  return false;
}

}  // namespace gocr
