// Grouped-query attention of a window of query rows against a contiguous
// per-request KV cache, with the two mask modes of the round expressed as one
// per-row key limit: row t reads keys 0..lim[t].
//   draft  (GravityOCR review §3.2): boundary row lim = p (causal), [M] rows
//          lim = p + B (the cache plus the whole window, bidirectional);
//   verify / AR / prefill: lim = the row's own position (token-causal).
//
// Keys are visited in fixed chunks at absolute positions (64 keys for the
// CUDA-core kernel, 32 for the tensor-core one).  A chunk with no key visible
// to a row leaves that row's running (max, sum, output) bit-for-bit unchanged
// (scale exp(0) = 1, zero contributions), so a row's result does not depend
// on how many other rows share the launch: the AR step and the verify row at
// the same position give identical bits.
//
// bf16 models: tensor-core kernels.  q and the KV cache are stored as bf16
// hi + lo planes (written once by the QKV epilogue); QK^T takes qh kh + qh kl
// + ql kh and PV takes P vh + P vl (P in bf16), accumulating in fp32.  The R
// CTAs of one (kv head, query-row group) split the chunks, rank r visiting
// chunks r, r + R, ... with an online softmax, and write partial (max, sum,
// output) rows to global memory; a merge kernel adds them in rank order.  R
// is fixed per handle (attention_ranks: 48 for one request, fewer for a
// batch).  Two partial kernels, one per handle:
//   attention_part_kernel: 64-row groups on mma.sync tiles (this file and
//     attn_core.cuh), the lighter footprint that wins when a rank reads one
//     or two chunks;
//   attention_tc_part_kernel: 128-row groups on tcgen05 (attn_tc.cuh), for
//     handles whose ranks average at least four chunks.
// Both have an instantiation for rows with a second key interval (the
// joint-training mask).  The partial rows of the ranks are then added in rank
// order by attention_merge_kernel, or with at most eight ranks by
// attention_merge_few_kernel (one warp per row, no barrier).
// There is no thread-block cluster: the CTAs need no co-scheduling.  Under
// programmatic dependent launch a CTA fetches its first chunk before the
// grid-dependency wait when that chunk holds only committed cache positions
// (below the round-start cache length, which no kernel of the forward
// writes).  The result is written as the O projection's input planes.
// fp32 models: CUDA-core kernel with one CTA sweeping every chunk.
#include <cstdlib>
#include <cstring>

#include "attn_core.cuh"
#include "attn_tc.cuh"
#include "tc.cuh"

namespace gocr {

namespace {
constexpr int ROWS = 128;   // CUDA-core kernel: query rows (token, q head) per CTA
constexpr int CH = 64;      // keys per chunk
}  // namespace

// ---------------------------------------------------------------- CUDA-core path (fp32)

template <int D>
__global__ void __launch_bounds__(ROWS) attention_simt_kernel(AttnArgs a) {
  extern __shared__ float sm[];
  float* Qs = sm;                     // [ROWS][D + 1]
  float* Os = Qs + ROWS * (D + 1);    // [ROWS][D + 1]
  float* Ks = Os + ROWS * (D + 1);    // [CH][D]
  float* Vs = Ks + CH * D;            // [CH][D]
  __shared__ int s_maxlim;

  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int G = a.Hq / a.Hkv;
  const int kvh = blockIdx.y;
  const int slot = blockIdx.z;
  int req = 0, row0 = 0, nrows = a.T;
  if (a.plan) {
    req = a.plan->slot_req[slot];
    row0 = a.plan->slot_row0[slot];
    nrows = a.plan->slot_nrows[slot];
  }
  const int qr0 = blockIdx.x * ROWS;
  if (qr0 >= nrows * G) return;

  const float* kc = reinterpret_cast<const float*>(a.k_hi) + (size_t)req * a.req_stride + (size_t)kvh * a.cap * D;
  const float* vc = reinterpret_cast<const float*>(a.v_hi) + (size_t)req * a.req_stride + (size_t)kvh * a.cap * D;
  const float* qf = reinterpret_cast<const float*>(a.q_hi);
  float* o = reinterpret_cast<float*>(a.o_hi);

  const int i = threadIdx.x;
  const int gi = qr0 + i;
  const bool valid = gi < nrows * G;
  const int t = row0 + (valid ? gi / G : 0);
  const int hq = kvh * G + (valid ? gi % G : 0);
  const int lim = valid ? a.row_lim[t] : -1;
  const int lo2 = valid && a.row_lo2 ? a.row_lo2[t] : 1;
  const int hi2 = valid && a.row_hi2 ? a.row_hi2[t] : 0;

  if (i == 0) s_maxlim = -1;
  __syncthreads();
  if (valid) atomicMax(&s_maxlim, lim);
  if (valid && hi2 >= lo2) atomicMax(&s_maxlim, hi2);
  for (int dd = 0; dd < D; ++dd) {
    Qs[i * (D + 1) + dd] = valid ? qf[((size_t)t * a.Hq + hq) * D + dd] : 0.f;
    Os[i * (D + 1) + dd] = 0.f;
  }
  __syncthreads();
  const int maxlim = min(s_maxlim, a.cap - 1);
  const int n_chunks = maxlim < 0 ? 0 : maxlim / CH + 1;

  float m = -INFINITY, l = 0.f;
  for (int c = 0; c < n_chunks; ++c) {
    const int kbase = c * CH;
    for (int x = i; x < CH * D; x += ROWS) {
      int j = x / D, dd = x % D;
      bool in = kbase + j <= maxlim;
      Ks[x] = in ? kc[(size_t)(kbase + j) * D + dd] : 0.f;
      Vs[x] = in ? vc[(size_t)(kbase + j) * D + dd] : 0.f;
    }
    __syncthreads();
    float s[CH];
    float mc = -INFINITY;
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      if (kbase + j <= lim || (kbase + j >= lo2 && kbase + j <= hi2)) {
        float dot = 0.f;
#pragma unroll 1
        for (int dd = 0; dd < D; ++dd) dot = fmaf(Qs[i * (D + 1) + dd], Ks[j * D + dd], dot);
        s[j] = dot * a.scale;
        mc = fmaxf(mc, s[j]);
      } else {
        s[j] = -INFINITY;
      }
    }
    const float m_new = fmaxf(m, mc);
    if (m_new != -INFINITY) {
      const float corr = (m == -INFINITY) ? 0.f : expf(m - m_new);
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        float p = (s[j] == -INFINITY) ? 0.f : expf(s[j] - m_new);
        s[j] = p;
        psum += p;
      }
      l = l * corr + psum;
#pragma unroll 1
      for (int dd = 0; dd < D; ++dd) {
        float acc = Os[i * (D + 1) + dd] * corr;
#pragma unroll
        for (int j = 0; j < CH; ++j) acc = fmaf(s[j], Vs[j * D + dd], acc);
        Os[i * (D + 1) + dd] = acc;
      }
      m = m_new;
    }
    __syncthreads();
  }
  if (valid) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    for (int dd = 0; dd < D; ++dd) o[((size_t)t * a.Hq + hq) * D + dd] = Os[i * (D + 1) + dd] * inv;
  }
}

// ---------------------------------------------------------------- tensor-core path (bf16 models)

// Partial kernel: one CTA per (kv head x row group, rank, slot) tile; the
// rank is the second grid dimension so that low ranks, which hold chunks at
// every context length, dispatch first.  Ranks whose first chunk lies past
// the group's last visible key exit after the row limits are read; the others
// write their partial rows to a.part.
template <int D, bool TRACE, bool R2 = false>
__global__ void __launch_bounds__(256, 2)
    attention_part_kernel(const __grid_constant__ attn::KvMaps tms, AttnArgs a) {
  using Gm = attn::Geo<D>;
  constexpr int RLD = Gm::RLD;
  extern __shared__ __align__(16) uint8_t sm_in[];
  uint8_t* sm_raw = attn::tile_base(sm_in);
  __shared__ int s_maxlim;
  __shared__ __align__(8) uint64_t s_kbar, s_vbar;  // a chunk's K, V landed
  const Grp grp = Grp::block();
  const int group = blockIdx.x, rank = blockIdx.y, R = gridDim.y;
  const int slot = blockIdx.z;
  const int kvh = group % a.Hkv, rg = group / a.Hkv;
  const int G = a.Hq / a.Hkv;
  const int tid = threadIdx.x;

  if (tid == 0) {
    if (TRACE) trace_at(a, 0);
    tc::mbar_init(&s_kbar, 1);
    tc::mbar_init(&s_vbar, 1);
    tc::fence_mbar_init();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  __syncthreads();
  // cache row of key 0 of this CTA's (request, kv head): the planes' tensor
  // maps span every request and layer
  auto kv_row = [&](int req) { return a.kv_row0 + (long long)req * a.kv_req_rows + (long long)kvh * a.cap; };
  // committed cache before the dependency wait (decode launches only)
  int req_pre = -1, kv_kmax = -1;
  bool pre = false;
  if (a.st && a.slot_req) {
    req_pre = a.slot_req[slot];
    const int pc = a.st[req_pre].cache_len;
    pre = attn::tile_prefetch<D>(sm_raw, tms, attn::kv_planes(a, req_pre, kvh, D), kv_row(req_pre), rank, R, pc,
                                 tid, &s_kbar, &s_vbar);
    // no row of this forward reads past the round-start length plus its rows
    kv_kmax = min(a.cap - 1, pc + a.rows_per_slot);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (TRACE && tid == 0) trace_at(a, 1);

  int req = 0, row0 = 0, nrows = a.T;
  if (a.rows_per_slot > 0) {
    req = req_pre >= 0 ? req_pre : a.slot_req[slot];  // the slot table is constant during a decode
    row0 = slot * a.rows_per_slot;
    nrows = a.rows_per_slot;
  } else if (a.plan) {
    req = a.plan->slot_req[slot];
    row0 = a.plan->slot_row0[slot];
    nrows = a.plan->slot_nrows[slot];
  }
  const int qr0 = rg * attn::QR;
  if (qr0 >= nrows * G) {  // uniform: a row group past the window
    if (pre && !(tc::mbar_wait(&s_kbar, 0) && tc::mbar_wait(&s_vbar, 0)) && tid == 0)
      set_err(a.err, DERR_TIMEOUT);  // no copy outlives the CTA
    return;
  }
  const int n_chunks = attn::tile_partial<D, TRACE, R2>(a, sm_raw, grp, tms, kv_row(req), &s_kbar, &s_vbar, rank, R,
                                                        kvh, qr0, row0, nrows, pre, &s_maxlim, kv_kmax);
  if (rank == 0 && tid == 0) a.part_chunks[(size_t)slot * gridDim.x + group] = n_chunks;
  if (rank >= n_chunks) return;
  // all 64 rows, also those past the window (which the merge reads but does
  // not output): a fixed trip count measured faster than writing fewer rows
  const float4* src = reinterpret_cast<const float4*>(attn::staged_rows<D>(sm_raw));
  float4* dst = reinterpret_cast<float4*>(
      a.part + (((size_t)slot * gridDim.x + group) * R + rank) * attn::QR * RLD);
  for (int x = tid; x < attn::QR * RLD / 4; x += 256) dst[x] = src[x];
  if (TRACE && tid == 0) trace_at(a, 3);
}

// Merge kernel: one CTA per (PPC pairs of rows, kv head x row group, slot);
// tiles of TQR rows.
template <int D, int TQR, int PPC, bool TRACE>
__global__ void __launch_bounds__(256) attention_merge_kernel(AttnArgs a, int R) {
  constexpr int RLD = attn::Geo<D>::RLD;
  __shared__ float WS[2 * 64];
  __shared__ float IL[2];
  __shared__ float4 AC[4 * 64];
  const Grp grp = Grp::block();
  const int group = blockIdx.y, slot = blockIdx.z;
  const int kvh = group % a.Hkv, rg = group / a.Hkv;
  const int G = a.Hq / a.Hkv;
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (TRACE && a.trace_cta && threadIdx.x == 0) trace_at(a, 0, TRACE_MERGE_SLOT);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (TRACE && a.trace_cta && threadIdx.x == 0) trace_at(a, 1, TRACE_MERGE_SLOT);
  if (TRACE && threadIdx.x == 0) trace_at(a, 6, TRACE_MERGE_SLOT);
  int row0 = 0, nrows = a.T;
  if (a.rows_per_slot > 0) {
    row0 = slot * a.rows_per_slot;
    nrows = a.rows_per_slot;
  } else if (a.plan) {
    row0 = a.plan->slot_row0[slot];
    nrows = a.plan->slot_nrows[slot];
  }
  const int qr0 = rg * TQR;
  if (qr0 + 2 * blockIdx.x * PPC >= nrows * G) return;
  const int n_chunks = a.part_chunks[(size_t)slot * gridDim.y + group];
  const int n_ranks = n_chunks < R ? n_chunks : R;
  const float* base = a.part + ((size_t)slot * gridDim.y + group) * R * TQR * RLD;
  auto part = [&](int c, int i) -> const float* { return base + ((size_t)c * TQR + i) * RLD; };
#pragma unroll
  for (int k = 0; k < PPC; ++k) {
    const int pair = blockIdx.x * PPC + k;
    if (qr0 + 2 * pair >= nrows * G) break;  // uniform over the CTA
    attn::merge_rows<D, false>(a, grp, part, WS, IL, AC, n_ranks, R, 2 * pair, 1, 2, kvh, qr0, row0, nrows);
  }
  if (TRACE && threadIdx.x == 0) trace_at(a, 3, TRACE_MERGE_SLOT);
}

// Merge for few ranks (R <= MERGE_FEW): one warp per (row, head) pair, each
// lane a run of D / 32 output columns; every load in one round trip, no CTA
// barrier.  Ranks are added in rank order.  The choice depends on R alone,
// which a handle fixes, so every forward of a handle merges the same way.
constexpr int MERGE_FEW = 8;
template <int D, int TQR, bool TRACE>
__global__ void __launch_bounds__(256) attention_merge_few_kernel(AttnArgs a, int R) {
  constexpr int RLD = (TQR == attn::QR ? attn::Geo<D>::RLD : attn_tc::Geo<D>::RLD);
  constexpr int CL = D / 32;  // columns per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int group = blockIdx.y, slot = blockIdx.z;
  const int kvh = group % a.Hkv, rg = group / a.Hkv;
  const int G = a.Hq / a.Hkv;
  const int i = blockIdx.x * 8 + warp;  // row of the group's tile
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (TRACE && a.trace_cta && threadIdx.x == 0) trace_at(a, 0, TRACE_MERGE_SLOT);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (TRACE && a.trace_cta && threadIdx.x == 0) trace_at(a, 1, TRACE_MERGE_SLOT);
  if (TRACE && threadIdx.x == 0) trace_at(a, 6, TRACE_MERGE_SLOT);
  int row0 = 0, nrows = a.T;
  if (a.rows_per_slot > 0) {
    row0 = slot * a.rows_per_slot;
    nrows = a.rows_per_slot;
  } else if (a.plan) {
    row0 = a.plan->slot_row0[slot];
    nrows = a.plan->slot_nrows[slot];
  }
  const int nq = nrows * G, gi = rg * TQR + i;
  if (i < TQR && gi < nq) {
    const size_t gs = (size_t)slot * gridDim.y + group;
    const int n_chunks = a.part_chunks[gs];
    const int n_ranks = n_chunks < R ? n_chunks : R;
    const float* base = a.part + gs * R * TQR * RLD + (size_t)i * RLD;
    float m[MERGE_FEW], l[MERGE_FEW], v[MERGE_FEW][CL];
#pragma unroll
    for (int r = 0; r < MERGE_FEW; ++r) {
      m[r] = -INFINITY;
      l[r] = 0.f;
#pragma unroll
      for (int j = 0; j < CL; ++j) v[r][j] = 0.f;
      if (r < n_ranks) {
        const float* p = base + (size_t)r * TQR * RLD;
        m[r] = __ldcg(p + D);
        l[r] = __ldcg(p + D + 1);
        if constexpr (CL == 4) {
          const float4 x = __ldcg(reinterpret_cast<const float4*>(p + lane * 4));
          v[r][0] = x.x; v[r][1] = x.y; v[r][2] = x.z; v[r][3] = x.w;
        } else {
          const float2 x = __ldcg(reinterpret_cast<const float2*>(p + lane * 2));
          v[r][0] = x.x; v[r][1] = x.y;
        }
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < MERGE_FEW; ++r) M = fmaxf(M, m[r]);
    float L = 0.f, o[CL];
#pragma unroll
    for (int j = 0; j < CL; ++j) o[j] = 0.f;
#pragma unroll
    for (int r = 0; r < MERGE_FEW; ++r) {
      const float w = m[r] == -INFINITY ? 0.f : exp2f(m[r] - M);
      L = fmaf(w, l[r], L);
#pragma unroll
      for (int j = 0; j < CL; ++j) o[j] = fmaf(w, v[r][j], o[j]);
    }
    const float il = L > 0.f ? 1.f / L : 0.f;
    const int tq = attn::div_small(gi, G, 0xFFFFFFFFu / (unsigned)G + 1u);
    const size_t off = ((size_t)(row0 + tq) * a.Hq + kvh * G + (gi - tq * G)) * D + lane * CL;
#pragma unroll
    for (int j = 0; j < CL; ++j) put_plane(a.o_hi, a.o_lo, a.out_bf16, off + j, o[j] * il);
  }
  if (TRACE && threadIdx.x == 0) trace_at(a, 3, TRACE_MERGE_SLOT);
}

size_t attention_part_floats(int n_slots, int max_rows, int Hq, int Hkv, int d, int R) {
  const int G = Hq / Hkv;
  size_t best = 0;
  for (int qr : {attn::QR, attn_tc::QR}) {
    const size_t groups = (size_t)Hkv * ((max_rows * G + qr - 1) / qr);
    const size_t f = (size_t)n_slots * groups * R * qr * (d + 4);
    if (f > best) best = f;
  }
  return best;
}

// The merge after a partial kernel of TQR-row tiles (always ordered after it).
template <int D, int TQR, bool TRACE>
static bool launch_attn_merge(const AttnArgs& a, int R, int n_groups, int n_slots, cudaStream_t s) {
  if (R <= MERGE_FEW) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(TQR / 8, n_groups, n_slots);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attention_merge_few_kernel<D, TQR, TRACE>, a, R) == cudaSuccess;
  }
  // with few ranks a row pair is little work: four pairs per CTA then
  const int ppc = R <= 16 ? 4 : 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(TQR / 2 / ppc, n_groups, n_slots);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return (ppc == 4 ? cudaLaunchKernelEx(&cfg, attention_merge_kernel<D, TQR, 4, TRACE>, a, R)
                   : cudaLaunchKernelEx(&cfg, attention_merge_kernel<D, TQR, 1, TRACE>, a, R)) == cudaSuccess;
}

template <int D, bool TRACE, bool R2 = false>
static bool launch_attn_tc_t(const AttnArgs& a, int n_slots, int max_rows, cudaStream_t s, bool pdl) {
  using Gm = attn_tc::Geo<D>;
  const int G = a.Hq / a.Hkv;
  const int n_rg = (max_rows * G + attn_tc::QR - 1) / attn_tc::QR;
  if (!kernel_smem_at_least(reinterpret_cast<const void*>(attention_tc_part_kernel<D, TRACE, R2>), Gm::SMEM))
    return false;
  const int R = a.ranks > 0 ? a.ranks : attention_ranks(a.cap, 1);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.Hkv * n_rg, R, n_slots);
  cfg.blockDim = dim3(attn_tc::THREADS);
  cfg.dynamicSmemBytes = Gm::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, attention_tc_part_kernel<D, TRACE, R2>, a) != cudaSuccess) return false;
  return launch_attn_merge<D, attn_tc::QR, TRACE>(a, R, a.Hkv * n_rg, n_slots, s);
}

template <int D, bool TRACE, bool R2 = false>
static bool launch_attn_mma_t(const AttnArgs& a, int n_slots, int max_rows, cudaStream_t s, bool pdl) {
  if (!a.kv_maps) return false;
  attn::KvMaps tms;
  memcpy(&tms, a.kv_maps, sizeof(tms));
  const int G = a.Hq / a.Hkv;
  const int n_rg = (max_rows * G + attn::QR - 1) / attn::QR;
  const size_t smem = R2 ? attn::Geo<D>::TILE_SMEM_R2 : attn::Geo<D>::TILE_SMEM;
  if (!kernel_smem_at_least(reinterpret_cast<const void*>(attention_part_kernel<D, TRACE, R2>), smem))
    return false;
  cudaLaunchConfig_t cfg{};
  const int R = a.ranks > 0 ? a.ranks : attention_ranks(a.cap, 1);
  cfg.gridDim = dim3(a.Hkv * n_rg, R, n_slots);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, attention_part_kernel<D, TRACE, R2>, tms, a) != cudaSuccess) return false;
  return launch_attn_merge<D, attn::QR, TRACE>(a, R, a.Hkv * n_rg, n_slots, s);
}

template <int D>
static bool launch_attn_mma(const AttnArgs& a, int n_slots, int max_rows, cudaStream_t s, bool pdl) {
  // rows with a second key interval (the joint-training mask): the R2
  // instantiation of the kernel of a.kind
  if (a.row_lo2)
    return a.kind == ATTN_TCGEN05 ? launch_attn_tc_t<D, false, true>(a, n_slots, max_rows, s, pdl)
                                  : launch_attn_mma_t<D, false, true>(a, n_slots, max_rows, s, pdl);
  if (a.kind == ATTN_TCGEN05)
    return a.trace ? launch_attn_tc_t<D, true>(a, n_slots, max_rows, s, pdl)
                   : launch_attn_tc_t<D, false>(a, n_slots, max_rows, s, pdl);
  return a.trace ? launch_attn_mma_t<D, true>(a, n_slots, max_rows, s, pdl)
                 : launch_attn_mma_t<D, false>(a, n_slots, max_rows, s, pdl);
}

template <int D>
static bool launch_attn_simt(const AttnArgs& a, int n_slots, int max_rows, cudaStream_t s, bool pdl) {
  const int G = a.Hq / a.Hkv;
  dim3 grid((max_rows * G + ROWS - 1) / ROWS, a.Hkv, n_slots);
  const size_t smem = sizeof(float) * (2 * ROWS * (D + 1) + 2 * CH * D);
  if (!kernel_smem_at_least(reinterpret_cast<const void*>(attention_simt_kernel<D>), smem)) return false;
  return launch_k(attention_simt_kernel<D>, grid, dim3(ROWS), smem, s, pdl, a) == cudaSuccess;
}

bool launch_attention(int dtype, const AttnArgs& a, int n_slots, int max_rows, cudaStream_t s, bool pdl) {
  if (dtype == 1) return a.d == 128 ? launch_attn_mma<128>(a, n_slots, max_rows, s, pdl)
                                    : launch_attn_mma<64>(a, n_slots, max_rows, s, pdl);
  return a.d == 128 ? launch_attn_simt<128>(a, n_slots, max_rows, s, pdl)
                    : launch_attn_simt<64>(a, n_slots, max_rows, s, pdl);
}

}  // namespace gocr
