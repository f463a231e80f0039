// Grouped-query attention of a window of query rows against a contiguous
// per-request KV cache, with the two mask modes of the round expressed as one
// per-row key limit: row t reads keys 0..lim[t].
//   draft  (GravityOCR review §3.2): boundary row lim = p (causal), [M] rows
//          lim = p + B (the cache plus the whole window, bidirectional);
//   verify / AR / prefill: lim = the row's own position (token-causal).
//
// Keys are visited in fixed 64-key chunks at absolute positions.  A chunk with
// no key visible to a row leaves that row's running (max, sum, output)
// bit-for-bit unchanged (scale exp(0) = 1, zero contributions), so a row's
// result does not depend on how many other rows share the launch: the AR step
// and the verify row at the same position give identical bits.
//
// bf16 models: tensor-core kernel.  q and the KV cache are stored as bf16
// hi + lo planes (written once by the QKV epilogue), QK^T takes
// qh kh + qh kl + ql kh and PV takes P vh + P vl on mma.sync tiles (P in
// bf16), accumulating in fp32.  A cluster of CL CTAs shares one (kv head,
// 64-query-row group): CTA r visits chunks r, r + CL, ... with an online
// softmax, K/V tiles double-buffered through cp.async, then the cluster merges
// its CL partial (max, sum, output) triples through distributed shared memory
// in rank order.  Under programmatic dependent launch a CTA fetches its first
// chunk before the grid-dependency wait when that chunk holds only committed
// cache positions (below the round-start cache length, which no kernel of the
// forward writes).  The result is written as the O projection's input planes.
// fp32 models: CUDA-core kernel with one CTA sweeping every chunk.
#include <cooperative_groups.h>

#include "attn_core.cuh"
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

  if (i == 0) s_maxlim = -1;
  __syncthreads();
  if (valid) atomicMax(&s_maxlim, lim);
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
      if (kbase + j <= lim) {
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

// One CTA per (cluster rank, kv head x row group, slot) tile; the cluster's
// CL tiles split the key chunks and merge over distributed shared memory.
// At most 128 registers a thread: one attention CTA (32 K registers) and two
// GEMM CTAs of the next kernels then fit one SM's register file together, so
// under programmatic dependent launch those CTAs become resident, and start
// their weight loads, while attention still runs.
template <int D, int CL, bool TRACE>
__global__ void __launch_bounds__(256, 2) attention_mma_kernel(AttnArgs a) {
  namespace cg = cooperative_groups;
  using Gm = attn::Geo<D>;
  constexpr int RLD = Gm::RLD;
  constexpr int RPC = attn::QR / CL; // rows owned per CTA
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) uint8_t sm_raw[];
  float* RX = reinterpret_cast<float*>(sm_raw + Gm::TILE_SMEM);  // [CL][RPC][RLD] partial rows from each rank
  float* WS = RX + CL * RPC * RLD;                               // [RPC][CL] merge weights
  float* IL = WS + RPC * CL;                                     // [RPC] 1 / total sum
  __shared__ __align__(8) uint64_t rxbar;
  __shared__ int s_maxlim;
  const Grp grp = Grp::block();

  const int rank = blockIdx.x;  // == cluster rank (the cluster spans grid x)
  const int kvh = blockIdx.y % a.Hkv;
  const int rg = blockIdx.y / a.Hkv;
  const int slot = blockIdx.z;
  const int G = a.Hq / a.Hkv;
  const int tid = threadIdx.x;

  if (tid == 0) {
    if (TRACE) trace_mark(a.trace, 0);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tc::mbar_init(&rxbar, 1);
    tc::fence_mbar_init();
    tc::mbar_expect_tx(&rxbar, (uint32_t)(CL * RPC * RLD * 4));  // one block of rows from every rank
  }
  cluster.sync();  // every receive barrier is armed before any rank sends
  // committed cache before the dependency wait (decode launches only)
  int req_pre = -1;
  bool pre = false;
  if (a.st && a.slot_req) {
    req_pre = a.slot_req[slot];
    pre = attn::tile_prefetch<D, CL>(sm_raw, attn::kv_planes(a, req_pre, kvh, D), rank, a.st[req_pre].cache_len,
                                     tid);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (TRACE && tid == 0) trace_mark(a.trace, 1);

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
  if (qr0 >= nrows * G) {  // uniform across the cluster
    attn::cp_async_wait<0>();
    return;
  }
  attn::tile_partial<D, CL, TRACE>(a, sm_raw, grp, attn::kv_planes(a, req, kvh, D), rank, kvh, qr0, row0, nrows,
                                   pre, &s_maxlim);
  float* ST = attn::staged_rows<D>(sm_raw);
  tc::fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0) {
    // one bulk copy per owner: this CTA's rows of that owner -> its RX[rank]
    for (int r = 0; r < CL; ++r)
      tc::bulk_s2s(tc::mapa(tc::smem_u32(RX + (size_t)rank * RPC * RLD), r), ST + (size_t)r * RPC * RLD,
                   (uint32_t)(RPC * RLD * 4), tc::mapa(tc::smem_u32(&rxbar), r));
    tc::bulk_commit();
  }
  const bool rx_ok = tc::mbar_wait(&rxbar, 0);
  if (TRACE && tid == 0) trace_mark(a.trace, 6);
  auto row = [&](int c, int i) -> const float* { return RX + (c * RPC + i) * RLD; };
  attn::merge_owned<D, CL>(a, grp, row, WS, IL, rank, kvh, qr0, row0, nrows, rx_ok);
  if (tid == 0) tc::bulk_wait_read();  // the copies have read this CTA's staged rows
  if (TRACE && tid == 0) trace_mark(a.trace, 3);
}

template <int D, int CL>
static size_t attn_mma_smem() {
  constexpr int RPC = attn::QR / CL, RLD = attn::Geo<D>::RLD;
  return attn::Geo<D>::TILE_SMEM + ((size_t)CL * RPC * RLD + RPC * CL + RPC) * 4;
}

template <int D, int CL, bool TRACE>
static cudaError_t launch_attn_cl(const AttnArgs& a, dim3 grid, cudaStream_t s, bool pdl) {
  const size_t smem = attn_mma_smem<D, CL>();
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = CL;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, attention_mma_kernel<D, CL, TRACE>, a);
}

// Kernel attributes of one cluster width (both trace instantiations).
template <int D, int CL>
static bool attn_configure() {
  const int smem = (int)attn_mma_smem<D, CL>();
  bool ok = true;
  for (const void* fn : {reinterpret_cast<const void*>(attention_mma_kernel<D, CL, false>),
                         reinterpret_cast<const void*>(attention_mma_kernel<D, CL, true>)}) {
    prefer_shared(fn);
    if (CL > 8) ok &= cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    ok &= cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess;
  }
  return ok;
}

// Cluster width: 16 CTAs when the device keeps the eight 16-CTA clusters of
// a 33-row decode window (4 kv heads x 2 row groups) resident at once, else
// 8.  The width fixes which rank reads which key chunk and the order of the
// merge, so it is chosen once per process: every launch, AR or
// self-speculative, adds the same partials in the same order.
template <int D>
static int attn_cluster_width() {
  static int width = 0;
  if (width) return width;
  width = 8;
  if (attn_configure<D, 16>()) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(16, 1, 1);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = attn_mma_smem<D, 16>();
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 16;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attention_mma_kernel<D, 16, false>, &cfg) == cudaSuccess && n >= 8)
      width = 16;
  }
  cudaGetLastError();
  if (width == 8) attn_configure<D, 8>();
  return width;
}

int attention_cluster_width(int d) { return d == 128 ? attn_cluster_width<128>() : attn_cluster_width<64>(); }

template <int D>
static bool launch_attn_mma(const AttnArgs& a, int n_slots, int max_rows, cudaStream_t s, bool pdl) {
  const int G = a.Hq / a.Hkv;
  const int n_rg = (max_rows * G + attn::QR - 1) / attn::QR;
  const int cl = attn_cluster_width<D>();
  const dim3 grid(cl, a.Hkv * n_rg, n_slots);
  cudaError_t e;
  if (a.trace)
    e = cl == 16 ? launch_attn_cl<D, 16, true>(a, grid, s, pdl) : launch_attn_cl<D, 8, true>(a, grid, s, pdl);
  else
    e = cl == 16 ? launch_attn_cl<D, 16, false>(a, grid, s, pdl) : launch_attn_cl<D, 8, false>(a, grid, s, pdl);
  return e == cudaSuccess;
}

template <int D>
static bool launch_attn_simt(const AttnArgs& a, int n_slots, int max_rows, cudaStream_t s, bool pdl) {
  const int G = a.Hq / a.Hkv;
  dim3 grid((max_rows * G + ROWS - 1) / ROWS, a.Hkv, n_slots);
  const size_t smem = sizeof(float) * (2 * ROWS * (D + 1) + 2 * CH * D);
  static bool init = false;
  if (!init) {
    if (cudaFuncSetAttribute(attention_simt_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return false;
    init = true;
  }
  return launch_k(attention_simt_kernel<D>, grid, dim3(ROWS), smem, s, pdl, a) == cudaSuccess;
}

bool launch_attention(int dtype, const AttnArgs& a, int n_slots, int max_rows, cudaStream_t s, bool pdl) {
  if (dtype == 1) return a.d == 128 ? launch_attn_mma<128>(a, n_slots, max_rows, s, pdl)
                                    : launch_attn_mma<64>(a, n_slots, max_rows, s, pdl);
  return a.d == 128 ? launch_attn_simt<128>(a, n_slots, max_rows, s, pdl)
                    : launch_attn_simt<64>(a, n_slots, max_rows, s, pdl);
}

}  // namespace gocr
