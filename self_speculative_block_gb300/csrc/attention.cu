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

#include "epilogue.cuh"
#include "tc.cuh"

namespace gocr {

namespace {
constexpr int ROWS = 128;   // CUDA-core kernel: query rows (token, q head) per CTA
constexpr int CH = 64;      // keys per chunk
constexpr int QR = 64;      // tensor-core kernel: query rows per cluster
constexpr float LOG2E = 1.4426950408889634f;
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

__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Four 8x8 bf16 matrices, transposed on load: each lane gets the pair
// (row 2t, col g), (row 2t+1, col g) of the matrix whose row addresses lanes
// 8i..8i+7 supply, which is the B-fragment layout of m16n8k16.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Hint a contiguous global range into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, int bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// 16-byte asynchronous global -> shared copy; src_bytes = 0 fills zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Tensor-core kernel: 256 threads, keys in chunks of AC = 32.  Warp w owns
// query rows 16 (w % 4) .. 16 (w % 4) + 15 of the row group and key half w / 4
// (keys 16 (w / 4) .. 16 (w / 4) + 15 of every chunk), so each (cluster rank,
// key half) runs its own online softmax over a fixed set of absolute key
// positions.  The two halves of a CTA are merged in shared memory (half 0,
// then half 1), then every CTA pushes its partial rows to the rows' owner CTAs
// over distributed shared memory (row r belongs to rank r % CL) and, after one
// cluster barrier, each owner adds the CL partials in rank order.
constexpr int AC = 32;  // keys per chunk of the tensor-core kernel

template <int D, int CL>
__global__ void __launch_bounds__(256) attention_mma_kernel(AttnArgs a) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  constexpr int QLD = D + 8;   // bf16 row stride of the Q, K and V tiles
  constexpr int OLD = D + 4;   // fp32 row stride of the half-1 partial
  constexpr int TILE = AC * QLD;
  constexpr int RPC = QR / CL; // rows owned per CTA
  extern __shared__ __align__(16) uint8_t sm_raw[];
  bf16* Qh = reinterpret_cast<bf16*>(sm_raw);            // [QR][QLD]
  bf16* Ql = Qh + QR * QLD;
  bf16* KV = Ql + QR * QLD;                              // {Kh, Kl, Vh, Vl} [AC][QLD]
  float* Oh = reinterpret_cast<float*>(Qh);              // [QR][OLD] half-1 partial (Q is dead by then)
  float* Mh = Oh + QR * OLD;                             // [QR]
  float* Lh = Mh + QR;                                   // [QR]
  constexpr int RLD = D + 4;   // fp32 stride of a partial row: D outputs, max, sum, pad
  float* RX = reinterpret_cast<float*>(KV + 4 * TILE);   // [CL][RPC][RLD] partial rows from each rank
  float* ST = reinterpret_cast<float*>(KV);              // [CL][RPC][RLD] rows to send, after the loop
  float* WS = RX + CL * RPC * RLD;                       // [RPC][CL] merge weights
  float* IL = WS + RPC * CL;                             // [RPC] 1 / total sum
  int* Lim = reinterpret_cast<int*>(IL + RPC);           // [QR]
  __shared__ __align__(8) uint64_t rxbar;
  __shared__ int s_maxlim;

  const int rank = blockIdx.x;  // == cluster rank (the cluster spans grid x)
  const int kvh = blockIdx.y % a.Hkv;
  const int rg = blockIdx.y / a.Hkv;
  const int slot = blockIdx.z;
  const int G = a.Hq / a.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = warp & 3, kh = warp >> 2;
  const int g = lane >> 2, tq = lane & 3;

  // cp.async copies of the two planes of K (tile 0) or V (tile 2) of chunk c
  // (keys c*AC .. c*AC+AC-1, zero past kmax)
  auto load_part = [&](const bf16* p_h, const bf16* p_l, int tile0, int c, int kmax) {
    for (int x = tid; x < 2 * AC * (D / 8); x += 256) {
      const int pl = x / (AC * (D / 8)), rem = x % (AC * (D / 8));
      const int j = rem / (D / 8), v = rem % (D / 8);
      const int key = c * AC + j;
      const bf16* base = pl == 0 ? p_h : p_l;
      const bool in = key <= kmax;
      cp_async16(KV + (tile0 + pl) * TILE + j * QLD + v * 8, base + (size_t)(in ? key : 0) * D + v * 8, in ? 16 : 0);
    }
  };
  // cp.async copies of chunk c (keys c*AC .. c*AC+AC-1, zero past kmax)
  auto load_chunk = [&](const bf16* k_h, const bf16* k_l, const bf16* v_h, const bf16* v_l, int c, int kmax) {
    for (int x = tid; x < 4 * AC * (D / 8); x += 256) {
      const int pl = x / (AC * (D / 8)), rem = x % (AC * (D / 8));
      const int j = rem / (D / 8), v = rem % (D / 8);
      const int key = c * AC + j;
      const bf16* base = pl == 0 ? k_h : pl == 1 ? k_l : pl == 2 ? v_h : v_l;
      const bool in = key <= kmax;
      cp_async16(KV + pl * TILE + j * QLD + v * 8, base + (size_t)(in ? key : 0) * D + v * 8, in ? 16 : 0);
    }
  };

  if (tid == 0) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tc::mbar_init(&rxbar, 1);
    tc::fence_mbar_init();
    tc::mbar_expect_tx(&rxbar, (uint32_t)(CL * RPC * RLD * 4));  // one block of rows from every rank
  }
  cluster.sync();  // every receive barrier is armed before any rank sends
  // committed cache before the dependency wait (decode launches only): the
  // first chunk into shared memory, the CTA's later committed chunks into L2
  int req_pre = -1, pc = 0;
  if (a.st && a.slot_req) {
    req_pre = a.slot_req[slot];
    pc = a.st[req_pre].cache_len;
  }
  const bool pre = req_pre >= 0 && (rank + 1) * AC <= pc;
  if (pre) {
    const size_t o = (size_t)req_pre * a.req_stride + (size_t)kvh * a.cap * D;
    const bf16* pk[4] = {reinterpret_cast<const bf16*>(a.k_hi) + o, reinterpret_cast<const bf16*>(a.k_lo) + o,
                         reinterpret_cast<const bf16*>(a.v_hi) + o, reinterpret_cast<const bf16*>(a.v_lo) + o};
    load_chunk(pk[0], pk[1], pk[2], pk[3], rank, pc - 1);
    cp_async_commit();
    // later committed chunks of this CTA: rank + CL, rank + 2 CL, ... (4 planes each)
    for (int i = tid; i < 4 * 8; i += 256) {
      const int c = rank + (1 + i / 4) * CL;
      if ((c + 1) * AC <= pc) prefetch_l2(pk[i % 4] + (size_t)c * AC * D, AC * D * 2);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");

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
  const int nq = nrows * G;
  const int qr0 = rg * QR;
  if (qr0 >= nq) {  // uniform across the cluster
    cp_async_wait<0>();
    return;
  }
  const size_t kv_off = (size_t)req * a.req_stride + (size_t)kvh * a.cap * D;
  const bf16* k_h = reinterpret_cast<const bf16*>(a.k_hi) + kv_off;
  const bf16* k_l = reinterpret_cast<const bf16*>(a.k_lo) + kv_off;
  const bf16* v_h = reinterpret_cast<const bf16*>(a.v_hi) + kv_off;
  const bf16* v_l = reinterpret_cast<const bf16*>(a.v_lo) + kv_off;
  const bf16* qh = reinterpret_cast<const bf16*>(a.q_hi);
  const bf16* ql = reinterpret_cast<const bf16*>(a.q_lo);

  if (tid == 0) s_maxlim = -1;
  __syncthreads();
  // Q planes of this row group (zero past the window) and the rows' key limits
  for (int x = tid; x < 2 * QR * (D / 8); x += 256) {
    const int pl = x / (QR * (D / 8)), rem = x % (QR * (D / 8));
    const int r = rem / (D / 8), v = rem % (D / 8);
    const int gi = qr0 + r;
    size_t src = 0;
    if (gi < nq) src = ((size_t)(row0 + gi / G) * a.Hq + kvh * G + gi % G) * D + v * 8;
    cp_async16((pl ? Ql : Qh) + r * QLD + v * 8, (pl ? ql : qh) + src, gi < nq ? 16 : 0);
  }
  cp_async_commit();
  if (tid < QR) {
    const int gi = qr0 + tid;
    int lim = -1;
    if (gi < nq) lim = min(a.row_lim[row0 + gi / G], a.cap - 1);
    Lim[tid] = lim;
    if (lim >= 0) atomicMax(&s_maxlim, lim);
  }
  __syncthreads();
  const int maxlim = s_maxlim;
  const int n_chunks = maxlim < 0 ? 0 : maxlim / AC + 1;
  const float sl2 = a.scale * LOG2E;

  const int r_lo = mt * 16 + g, r_hi = r_lo + 8;
  const int lim_lo = Lim[r_lo], lim_hi = Lim[r_hi];
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  float oacc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int lcol = (lane >> 4) * 8;
  const bf16* Kh = KV + kh * 16 * QLD;  // this warp's 16 keys of the chunk
  const bf16* Kl = Kh + TILE;
  const bf16* Vh = Kl + TILE;
  const bf16* Vl = Vh + TILE;

  // K and V of a chunk are separate cp.async groups: K of the next chunk
  // streams in while this chunk's softmax and PV run, V of the next chunk
  // while the next QK^T runs.  Group order: [K+V of the first chunk] (issued
  // before the wait when it is committed cache), Q, then K, V per chunk.
  if (!pre && rank < n_chunks) {
    load_part(k_h, k_l, 0, rank, maxlim);
    load_part(v_h, v_l, 2, rank, maxlim);
  }
  cp_async_commit();
  int it = 0;
  for (int c = rank; c < n_chunks; c += CL, ++it) {
    const int kbase = c * AC + kh * 16;
    const bool next = c + CL < n_chunks;
    if (it == 0) cp_async_wait<0>(); else cp_async_wait<1>();  // this chunk's K (and Q, first chunk)
    __syncthreads();
    // S = Q K^T for this warp's 16 rows and 16 keys
    float sacc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t ah[4], al[4];
      const int qo = (mt * 16 + g) * QLD + ks * 16 + tq * 2;
      ah[0] = *reinterpret_cast<const uint32_t*>(Qh + qo);
      ah[1] = *reinterpret_cast<const uint32_t*>(Qh + qo + 8 * QLD);
      ah[2] = *reinterpret_cast<const uint32_t*>(Qh + qo + 8);
      ah[3] = *reinterpret_cast<const uint32_t*>(Qh + qo + 8 * QLD + 8);
      al[0] = *reinterpret_cast<const uint32_t*>(Ql + qo);
      al[1] = *reinterpret_cast<const uint32_t*>(Ql + qo + 8 * QLD);
      al[2] = *reinterpret_cast<const uint32_t*>(Ql + qo + 8);
      al[3] = *reinterpret_cast<const uint32_t*>(Ql + qo + 8 * QLD + 8);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int ko = (nt * 8 + g) * QLD + ks * 16 + tq * 2;
        uint32_t bh[2], bl[2];
        bh[0] = *reinterpret_cast<const uint32_t*>(Kh + ko);
        bh[1] = *reinterpret_cast<const uint32_t*>(Kh + ko + 8);
        bl[0] = *reinterpret_cast<const uint32_t*>(Kl + ko);
        bl[1] = *reinterpret_cast<const uint32_t*>(Kl + ko + 8);
        mma16816(sacc[nt], al, bh);
        mma16816(sacc[nt], ah, bl);
        mma16816(sacc[nt], ah, bh);
      }
    }
    __syncthreads();  // every warp is done with this chunk's K
    if (next) load_part(k_h, k_l, 0, c + CL, maxlim);
    cp_async_commit();
    // mask, scale to log2 units, row maxima over the 16 keys
    float mc_lo = -INFINITY, mc_hi = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = kbase + nt * 8 + tq * 2 + e;
        float s0 = key <= lim_lo ? sacc[nt][e] * sl2 : -INFINITY;
        float s1 = key <= lim_hi ? sacc[nt][2 + e] * sl2 : -INFINITY;
        sacc[nt][e] = s0;
        sacc[nt][2 + e] = s1;
        mc_lo = fmaxf(mc_lo, s0);
        mc_hi = fmaxf(mc_hi, s1);
      }
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mc_lo = fmaxf(mc_lo, __shfl_xor_sync(0xffffffffu, mc_lo, off));
      mc_hi = fmaxf(mc_hi, __shfl_xor_sync(0xffffffffu, mc_hi, off));
    }
    const float mn_lo = fmaxf(m_lo, mc_lo), mn_hi = fmaxf(m_hi, mc_hi);
    const float corr_lo = mn_lo == -INFINITY ? 1.f : (m_lo == -INFINITY ? 0.f : exp2f(m_lo - mn_lo));
    const float corr_hi = mn_hi == -INFINITY ? 1.f : (m_hi == -INFINITY ? 0.f : exp2f(m_hi - mn_hi));
    float ps_lo = 0.f, ps_hi = 0.f;
    uint32_t pf[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      float p0 = sacc[nt][0] == -INFINITY ? 0.f : exp2f(sacc[nt][0] - mn_lo);
      float p1 = sacc[nt][1] == -INFINITY ? 0.f : exp2f(sacc[nt][1] - mn_lo);
      float p2 = sacc[nt][2] == -INFINITY ? 0.f : exp2f(sacc[nt][2] - mn_hi);
      float p3 = sacc[nt][3] == -INFINITY ? 0.f : exp2f(sacc[nt][3] - mn_hi);
      ps_lo += p0 + p1;
      ps_hi += p2 + p3;
      pf[nt][0] = pack_bf16(p0, p1);
      pf[nt][1] = pack_bf16(p2, p3);
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      ps_lo += __shfl_xor_sync(0xffffffffu, ps_lo, off);
      ps_hi += __shfl_xor_sync(0xffffffffu, ps_hi, off);
    }
    l_lo = l_lo * corr_lo + ps_lo;
    l_hi = l_hi * corr_hi + ps_hi;
    m_lo = mn_lo;
    m_hi = mn_hi;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      oacc[dn][0] *= corr_lo; oacc[dn][1] *= corr_lo;
      oacc[dn][2] *= corr_hi; oacc[dn][3] *= corr_hi;
    }
    if (it > 0) {
      cp_async_wait<1>();  // this chunk's V (the next chunk's K may still be in flight)
      __syncthreads();
    }
    // O += P (V_hi + V_lo); B fragments of two d-tiles per ldmatrix.x4.trans
    uint32_t af[4] = {pf[0][0], pf[0][1], pf[1][0], pf[1][1]};
#pragma unroll
    for (int dn = 0; dn < D / 8; dn += 2) {
      const int vo = lrow * QLD + dn * 8 + lcol;
      uint32_t bh[4], bl[4];
      ldsm_x4_trans(bh, Vh + vo);
      ldsm_x4_trans(bl, Vl + vo);
      mma16816(oacc[dn], af, bl);
      mma16816(oacc[dn], af, bh);
      mma16816(oacc[dn + 1], af, bl + 2);
      mma16816(oacc[dn + 1], af, bh + 2);
    }
    __syncthreads();  // every warp is done with this chunk's V
    if (next) load_part(v_h, v_l, 2, c + CL, maxlim);
    cp_async_commit();
  }
  cp_async_wait<0>();
  __syncthreads();
  // merge the two key halves of this CTA: half 0 + half 1, in that order
  if (kh == 1) {
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      Oh[r_lo * OLD + dn * 8 + tq * 2] = oacc[dn][0];
      Oh[r_lo * OLD + dn * 8 + tq * 2 + 1] = oacc[dn][1];
      Oh[r_hi * OLD + dn * 8 + tq * 2] = oacc[dn][2];
      Oh[r_hi * OLD + dn * 8 + tq * 2 + 1] = oacc[dn][3];
    }
    if (tq == 0) {
      Mh[r_lo] = m_lo; Lh[r_lo] = l_lo;
      Mh[r_hi] = m_hi; Lh[r_hi] = l_hi;
    }
  }
  __syncthreads();
  if (kh == 0) {
    const float m1_lo = Mh[r_lo], m1_hi = Mh[r_hi];
    const float M_lo = fmaxf(m_lo, m1_lo), M_hi = fmaxf(m_hi, m1_hi);
    const float w0_lo = m_lo == -INFINITY ? 0.f : exp2f(m_lo - M_lo);
    const float w1_lo = m1_lo == -INFINITY ? 0.f : exp2f(m1_lo - M_lo);
    const float w0_hi = m_hi == -INFINITY ? 0.f : exp2f(m_hi - M_hi);
    const float w1_hi = m1_hi == -INFINITY ? 0.f : exp2f(m1_hi - M_hi);
    const float L_lo = w0_lo * l_lo + w1_lo * Lh[r_lo];
    const float L_hi = w0_hi * l_hi + w1_hi * Lh[r_hi];
    // stage this CTA's partial rows by owner: row r -> rank r % CL, slot r / CL
    float* st_lo = ST + ((r_lo % CL) * RPC + r_lo / CL) * RLD;
    float* st_hi = ST + ((r_hi % CL) * RPC + r_hi / CL) * RLD;
    float o1[D / 8][4];
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      const int col = dn * 8 + tq * 2;
      o1[dn][0] = Oh[r_lo * OLD + col];
      o1[dn][1] = Oh[r_lo * OLD + col + 1];
      o1[dn][2] = Oh[r_hi * OLD + col];
      o1[dn][3] = Oh[r_hi * OLD + col + 1];
    }
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      const int col = dn * 8 + tq * 2;
      st_lo[col] = w0_lo * oacc[dn][0] + w1_lo * o1[dn][0];
      st_lo[col + 1] = w0_lo * oacc[dn][1] + w1_lo * o1[dn][1];
      st_hi[col] = w0_hi * oacc[dn][2] + w1_hi * o1[dn][2];
      st_hi[col + 1] = w0_hi * oacc[dn][3] + w1_hi * o1[dn][3];
    }
    if (tq == 0) {
      st_lo[D] = M_lo; st_lo[D + 1] = L_lo;
      st_hi[D] = M_hi; st_hi[D + 1] = L_hi;
    }
  }
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
  // owner: rows rank + i * CL.  Warp i computes the merge weights of row i,
  // lane c holding rank c's (max, sum); the butterfly order is fixed
  if (warp < RPC) {
    const int i = warp;
    const float m = lane < CL ? RX[(lane * RPC + i) * RLD + D] : -INFINITY;
    const float l = lane < CL ? RX[(lane * RPC + i) * RLD + D + 1] : 0.f;
    float M = m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float w = m == -INFINITY ? 0.f : exp2f(m - M);
    float L = w * l;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (lane < CL) WS[i * CL + lane] = w;
    if (lane == 0) IL[i] = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();
  if (rx_ok) {
    // thread x: row x / (D / 4), outputs 4 (x % (D / 4)) .. +3; all CL partials
    // are loaded first, then weighted and added in rank order
    for (int x = tid; x < RPC * (D / 4); x += 256) {
      const int i = x / (D / 4), d4 = (x % (D / 4)) * 4;
      const int gi = qr0 + rank + i * CL;
      if (gi >= nq) continue;
      float4 pv[CL];
#pragma unroll
      for (int c = 0; c < CL; ++c) pv[c] = *reinterpret_cast<const float4*>(RX + (c * RPC + i) * RLD + d4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int c = 0; c < CL; ++c) {
        const float w = WS[i * CL + c];
        acc.x += w * pv[c].x;
        acc.y += w * pv[c].y;
        acc.z += w * pv[c].z;
        acc.w += w * pv[c].w;
      }
      const float il = IL[i];
      const int t = row0 + gi / G, hq = kvh * G + gi % G;
      const size_t o = ((size_t)t * a.Hq + hq) * D + d4;
      put_plane(a.o_hi, a.o_lo, a.out_bf16, o, acc.x * il);
      put_plane(a.o_hi, a.o_lo, a.out_bf16, o + 1, acc.y * il);
      put_plane(a.o_hi, a.o_lo, a.out_bf16, o + 2, acc.z * il);
      put_plane(a.o_hi, a.o_lo, a.out_bf16, o + 3, acc.w * il);
    }
  }
  if (tid == 0) tc::bulk_wait_read();  // the copies have read this CTA's staged rows
}

template <int D, int CL>
static size_t attn_mma_smem() {
  constexpr int QLD = D + 8, RPC = QR / CL, RLD = D + 4;
  return (size_t)(2 * QR * QLD + 4 * AC * QLD) * 2 + ((size_t)CL * RPC * RLD + RPC * CL + RPC) * 4 + QR * 4;
}

template <int D, int CL>
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
  return cudaLaunchKernelEx(&cfg, attention_mma_kernel<D, CL>, a);
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
  prefer_shared(reinterpret_cast<const void*>(attention_mma_kernel<D, 16>));
  prefer_shared(reinterpret_cast<const void*>(attention_mma_kernel<D, 8>));
  const size_t smem16 = attn_mma_smem<D, 16>();
  if (cudaFuncSetAttribute(attention_mma_kernel<D, 16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
          cudaSuccess &&
      cudaFuncSetAttribute(attention_mma_kernel<D, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem16) ==
          cudaSuccess) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(16, 1, 1);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem16;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 16;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attention_mma_kernel<D, 16>, &cfg) == cudaSuccess && n >= 8) width = 16;
  }
  cudaGetLastError();
  if (width == 8)
    cudaFuncSetAttribute(attention_mma_kernel<D, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)attn_mma_smem<D, 8>());
  return width;
}

template <int D>
static bool launch_attn_mma(const AttnArgs& a, int n_slots, int max_rows, cudaStream_t s, bool pdl) {
  const int G = a.Hq / a.Hkv;
  const int n_rg = (max_rows * G + QR - 1) / QR;
  const int cl = attn_cluster_width<D>();
  const dim3 grid(cl, a.Hkv * n_rg, n_slots);
  return (cl == 16 ? launch_attn_cl<D, 16>(a, grid, s, pdl) : launch_attn_cl<D, 8>(a, grid, s, pdl)) ==
         cudaSuccess;
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
