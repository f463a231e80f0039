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
// bf16 models: tensor-core kernel.  A cluster of CL CTAs shares one
// (kv head, 64-query-row group); CTA r visits chunks r, r + CL, ... with an
// online softmax on mma.sync tiles, then the cluster merges its CL partial
// (max, sum, output) triples through distributed shared memory in rank order.
// fp32 models: CUDA-core kernel with one CTA sweeping every chunk.
#include <cooperative_groups.h>

#include "kernels.cuh"

namespace gocr {

namespace {
constexpr int ROWS = 128;   // query rows (token, q-head-in-group) per CTA
constexpr int CH = 64;      // keys per chunk
}

template <typename T, int D>
__global__ void __launch_bounds__(ROWS) attention_simt_kernel(AttnArgs a) {
  extern __shared__ float sm[];
  float* Qs = sm;                     // [ROWS][D + 1]
  float* Os = Qs + ROWS * (D + 1);    // [ROWS][D + 1]
  float* Ks = Os + ROWS * (D + 1);    // [CH][D]
  float* Vs = Ks + CH * D;            // [CH][D]
  __shared__ int s_maxlim;

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

  const T* q = reinterpret_cast<const T*>(a.q);
  const T* kc = reinterpret_cast<const T*>(a.kc) + (size_t)req * a.req_stride + (size_t)kvh * a.cap * D;
  const T* vc = reinterpret_cast<const T*>(a.vc) + (size_t)req * a.req_stride + (size_t)kvh * a.cap * D;
  T* o = reinterpret_cast<T*>(a.o);

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
    Qs[i * (D + 1) + dd] = valid ? to_f32<T>(q[((size_t)t * a.Hq + hq) * D + dd]) : 0.f;
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
      Ks[x] = in ? to_f32<T>(kc[(size_t)(kbase + j) * D + dd]) : 0.f;
      Vs[x] = in ? to_f32<T>(vc[(size_t)(kbase + j) * D + dd]) : 0.f;
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
    for (int dd = 0; dd < D; ++dd)
      o[((size_t)t * a.Hq + hq) * D + dd] = from_f32<T>(Os[i * (D + 1) + dd] * inv);
  }
}

// ---------------------------------------------------------------- tensor-core path

namespace {
constexpr int CL = 8;        // CTAs per cluster (key-chunk split)
constexpr int QR = 64;       // query rows per cluster
constexpr float LOG2E = 1.4426950408889634f;
}

__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int D>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(128) attention_mma_kernel(AttnArgs a, int n_rg) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  constexpr int QLD = D + 8;   // bf16 row stride of Q and K tiles
  constexpr int VLD = 64 + 8;  // bf16 row stride of the transposed V tile
  constexpr int OLD = D + 4;   // fp32 row stride of the partial output
  extern __shared__ __align__(16) uint8_t sm_raw[];
  bf16* Qs = reinterpret_cast<bf16*>(sm_raw);            // [QR][QLD]
  bf16* Ks = Qs + QR * QLD;                              // [64][QLD]
  bf16* Vt = Ks + 64 * QLD;                              // [D][VLD]
  float* Ob = reinterpret_cast<float*>(Vt + D * VLD);    // [QR][OLD]
  float* Ms = Ob + QR * OLD;                             // [QR] running max (log2 units)
  float* Ls = Ms + QR;                                   // [QR] running sum
  int* Lim = reinterpret_cast<int*>(Ls + QR);            // [QR]
  __shared__ int s_maxlim;

  const int rank = blockIdx.x;  // == cluster rank (cluster spans grid x)
  const int kvh = blockIdx.y % a.Hkv;
  const int rg = blockIdx.y / a.Hkv;
  const int slot = blockIdx.z;
  const int G = a.Hq / a.Hkv;
  int req = 0, row0 = 0, nrows = a.T;
  if (a.plan) {
    req = a.plan->slot_req[slot];
    row0 = a.plan->slot_row0[slot];
    nrows = a.plan->slot_nrows[slot];
  }
  const int nq = nrows * G;
  const int qr0 = rg * QR;
  if (qr0 >= nq) return;  // uniform across the cluster
  const bf16* q = reinterpret_cast<const bf16*>(a.q);
  const bf16* kc = reinterpret_cast<const bf16*>(a.kc) + (size_t)req * a.req_stride + (size_t)kvh * a.cap * D;
  const bf16* vc = reinterpret_cast<const bf16*>(a.vc) + (size_t)req * a.req_stride + (size_t)kvh * a.cap * D;
  bf16* o = reinterpret_cast<bf16*>(a.o);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;

  if (tid == 0) s_maxlim = -1;
  __syncthreads();
  // stage Q rows (zero for rows past the window) and their key limits
  for (int x = tid; x < QR * (D / 8); x += 128) {
    const int r = x / (D / 8), v = x % (D / 8);
    const int gi = qr0 + r;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (gi < nq) {
      const int t = row0 + gi / G, hq = kvh * G + gi % G;
      val = *reinterpret_cast<const uint4*>(q + ((size_t)t * a.Hq + hq) * D + v * 8);
    }
    *reinterpret_cast<uint4*>(Qs + r * QLD + v * 8) = val;
  }
  if (tid < QR) {
    const int gi = qr0 + tid;
    int lim = -1;
    if (gi < nq) lim = min(a.row_lim[row0 + gi / G], a.cap - 1);
    Lim[tid] = lim;
    if (lim >= 0) atomicMax(&s_maxlim, lim);
  }
  __syncthreads();
  const int maxlim = s_maxlim;
  const int n_chunks = maxlim < 0 ? 0 : maxlim / 64 + 1;
  const float sl2 = a.scale * LOG2E;

  const int r_lo = warp * 16 + g, r_hi = r_lo + 8;
  const int lim_lo = Lim[r_lo], lim_hi = Lim[r_hi];
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  float oacc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

  for (int c = rank; c < n_chunks; c += CL) {
    const int kbase = c * 64;
    for (int x = tid; x < 64 * (D / 8); x += 128) {
      const int j = x / (D / 8), v = x % (D / 8);
      uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
      if (kbase + j <= maxlim) {
        kv = *reinterpret_cast<const uint4*>(kc + (size_t)(kbase + j) * D + v * 8);
        vv = *reinterpret_cast<const uint4*>(vc + (size_t)(kbase + j) * D + v * 8);
      }
      *reinterpret_cast<uint4*>(Ks + j * QLD + v * 8) = kv;
      const bf16* ve = reinterpret_cast<const bf16*>(&vv);
#pragma unroll
      for (int e = 0; e < 8; ++e) Vt[(v * 8 + e) * VLD + j] = ve[e];
    }
    __syncthreads();
    // S = Q K^T for this warp's 16 rows and the chunk's 64 keys
    float sacc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t af[4];
      const bf16* qa = Qs + (warp * 16 + g) * QLD + ks * 16 + tq * 2;
      af[0] = *reinterpret_cast<const uint32_t*>(qa);
      af[1] = *reinterpret_cast<const uint32_t*>(qa + 8 * QLD);
      af[2] = *reinterpret_cast<const uint32_t*>(qa + 8);
      af[3] = *reinterpret_cast<const uint32_t*>(qa + 8 * QLD + 8);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        uint32_t bfr[2];
        const bf16* kb = Ks + (nt * 8 + g) * QLD + ks * 16 + tq * 2;
        bfr[0] = *reinterpret_cast<const uint32_t*>(kb);
        bfr[1] = *reinterpret_cast<const uint32_t*>(kb + 8);
        mma16816(sacc[nt], af, bfr);
      }
    }
    // mask, scale to log2 units, chunk row maxima
    float mc_lo = -INFINITY, mc_hi = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
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
    uint32_t pf[8][2];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
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
    // O += P V
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      uint32_t af[4] = {pf[2 * kt][0], pf[2 * kt][1], pf[2 * kt + 1][0], pf[2 * kt + 1][1]};
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        uint32_t bfr[2];
        const bf16* vb = Vt + (dn * 8 + g) * VLD + kt * 16 + tq * 2;
        bfr[0] = *reinterpret_cast<const uint32_t*>(vb);
        bfr[1] = *reinterpret_cast<const uint32_t*>(vb + 8);
        mma16816(oacc[dn], af, bfr);
      }
    }
    __syncthreads();
  }
  // publish this CTA's partial (unnormalised output, max, sum)
#pragma unroll
  for (int dn = 0; dn < D / 8; ++dn) {
    Ob[r_lo * OLD + dn * 8 + tq * 2] = oacc[dn][0];
    Ob[r_lo * OLD + dn * 8 + tq * 2 + 1] = oacc[dn][1];
    Ob[r_hi * OLD + dn * 8 + tq * 2] = oacc[dn][2];
    Ob[r_hi * OLD + dn * 8 + tq * 2 + 1] = oacc[dn][3];
  }
  if (tq == 0) {
    Ms[r_lo] = m_lo; Ls[r_lo] = l_lo;
    Ms[r_hi] = m_hi; Ls[r_hi] = l_hi;
  }
  cluster.sync();
  // merge: CTA `rank` finalises rows rank, rank + CL, ... in cluster-rank order
  for (int r = rank; r < QR; r += CL) {
    const int gi = qr0 + r;
    if (gi >= nq) break;
    float mv[CL], lv[CL];
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < CL; ++c) {
      mv[c] = *cluster.map_shared_rank(Ms + r, c);
      lv[c] = *cluster.map_shared_rank(Ls + r, c);
      M = fmaxf(M, mv[c]);
    }
    float L = 0.f;
    float wv[CL];
#pragma unroll
    for (int c = 0; c < CL; ++c) {
      wv[c] = mv[c] == -INFINITY ? 0.f : exp2f(mv[c] - M);
      L += wv[c] * lv[c];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int t = row0 + gi / G, hq = kvh * G + gi % G;
    for (int d = tid; d < D; d += 128) {
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < CL; ++c) acc += wv[c] * *cluster.map_shared_rank(Ob + r * OLD + d, c);
      o[((size_t)t * a.Hq + hq) * D + d] = __float2bfloat16_rn(acc * inv);
    }
  }
  cluster.sync();
}

template <int D>
static void launch_attn_mma(const AttnArgs& a, int n_slots, int max_rows, cudaStream_t s) {
  const int G = a.Hq / a.Hkv;
  const int n_rg = (max_rows * G + QR - 1) / QR;
  dim3 grid(CL, a.Hkv * n_rg, n_slots);
  constexpr int QLD = D + 8, VLD = 72, OLD = D + 4;
  size_t smem = (size_t)(QR * QLD + 64 * QLD + D * VLD) * 2 + (size_t)QR * OLD * 4 + QR * 12;
  static bool init = false;
  if (!init) {
    cudaFuncSetAttribute(attention_mma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    init = true;
  }
  attention_mma_kernel<D><<<grid, 128, smem, s>>>(a, n_rg);
}

template <typename T, int D>
static void launch_attn_t(const AttnArgs& a, int n_slots, int max_rows, cudaStream_t s) {
  const int G = a.Hq / a.Hkv;
  dim3 grid((max_rows * G + ROWS - 1) / ROWS, a.Hkv, n_slots);
  size_t smem = sizeof(float) * (2 * ROWS * (D + 1) + 2 * CH * D);
  static bool init = false;
  if (!init) {
    cudaFuncSetAttribute(attention_simt_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    init = true;
  }
  attention_simt_kernel<T, D><<<grid, ROWS, smem, s>>>(a);
}

void launch_attention(int dtype, const AttnArgs& a, int n_slots, int max_rows, cudaStream_t s) {
  if (dtype == 1) {
    if (a.d == 128) launch_attn_mma<128>(a, n_slots, max_rows, s);
    else launch_attn_mma<64>(a, n_slots, max_rows, s);
  } else {
    if (a.d == 128) launch_attn_t<float, 128>(a, n_slots, max_rows, s);
    else launch_attn_t<float, 64>(a, n_slots, max_rows, s);
  }
}

}  // namespace gocr
