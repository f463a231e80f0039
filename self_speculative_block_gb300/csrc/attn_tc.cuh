// Tensor-core attention on tcgen05: the partial kernel of the bf16 decoder's
// split-KV attention (rank r of the R ranks of a (request, kv head, 128-row
// group) visits key chunks r, r + R, ... of AC = 32 keys) with both
// contractions of a chunk on the 5th-generation tensor cores and their
// accumulators in tensor memory:
//   S  = Qh Kh^T + Qh Kl^T + Ql Kh^T       M = 128 query rows, N = 32 keys, K = d
//   PV = P Vh + P Vl                       M = 128 query rows, N = d, K = 32 keys
// (q and the cache as bf16 hi + lo planes, P in bf16, fp32 accumulation).
// Operands sit in shared memory in the 128-byte swizzled K-major layout: Q
// and K as loaded (cp.async into the swizzled positions), V transposed on
// the way (ldmatrix.trans from a row-major staging copy), P written by the
// softmax threads.  One thread issues the MMAs; warps 4-7 run the online
// softmax with one thread per query row (a row's 32 scores come from its own
// TMEM lane, so no cross-thread reduction); all eight warps fold each chunk's
// PV into the running output, O = O * corr + PV (warp w: rows 32 (w % 4) ..
// +31, output columns (w / 4) d/2 .. +d/2).  Two score buffers let the next
// chunk's QK^T run under this chunk's softmax; K/V are fetched two chunks
// ahead.
//
// A chunk with no key visible to a row leaves that row's (max, sum, output)
// bit for bit unchanged (corr = 1, P = 0), so a row's result does not depend
// on which other rows share the tile: the AR step, a verify row and a batched
// row at the same position give identical bits.  Partial rows (d outputs,
// max, sum) go to global memory for the fixed-order merge kernel.
#pragma once
#include "attn_core.cuh"
#include "tc.cuh"

namespace gocr {
namespace attn_tc {

constexpr int QR = 128;       // query rows per tile (MMA M)
constexpr int AC = attn::AC;  // keys per chunk: the rank split is shared with every other path
constexpr int THREADS = 256;
constexpr uint32_t S_COL = 0;     // TMEM columns of the two score accumulators [2][QR x AC]
constexpr uint32_t PV_COL = 128;  // TMEM columns of the chunk's P V accumulator [QR x d]
constexpr uint32_t TMEM_COLS = 256;

template <int D> struct Geo {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static constexpr int KB = D / 64;                // 64-element (128-byte) K blocks of a q / k row
  static constexpr int Q_PLANE = KB * QR * 128;    // [KB][QR rows][128 B], swizzled
  static constexpr int K_PLANE = KB * AC * 128;    // [KB][AC rows][128 B], swizzled
  static constexpr int VLD = D + 8;                // row stride (elements) of the row-major V staging
  static constexpr int V_PLANE = AC * VLD * 2;
  static constexpr int VT_PLANE = D * 128;         // [D rows][128 B], swizzled; keys in the first 64 B
  static constexpr int P_BYTES = QR * 128;         // [QR rows][128 B], swizzled; keys in the first 64 B
  static constexpr int OFF_Q = 0;                            // hi, lo
  static constexpr int OFF_K = OFF_Q + 2 * Q_PLANE;          // [stage][hi, lo]
  static constexpr int OFF_VT = OFF_K + 4 * K_PLANE;         // hi, lo
  static constexpr int OFF_P = OFF_VT + 2 * VT_PLANE;
  static constexpr int OFF_V = OFF_P + P_BYTES;              // [stage][hi, lo]
  static constexpr int OFF_LIM = OFF_V + 4 * V_PLANE;        // int [QR]
  static constexpr int OFF_LO2 = OFF_LIM + QR * 4;           // int [QR]: second key interval (training mask)
  static constexpr int OFF_HI2 = OFF_LO2 + QR * 4;           // int [QR]
  static constexpr int OFF_CORR = OFF_HI2 + QR * 4;          // float [QR]
  static constexpr int OFF_BAR = OFF_CORR + QR * 4;          // three mbarriers, the TMEM address
  static constexpr int SMEM = OFF_BAR + 32 + 1024;           // + slack for the 1024-byte alignment
  static constexpr int RLD = D + 4;                          // fp32 stride of a staged partial row
  static_assert(QR * RLD * 4 <= OFF_VT, "staged partial rows fit over Q and K");
  static_assert(OFF_K % 1024 == 0 && OFF_VT % 1024 == 0 && OFF_P % 1024 == 0, "1024-byte operand tiles");
};

// Byte offset of 16-byte chunk c of row r in a 128-byte swizzled tile.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// K (swizzled, both K blocks) and V (row-major staging) of chunk c into stage
// st, hi and lo planes; keys past kmax read as zero.
template <int D>
__device__ __forceinline__ void load_kv(uint8_t* sm, const attn::KvPlanes& kv, int st, int c, int kmax, int tid) {
  using Gm = Geo<D>;
  constexpr int CPR = D / 8;  // 16-byte chunks per key row
  for (int x = tid; x < 2 * AC * CPR; x += THREADS) {
    const int pl = x / (AC * CPR), rem = x % (AC * CPR);
    const int j = rem / CPR, v = rem % CPR;
    const int key = c * AC + j;
    const bool in = key <= kmax;
    const size_t src = (size_t)(in ? key : 0) * D + v * 8;
    uint8_t* kd = sm + Gm::OFF_K + (st * 2 + pl) * Gm::K_PLANE + (v >> 3) * (AC * 128) + sw128(j, v & 7);
    attn::cp_async16(kd, kv.p[pl] + src, in ? 16 : 0);
    uint8_t* vd = sm + Gm::OFF_V + (st * 2 + pl) * Gm::V_PLANE + (j * Gm::VLD + v * 8) * 2;
    attn::cp_async16(vd, kv.p[2 + pl] + src, in ? 16 : 0);
  }
}

// Transposed copy of the staged V planes of stage st: VT[d][key], key pairs as
// 32-bit words, through ldmatrix.trans on 8 x 8 blocks.
template <int D>
__device__ __forceinline__ void transpose_v(uint8_t* sm, int st, int warp, int lane) {
  using Gm = Geo<D>;
  constexpr int DB = D / 8;              // 8-wide d blocks
  constexpr int BLOCKS = 2 * (AC / 8) * DB;  // both planes
  for (int b0 = warp * 4; b0 < BLOCKS; b0 += 32) {
    // matrix m of this x4 load: block b0 + m; lanes 8m .. 8m+7 give its rows
    const int bm = b0 + (lane >> 3);
    const int pl = bm / ((AC / 8) * DB), rem = bm % ((AC / 8) * DB);
    const int kb = rem / DB, db = rem % DB;
    const uint8_t* src = sm + Gm::OFF_V + (st * 2 + pl) * Gm::V_PLANE + ((kb * 8 + (lane & 7)) * Gm::VLD + db * 8) * 2;
    uint32_t r[4];
    attn::ldsm_x4_trans(r, src);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int b = b0 + m;
      const int pl2 = b / ((AC / 8) * DB), rem2 = b % ((AC / 8) * DB);
      const int kb2 = rem2 / DB, db2 = rem2 % DB;
      const int d = db2 * 8 + (lane >> 2), key = kb2 * 8 + 2 * (lane & 3);
      uint8_t* dst = sm + Gm::OFF_VT + pl2 * Gm::VT_PLANE + sw128(d, key >> 3) + (key & 7) * 2;
      *reinterpret_cast<uint32_t*>(dst) = r[m];
    }
  }
}

}  // namespace attn_tc
}  // namespace gocr

namespace gocr {

// Partial kernel: one CTA per (kv head x 128-row group, rank, slot).  R2: rows
// also read a second key interval lo2..hi2 (the joint-training mask), and the
// rank skips the chunks that are masked for every row of its tile.
template <int D, bool TRACE, bool R2 = false>
__global__ void __launch_bounds__(attn_tc::THREADS, 1) attention_tc_part_kernel(AttnArgs a) {
  using namespace attn_tc;
  using Gm = Geo<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  int* Lim = reinterpret_cast<int*>(sm + Gm::OFF_LIM);
  int* Lo2 = reinterpret_cast<int*>(sm + Gm::OFF_LO2);
  int* Hi2 = reinterpret_cast<int*>(sm + Gm::OFF_HI2);
  float* Corr = reinterpret_cast<float*>(sm + Gm::OFF_CORR);
  uint64_t* s_full = reinterpret_cast<uint64_t*>(sm + Gm::OFF_BAR);  // [2] score buffers
  uint64_t* pv_full = s_full + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(pv_full + 1);
  __shared__ int s_maxlim;
  __shared__ int s_lim1, s_lo2min;  // R2: the rows' largest limit, smallest second-interval start
  __shared__ int s_fail;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int group = blockIdx.x, rank = blockIdx.y, R = gridDim.y, slot = blockIdx.z;
  const int kvh = group % a.Hkv, rg = group / a.Hkv;
  const int G = a.Hq / a.Hkv;

  if (tid == 0) {
    if (TRACE) trace_at(a, 0);
    tc::grid_dep_launch();
    tc::mbar_init(s_full, 1);
    tc::mbar_init(s_full + 1, 1);
    tc::mbar_init(pv_full, 1);
    tc::fence_mbar_init();
    s_maxlim = -1;
    s_lim1 = -1;
    s_lo2min = 0x7fffffff;
    s_fail = 0;
  }
  // committed cache before the dependency wait (decode launches only): the
  // first chunk into stage 0 when it holds only positions below the
  // round-start cache length, which no kernel of the forward writes, and the
  // rank's later committed chunks into L2
  int req_pre = -1;
  bool pre = false;
  if (a.st && a.slot_req) {
    req_pre = a.slot_req[slot];
    const int pc = a.st[req_pre].cache_len;
    pre = (rank + 1) * AC <= pc;
    if (pre) {
      const attn::KvPlanes kvp = attn::kv_planes(a, req_pre, kvh, D);
      load_kv<D>(sm, kvp, 0, rank, pc - 1, tid);
      attn::cp_async_commit();
      for (int i = tid; i < 4 * 8; i += THREADS) {
        const int c = rank + (1 + i / 4) * R;
        if ((c + 1) * AC <= pc) attn::prefetch_l2(kvp.p[i % 4] + (size_t)c * AC * D, AC * D * 2);
      }
    }
  }
  __syncwarp();
  if (warp == 0) tc::tmem_alloc(tmem_holder, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_holder;
  tc::grid_dep_wait();
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
  const int nq = nrows * G;
  const int qr0 = rg * QR;
  int n_chunks = 0;
  if (qr0 < nq) {  // uniform
    // Q planes of the row group (swizzled; zero past the window) and the row limits
    const bf16* qp[2] = {reinterpret_cast<const bf16*>(a.q_hi), reinterpret_cast<const bf16*>(a.q_lo)};
    constexpr int CPR = D / 8;
    const unsigned gm = 0xFFFFFFFFu / (unsigned)G + 1u;
    for (int x = tid; x < 2 * QR * CPR; x += THREADS) {
      const int pl = x / (QR * CPR), rem = x % (QR * CPR);
      const int r = rem / CPR, v = rem % CPR;
      const int gi = qr0 + r;
      size_t src = 0;
      if (gi < nq) {
        const int tq = attn::div_small(gi, G, gm);
        src = ((size_t)(row0 + tq) * a.Hq + kvh * G + (gi - tq * G)) * D + v * 8;
      }
      attn::cp_async16(sm + Gm::OFF_Q + pl * Gm::Q_PLANE + (v >> 3) * (QR * 128) + sw128(r, v & 7), qp[pl] + src,
                       gi < nq ? 16 : 0);
    }
    if (tid < QR) {
      const int gi = qr0 + tid;
      int lim = -1;
      const int t = gi < nq ? row0 + attn::div_small(gi, G, gm) : 0;
      if (gi < nq) lim = min(a.row_lim[t], a.cap - 1);
      Lim[tid] = lim;
      if (lim >= 0) {
        atomicMax(&s_maxlim, lim);
        if (R2) atomicMax(&s_lim1, lim);
      }
      if (R2) {
        int lo2 = 1, hi2 = 0;
        if (gi < nq) {
          lo2 = max(a.row_lo2[t], 0);
          hi2 = min(a.row_hi2[t], a.cap - 1);
        }
        Lo2[tid] = lo2;
        Hi2[tid] = hi2;
        if (hi2 >= lo2) {
          atomicMax(&s_maxlim, hi2);
          atomicMin(&s_lo2min, lo2);
        }
      }
    }
    __syncthreads();
    const int maxlim = s_maxlim;
    n_chunks = maxlim < 0 ? 0 : maxlim / AC + 1;
    if (rank == 0 && tid == 0) a.part_chunks[(size_t)slot * gridDim.x + group] = n_chunks;
    if (rank < n_chunks) {  // uniform
      const attn::KvPlanes kv = attn::kv_planes(a, req, kvh, D);
      // a rank's chunks: rank, rank + R, ... below n_chunks; with a second
      // interval (R2) minus the chunks cA .. c0 - 1, whose keys all lie past
      // every row's limit and before every row's second interval (for those
      // a row's state would not change).  chunk(it) is the it-th of them, in
      // increasing order: chunk it sits in stage it & 1 (K swizzled, V
      // row-major), its scores in S buffer it & 1.  n_it may be 0 (R2): the
      // rank then writes the empty partial (m = -inf, l = 0, O = 0).
      int cA = n_chunks, c0 = n_chunks;
      if (R2) {
        cA = s_lim1 < 0 ? 0 : s_lim1 / AC + 1;
        c0 = s_lo2min / AC < n_chunks ? s_lo2min / AC : n_chunks;
        if (c0 <= cA) cA = c0 = n_chunks;  // nothing to skip
      }
      const int n_a = rank < cA ? (cA - rank + R - 1) / R : 0;  // chunks below the skipped range
      const int cB = c0 + ((rank - c0) % R + R) % R;             // the first chunk past it
      const int n_it = n_a + (cB < n_chunks ? (n_chunks - cB + R - 1) / R : 0);
      auto chunk = [&](int it) { return it < n_a ? rank + it * R : cB + (it - n_a) * R; };
      if (!pre && n_it > 0) load_kv<D>(sm, kv, 0, chunk(0), maxlim, tid);
      attn::cp_async_commit();  // Q (and chunk 0)
      if (n_it > 1) load_kv<D>(sm, kv, 1, chunk(1), maxlim, tid);
      attn::cp_async_commit();  // chunk 1
      const float sl2 = a.scale * attn::LOG2E;
      const int q4 = warp & 3, h = warp >> 2;
      const int r = q4 * 32 + lane;  // this thread's tile row
      const int lim_r = Lim[r];
      const int lo2_r = R2 ? Lo2[r] : 1, hi2_r = R2 ? Hi2[r] : 0;
      const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
      constexpr int OH = D / 2;  // output columns per warp
      float O[OH];
#pragma unroll
      for (int j = 0; j < OH; ++j) O[j] = 0.f;
      float m = -INFINITY, l = 0.f;  // warps 4-7
      constexpr uint32_t idesc_s = tc::idesc_bf16(QR, AC);
      constexpr uint32_t idesc_pv = tc::idesc_bf16(QR, D);
      const uint32_t q_hi = tc::smem_u32(sm + Gm::OFF_Q), q_lo = q_hi + Gm::Q_PLANE;
      const uint32_t vt_hi = tc::smem_u32(sm + Gm::OFF_VT), vt_lo = vt_hi + Gm::VT_PLANE;
      const uint32_t p_s = tc::smem_u32(sm + Gm::OFF_P);
      // S(it) = Qh Kh^T, += Qh Kl^T, += Ql Kh^T over d in 16-element steps (one thread)
      auto issue_qk = [&](int it) {
        const int st = it & 1;
        const uint32_t k_hi = tc::smem_u32(sm + Gm::OFF_K + (st * 2) * Gm::K_PLANE), k_lo = k_hi + Gm::K_PLANE;
        const uint32_t as[3] = {q_hi, q_hi, q_lo}, bs[3] = {k_hi, k_lo, k_hi};
#pragma unroll
        for (int t = 0; t < 3; ++t)
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t ao = (ks >> 2) * (QR * 128) + (ks & 3) * 32;
            const uint32_t bo = (ks >> 2) * (AC * 128) + (ks & 3) * 32;
            tc::mma_bf16(tmem + S_COL + st * AC, tc::sdesc_sw128(as[t] + ao), tc::sdesc_sw128(bs[t] + bo), idesc_s,
                         (t > 0 || ks > 0) ? 1u : 0u);
          }
        tc::mma_commit(s_full + st);
      };
      // prologue: Q and chunk 0 in shared memory, its scores on the way
      if (n_it > 1) attn::cp_async_wait<1>(); else attn::cp_async_wait<0>();
      tc::fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0 && n_it > 0) {
        tc::fence_after_sync();
        issue_qk(0);
      }
      for (int it = 0; it < n_it; ++it) {
        const int st = it & 1, c = chunk(it);
        // chunk it + 1 landed; V of chunk it transposed (the last P V has completed)
        attn::cp_async_wait<0>();
        transpose_v<D>(sm, st, warp, lane);
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        if (TRACE && it == 0 && tid == 0) trace_at(a, 4);
        // the next chunk's scores while this chunk's softmax runs
        if (tid == 0 && it + 1 < n_it) {
          tc::fence_after_sync();
          issue_qk(it + 1);
        }
        if (warp >= 4) {
          // online softmax of row r over the chunk's 32 keys
          if (!tc::mbar_wait(s_full + st, (it >> 1) & 1)) s_fail = 1;
          tc::fence_after_sync();
          float sv[AC];
          tc::tmem_ld32(lane_base + S_COL + st * AC, sv);
          float mc = -INFINITY;
#pragma unroll
          for (int j = 0; j < AC; ++j) {
            const int key = c * AC + j;
            const bool vis = key <= lim_r || (R2 && key >= lo2_r && key <= hi2_r);
            const float v = vis ? sv[j] * sl2 : -INFINITY;
            sv[j] = v;
            mc = fmaxf(mc, v);
          }
          const float mn = fmaxf(m, mc);
          const float corr = mn == -INFINITY ? 1.f : (m == -INFINITY ? 0.f : exp2f(m - mn));
          float ps = 0.f;
          uint32_t pk[AC / 2];
#pragma unroll
          for (int j = 0; j < AC; j += 2) {
            const float p0 = sv[j] == -INFINITY ? 0.f : exp2f(sv[j] - mn);
            const float p1 = sv[j + 1] == -INFINITY ? 0.f : exp2f(sv[j + 1] - mn);
            ps += p0;
            ps += p1;
            pk[j / 2] = attn::pack_bf16(p0, p1);
          }
          l = fmaf(l, corr, ps);
          m = mn;
          Corr[r] = corr;
          uint8_t* prow = sm + Gm::OFF_P;
#pragma unroll
          for (int cc = 0; cc < AC / 8; ++cc)
            *reinterpret_cast<uint4*>(prow + sw128(r, cc)) =
                make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
          tc::fence_proxy_async_smem();
        }
        tc::fence_before_sync();
        __syncthreads();  // P and the corrections are in shared memory; S(it) and K(it) are consumed
        if (tid == 0) {
          tc::fence_after_sync();
          // PV = P Vh, += P Vl; over the chunk's keys in 16-element steps
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int ks = 0; ks < AC / 16; ++ks)
              tc::mma_bf16(tmem + PV_COL, tc::sdesc_sw128(p_s + ks * 32),
                           tc::sdesc_sw128((t ? vt_lo : vt_hi) + ks * 32), idesc_pv, (t > 0 || ks > 0) ? 1u : 0u);
          tc::mma_commit(pv_full);
        }
        // chunk it + 2 into this chunk's stage
        if (it + 2 < n_it) load_kv<D>(sm, kv, st, chunk(it + 2), maxlim, tid);
        attn::cp_async_commit();
        // O = O * corr + PV for this warp's rows and output columns
        if (!tc::mbar_wait(pv_full, it & 1)) s_fail = 1;
        tc::fence_after_sync();
        const float corr = Corr[r];
#pragma unroll
        for (int j0 = 0; j0 < OH; j0 += 32) {
          float pv[32];
          tc::tmem_ld32(lane_base + PV_COL + h * OH + j0, pv);
#pragma unroll
          for (int j = 0; j < 32; ++j) O[j0 + j] = fmaf(O[j0 + j], corr, pv[j]);
        }
        tc::fence_before_sync();
      }
      if (TRACE && tid == 0) trace_at(a, 5);
      __syncthreads();  // every MMA is complete: Q and K are dead
      float* ST = reinterpret_cast<float*>(sm);  // [QR][RLD] staged partial rows
#pragma unroll
      for (int j = 0; j < OH; j += 4)
        *reinterpret_cast<float4*>(ST + r * Gm::RLD + h * OH + j) = make_float4(O[j], O[j + 1], O[j + 2], O[j + 3]);
      if (warp >= 4) {
        ST[r * Gm::RLD + D] = m;
        ST[r * Gm::RLD + D + 1] = l;
      }
      __syncthreads();
      const float4* src = reinterpret_cast<const float4*>(ST);
      float4* dst = reinterpret_cast<float4*>(a.part + (((size_t)slot * gridDim.x + group) * R + rank) * QR * Gm::RLD);
      for (int x = tid; x < QR * Gm::RLD / 4; x += THREADS) dst[x] = src[x];
      if (s_fail && tid == 0) set_err(a.err, DERR_TIMEOUT);
      if (TRACE && tid == 0) trace_at(a, 3);
    }
  }
  attn::cp_async_wait<0>();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace gocr
