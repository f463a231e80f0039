// Tensor-core attention of one (request, kv head, 64-query-row group) tile
// over a fixed subset of key chunks, and the fixed-order merge of the
// partial results of the R tiles ("ranks") that share those query rows.
//
// The attention partial kernel runs one tile per CTA; the merge adds the
// ranks' partial rows in rank order.
//
// Layout of the work: keys sit in chunks of AC = 32 at absolute positions;
// rank r of the R ranks visits chunks r, r + R, ... (with a second key
// interval per row, minus the chunks masked for every row of its tile, which
// would change nothing).  In a tile,
// warp w owns query rows 16 (w % 4) .. +15 and key half w / 4 (keys
// 16 (w / 4) .. +15 of every chunk), so each (rank, key half) runs its own
// online softmax over a fixed set of key positions.  A chunk with no key
// visible to a row leaves that row's running (max, sum, output) bit for bit
// unchanged, so a row's result does not depend on the other rows.  q and the
// KV cache are bf16 hi + lo planes: QK^T takes qh kh + qh kl + ql kh and PV
// takes P vh + P vl on mma.sync tiles (P in bf16), accumulating in fp32.
// K and V chunks come into shared memory by TMA (128-byte swizzled 32 x 64
// boxes of the cache planes, counted on one mbarrier for K and one for V);
// q rows by cp.async.
#pragma once
#include <cuda.h>

#include "epilogue.cuh"
#include "tc.cuh"

namespace gocr {
namespace attn {

constexpr int QR = 64;      // query rows (token, q head) per tile
constexpr int AC = 32;      // keys per chunk
constexpr float LOG2E = 1.4426950408889634f;

template <int D> struct Geo {
  static constexpr int QLD = D + 8;    // bf16 row stride of the Q tiles
  static constexpr int OLD = D + 4;    // fp32 row stride of the half-1 partial
  static constexpr int KVP = AC * D;   // bf16 elements of one K/V chunk plane (swizzled 128-byte rows)
  static constexpr int RLD = D + 4;    // fp32 stride of a partial row: D outputs, max, sum, pad
  // shared memory of one tile (from a 1024-byte aligned base): Q planes, the
  // four K/V chunk planes (their region also holds the staged partial rows),
  // row limits; 1024 bytes of slack for the alignment
  static constexpr size_t Q_BYTES = (size_t)2 * QR * QLD * 2;
  static constexpr size_t KV_MIN = (size_t)4 * KVP * 2 > (size_t)QR * RLD * 4 ? (size_t)4 * KVP * 2 : (size_t)QR * RLD * 4;
  static constexpr size_t KV_BYTES = (KV_MIN + 1023) / 1024 * 1024;
  static constexpr size_t LIM_BYTES = QR * 4;
  static constexpr size_t TILE_SMEM = 1024 + Q_BYTES + KV_BYTES + LIM_BYTES + 16;
  // tiles with a second key interval per row: its bounds after the limits
  static constexpr size_t TILE_SMEM_R2 = TILE_SMEM + 2 * LIM_BYTES;
  static_assert(Q_BYTES % 1024 == 0, "the K/V planes start on a 1024-byte boundary (128-byte swizzle)");
  static_assert((size_t)QR * OLD * 4 + 2 * QR * 4 <= Q_BYTES, "half-1 partial fits the Q region");
};

// The four cache planes (K hi, K lo, V hi, V lo) as 2-D tensor maps over rows
// of D values, boxes of AC rows x 64 values with the 128-byte swizzle; passed
// to the kernels as one __grid_constant__ parameter.
struct KvMaps {
  CUtensorMap m[4];
};

// The tile's shared memory from a 1024-byte aligned address.
__device__ __forceinline__ uint8_t* tile_base(uint8_t* raw) {
  return raw + ((1024u - (tc::smem_u32(raw) & 1023u)) & 1023u);
}

// Element offset of (key row r, value c) in a K/V chunk plane as TMA writes
// it: 64-value halves of AC rows, 128-byte rows whose 16-byte chunks are
// XOR-swizzled by r % 8.
__device__ __forceinline__ int kv_el(int r, int c) {
  return (c >> 6) * (AC * 64) + r * 64 + ((((c & 63) >> 3) ^ (r & 7)) << 3) + (c & 7);
}

// TMA loads of the two planes [pl0, pl0 + 2) (K or V) of the chunk whose first
// key is cache row `row`, counted on `bar`; one thread issues them.
template <int D>
__device__ __forceinline__ void tma_planes(bf16* KV, const KvMaps& tms, int pl0, long long row, uint64_t* bar) {
  constexpr int HALVES = D / 64;
  tc::mbar_expect_tx(bar, (uint32_t)(2 * HALVES * AC * 64 * 2));
#pragma unroll
  for (int pl = pl0; pl < pl0 + 2; ++pl)
#pragma unroll
    for (int h = 0; h < HALVES; ++h)
      tc::tma_load_2d(KV + pl * Geo<D>::KVP + h * AC * 64, &tms.m[pl], h * 64, (int)row, bar);
}

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

// floor(n / g) for 0 <= n < 2^20 and 1 <= g <= 64 by a multiply-high with
// gm = floor((2^32 - 1) / g) + 1 (exact in that range; g = 1 passes n through).
__device__ __forceinline__ int div_small(int n, int g, unsigned gm) {
  return g == 1 ? n : (int)__umulhi((unsigned)n, gm);
}

// Cache planes of one (request, kv head): K hi, K lo, V hi, V lo.
struct KvPlanes {
  const bf16* p[4];
};

__device__ __forceinline__ KvPlanes kv_planes(const AttnArgs& a, int req, int kvh, int D) {
  const size_t o = (size_t)req * a.req_stride + (size_t)kvh * a.cap * D;
  KvPlanes k;
  k.p[0] = reinterpret_cast<const bf16*>(a.k_hi) + o;
  k.p[1] = reinterpret_cast<const bf16*>(a.k_lo) + o;
  k.p[2] = reinterpret_cast<const bf16*>(a.v_hi) + o;
  k.p[3] = reinterpret_cast<const bf16*>(a.v_lo) + o;
  return k;
}

// Work a tile may start before the rows' q and the window's K/V exist: when
// its first chunk holds only committed cache positions (below the round-start
// cache length pc, which no kernel of the forward writes), that chunk's K and
// V go to shared memory (TMA on kbar and vbar; kvrow is the cache row of key
// 0 of this tile's (request, kv head)) and the tile's later committed chunks
// (rank + stride, ...) into L2.  Returns whether the first chunk was issued.
template <int D>
__device__ __forceinline__ bool tile_prefetch(uint8_t* sm, const KvMaps& tms, const KvPlanes& kv, long long kvrow,
                                              int rank, int stride, int pc, int tid, uint64_t* kbar, uint64_t* vbar) {
  bf16* KV = reinterpret_cast<bf16*>(sm + Geo<D>::Q_BYTES);
  const bool pre = (rank + 1) * AC <= pc;
  if (pre) {
    if (tid == 0) {
      tma_planes<D>(KV, tms, 0, kvrow + (long long)rank * AC, kbar);
      tma_planes<D>(KV, tms, 2, kvrow + (long long)rank * AC, vbar);
    }
    for (int i = tid; i < 4 * 8; i += 256) {
      const int c = rank + (1 + i / 4) * stride;
      if ((c + 1) * AC <= pc) prefetch_l2(kv.p[i % 4] + (size_t)c * AC * D, AC * D * 2);
    }
  }
  return pre;
}

// One tile: query rows qr0 .. qr0+63 of the (row, q head) list of a request
// window (rows row0 .. row0+nrows-1, G = Hq / Hkv heads per kv head), keys
// of chunks rank, rank + stride, ...  `pre`: tile_prefetch issued the first
// chunk.  Returns the number of chunks the rows read (the last visible key
// of any row, over AC).  When rank < that number the tile's partial rows (D
// outputs, max, sum; stride RLD, row r at r * RLD) sit in shared memory at
// staged_rows(sm) on return; otherwise nothing is staged (the rank holds
// no chunk).  Every thread of the 256-thread group calls it.
template <int D>
__device__ __forceinline__ float* staged_rows(uint8_t* sm) {
  return reinterpret_cast<float*>(sm + Geo<D>::Q_BYTES);
}

// TRACE: record timeline marks in a.trace (first chunk ready, loop done).
// kv_kmax >= 0 (decode launches): no row of the forward reads past cache
// position kv_kmax, so a first chunk that tile_prefetch did not fetch and
// that starts at or below it is loaded right away, together with Q, instead
// of after the rows' key limits are known.  Keys past a row's limit
// contribute exact zeros: their scores are masked before the softmax, and
// the V rows past the tile's last visible key are zeroed after they land.
// R2: rows also read a second key interval (a.row_lo2 / a.row_hi2), whose
// bounds sit in TILE_SMEM_R2's extra shared memory.
template <int D, bool TRACE = false, bool R2 = false>
__device__ int tile_partial(const AttnArgs& a, uint8_t* sm, const Grp& grp, const KvMaps& tms, long long kvrow,
                            uint64_t* kbar, uint64_t* vbar, int rank, int stride, int kvh, int qr0, int row0,
                            int nrows, bool pre, int* s_maxlim, int kv_kmax = -1) {
  using Gm = Geo<D>;
  constexpr int QLD = Gm::QLD, OLD = Gm::OLD, KVP = Gm::KVP, RLD = Gm::RLD;
  bf16* Qh = reinterpret_cast<bf16*>(sm);               // [QR][QLD]
  bf16* Ql = Qh + QR * QLD;
  bf16* KV = Ql + QR * QLD;                             // {Kh, Kl, Vh, Vl} [AC][D] swizzled (kv_el)
  int* Lim = reinterpret_cast<int*>(sm + Gm::Q_BYTES + Gm::KV_BYTES);  // [QR]
  int* Lo2 = Lim + QR;                                  // [QR] (R2 only)
  int* Hi2 = Lo2 + QR;                                  // [QR] (R2 only)
  float* Oh = reinterpret_cast<float*>(Qh);             // [QR][OLD] half-1 partial (Q is dead by then)
  float* Mh = Oh + QR * OLD;                            // [QR]
  float* Lh = Mh + QR;                                  // [QR]
  float* ST = reinterpret_cast<float*>(KV);             // [QR][RLD] staged rows

  const int G = a.Hq / a.Hkv;
  const int tid = grp.tid, warp = tid >> 5, lane = tid & 31;
  const int mt = warp & 3, kh = warp >> 2;
  const int g = lane >> 2, tq = lane & 3;
  const int nq = nrows * G;
  const bf16* qh = reinterpret_cast<const bf16*>(a.q_hi);
  const bf16* ql = reinterpret_cast<const bf16*>(a.q_lo);

  __shared__ int s_lim1, s_lo2min;  // R2: the rows' largest limit, smallest second-interval start
  if (tid == 0) {
    *s_maxlim = -1;
    s_lim1 = -1;
    s_lo2min = 0x7fffffff;
  }
  grp.sync();
  const bool early = !pre && kv_kmax >= 0 && rank * AC <= kv_kmax;
  if (early && tid == 0) {
    tma_planes<D>(KV, tms, 0, kvrow + (long long)rank * AC, kbar);
    tma_planes<D>(KV, tms, 2, kvrow + (long long)rank * AC, vbar);
  }
  // Q planes of this row group (zero past the window) and the rows' key limits
  const unsigned gm = 0xFFFFFFFFu / (unsigned)G + 1u;
  for (int x = tid; x < 2 * QR * (D / 8); x += 256) {
    const int pl = x / (QR * (D / 8)), rem = x % (QR * (D / 8));
    const int r = rem / (D / 8), v = rem % (D / 8);
    const int gi = qr0 + r;
    size_t src = 0;
    if (gi < nq) {
      const int tq = div_small(gi, G, gm);
      src = ((size_t)(row0 + tq) * a.Hq + kvh * G + (gi - tq * G)) * D + v * 8;
    }
    cp_async16((pl ? Ql : Qh) + r * QLD + v * 8, (pl ? ql : qh) + src, gi < nq ? 16 : 0);
  }
  cp_async_commit();
  if (tid < QR) {
    const int gi = qr0 + tid;
    int lim = -1;
    if (gi < nq) lim = min(a.row_lim[row0 + div_small(gi, G, gm)], a.cap - 1);
    Lim[tid] = lim;
    if (lim >= 0) {
      atomicMax(s_maxlim, lim);
      if (R2) atomicMax(&s_lim1, lim);
    }
    if (R2) {
      int lo2 = 1, hi2 = 0;
      if (gi < nq) {
        lo2 = max(a.row_lo2[row0 + div_small(gi, G, gm)], 0);
        hi2 = min(a.row_hi2[row0 + div_small(gi, G, gm)], a.cap - 1);
      }
      Lo2[tid] = lo2;
      Hi2[tid] = hi2;
      if (hi2 >= lo2) {
        atomicMax(s_maxlim, hi2);
        atomicMin(&s_lo2min, lo2);
      }
    }
  }
  grp.sync();
  const int maxlim = *s_maxlim;
  const int n_chunks = maxlim < 0 ? 0 : maxlim / AC + 1;
  // R2: a chunk whose keys all lie past every row's limit and before every
  // row's second interval is an exact no-op for the tile: the rank skips it.
  // next_chunk(c): the rank's next chunk after c that is not skipped.
  const int lim1 = R2 ? s_lim1 : maxlim, lo2min = R2 ? s_lo2min : 0x7fffffff;
  auto skip = [&](int c) { return R2 && c * AC > lim1 && (c + 1) * AC - 1 < lo2min; };
  auto next_chunk = [&](int c) {
    c += stride;
    if (skip(c)) {
      // the chunk of the smallest start (not skipped, nor any after it), at most n_chunks
      const int c0 = lo2min / AC < n_chunks ? lo2min / AC : n_chunks;
      c = c0 + ((rank - c0) % stride + stride) % stride;
    }
    return c;
  };
  if (rank >= n_chunks) {  // uniform: this rank holds no chunk
    cp_async_wait<0>();
    if (pre || early) {  // no copy outlives the CTA
      const bool ok = tc::mbar_wait(kbar, 0) && tc::mbar_wait(vbar, 0);
      if (!ok && tid == 0) set_err(a.err, DERR_TIMEOUT);
    }
    return n_chunks;
  }
  const float sl2 = a.scale * LOG2E;

  const int r_lo = mt * 16 + g, r_hi = r_lo + 8;
  const int lim_lo = Lim[r_lo], lim_hi = Lim[r_hi];
  const int a_lo = R2 ? Lo2[r_lo] : 1, b_lo = R2 ? Hi2[r_lo] : 0;
  const int a_hi = R2 ? Lo2[r_hi] : 1, b_hi = R2 ? Hi2[r_hi] : 0;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  float oacc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int lcol = (lane >> 4) * 8;
  const bf16* Kh = KV;  // this warp's 16 keys of the chunk: rows kh * 16 .. of each plane
  const bf16* Kl = KV + KVP;
  const bf16* Vh = KV + 2 * KVP;
  const bf16* Vl = KV + 3 * KVP;

  // K and V of a chunk arrive on kbar and vbar (one phase per chunk): K of the
  // next chunk streams in while this chunk's softmax and PV run, V of the next
  // chunk while the next QK^T runs.  The first chunk went out before the
  // dependency wait (pre), right after it (early), or goes out now.
  // (the first chunk issued before the limits were known is chunk `rank`)
  const int c_first = (!pre && !early && skip(rank)) ? next_chunk(rank - stride) : rank;
  if (!pre && !early && tid == 0 && c_first < n_chunks) {
    tma_planes<D>(KV, tms, 0, kvrow + (long long)c_first * AC, kbar);
    tma_planes<D>(KV, tms, 2, kvrow + (long long)c_first * AC, vbar);
  }
  if (c_first >= n_chunks) cp_async_wait<0>();  // every chunk of this rank skipped: q only
  int it = 0;
  for (int c = c_first; c < n_chunks; ++it) {
    const int kbase = c * AC + kh * 16;
    const int cn = next_chunk(c);
    const bool next = cn < n_chunks;
    if (it == 0) cp_async_wait<0>();  // q
    if (!tc::mbar_wait(kbar, it & 1) && tid == 0) set_err(a.err, DERR_TIMEOUT);  // this chunk's K
    grp.sync();
    if (TRACE && it == 0 && tid == 0) trace_at(a, 4);
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
        const int kr = kh * 16 + nt * 8 + g, kc = ks * 16 + tq * 2;
        const int ko0 = kv_el(kr, kc), ko1 = kv_el(kr, kc + 8);
        uint32_t bh[2], bl[2];
        bh[0] = *reinterpret_cast<const uint32_t*>(Kh + ko0);
        bh[1] = *reinterpret_cast<const uint32_t*>(Kh + ko1);
        bl[0] = *reinterpret_cast<const uint32_t*>(Kl + ko0);
        bl[1] = *reinterpret_cast<const uint32_t*>(Kl + ko1);
        mma16816(sacc[nt], al, bh);
        mma16816(sacc[nt], ah, bl);
        mma16816(sacc[nt], ah, bh);
      }
    }
    grp.sync();  // every warp is done with this chunk's K
    if (next && tid == 0) tma_planes<D>(KV, tms, 0, kvrow + (long long)cn * AC, kbar);
    // mask, scale to log2 units, row maxima over the 16 keys
    float mc_lo = -INFINITY, mc_hi = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = kbase + nt * 8 + tq * 2 + e;
        const bool in_lo = key <= lim_lo || (R2 && key >= a_lo && key <= b_lo);
        const bool in_hi = key <= lim_hi || (R2 && key >= a_hi && key <= b_hi);
        float s0 = in_lo ? sacc[nt][e] * sl2 : -INFINITY;
        float s1 = in_hi ? sacc[nt][2 + e] * sl2 : -INFINITY;
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
    // this chunk's V (the next chunk's K may still be in flight)
    if (!tc::mbar_wait(vbar, it & 1) && tid == 0) set_err(a.err, DERR_TIMEOUT);
    if (c * AC + AC - 1 > maxlim) {  // uniform: the chunk of the tile's last visible key
      // keys past it may hold stale (even non-finite) cache contents, which
      // TMA copies as they are: zero their V rows so that P = 0 adds exact zeros
      const int r0 = maxlim - c * AC + 1, nr = AC - r0;
      for (int x = tid; x < 2 * nr * (D / 8); x += 256) {
        const int pl = 2 + x / (nr * (D / 8)), rem = x % (nr * (D / 8));
        *reinterpret_cast<uint4*>(KV + pl * KVP + kv_el(r0 + rem / (D / 8), (rem % (D / 8)) * 8)) =
            make_uint4(0u, 0u, 0u, 0u);
      }
      grp.sync();
    }
    // O += P (V_hi + V_lo); B fragments of two d-tiles per ldmatrix.x4.trans
    uint32_t af[4] = {pf[0][0], pf[0][1], pf[1][0], pf[1][1]};
#pragma unroll
    for (int dn = 0; dn < D / 8; dn += 2) {
      const int vo = kv_el(kh * 16 + lrow, dn * 8 + lcol);
      uint32_t bh[4], bl[4];
      ldsm_x4_trans(bh, Vh + vo);
      ldsm_x4_trans(bl, Vl + vo);
      mma16816(oacc[dn], af, bl);
      mma16816(oacc[dn], af, bh);
      mma16816(oacc[dn + 1], af, bl + 2);
      mma16816(oacc[dn + 1], af, bh + 2);
    }
    grp.sync();  // every warp is done with this chunk's V
    if (next && tid == 0) tma_planes<D>(KV, tms, 2, kvrow + (long long)cn * AC, vbar);
    c = cn;
  }
  grp.sync();
  if (TRACE && tid == 0) trace_at(a, 5);
  // merge the two key halves of this tile: half 0 + half 1, in that order
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
  grp.sync();
  if (kh == 0) {
    const float m1_lo = Mh[r_lo], m1_hi = Mh[r_hi];
    const float M_lo = fmaxf(m_lo, m1_lo), M_hi = fmaxf(m_hi, m1_hi);
    const float w0_lo = m_lo == -INFINITY ? 0.f : exp2f(m_lo - M_lo);
    const float w1_lo = m1_lo == -INFINITY ? 0.f : exp2f(m1_lo - M_lo);
    const float w0_hi = m_hi == -INFINITY ? 0.f : exp2f(m_hi - M_hi);
    const float w1_hi = m1_hi == -INFINITY ? 0.f : exp2f(m1_hi - M_hi);
    const float L_lo = w0_lo * l_lo + w1_lo * Lh[r_lo];
    const float L_hi = w0_hi * l_hi + w1_hi * Lh[r_hi];
    // stage this tile's partial rows
    float* st_lo = ST + r_lo * RLD;
    float* st_hi = ST + r_hi * RLD;
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
  grp.sync();
  return n_chunks;
}

// Merge of tile rows i0 and i0 + step (cnt = 1 or 2 of them, < QR) from the
// partial rows of ranks 0 .. n_ranks-1 (n_ranks <= r_all <= 64, r_all the
// rank slots part() may address): part(c, i) -> D
// outputs, max, sum of rank c's partial of row i.  Ranks whose chunks a row
// cannot see hold (-inf, 0, 0) and add exact zeros, so the result does not
// depend on n_ranks beyond the row's own chunks.  Fixed order: warp k reduces
// row k's maxima and weighted sums over lanes (lane l holds ranks l and
// l + 32, added in that order, then a fixed butterfly); the outputs are four
// sums over the ranks of each residue mod 4 (in rank order), added as
// ((s0 + s1) + s2) + s3.  The group has 256 threads.  WS: [2][64], IL: [2]
// and AC: [4][64] float4 shared scratch; writes the rows' output planes.
template <int D, bool GLOBAL, class Part>
__device__ void merge_rows(const AttnArgs& a, const Grp& grp, const Part& part, float* WS, float* IL, float4* AC,
                           int n_ranks, int r_all, int i0, int step, int cnt, int kvh, int qr0, int row0,
                           int nrows) {
  static_assert(D <= 128 && D % 4 == 0, "two rows of output quads per 64 threads");
  const int tid = grp.tid, warp = tid >> 5, lane = tid & 31;
  const int G = a.Hq / a.Hkv;
  const int nq = nrows * G;
  auto ld = [&](const float* p) -> float { return GLOBAL ? __ldcg(p) : *p; };
  // thread: residue q = tid / 64 of the ranks, output quad (row k, d4) = tid % 64
  const int q = tid >> 6, slot = tid & 63, k = slot / (D / 4), d4 = (slot % (D / 4)) * 4;
  // the (at most 16) partials of this residue: every rank slot is loaded,
  // before n_ranks is used, so that these loads, the (max, sum) loads below
  // and the caller's share one round trip; slots past n_ranks are not added
  float4 v[16];
  if (k < cnt) {
    const int i = i0 + k * step;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int c = q + 4 * u;
      if (c < r_all)
        v[u] = GLOBAL ? __ldcg(reinterpret_cast<const float4*>(part(c, i) + d4))
                      : *reinterpret_cast<const float4*>(part(c, i) + d4);
    }
  }
  if (warp < cnt) {
    const int kw = warp;
    const int i = i0 + kw * step;
    // every rank slot's (max, sum) is read before n_ranks is used; slots
    // past n_ranks hold stale values and are masked
    const float lm0 = lane < r_all ? ld(part(lane, i) + D) : 0.f;
    const float lm1 = lane + 32 < r_all ? ld(part(lane + 32, i) + D) : 0.f;
    const float ll0 = lane < r_all ? ld(part(lane, i) + D + 1) : 0.f;
    const float ll1 = lane + 32 < r_all ? ld(part(lane + 32, i) + D + 1) : 0.f;
    const float m0 = lane < n_ranks ? lm0 : -INFINITY;
    const float m1 = lane + 32 < n_ranks ? lm1 : -INFINITY;
    float M = fmaxf(m0, m1);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float w0 = m0 == -INFINITY ? 0.f : exp2f(m0 - M);
    const float w1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M);
    float L = w0 * (lane < n_ranks ? ll0 : 0.f);
    L += w1 * (lane + 32 < n_ranks ? ll1 : 0.f);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    WS[kw * 64 + lane] = w0;
    WS[kw * 64 + lane + 32] = w1;
    if (lane == 0) IL[kw] = L > 0.f ? 1.f / L : 0.f;
  }
  grp.sync();
  if (k < cnt) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // add in rank order
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int c = q + 4 * u;
      if (c < n_ranks) {
        const float w = WS[k * 64 + c];
        acc.x += w * v[u].x;
        acc.y += w * v[u].y;
        acc.z += w * v[u].z;
        acc.w += w * v[u].w;
      }
    }
    AC[q * 64 + slot] = acc;
  }
  grp.sync();
  if (q == 0 && k < cnt) {
    const int i = i0 + k * step;
    const int gi = qr0 + i;
    if (gi < nq) {
      const float4 s0 = AC[slot], s1 = AC[64 + slot], s2 = AC[128 + slot], s3 = AC[192 + slot];
      const float il = IL[k];
      const float ox = ((s0.x + s1.x) + s2.x) + s3.x, oy = ((s0.y + s1.y) + s2.y) + s3.y;
      const float oz = ((s0.z + s1.z) + s2.z) + s3.z, ow = ((s0.w + s1.w) + s2.w) + s3.w;
      const int tq = div_small(gi, G, 0xFFFFFFFFu / (unsigned)G + 1u);
      const int t = row0 + tq, hq = kvh * G + (gi - tq * G);
      const size_t o = ((size_t)t * a.Hq + hq) * D + d4;
      put_plane(a.o_hi, a.o_lo, a.out_bf16, o, ox * il);
      put_plane(a.o_hi, a.o_lo, a.out_bf16, o + 1, oy * il);
      put_plane(a.o_hi, a.o_lo, a.out_bf16, o + 2, oz * il);
      put_plane(a.o_hi, a.o_lo, a.out_bf16, o + 3, ow * il);
    }
  }
  grp.sync();
}

}  // namespace attn

}  // namespace gocr
