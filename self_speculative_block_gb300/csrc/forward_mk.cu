// Persistent decode forward: one kernel, one CTA per SM, runs every layer of
// a draft, verify or AR forward and the LM head.
//
// A decode forward moves ~1 GB of weights for 1 to 128 token rows, so its
// floor is the time HBM needs to stream the weights once (GravityOCR's round
// reads all weights twice, once per forward).  Launched as ~80 separate
// kernels, each GEMM pays a launch, a pipeline fill and a tail, and HBM idles
// in between.  Here the weights of the whole forward form one stream per CTA
// that never waits on activations:
//
//   warp 0   TMA weight producer: walks the CTA's GEMM work items in forward
//            order and keeps a ring of 128 x 64 weight tiles full, with
//            L2 prefetches running further ahead; it never waits for data.
//   warp 1   TMA activation producer: before the first tile of an item it
//            waits until the phase that writes the item's input is complete
//            (a device counter), then streams the input planes.
//   warp 2   tcgen05 MMA issuer into two TMEM accumulators (double buffer).
//   warps 4-11  compute group: drains accumulators, reduces split-K tiles,
//            runs the fused epilogues and the attention tiles.
//
// Work items: per layer QKV, attention, O, gate/up, down, then the LM head;
// a GEMM item is one (128-row weight tile, K split) as in the per-operation
// kernel, an attention item one (slot, kv head, row group, cluster rank)
// tile.  Items are dealt round robin over the CTAs in forward order.
// Split-K: each item writes its fp32 partial tile to global memory and bumps
// the tile's counter; the item that completes the count adds the partials in
// split order and runs the epilogue, then bumps the phase counter.  Attention
// tiles write their partial rows; once a (slot, kv head, row group) has all
// its CL tiles, each tile's CTA merges the rows it owns.  These are the
// per-operation kernels' reductions in the same order, so the persistent
// forward and the per-operation forward give the same bits.
//
// Counters only grow: a forward with epoch e waits for (e + 1) x items; the
// last CTA to finish advances the epoch.  Every wait is bounded (wall clock);
// a wait that runs out raises a device error and an abort word that ends the
// other CTAs' waits, and each role drains its copies in flight before exit.
#include "attn_core.cuh"
#include "tc.cuh"

#include <cuda.h>

namespace gocr {
namespace mk {

constexpr int THREADS = 384;
constexpr int W_BYTES = NTILE * 64 * 2;     // one 128 x 64 bf16 weight tile
constexpr int EG = 32;                      // tokens per epilogue pass
constexpr int YLD = NTILE + 4;              // fp32 row stride of reduced rows
constexpr int D = 128;                      // head dim of the attention tiles
constexpr unsigned long long WAIT_NS = 200ull * 1000 * 1000;
constexpr int GRP_BAR = 1;                  // named barrier of the compute group

constexpr size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }
constexpr size_t EPI_BYTES = (size_t)EG * YLD * 4 + (size_t)EPI_SCRATCH_FLOATS * 4;
constexpr size_t ATT_BYTES = attn::Geo<D>::TILE_SMEM + (size_t)(2 * 64 + 4) * 4 + 4 * 64 * 16;  // + merge scratch
// fixup inputs fetched with the partial sums: row scales, sums of squares,
// then residual rows (RESID) or RoPE rows (QKV), and the next-norm gains
constexpr size_t PF_FLOATS = EG + EG * EPI_MAX_SSQ + EG * NTILE + NTILE;
constexpr size_t GEMM_BYTES = EPI_BYTES + PF_FLOATS * 4;
constexpr size_t C_BYTES = align16(ATT_BYTES > GEMM_BYTES ? ATT_BYTES : GEMM_BYTES);
constexpr size_t GA_BYTES = align16(sizeof(GemmArgs));
constexpr size_t AA_BYTES = align16(sizeof(AttnArgs));
static_assert(sizeof(GemmArgs) % 16 == 0 && sizeof(AttnArgs) % 16 == 0, "tables are copied by 16-byte loads");

__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Event record of writer w (0: activation producer, 1: compute group) of this CTA.
__device__ __forceinline__ void trace_ev(const MkArgs& a, int w, int& n, int ph, int ev) {
  if (!a.trace || n >= a.trace_cap) return;
  unsigned long long* r = a.trace + (((size_t)blockIdx.x * 2 + w) * a.trace_cap + n) * 2;
  r[0] = gtimer();
  r[1] = ((unsigned long long)ph << 8) | (unsigned)ev;
  ++n;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_relaxed(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// Release by one thread on behalf of a thread group that synchronised just
// before: a GPU-scope fence (cumulative over the writes the group ordered
// before the barrier), then a relaxed add.
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("fence.acq_rel.gpu;\n\tred.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Abort state of a CTA: the shared flag, mirrored by the grid-wide word.
struct Abort {
  volatile int* s;        // shared
  unsigned* word;         // global (ctr[CTR_ABORT])
  int* err;
  __device__ bool raised() const {
    if (*s) return true;
    if (ld_relaxed(word)) { *s = 1; return true; }
    return false;
  }
  __device__ void raise() const {
    *s = 1;
    atomicExch(word, 1u);
    set_err(err, DERR_TIMEOUT);
  }
};

// Bounded mbarrier wait; false when the CTA or the grid aborted or time ran out.
__device__ bool wait_bar(uint64_t* bar, uint32_t parity, const Abort& ab) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = gtimer();
  for (unsigned n = 1;; ++n) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((n & 15) == 0) {
      if (ab.raised()) return false;
      if (gtimer() - t0 > WAIT_NS) { ab.raise(); return false; }
    }
  }
}

// Wait for copies already in flight (they complete whatever the other roles
// do); bounded by time only.
__device__ void wait_bar_drain(uint64_t* bar, uint32_t parity, const Abort& ab) {
  const unsigned long long t0 = gtimer();
  while (!tc::mbar_try_wait(bar, parity))
    if (gtimer() - t0 > WAIT_NS) { ab.raise(); return; }
}

// Bounded wait until a counter reaches `target` (acquire).
__device__ bool wait_ctr(const unsigned* p, unsigned target, const Abort& ab) {
  if ((int)(ld_acquire(p) - target) >= 0) return true;
  const unsigned long long t0 = gtimer();
  for (unsigned n = 1;; ++n) {
    if ((int)(ld_acquire(p) - target) >= 0) return true;
    if ((n & 7) == 0) {
      if (ab.raised()) return false;
      if (gtimer() - t0 > WAIT_NS) { ab.raise(); return false; }
    }
  }
}

// ---------------------------------------------------------------- schedule

__device__ __forceinline__ bool is_att(const MkArgs& a, int ph) { return ph < 5 * a.L && ph % 5 == 1; }
// GEMM kind of a phase: 0 QKV, 1 O, 2 GU, 3 DN, 4 LM
__device__ __forceinline__ int gemm_kind(const MkArgs& a, int ph) {
  if (ph == 5 * a.L) return 4;
  const int k = ph % 5;
  return k == 0 ? 0 : k - 1;
}
__device__ __forceinline__ int n_items(const MkArgs& a, int ph) {
  return ph == 5 * a.L ? a.tiles[4] * a.splits[4] : a.n_items[ph % 5];
}
// increments of phase ph's counter when it is complete: every GEMM item
// publishes once (its token slice of the tile, or the whole one-split tile),
// every attention item once (its merged rows)
__device__ __forceinline__ int n_done(const MkArgs& a, int ph) { return n_items(a, ph); }
__device__ __forceinline__ int first_item(const MkArgs& a, int ph, int cta) {
  const int base = ph == 5 * a.L ? a.L * a.per_layer : (ph / 5) * a.per_layer + a.prefix[ph % 5];
  return ((cta - base) % a.G + a.G) % a.G;
}

struct Item {
  int ph = -1, j = 0;
};
// Advance to this CTA's next GEMM item in forward order; false at the end.
__device__ bool next_gemm(const MkArgs& a, int cta, Item& it) {
  int ph = it.ph, j;
  if (ph < 0) {
    ph = 0;
    j = first_item(a, 0, cta);
  } else {
    j = it.j + a.G;
  }
  for (;;) {
    if (ph > 5 * a.L) return false;
    if (!is_att(a, ph) && j < n_items(a, ph)) {
      it.ph = ph;
      it.j = j;
      return true;
    }
    ++ph;
    if (ph > 5 * a.L) return false;
    j = first_item(a, ph, cta);
  }
}

struct Geo {
  int gk, layer, tile, split, n0, k0, nkb;
};
__device__ __forceinline__ Geo item_geo(const MkArgs& a, const Item& it) {
  Geo g;
  g.gk = gemm_kind(a, it.ph);
  g.layer = it.ph / 5;
  const int S = a.splits[g.gk];
  g.tile = it.j / S;
  g.split = it.j % S;
  g.n0 = g.tile * NTILE;
  g.k0 = g.split * a.kchunk[g.gk];
  const int k1 = min(a.K[g.gk], g.k0 + a.kchunk[g.gk]);
  g.nkb = (k1 - g.k0 + 63) / 64;
  return g;
}
__device__ __forceinline__ const void* wmap(const MkArgs& a, const Geo& g) {
  const int idx = g.gk == 4 ? 4 * a.L : g.layer * 4 + g.gk;
  return reinterpret_cast<const uint8_t*>(a.maps) + (size_t)idx * 128;
}
// activation maps: 0/1 GEMM-input planes (QKV, GU, LM), 2/3 attention output (O), 4/5 SwiGLU output (DN)
__device__ __forceinline__ const void* amap(const MkArgs& a, int gk, int lo) {
  const int base = gk == 1 ? 2 : (gk == 3 ? 4 : 0);
  return reinterpret_cast<const uint8_t*>(a.maps) + (size_t)(4 * a.L + 1 + base + lo) * 128;
}
__device__ __forceinline__ int gemm_args_index(const MkArgs& a, const Geo& g) {
  return g.gk == 4 ? 4 * a.L : g.layer * 4 + g.gk;
}

// ---------------------------------------------------------------- roles

__device__ void weight_producer(const MkArgs& a, uint8_t* sW, uint64_t* w_full, uint64_t* w_empty, const Abort& ab) {
  const int cta = blockIdx.x, WS = a.ws_stages;
  const uint64_t pol = tc::policy_evict_first();
  for (int i = 0; i < 4 * a.L + 1 + 6; ++i)
    tc::prefetch_tmap(reinterpret_cast<const uint8_t*>(a.maps) + (size_t)i * 128);
  Item ld, pf;
  bool ld_ok = next_gemm(a, cta, ld), pf_ok = next_gemm(a, cta, pf);
  Geo lg{}, pg{};
  if (ld_ok) lg = item_geo(a, ld);
  if (pf_ok) pg = item_geo(a, pf);
  int ld_kb = 0, pf_kb = 0;
  long long issued = 0, pf_pos = 0;
  while (ld_ok) {
    // L2 prefetch of the tiles beyond the ring, up to pf_blocks ahead
    while (pf_ok && pf_pos < issued + WS + a.pf_blocks) {
      if (pf_pos >= issued + WS) tc::tma_prefetch_2d(wmap(a, pg), pg.k0 + pf_kb * 64, pg.n0);
      ++pf_pos;
      if (++pf_kb == pg.nkb) {
        pf_kb = 0;
        pf_ok = next_gemm(a, cta, pf);
        if (pf_ok) pg = item_geo(a, pf);
      }
    }
    const int s = (int)(issued % WS);
    const long long u = issued / WS;
    if (u > 0 && !wait_bar(&w_empty[s], (uint32_t)((u - 1) & 1), ab)) break;
    tc::mbar_expect_tx(&w_full[s], W_BYTES);
    tc::tma_load_2d_hint(sW + (size_t)s * W_BYTES, wmap(a, lg), lg.k0 + ld_kb * 64, lg.n0, &w_full[s], pol);
    ++issued;
    if (++ld_kb == lg.nkb) {
      ld_kb = 0;
      ld_ok = next_gemm(a, cta, ld);
      if (ld_ok) lg = item_geo(a, ld);
    }
  }
  for (long long i = issued > WS ? issued - WS : 0; i < issued; ++i)
    wait_bar_drain(&w_full[i % WS], (uint32_t)((i / WS) & 1), ab);
}

__device__ void act_producer(const MkArgs& a, uint8_t* sA, uint64_t* a_full, uint64_t* a_empty, unsigned e1,
                             const Abort& ab) {
  const int cta = blockIdx.x, AS = a.as_stages;
  const int ast = 2 * a.nt * 128;
  const unsigned* ctr = a.ctr;
  Item it;
  int dep_done = -1, ntr = 0;
  long long issued = 0;
  bool ok = true;
  trace_ev(a, 0, ntr, 0, EV_START);
  while (ok && next_gemm(a, cta, it)) {
    const Geo g = item_geo(a, it);
    const int dep = it.ph - 1;  // the phase that writes this item's input
    if (dep >= 0 && dep > dep_done) {
      if (!wait_ctr(ctr + CTR_PHASE + dep, e1 * (unsigned)n_done(a, dep), ab)) break;
      fence_proxy_async_global();  // other CTAs' generic writes -> this thread's TMA reads
      dep_done = dep;
      trace_ev(a, 0, ntr, it.ph, EV_DEP);
    }
    const void* mh = amap(a, g.gk, 0);
    const void* ml = amap(a, g.gk, 1);
    for (int kb = 0; kb < g.nkb; ++kb) {
      const int s = (int)(issued % AS);
      const long long u = issued / AS;
      if (u > 0 && !wait_bar(&a_empty[s], (uint32_t)((u - 1) & 1), ab)) { ok = false; break; }
      uint8_t* dst = sA + (size_t)s * ast;
      tc::mbar_expect_tx(&a_full[s], (uint32_t)ast);
      tc::tma_load_2d(dst, mh, g.k0 + kb * 64, 0, &a_full[s]);
      tc::tma_load_2d(dst + a.nt * 128, ml, g.k0 + kb * 64, 0, &a_full[s]);
      ++issued;
    }
  }
  for (long long i = issued > AS ? issued - AS : 0; i < issued; ++i)
    wait_bar_drain(&a_full[i % AS], (uint32_t)((i / AS) & 1), ab);
}

__device__ void mma_issuer(const MkArgs& a, uint8_t* sW, uint8_t* sA, uint64_t* w_full, uint64_t* w_empty,
                           uint64_t* a_full, uint64_t* a_empty, uint64_t* acc_full, uint64_t* acc_empty,
                           uint64_t* mma_done, uint32_t tmem, const Abort& ab) {
  const int cta = blockIdx.x, WS = a.ws_stages, AS = a.as_stages;
  const int ast = 2 * a.nt * 128;
  const uint32_t idesc = tc::idesc_bf16(NTILE, 2 * a.nt);
  Item it;
  long long wc = 0, ac = 0;
  int gi = 0;
  bool ok = true;
  while (ok && next_gemm(a, cta, it)) {
    const Geo g = item_geo(a, it);
    const int b = gi & 1, u = gi >> 1;
    if (u > 0 && !wait_bar(&acc_empty[b], (uint32_t)((u - 1) & 1), ab)) break;
    tc::fence_after_sync();
    const uint32_t d = tmem + (uint32_t)(b * 256);
    for (int kb = 0; kb < g.nkb; ++kb) {
      const int ws = (int)(wc % WS), as = (int)(ac % AS);
      if (!wait_bar(&w_full[ws], (uint32_t)((wc / WS) & 1), ab) ||
          !wait_bar(&a_full[as], (uint32_t)((ac / AS) & 1), ab)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t wb = tc::smem_u32(sW + (size_t)ws * W_BYTES);
      const uint32_t xb = tc::smem_u32(sA + (size_t)as * ast);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_bf16(d, tc::sdesc_sw128(wb + kk * 32), tc::sdesc_sw128(xb + kk * 32), idesc,
                     (kb > 0 || kk > 0) ? 1u : 0u);
      tc::mma_commit(&w_empty[ws]);
      tc::mma_commit(&a_empty[as]);
      ++wc;
      ++ac;
    }
    if (!ok) break;
    tc::mma_commit(&acc_full[b]);
    ++gi;
  }
  // every MMA this thread issued has completed before TMEM is released
  tc::mma_commit(mma_done);
  wait_bar_drain(mma_done, 0, ab);
}

// ---------------------------------------------------------------- compute group

struct Ctx {
  const MkArgs* a;
  Grp grp;
  uint8_t* sC;
  GemmArgs* sGA;
  AttnArgs* sAA;
  uint64_t* acc_full;
  uint64_t* acc_empty;
  volatile int* s_flag;
  int* s_maxlim;
  Abort ab;
  unsigned e1;
  uint32_t tmem;
  int* ntr;       // trace records written by the group's thread 0
  const int* s_pos;  // [T] row positions of the forward
  const int* s_req;  // [T] row requests
  float* s_rs;       // [T] rstd of every row for the running phase's input (one-split tiles)
  __device__ void ev(int ph, int e) const {
    if (grp.tid == 0) trace_ev(*a, 1, *ntr, ph, e);
  }
};

// Thread 0 of the group waits; the group agrees on the outcome.
__device__ bool grp_wait_ctr(const Ctx& c, const unsigned* p, unsigned target) {
  if (c.grp.tid == 0) *c.s_flag = wait_ctr(p, target, c.ab) ? 1 : 0;
  c.grp.sync();
  const bool ok = *c.s_flag != 0;
  c.grp.sync();
  return ok;
}
__device__ bool grp_wait_bar(const Ctx& c, uint64_t* bar, uint32_t parity) {
  if (c.grp.tid == 0) *c.s_flag = wait_bar(bar, parity, c.ab) ? 1 : 0;
  c.grp.sync();
  const bool ok = *c.s_flag != 0;
  c.grp.sync();
  return ok;
}

// Release this group's writes to their consumers and count one item on *p:
// the group synchronises, then one thread's release makes every write the
// group made before the barrier visible at GPU scope (a release is
// cumulative).  tma: the writes will be read by TMA (the async proxy) too.
__device__ void grp_publish(const Ctx& c, unsigned* p, bool tma) {
  if (tma) fence_proxy_async_global();
  c.grp.sync();
  if (c.grp.tid == 0) red_release_add(p, 1u);
}
// The same, returning the counter value before the increment (group-uniform).
__device__ unsigned grp_publish_ret(const Ctx& c, unsigned* p, bool tma) {
  if (tma) fence_proxy_async_global();
  c.grp.sync();
  if (c.grp.tid == 0) *c.s_flag = (int)atom_add_acq_rel(p, 1u);
  c.grp.sync();
  const unsigned old = (unsigned)*c.s_flag;
  c.grp.sync();
  return old;
}

__device__ void copy_to_shared(void* dst, const void* src, int bytes, const Grp& grp) {
  const int4* s = reinterpret_cast<const int4*>(src);
  int4* d = reinterpret_cast<int4*>(dst);
  for (int i = grp.tid; i < bytes / 16; i += grp.n) d[i] = s[i];
}

// Split-K fixup of tokens [t0, t1) of one tile: the S partials added in split
// order (the per-operation kernel's order), then the epilogue.  The
// epilogue's inputs (sums of squares, residual or RoPE rows, gains) are
// fetched in the same memory round trip as the partials.
template <int EPI>
__device__ void fixup_tile(const Ctx& c, const Geo& g, int t0, int t1) {
  const MkArgs& a = *c.a;
  const EpiArgs& e = c.sGA->e;
  const int T = a.T, N = a.N[g.gk], S = a.splits[g.gk], gs = a.kgroup[g.gk];
  float* Ys = reinterpret_cast<float*>(c.sC);
  float* scratch = Ys + EG * YLD;
  float* pf_rs = scratch + EPI_SCRATCH_FLOATS;  // [EG]
  float* pf_sq = pf_rs + EG;                    // [EG][n_ssq]
  float* pf_rr = pf_sq + EG * EPI_MAX_SSQ;      // [EG][NTILE] residual rows, or
  float2* pf_rope = reinterpret_cast<float2*>(pf_rr);  // [EG][head_dim / 2] RoPE rows
  float* pf_gn = pf_rr + EG * NTILE;            // [NTILE]
  const bool norm = e.ssq_in != nullptr;
  const size_t sstride = (size_t)T * N;
  for (int g0 = t0; g0 < t1; g0 += EG) {
    const int cnt = min(EG, t1 - g0);
    for (int x = c.grp.tid; x < cnt * (NTILE / 4); x += c.grp.n) {
      const int j = x / (NTILE / 4), c4 = (x % (NTILE / 4)) * 4;
      const float* src = a.part + ((size_t)g0 + j) * N + g.n0 + c4;
      // chunk sums added in split order within each reduction group of gs
      // splits, the group sums in group order; the unrolled loads go out together
      float4 acc = __ldcg(reinterpret_cast<const float4*>(src)), gsum = acc;
#pragma unroll 12
      for (int sp = 1; sp < S; ++sp) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(src + sp * sstride));
        if (sp % gs == 0) {
          gsum = v;
        } else {
          gsum.x += v.x;
          gsum.y += v.y;
          gsum.z += v.z;
          gsum.w += v.w;
        }
        if (sp % gs == gs - 1 || sp == S - 1) {
          if (sp < gs) {
            acc = gsum;
          } else {
            acc.x += gsum.x;
            acc.y += gsum.y;
            acc.z += gsum.z;
            acc.w += gsum.w;
          }
        }
      }
      *reinterpret_cast<float4*>(Ys + (size_t)j * YLD + c4) = acc;
    }
    if (norm)
      for (int x = c.grp.tid; x < cnt * e.n_ssq; x += c.grp.n)
        pf_sq[x] = __ldcg(e.ssq_in + (size_t)(g0 + x / e.n_ssq) * e.n_ssq + x % e.n_ssq);
    if (EPI == EPI_RESID) {
      for (int x = c.grp.tid; x < cnt * NTILE; x += c.grp.n)
        pf_rr[x] = __ldcg(e.resid + (size_t)(g0 + x / NTILE) * e.H + g.n0 + x % NTILE);
      for (int x = c.grp.tid; x < NTILE; x += c.grp.n) pf_gn[x] = e.g_next[g.n0 + x];
    }
    const bool rope = EPI == EPI_QKV && e.head_dim <= NTILE && g.n0 < e.q_dim + e.kv_dim;
    if (rope) {
      const int half = e.head_dim / 2;
      for (int x = c.grp.tid; x < cnt * half; x += c.grp.n) {
        const int pc = min(max(c.s_pos[g0 + x / half], 0), e.cap - 1);  // a bad position is flagged by the epilogue
        pf_rope[x] = e.rope[(size_t)pc * half + x % half];
      }
    }
    c.grp.sync();
    if (norm) {
      // rstd = 1 / sqrt(mean(x^2) + eps), partial sums added in column order
      for (int tl = c.grp.tid; tl < cnt; tl += c.grp.n) {
        float ssum = 0.f;
        for (int i = 0; i < e.n_ssq; ++i) ssum += pf_sq[tl * e.n_ssq + i];
        pf_rs[tl] = rsqrtf(ssum / (float)e.norm_H + e.eps);
      }
      c.grp.sync();
    }
    EpiPre pre;
    if (norm) pre.rs = pf_rs;
    if (EPI == EPI_RESID) {
      pre.rr = pf_rr;
      pre.gn = pf_gn;
    }
    if (EPI == EPI_QKV) {
      pre.pos = c.s_pos + g0;
      pre.req = c.s_req + g0;
      if (rope) pre.rope = pf_rope;
    }
    apply_epilogue_k<EPI>(*c.sGA, Ys, YLD, g.tile, g0, cnt, scratch, pre, c.grp);
  }
}

// One-split tile (the LM head): accumulator -> reduced rows -> epilogue, by
// 32-token groups straight from TMEM.
template <int EPI>
__device__ void direct_tile(const Ctx& c, const Geo& g, uint32_t taddr, int half, int row) {
  const MkArgs& a = *c.a;
  const EpiArgs& e = c.sGA->e;
  float* Ys = reinterpret_cast<float*>(c.sC);
  float* scratch = Ys + EG * YLD;
  float* pf_rr = scratch + EPI_SCRATCH_FLOATS + EG + EG * EPI_MAX_SSQ;  // [EG][NTILE] residual rows
  float* pf_gn = pf_rr + EG * NTILE;                                     // [NTILE]
  for (int g0 = 0; g0 < a.T; g0 += EG) {
    const int cnt = min(EG, a.T - g0);
    if (EPI == EPI_RESID) {
      // residual rows written by other CTAs of this kernel: through L2
      for (int x = c.grp.tid; x < cnt * NTILE; x += c.grp.n)
        pf_rr[x] = __ldcg(e.resid + (size_t)(g0 + x / NTILE) * e.H + g.n0 + x % NTILE);
      for (int x = c.grp.tid; x < NTILE; x += c.grp.n) pf_gn[x] = e.g_next[g.n0 + x];
    }
    const int g16 = g0 / 16 + half;
    if (g16 * 16 < a.nt) {  // warp-uniform
      float vh[16], vl[16];
      tc::tmem_ld16(taddr + g16 * 16, vh);
      tc::tmem_ld16(taddr + a.nt + g16 * 16, vl);
#pragma unroll
      for (int j = 0; j < 16; ++j) Ys[(half * 16 + j) * YLD + row] = vh[j] + vl[j];
    }
    c.grp.sync();
    EpiPre pre;
    if (e.ssq_in) pre.rs = c.s_rs + g0;
    if (EPI == EPI_RESID) {
      pre.rr = pf_rr;
      pre.gn = pf_gn;
    }
    if (EPI == EPI_QKV) {
      pre.pos = c.s_pos + g0;
      pre.req = c.s_req + g0;
    }
    apply_epilogue_k<EPI>(*c.sGA, Ys, YLD, g.tile, g0, cnt, scratch, pre, c.grp);
  }
}

template <int EPI>
__device__ void epilogue_kind(const Ctx& c, const Geo& g, bool split, int t0, int t1, uint32_t taddr, int half,
                              int row) {
  if (split) fixup_tile<EPI>(c, g, t0, t1);
  else direct_tile<EPI>(c, g, taddr, half, row);
}

__device__ void run_epilogue(const Ctx& c, const Geo& g, bool split, int t0, int t1, uint32_t taddr, int half,
                             int row) {
  switch (c.sGA->epi) {
    case EPI_QKV: epilogue_kind<EPI_QKV>(c, g, split, t0, t1, taddr, half, row); break;
    case EPI_RESID: epilogue_kind<EPI_RESID>(c, g, split, t0, t1, taddr, half, row); break;
    case EPI_SWIGLU: epilogue_kind<EPI_SWIGLU>(c, g, split, t0, t1, taddr, half, row); break;
    case EPI_ARGMAX: epilogue_kind<EPI_ARGMAX>(c, g, split, t0, t1, taddr, half, row); break;
    default: epilogue_kind<EPI_STORE>(c, g, split, t0, t1, taddr, half, row); break;
  }
}

__device__ void load_gemm_args(const Ctx& c, const Geo& g, int& ga_loaded) {
  const int gidx = gemm_args_index(*c.a, g);
  if (gidx != ga_loaded) {
    c.grp.sync();  // nobody still reads the previous table
    copy_to_shared(c.sGA, c.a->gemm + gidx, (int)GA_BYTES, c.grp);
    c.grp.sync();
    ga_loaded = gidx;
  }
}

// The forward's last LM-head item publishes the argmax of every row.
__device__ void publish_argmax(const Ctx& c, unsigned old, int ph) {
  if (old != c.e1 * (unsigned)n_done(*c.a, ph) - 1) return;
  __threadfence();
  const EpiArgs& e = c.sGA->e;
  for (int t = c.grp.tid; t < c.a->T; t += c.grp.n) {
    const unsigned long long k = atomicExch(e.amax + t, 0ull);
    e.am_out[t] = k ? (int)(0xFFFFFFFFu - (unsigned)(k & 0xFFFFFFFFull)) : 0;
  }
}

__device__ void publish_item(const Ctx& c, const Item& it) {
  unsigned* p = c.a->ctr + CTR_PHASE + it.ph;
  if (c.sGA->epi == EPI_ARGMAX) publish_argmax(c, grp_publish_ret(c, p, true), it.ph);
  else grp_publish(c, p, true);
  c.ev(it.ph, EV_FIXED);
}

// First pass over a GEMM item (the CTA's gi-th): drain the accumulator.  A
// split item writes its partial tile and counts it on the tile counter; a
// one-split item runs its epilogue straight from TMEM and is complete.
// False on abort.
__device__ bool gemm_drain(const Ctx& c, const Item& it, int gi, int& ga_loaded) {
  const MkArgs& a = *c.a;
  const Geo g = item_geo(a, it);
  const int S = a.splits[g.gk];
  load_gemm_args(c, g, ga_loaded);
  const int b = gi & 1;
  if (!grp_wait_bar(c, &c.acc_full[b], (uint32_t)((gi >> 1) & 1))) return false;
  tc::fence_after_sync();
  c.ev(it.ph, EV_ACC);
  const int warp = (int)(threadIdx.x >> 5), lane = (int)(threadIdx.x & 31);
  const int q = warp & 3;                 // TMEM lane quarter this warp may read
  const int half = (c.grp.tid >> 5) >> 2; // token half of the drain
  const int row = q * 32 + lane;          // weight row = output column of the tile
  const uint32_t taddr = c.tmem + (uint32_t)(b * 256) + ((uint32_t)(q * 32) << 16);
  if (S > 1) {
    // partial tile -> global [split][token][column]
    const int N = a.N[g.gk];
    for (int g16 = half; g16 < a.nt / 16; g16 += 2) {
      float vh[16], vl[16];
      tc::tmem_ld16(taddr + g16 * 16, vh);
      tc::tmem_ld16(taddr + a.nt + g16 * 16, vl);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = g16 * 16 + j;
        if (t < a.T) __stcg(a.part + ((size_t)g.split * a.T + t) * N + g.n0 + row, vh[j] + vl[j]);
      }
    }
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&c.acc_empty[b]);
    grp_publish(c, a.ctr + tile_ctr_base(a.L) + (size_t)it.ph * MAXT + g.tile, false);
    c.ev(it.ph, EV_DRAINED);
    return true;
  }
  run_epilogue(c, g, false, 0, 0, taddr, half, row);
  tc::fence_before_sync();
  __syncwarp();
  if (lane == 0) tc::mbar_arrive(&c.acc_empty[b]);
  publish_item(c, it);
  return true;
}

// Second pass over a split item: once all S partial tiles are written, reduce
// this split's token slice (the per-operation kernel's cluster-rank slice)
// and run its epilogue.  False on abort.
__device__ bool gemm_fixup(const Ctx& c, const Item& it, int& ga_loaded) {
  const MkArgs& a = *c.a;
  const Geo g = item_geo(a, it);
  const int S = a.splits[g.gk];
  load_gemm_args(c, g, ga_loaded);
  if (!grp_wait_ctr(c, a.ctr + tile_ctr_base(a.L) + (size_t)it.ph * MAXT + g.tile, c.e1 * (unsigned)S))
    return false;
  // (the phase's inputs were acquired in compute_group before its drains)
  const int per = (a.T + S - 1) / S;
  const int t0 = min(a.T, g.split * per), t1 = min(a.T, t0 + per);
  if (t1 > t0) run_epilogue(c, g, true, t0, t1, 0, 0, 0);
  publish_item(c, it);
  return true;
}

// The attention items of one layer: first every tile's partial rows (which
// wait only for the QKV phase), then every rank's row merges (which wait for
// the R ranks of its group).  Rank r merges rows r, r + R, ...  False on abort.
__device__ bool attention_phase(const Ctx& c, int ph) {
  const MkArgs& a = *c.a;
  using Gm = attn::Geo<D>;
  constexpr int RLD = Gm::RLD, QR = attn::QR;
  const int R = a.ranks;
  const int l = ph / 5;
  const int n = a.n_items[1];
  const int j0 = first_item(a, ph, blockIdx.x);
  if (j0 >= n) return true;
  copy_to_shared(c.sAA, a.att + l, (int)AA_BYTES, c.grp);
  c.grp.sync();
  const AttnArgs& at = *c.sAA;
  const int per_slot = a.Hkv * a.n_rg;
  const int G = at.Hq / at.Hkv;
  unsigned* tctr = a.ctr + tile_ctr_base(a.L) + (size_t)ph * MAXT;
  float* WSm = reinterpret_cast<float*>(c.sC + Gm::TILE_SMEM);  // [2][64]
  float* ILm = WSm + 2 * 64;                                      // [2] (+ pad)
  float4* ACm = reinterpret_cast<float4*>(ILm + 4);               // [4][64]
  const unsigned qkv_target = c.e1 * (unsigned)n_done(a, ph - 1);
  bool qkv_ready = false;
  for (int j = j0; j < n; j += a.G) {
    const int rank = j % R, grp_id = j / R;
    const int y = grp_id % per_slot, slot = grp_id / per_slot;
    const int kvh = y % a.Hkv, rg = y / a.Hkv;
    const int req = at.slot_req[slot];
    const attn::KvPlanes kv = attn::kv_planes(at, req, kvh, D);
    const bool pre = attn::tile_prefetch<D>(c.sC, kv, rank, R, at.st[req].cache_len, c.grp.tid);
    if (!qkv_ready) {
      if (!grp_wait_ctr(c, a.ctr + CTR_PHASE + ph - 1, qkv_target)) {
        attn::cp_async_wait<0>();
        return false;
      }
      qkv_ready = true;
      c.ev(ph, EV_ATT_READY);
    }
    const int row0 = slot * a.rows_per_slot, nrows = a.rows_per_slot, qr0 = rg * QR;
    const bool rows = qr0 < nrows * G;
    const int n_chunks =
        rows ? attn::tile_partial<D>(at, c.sC, c.grp, kv, rank, R, kvh, qr0, row0, nrows, pre, c.s_maxlim) : 0;
    if (rows && rank < n_chunks) {
      const float4* src = reinterpret_cast<const float4*>(attn::staged_rows<D>(c.sC));
      float4* dst = reinterpret_cast<float4*>(at.part + ((size_t)grp_id * R + rank) * QR * RLD);
      for (int x = c.grp.tid; x < QR * RLD / 4; x += c.grp.n) __stcg(dst + x, src[x]);
    } else {
      attn::cp_async_wait<0>();
    }
    grp_publish(c, tctr + grp_id, false);
    c.ev(ph, EV_ATT_PART);
  }
  for (int j = j0; j < n; j += a.G) {
    const int rank = j % R, grp_id = j / R;
    const int y = grp_id % per_slot, slot = grp_id / per_slot;
    const int kvh = y % a.Hkv, rg = y / a.Hkv;
    if (!grp_wait_ctr(c, tctr + grp_id, c.e1 * (unsigned)R)) return false;
    const int row0 = slot * a.rows_per_slot, nrows = a.rows_per_slot, qr0 = rg * QR;
    if (qr0 < nrows * G && rank < QR) {
      const int n_chunks = attn::tile_chunks(at, c.grp, qr0, row0, nrows, c.s_maxlim);
      const int n_ranks = n_chunks < R ? n_chunks : R;
      const float* base = at.part + (size_t)grp_id * R * QR * RLD;
      auto part = [&](int src, int i) -> const float* { return base + ((size_t)src * QR + i) * RLD; };
      const int cnt = (QR - rank + R - 1) / R;  // rows rank, rank + R, ... of the 64
      for (int k0 = 0; k0 < cnt; k0 += 2)
        attn::merge_rows<D, true>(at, c.grp, part, WSm, ILm, ACm, n_ranks, R, rank + k0 * R, R,
                                  cnt - k0 < 2 ? cnt - k0 : 2, kvh, qr0, row0, nrows);
    }
    grp_publish(c, a.ctr + CTR_PHASE + ph, true);
    c.ev(ph, EV_ATT_MERGED);
  }
  return true;
}

// Phase by phase: attention items, or every GEMM item's drain and then every
// split item's fixup.  Drains wait only for the previous phase, so no CTA
// waits on a tile whose partials sit behind its own pending fixup.
__device__ void compute_group(const Ctx& c) {
  const MkArgs& a = *c.a;
  int gi = 0, ga_loaded = -1;
  for (int ph = 0; ph <= 5 * a.L; ++ph) {
    if (is_att(a, ph)) {
      if (!attention_phase(c, ph)) return;
      continue;
    }
    const int n = n_items(a, ph);
    const int j0 = first_item(a, ph, blockIdx.x);
    if (j0 >= n) continue;
    // the epilogues read what the previous phase wrote (sums of squares,
    // residual rows): acquire its counter (complete by the time the first
    // accumulator of this phase is ready)
    if (ph > 0 && !grp_wait_ctr(c, a.ctr + CTR_PHASE + ph - 1, c.e1 * (unsigned)n_done(a, ph - 1))) return;
    const int S = a.splits[gemm_kind(a, ph)];
    if (S == 1) {
      // one-split tiles run their epilogue from TMEM: row scales of every row now
      Geo g0 = item_geo(a, Item{ph, j0});
      load_gemm_args(c, g0, ga_loaded);
      const EpiArgs& e = c.sGA->e;
      if (e.ssq_in)
        for (int t = c.grp.tid; t < a.T; t += c.grp.n) {
          // row_rstd's sum in column order, through L2 (other CTAs wrote the sums)
          const float* p = e.ssq_in + (size_t)(e.in_rows ? e.in_rows[t] : t) * e.n_ssq;
          float ssum = 0.f;
          for (int i = 0; i < e.n_ssq; ++i) ssum += __ldcg(p + i);
          c.s_rs[t] = rsqrtf(ssum / (float)e.norm_H + e.eps);
        }
      c.grp.sync();
    }
    Item it;
    it.ph = ph;
    for (int j = j0; j < n; j += a.G) {
      it.j = j;
      if (!gemm_drain(c, it, gi, ga_loaded)) return;
      ++gi;
    }
    if (S > 1)
      for (int j = j0; j < n; j += a.G) {
        it.j = j;
        if (!gemm_fixup(c, it, ga_loaded)) return;
      }
  }
}

// ---------------------------------------------------------------- kernel

__global__ void __launch_bounds__(THREADS, 1) forward_mk_kernel(const MkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int WS = a.ws_stages, AS = a.as_stages;
  const int ast = 2 * a.nt * 128;
  uint8_t* sW = smem;
  uint8_t* sA = sW + (size_t)WS * W_BYTES;
  uint8_t* sC = sA + (size_t)AS * ast;
  GemmArgs* sGA = reinterpret_cast<GemmArgs*>(sC + C_BYTES);
  AttnArgs* sAA = reinterpret_cast<AttnArgs*>(reinterpret_cast<uint8_t*>(sGA) + GA_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sAA) + AA_BYTES);
  uint64_t* w_full = bars;
  uint64_t* w_empty = w_full + WS;
  uint64_t* a_full = w_empty + WS;
  uint64_t* a_empty = a_full + AS;
  uint64_t* acc_full = a_empty + AS;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_empty + 2;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_flag;
  __shared__ int s_maxlim;
  __shared__ int s_pos[128], s_req[128];
  __shared__ float s_rs[128];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < WS; ++s) {
      tc::mbar_init(&w_full[s], 1);
      tc::mbar_init(&w_empty[s], 1);
    }
    for (int s = 0; s < AS; ++s) {
      tc::mbar_init(&a_full[s], 1);
      tc::mbar_init(&a_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], 8);  // one arrival per compute warp
    }
    tc::mbar_init(mma_done, 1);
    tc::fence_mbar_init();
    s_abort = 0;
    tc::grid_dep_launch();
  }
  if (warp == 2) tc::tmem_alloc(&s_tmem, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const Abort ab{&s_abort, a.ctr + CTR_ABORT, a.err};

  unsigned e1 = 0;
  if (warp == 0) {
    // weights do not depend on earlier kernels: no dependency wait
    if (lane == 0) weight_producer(a, sW, w_full, w_empty, ab);
  } else if (warp == 1) {
    if (lane == 0) {
      tc::grid_dep_wait();
      e1 = ld_acquire(a.ctr + CTR_EPOCH) + 1;
      act_producer(a, sA, a_full, a_empty, e1, ab);
    }
  } else if (warp == 2) {
    if (lane == 0) mma_issuer(a, sW, sA, w_full, w_empty, a_full, a_empty, acc_full, acc_empty, mma_done, s_tmem, ab);
  } else if (warp >= 4) {
    tc::grid_dep_wait();
    e1 = ld_acquire(a.ctr + CTR_EPOCH) + 1;
    Ctx c;
    c.a = &a;
    c.grp = Grp{tid - 128, THREADS - 128, GRP_BAR};
    c.sC = sC;
    c.sGA = sGA;
    c.sAA = sAA;
    c.acc_full = acc_full;
    c.acc_empty = acc_empty;
    c.s_flag = &s_flag;
    c.s_maxlim = &s_maxlim;
    c.ab = ab;
    c.e1 = e1;
    c.tmem = s_tmem;
    int ntr = 0;
    c.ntr = &ntr;
    // the forward's row table (positions, requests), constant for the kernel
    {
      const EpiArgs& e0 = a.gemm[0].e;
      for (int t = c.grp.tid; t < a.T; t += c.grp.n) {
        s_pos[t] = e0.row_pos[t];
        s_req[t] = e0.plan->slot_req[e0.row_slot[t]];
      }
      c.grp.sync();
    }
    c.s_pos = s_pos;
    c.s_req = s_req;
    c.s_rs = s_rs;
    c.ev(0, EV_START);
    compute_group(c);
    c.ev(5 * a.L, EV_END);
    attn::cp_async_wait<0>();
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc::fence_after_sync();
    tc::tmem_dealloc(s_tmem, 512);
  }
  if (tid == 128) {
    // the last CTA of the forward advances the epoch
    __threadfence();
    const unsigned old = atom_add_acq_rel(a.ctr + CTR_DONE, 1u);
    if (old == e1 * (unsigned)a.G - 1) atom_add_acq_rel(a.ctr + CTR_EPOCH, 1u);
  }
}

}  // namespace mk

size_t forward_mk_smem(int nt, int ws_stages, int as_stages) {
  return 1024 + (size_t)ws_stages * mk::W_BYTES + (size_t)as_stages * 2 * nt * 128 + mk::C_BYTES + mk::GA_BYTES +
         mk::AA_BYTES + (size_t)(2 * ws_stages + 2 * as_stages + 5) * 8;
}

static bool mk_configure(size_t smem) {
  static size_t configured = 0;
  if (smem <= configured) return true;
  if (cudaFuncSetAttribute(mk::forward_mk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return false;
  prefer_shared(reinterpret_cast<const void*>(mk::forward_mk_kernel));
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, mk::forward_mk_kernel, mk::THREADS, smem) != cudaSuccess ||
      n < 1)
    return false;
  configured = smem;
  return true;
}

bool forward_mk_fits(int head_dim) { return head_dim == mk::D; }

bool launch_forward_mk(const MkArgs& a, int head_dim, cudaStream_t s, bool pdl) {
  if (!forward_mk_fits(head_dim) || a.ranks < 1 || a.ranks > 64) return false;
  const size_t smem = forward_mk_smem(a.nt, a.ws_stages, a.as_stages);
  if (smem > 227 * 1024) return false;
  if (!mk_configure(smem)) return false;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.G);
  cfg.blockDim = dim3(mk::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, mk::forward_mk_kernel, a) == cudaSuccess;
}

}  // namespace gocr
