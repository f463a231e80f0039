// Fused GEMM epilogues, applied by the CTA that owns a finished
// (128-column tile, token range) after the fixed-order split-K reduction.
// The reduced tile sits in shared memory as Ys[tl * ys_ld + c] (token tl < tn,
// column c < 128).  Each warp takes whole tokens; lane l handles columns
// l, l + 32, l + 64, l + 96, so per-token reductions are warp shuffles in a
// fixed order and every token's result is independent of the others.
#pragma once
#include "kernels.cuh"

namespace gocr {

__device__ __forceinline__ void set_err(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// The threads that run an epilogue: the whole CTA (barrier 0), or a set of
// whole warps that synchronise on a named barrier of their own while the
// CTA's other warps keep producing.
struct Grp {
  int tid;   // thread index within the group
  int n;     // threads in the group (a multiple of 32)
  int bar;   // 0: __syncthreads; else the named barrier id
  __device__ static Grp block() { return Grp{(int)threadIdx.x, (int)blockDim.x, 0}; }
  __device__ __forceinline__ void sync() const {
    if (bar == 0) __syncthreads();
    else asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(n) : "memory");
  }
};

// (value, index) maximum with the lowest index among equal values.
__device__ __forceinline__ void argmax_merge(float& v, int& i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
}

// Order-preserving 64-bit key: larger value wins, then the smaller index.
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  if (v == 0.f) v = 0.f;  // one zero
  unsigned u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)idx);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// GEMM-input plane element: bf16 hi + lo, or fp32.
__device__ __forceinline__ void put_plane(void* hi, void* lo, int bf, size_t idx, float v) {
  if (bf) {
    bf16 h = __float2bfloat16_rn(v);
    reinterpret_cast<bf16*>(hi)[idx] = h;
    reinterpret_cast<bf16*>(lo)[idx] = __float2bfloat16_rn(v - __bfloat162float(h));
  } else {
    reinterpret_cast<float*>(hi)[idx] = v;
  }
}

// rstd of one row from its per-128-column sums of squares, added in column order.
__device__ __forceinline__ float row_rstd(const EpiArgs& e, int row) {
  const float* p = e.ssq_in + (size_t)row * e.n_ssq;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = i < e.n_ssq ? p[i] : 0.f;
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (i < e.n_ssq) s += v[i];
  return rsqrtf(s / (float)e.norm_H + e.eps);
}

// Shared scratch of one epilogue call, in floats.
constexpr int EPI_GROUP = 32;                 // tokens per epilogue pass
constexpr int EPI_MAX_SSQ = 32;               // hidden <= 4096
constexpr int EPI_SCRATCH_FLOATS = EPI_GROUP + EPI_GROUP * EPI_MAX_SSQ + EPI_GROUP * NTILE;

// Epilogue inputs a GEMM kernel fetched ahead of time into shared memory,
// for the tokens t0 .. t0+tn-1 of one epilogue call (tn <= EPI_GROUP); a null
// pointer means "read it from global memory now".
struct EpiPre {
  const float* rs = nullptr;     // [tn] row scales
  const float* rr = nullptr;     // [tn][NTILE] residual rows of this tile (RESID)
  const float* gn = nullptr;     // [NTILE] next-norm gain of this tile's columns (RESID)
  const int* pos = nullptr;      // [tn] row positions (QKV)
  const int* req = nullptr;      // [tn] request of each row (QKV)
  const float2* rope = nullptr;  // [tn][head_dim / 2] (cos, sin) at each row's position (QKV)
};

// Epilogue EPI of tokens t0 .. t0+tn-1.  Every pass first issues all of its
// global loads (sums of squares, residual rows) into shared memory, so a pass
// costs one memory round trip rather than one per token; inputs in `pre`
// (tn <= EPI_GROUP) are not fetched again.  The loads here are plain (L1
// cached): a kernel that runs an epilogue on data other CTAs of the same
// kernel wrote must pass those inputs in `pre`.  The kind is a template argument
// so that a kernel carries only its own epilogue code.
template <int EPI>
__device__ inline void apply_epilogue_k(const GemmArgs& a, const float* Ys, int ys_ld, int tile, int t0, int tn,
                                        float* scratch, const EpiPre& pre, const Grp& grp) {
  const EpiArgs& e = a.e;
  const int n0 = tile * NTILE;
  const int tid = grp.tid, lane = tid & 31, warp = tid >> 5, nwarp = grp.n >> 5;
  float* rs_s = scratch;                                 // [EPI_GROUP] row scales
  float* sq = rs_s + EPI_GROUP;                          // [EPI_GROUP][n_ssq]
  float* rr_s = sq + EPI_GROUP * EPI_MAX_SSQ;            // [EPI_GROUP][NTILE] residual rows
  const float* rs_in = pre.rs;
  const float* rr_in = pre.rr;
  for (int g0 = 0; g0 < tn; g0 += EPI_GROUP) {
    const int gn = min(EPI_GROUP, tn - g0);
    const bool norm = e.ssq_in != nullptr;
    const bool resid = EPI == EPI_RESID;
    const bool load_rs = norm && !rs_in;
    const bool load_rr = resid && !rr_in;
    if (load_rs)
      for (int x = tid; x < gn * e.n_ssq; x += grp.n) {
        const int tl = x / e.n_ssq, i = x % e.n_ssq;
        const int row = e.in_rows ? e.in_rows[t0 + g0 + tl] : t0 + g0 + tl;
        sq[tl * e.n_ssq + i] = e.ssq_in[(size_t)row * e.n_ssq + i];
      }
    if (load_rr)
      for (int x = tid; x < gn * NTILE; x += grp.n) {
        const int tl = x / NTILE, c = x % NTILE;
        rr_s[x] = e.resid[(size_t)(t0 + g0 + tl) * e.H + n0 + c];
      }
    if (load_rs || load_rr) grp.sync();
    if (load_rs) {
      // rstd = 1 / sqrt(mean(x^2) + eps), partial sums added in column order
      for (int tl = tid; tl < gn; tl += grp.n) {
        float ssum = 0.f;
        for (int i = 0; i < e.n_ssq; ++i) ssum += sq[tl * e.n_ssq + i];
        rs_s[tl] = rsqrtf(ssum / (float)e.norm_H + e.eps);
      }
      grp.sync();
    }
    const bool first = g0 == 0;
    const float* rs = rs_in ? rs_in + g0 : rs_s;
    const float* rr = rr_in ? rr_in + (size_t)g0 * NTILE : rr_s;
    if (EPI == EPI_ARGMAX && !e.logits && !e.conf_part && grp.n >= 4 * EPI_GROUP) {
      // argmax alone: four threads per token scan the tile's columns q, q + 4,
      // ... in increasing order (a strict > keeps the lowest index among
      // equal maxima) and merge with the same rule: the tokens run side by
      // side instead of one warp reduction per token
      const int tl = tid >> 2, q = tid & 3;
      const bool act = tl < gn;
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      int nan = 0;
      if (act) {
        const float r = norm ? rs[tl] : 1.f;
        const float* yrow = Ys + (size_t)(g0 + tl) * ys_ld;
#pragma unroll 8
        for (int k = 0; k < NTILE / 4; ++k) {
          const int c = q + 4 * k, n = n0 + c;
          const float v = yrow[c] * r;
          if (n < a.N) {
            nan |= v != v;
            argmax_merge(bv, bi, v, n);
          }
        }
      }
      // every lane of the warp takes part; inactive lanes hold (-inf, none)
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        nan |= __shfl_xor_sync(0xffffffffu, nan, o);
        argmax_merge(bv, bi, ov, oi);
      }
      if (act && q == 0) {
        if (nan) set_err(e.err, DERR_NAN_LOGITS);
        if (bi != 0x7fffffff) atomicMax(e.amax + t0 + g0 + tl, argmax_key(bv, bi));
      }
      grp.sync();
      continue;
    }
    for (int tl = warp; tl < gn; tl += nwarp) {
      const int t = t0 + g0 + tl;
      const float r = norm ? rs[tl] : 1.f;
      const float* yrow = Ys + (size_t)(g0 + tl) * ys_ld;
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = yrow[lane + 32 * j] * r;
      switch (EPI) {
        case EPI_STORE:
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int n = n0 + lane + 32 * j;
            if (n < a.N) e.y[(size_t)t * e.ldy + n] = v[j];
          }
          break;
        case EPI_RESID: {
          float ss = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c = lane + 32 * j, n = n0 + c;
            const float x = rr[tl * NTILE + c] + v[j];
            e.resid[(size_t)t * e.H + n] = x;
            ss = fmaf(x, x, ss);
            put_plane(e.pl_hi, e.pl_lo, e.plane_bf16, (size_t)t * e.ld_pl + n, x * (pre.gn ? pre.gn[c] : e.g_next[n]));
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
          if (lane == 0) e.ssq_out[(size_t)t * (e.H / NTILE) + tile] = ss;
          break;
        }
        case EPI_SWIGLU: {
          // tile columns [0, 64) are gate rows, [64, 128) the up rows of the same 64 features
          const int f0 = tile * SWIGLU_GROUP;
#pragma unroll
          for (int j = 0; j < 2; ++j)
            put_plane(e.pl_hi, e.pl_lo, e.plane_bf16, (size_t)t * e.ld_pl + f0 + lane + 32 * j,
                      silu_f(v[j]) * v[j + 2]);
          break;
        }
        case EPI_QKV: {
          // head_dim is 64 or 128: index arithmetic by shifts and masks
          const int d = e.head_dim, half = d >> 1, dsh = d == 128 ? 7 : 6, dm = d - 1;
          const bool pq = first && pre.pos;
          const int pos = pq ? pre.pos[tl] : e.row_pos[t];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c = lane + 32 * j, n = n0 + c, jj = n & dm;
            float out = v[j];
            if (n < e.q_dim + e.kv_dim) {  // q and k are rotated, v is not
              const int ri = jj < half ? jj : jj - half;
              const float2 cs = (first && pre.rope) ? pre.rope[tl * half + ri] : e.rope[(size_t)pos * half + ri];
              const float partner = yrow[jj < half ? c + half : c - half] * r;
              out = jj < half ? (v[j] * cs.x - partner * cs.y) : (v[j] * cs.x + partner * cs.y);
            }
            if (n < e.q_dim) {
              put_plane(e.q_hi, e.q_lo, e.plane_bf16, (size_t)t * e.q_dim + n, out);
            } else {
              const int req = (first && pre.req) ? pre.req[tl] : e.plan->slot_req[e.row_slot[t]];
              if (pos < 0 || pos >= e.cap) { set_err(e.err, DERR_CAPACITY); continue; }
              const bool is_k = n < e.q_dim + e.kv_dim;
              const int nn = is_k ? n - e.q_dim : n - e.q_dim - e.kv_dim;
              const size_t off = (size_t)req * e.req_stride + (((size_t)(nn >> dsh) * e.cap + pos) << dsh) + (nn & dm);
              if (is_k) put_plane(e.k_hi, e.k_lo, e.plane_bf16, off, out);
              else put_plane(e.v_hi, e.v_lo, e.plane_bf16, off, out);
            }
          }
          break;
        }
        case EPI_ARGMAX: {
          float bv = -INFINITY;
          int bi = 0x7fffffff;
          bool nan = false;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int n = n0 + lane + 32 * j;
            if (n >= a.N) continue;
            if (v[j] != v[j]) nan = true;
            if (e.logits) e.logits[(size_t)t * e.ld_logits + n] = v[j];
            argmax_merge(bv, bi, v[j], n);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            argmax_merge(bv, bi, ov, oi);
          }
          if (__any_sync(0xffffffffu, nan) && lane == 0) set_err(e.err, DERR_NAN_LOGITS);
          if (lane == 0 && bi != 0x7fffffff) atomicMax(e.amax + t, argmax_key(bv, bi));
          if (e.conf_part) {
            // every lane holds the tile maximum bv; lane 0's sum takes one fixed order
            float se = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (n0 + lane + 32 * j < a.N) se += expf(v[j] - bv);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) se += __shfl_xor_sync(0xffffffffu, se, o);
            if (lane == 0) e.conf_part[(size_t)t * (a.N / NTILE) + tile] = make_float2(bv, se);
          }
          break;
        }
      }
    }
    grp.sync();
  }
}

// Epilogue with the kind taken from the launch arguments.
__device__ inline void apply_epilogue(const GemmArgs& a, const float* Ys, int ys_ld, int tile, int t0, int tn,
                                      float* scratch) {
  switch (a.epi) {
    case EPI_STORE: apply_epilogue_k<EPI_STORE>(a, Ys, ys_ld, tile, t0, tn, scratch, EpiPre(), Grp::block()); break;
    case EPI_RESID: apply_epilogue_k<EPI_RESID>(a, Ys, ys_ld, tile, t0, tn, scratch, EpiPre(), Grp::block()); break;
    case EPI_QKV: apply_epilogue_k<EPI_QKV>(a, Ys, ys_ld, tile, t0, tn, scratch, EpiPre(), Grp::block()); break;
    case EPI_SWIGLU: apply_epilogue_k<EPI_SWIGLU>(a, Ys, ys_ld, tile, t0, tn, scratch, EpiPre(), Grp::block()); break;
    case EPI_ARGMAX: apply_epilogue_k<EPI_ARGMAX>(a, Ys, ys_ld, tile, t0, tn, scratch, EpiPre(), Grp::block()); break;
  }
}

// Grid-level end of the LM-head argmax: the last CTA to arrive publishes the
// indices and clears the keys and the counter for the next launch.
__device__ __forceinline__ void argmax_grid_finish(const GemmArgs& a, int* s_flag) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int total = (int)(gridDim.x * gridDim.y * gridDim.z);
    const int prev = atomicAdd(a.e.grid_ctr, 1);
    *s_flag = (prev == total - 1);
  }
  __syncthreads();
  if (!*s_flag) return;
  __threadfence();
  for (int t = threadIdx.x; t < a.T; t += blockDim.x) {
    const unsigned long long k = atomicExch(a.e.amax + t, 0ull);
    a.e.am_out[t] = k ? (int)(0xFFFFFFFFu - (unsigned)(k & 0xFFFFFFFFull)) : 0;
  }
  if (threadIdx.x == 0) *a.e.grid_ctr = 0;
}

}  // namespace gocr
