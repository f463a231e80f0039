// Fused GEMM epilogues, applied by the CTA that completes a (128-row tile,
// token slice) after the fixed-order split-K reduction.  The reduced tile sits
// in shared memory as Ys[tl * ys_ld + c] for token tl < tn and column c < 128.
#pragma once
#include "kernels.cuh"

namespace gocr {

__device__ __forceinline__ void set_err(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// (value, index) maximum with the lowest index among equal values.
__device__ __forceinline__ void argmax_merge(float& v, int& i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Returns true when this CTA must take part in the grid-level argmax finish.
template <typename T>
__device__ void apply_epilogue(const GemmArgs& a, const float* Ys, int ys_ld, int tile, int t0,
                               int tn) {
  const EpiArgs& e = a.e;
  const int n0 = tile * NTILE;
  const int tid = threadIdx.x, nth = blockDim.x;
  switch (a.epi) {
    case EPI_STORE:
      for (int i = tid; i < tn * NTILE; i += nth) {
        int tl = i / NTILE, c = i % NTILE, n = n0 + c;
        if (n < a.N) e.y[(size_t)(t0 + tl) * e.ldy + n] = Ys[tl * ys_ld + c];
      }
      break;
    case EPI_RESID:
      for (int i = tid; i < tn * NTILE; i += nth) {
        int tl = i / NTILE, c = i % NTILE, n = n0 + c;
        if (n < a.N) {
          float* p = e.y + (size_t)(t0 + tl) * e.ldy + n;
          *p = *p + Ys[tl * ys_ld + c];
        }
      }
      break;
    case EPI_SWIGLU: {
      // tile rows [0, 64) are gate rows, [64, 128) the up rows of the same 64 features
      const int f0 = tile * SWIGLU_GROUP;
      for (int i = tid; i < tn * SWIGLU_GROUP; i += nth) {
        int tl = i / SWIGLU_GROUP, j = i % SWIGLU_GROUP;
        float g = Ys[tl * ys_ld + j], u = Ys[tl * ys_ld + SWIGLU_GROUP + j];
        T* h = reinterpret_cast<T*>(e.hbuf);
        h[(size_t)(t0 + tl) * e.ldh + f0 + j] = from_f32<T>(silu_f(g) * u);
      }
      break;
    }
    case EPI_QKV: {
      const int d = e.head_dim, half = d >> 1;
      T* q = reinterpret_cast<T*>(e.qbuf);
      T* kc = reinterpret_cast<T*>(e.kc);
      T* vc = reinterpret_cast<T*>(e.vc);
      for (int i = tid; i < tn * NTILE; i += nth) {
        int tl = i / NTILE, c = i % NTILE, n = n0 + c;
        int t = t0 + tl;
        int pos = e.row_pos[t];
        int j = n % d;  // tiles hold whole heads (128 % d == 0)
        float x = Ys[tl * ys_ld + c];
        float out = x;
        if (n < e.q_dim + e.kv_dim) {  // q and k are rotated, v is not
          int jj = j < half ? j : j - half;
          float2 cs = e.rope[(size_t)pos * half + jj];
          float partner = Ys[tl * ys_ld + (j < half ? c + half : c - half)];
          out = j < half ? (x * cs.x - partner * cs.y) : (x * cs.x + partner * cs.y);
        }
        if (n < e.q_dim) {
          q[(size_t)t * e.q_dim + n] = from_f32<T>(out);
        } else {
          int slot = e.row_slot[t];
          int req = e.plan->slot_req[slot];
          if (pos < 0 || pos >= e.cap) { set_err(e.err, DERR_CAPACITY); continue; }
          bool is_k = n < e.q_dim + e.kv_dim;
          int nn = is_k ? n - e.q_dim : n - e.q_dim - e.kv_dim;
          int kvh = nn / d;
          size_t off = (size_t)req * e.req_stride + ((size_t)kvh * e.cap + pos) * d + j;
          (is_k ? kc : vc)[off] = from_f32<T>(out);
        }
      }
      break;
    }
    case EPI_ARGMAX: {
      const int lane = tid & 31, warp = tid >> 5, nwarp = nth >> 5;
      for (int tl = warp; tl < tn; tl += nwarp) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        bool nan = false;
        for (int c = lane; c < NTILE; c += 32) {
          int n = n0 + c;
          if (n >= a.N) continue;
          float v = Ys[tl * ys_ld + c];
          if (v != v) nan = true;
          if (e.logits) e.logits[(size_t)(t0 + tl) * e.ld_logits + n] = v;
          argmax_merge(bv, bi, v, n);
        }
        for (int o = 16; o > 0; o >>= 1) {
          float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          argmax_merge(bv, bi, ov, oi);
        }
        if (__any_sync(0xffffffffu, nan) && lane == 0) set_err(e.err, DERR_NAN_LOGITS);
        if (lane == 0) {
          e.pmax[(size_t)tile * a.T + t0 + tl] = bv;
          e.pidx[(size_t)tile * a.T + t0 + tl] = bi;
        }
      }
      break;
    }
  }
}

// Grid-level finish of the LM-head argmax: merge every tile's partial maxima.
__device__ __forceinline__ void argmax_finish(const GemmArgs& a) {
  const EpiArgs& e = a.e;
  const int n_tiles = (a.N + NTILE - 1) / NTILE;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  for (int t = warp; t < a.T; t += nwarp) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int tile = lane; tile < n_tiles; tile += 32)
      argmax_merge(bv, bi, __ldcg(e.pmax + (size_t)tile * a.T + t),
                   __ldcg(e.pidx + (size_t)tile * a.T + t));
    for (int o = 16; o > 0; o >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      argmax_merge(bv, bi, ov, oi);
    }
    if (lane == 0) e.am_out[t] = (bi == 0x7fffffff) ? 0 : bi;
  }
}

}  // namespace gocr
