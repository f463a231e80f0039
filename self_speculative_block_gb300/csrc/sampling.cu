// Sampling decodes: AR sampling and self-speculative rounds with the
// speculative acceptance-rejection rule (GravityOCR review §2 "Speculative
// Decoding"; the Trillion Labs blog's AR-equivalence paragraph: with
// sampling the rejection rule preserves the AR distribution).
//
// Distributions are softmax(logits / T) of the LM head's rows (the forward
// writes its logits when it samples).  Random numbers are Philox4x32-10
// (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3", SC 2011)
// with key (seed low, seed high) and counter (v / 4, position, purpose,
// request), lane v % 4, as uniforms ((x >> 9) + 0.5) 2^-23 (exact in fp32: a
// 25-bit uniform would round near 1, where -log(-log u) is steep).  A draw from a
// distribution is a Gumbel-max: argmax over v of score_v - log(-log u_v)
// with score = l / T (or log of the rejection residual), lowest index among
// equal values.  Purposes: 0 a target token at its position (AR steps, a0,
// the bonus), 1 a draft token, 2 a draft's acceptance uniform (v = 0), 3 the
// replacement after a rejection.  The token at absolute position t uses
// position t, so a0 is the AR sample of its position.
#include "epilogue.cuh"
#include "round.cuh"

namespace gocr {

namespace {

constexpr int SAMPLE_THREADS = 256;

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
  constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u, W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(M0, c.x), lo0 = M0 * c.x;
    const uint32_t hi1 = __umulhi(M1, c.z), lo1 = M1 * c.z;
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    k.x += W0;
    k.y += W1;
  }
  return c;
}

__device__ __forceinline__ float philox_uniform(uint32_t x) {
  return ((float)(x >> 9) + 0.5f) * (1.0f / 8388608.0f);
}

// Four uniforms of vocabulary entries 4 blk .. 4 blk + 3 of one draw.
__device__ __forceinline__ uint4 draw4(unsigned long long seed, int req, int pos, int purpose, int blk) {
  return philox4x32_10(make_uint4((uint32_t)blk, (uint32_t)pos, (uint32_t)purpose, (uint32_t)req),
                       make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
}

__device__ __forceinline__ void best_merge(float& v, int& i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
}

// Block-wide (value, index) maximum, lowest index among equals; every thread gets it.
__device__ __forceinline__ int block_best(float v, int i, float* sv, int* si) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) best_merge(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) { sv[w] = v; si[w] = i; }
  __syncthreads();
  if (threadIdx.x == 0) {
    float bv = sv[0];
    int bi = si[0];
    for (int k = 1; k < nw; ++k) best_merge(bv, bi, sv[k], si[k]);
    sv[0] = bv;
    si[0] = bi;
  }
  __syncthreads();
  const int r = si[0];
  __syncthreads();
  return r;
}

// Gumbel-max draw over a row: score(v) from the functor; -INF scores never win.
template <class Score>
__device__ int gumbel_draw(Score score, int V, unsigned long long seed, int req, int pos, int purpose, float* sv,
                           int* si) {
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int blk = threadIdx.x; blk * 4 < V; blk += blockDim.x) {
    const uint4 x = draw4(seed, req, pos, purpose, blk);
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      const int v = blk * 4 + l;
      if (v >= V) break;
      const float s = score(v);
      if (s == -INFINITY) continue;
      const float g = s - logf(-logf(philox_uniform(xs[l])));
      best_merge(bv, bi, g, v);
    }
  }
  return block_best(bv, bi, sv, si);
}

// (max, sum of exp(z - max)) of z = l / T over a row, one CTA, fixed order:
// thread t folds entries t, t + n, ... in order, then a fixed tree.
__device__ float2 row_stats(const float* l, int V, float invT, float* sm, float* ss) {
  float m = -INFINITY;
  for (int v = threadIdx.x; v < V; v += blockDim.x) m = fmaxf(m, l[v] * invT);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) sm[w] = m;
  __syncthreads();
  float M = sm[0];
  for (int k = 1; k < nw; ++k) M = fmaxf(M, sm[k]);
  float s = 0.f;
  for (int v = threadIdx.x; v < V; v += blockDim.x) s += expf(l[v] * invT - M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) ss[w] = s;
  __syncthreads();
  float S = 0.f;
  for (int k = 0; k < nw; ++k) S += ss[k];
  __syncthreads();
  return make_float2(M, S);
}

}  // namespace

// One CTA per row of a forward whose rows need a draw: AR rows (purpose 0 at
// position p + 1) or draft rows (row 0: purpose 0 at p + 1; row r >= 1:
// purpose 1 at p + 1 + r), with p the request's cache length.
__global__ void __launch_bounds__(SAMPLE_THREADS) sample_rows_kernel(const ReqState* st, const int* slot_req,
                                                                     int rows_per_slot, const float* logits, int V,
                                                                     int* out) {
  __shared__ float sv[SAMPLE_THREADS / 32];
  __shared__ int si[SAMPLE_THREADS / 32];
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t = blockIdx.x, s = t / rows_per_slot, r = t % rows_per_slot;
  const int req = slot_req[s];
  const ReqState& q = st[req];
  const float invT = 1.f / q.temp;
  const float* l = logits + (size_t)t * V;
  const int tok = gumbel_draw([&](int v) { return l[v] * invT; }, V, q.seed, req, q.cache_len + 1 + r,
                              r == 0 ? 0 : 1, sv, si);
  if (threadIdx.x == 0) out[t] = tok;
}

// After the verify forward of a sampling round: one CTA per request.  Draft
// d_j (row j of the draft, position p + 1 + j) is judged by its draft
// probability q_j(d_j) (draft row j) and its target probability p_j(d_j)
// (verify row j - 1), accepted when u_j < min(1, p/q); at the first
// rejection the replacement is drawn from max(0, p_j - q_j) (from p_j when
// that has no mass), after B acceptances the bonus from verify row B.
__global__ void __launch_bounds__(1024) accept_sample_kernel(ReqState* st, const int* slot_req, int n_slots, int B,
                                                             const int* dbuf, const float* ld, const float* lv,
                                                             int V, int* out, int out_stride, const int* err,
                                                             unsigned long long cond, int use_cond) {
  __shared__ float sv[32], sm_[32], ss_[32];
  __shared__ int si[32];
  __shared__ int s_A;
  __shared__ float2 s_stat[2];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int s = blockIdx.x;
  const int req = slot_req[s];
  ReqState& q = st[req];
  const bool live = !q.done;  // uniform over the CTA
  const int* d = dbuf + s * (B + 1);  // d[0] = a0, d[j] = d_j
  const float* LD = ld + (size_t)s * (B + 1) * V;
  const float* LV = lv + (size_t)s * (B + 1) * V;
  const float invT = 1.f / q.temp;
  const int p = q.cache_len;
  int A = 0;
  if (live) {
    // the acceptance walk: row statistics computed by the whole CTA per step
    for (A = 0; A < B; ++A) {
      const int j = A + 1, dj = d[j];
      const float2 qs = row_stats(LD + (size_t)j * V, V, invT, sm_, ss_);
      const float2 ps = row_stats(LV + (size_t)(j - 1) * V, V, invT, sm_, ss_);
      if (threadIdx.x == 0) {
        const float qd = expf(LD[(size_t)j * V + dj] * invT - qs.x) / qs.y;
        const float pd = expf(LV[(size_t)(j - 1) * V + dj] * invT - ps.x) / ps.y;
        const float u = philox_uniform(draw4(q.seed, req, p + 1 + j, 2, 0).x);
        s_A = u < fminf(1.f, pd / qd) ? 1 : 0;
        s_stat[0] = qs;
        s_stat[1] = ps;
      }
      __syncthreads();
      const int ok = s_A;
      __syncthreads();
      if (!ok) break;
    }
  }
  int last = 0;
  if (live) {
    if (A < B) {
      const float2 qs = s_stat[0], ps = s_stat[1];
      const float* lq = LD + (size_t)(A + 1) * V;
      const float* lp = LV + (size_t)A * V;
      // is there residual mass?
      float any = 0.f;
      for (int v = threadIdx.x; v < V; v += blockDim.x)
        any = fmaxf(any, expf(lp[v] * invT - ps.x) / ps.y - expf(lq[v] * invT - qs.x) / qs.y);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) any = fmaxf(any, __shfl_xor_sync(0xffffffffu, any, o));
      if ((threadIdx.x & 31) == 0) sm_[threadIdx.x >> 5] = any;
      __syncthreads();
      float mass = 0.f;
      for (int k = 0; k < (int)(blockDim.x >> 5); ++k) mass = fmaxf(mass, sm_[k]);
      __syncthreads();
      if (mass > 0.f)
        last = gumbel_draw(
            [&](int v) {
              const float w = expf(lp[v] * invT - ps.x) / ps.y - expf(lq[v] * invT - qs.x) / qs.y;
              return w > 0.f ? logf(w) : -INFINITY;
            },
            V, q.seed, req, p + 2 + A, 3, sv, si);
      else
        last = gumbel_draw([&](int v) { return lp[v] * invT; }, V, q.seed, req, p + 2 + A, 3, sv, si);
    } else {
      const float* lb = LV + (size_t)B * V;
      last = gumbel_draw([&](int v) { return lb[v] * invT; }, V, q.seed, req, p + B + 2, 0, sv, si);
    }
    if (threadIdx.x == 0) {
      int commit[66];
      commit[0] = d[0];
      for (int j = 1; j <= A; ++j) commit[j] = d[j];
      commit[A + 1] = last;
      finish_round(q, out + (size_t)req * out_stride, commit, A + 2, A, p + A + 2, last, 2, err);
    }
  }
}

// Sets the device-loop condition after a sampling round: one thread.
__global__ void loop_condition_kernel(ReqState* st, const int* slot_req, int n_slots, unsigned long long cond,
                                      int use_cond) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  set_loop_condition(st, slot_req, n_slots, cond, use_cond);
}

void launch_sample_rows(const ReqState* st, const int* slot_req, int n_slots, int rows_per_slot, const float* logits,
                        int V, int* out, cudaStream_t s, bool pdl) {
  launch_k(sample_rows_kernel, dim3(n_slots * rows_per_slot), dim3(SAMPLE_THREADS), 0, s, pdl, st, slot_req,
           rows_per_slot, logits, V, out);
}

void launch_accept_sample(ReqState* st, const int* slot_req, int n_slots, int B, const int* dbuf, const float* ld,
                          const float* lv, int V, int* out, int out_stride, const int* err, unsigned long long cond,
                          int use_cond, cudaStream_t s, bool pdl) {
  launch_k(accept_sample_kernel, dim3(n_slots), dim3(1024), 0, s, pdl, st, slot_req, n_slots, B, dbuf, ld, lv, V, out,
           out_stride, err, cond, use_cond);
  launch_k(loop_condition_kernel, dim3(1), dim3(1), 0, s, pdl, st, slot_req, n_slots, cond, use_cond);
}

}  // namespace gocr
