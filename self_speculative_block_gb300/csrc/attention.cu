// Grouped-query attention of a window of query rows against a contiguous
// per-request KV cache, with the two mask modes of the round expressed as one
// per-row key limit: row t reads keys 0..lim[t].
//   draft  (GravityOCR review §3.2): boundary row lim = p (causal), [M] rows
//          lim = p + B (the cache plus the whole window, bidirectional);
//   verify / AR / prefill: lim = the row's own position (token-causal).
//
// Keys are swept in fixed 64-key chunks at absolute positions with an online
// softmax in fp32.  A chunk with no key visible to a row leaves that row's
// running (max, sum, output) bit-for-bit unchanged (scale exp(0) = 1 and zero
// contributions), so a row's result does not depend on how many other rows
// share the launch: the AR step and the verify row at the same position give
// identical bits.
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
    if (a.d == 128) launch_attn_t<bf16, 128>(a, n_slots, max_rows, s);
    else launch_attn_t<bf16, 64>(a, n_slots, max_rows, s);
  } else {
    if (a.d == 128) launch_attn_t<float, 128>(a, n_slots, max_rows, s);
    else launch_attn_t<float, 64>(a, n_slots, max_rows, s);
  }
}

}  // namespace gocr
