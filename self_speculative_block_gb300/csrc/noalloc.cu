// Allocation-free variant of the single-GEMM entry point.
//
// Some callers cannot allocate device memory: a plug-in running inside a host
// application that owns every allocation (a fixed-size memory pool, a
// real-time loop that must never call the driver allocator, a sandbox that
// forbids cudaMalloc).  gocr_op_linear_static gives them the decoder's
// split-K GEMM without a caller-provided workspace: its split-K partial sums
// and tile counters live in one file-scope device array of fixed size that
// every GPU loading this library holds until the process exits.
#include "../../include/gocr.h"
#include "kernels.cuh"

#include <cstdio>
#include <mutex>

using namespace gocr;

namespace {

// GOCR_STATIC_SCRATCH_BYTES of scratch per device: tile counters, then fp32 partial sums.
constexpr size_t STATIC_SCRATCH_BYTES = GOCR_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_static_scratch[STATIC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
void* g_scratch_ptr[MAX_DEVICES] = {};  // device address of g_static_scratch, per device
int set_error(int code, const char* msg) {
  set_lib_error(msg);
  return code;
}

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.  With lazy module
// loading (the CUDA default) this first lookup is also where the driver loads
// the module and reserves the array on that device, so it can fail there for
// lack of device memory (GOCR_ECUDA).
int scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
    return set_error(GOCR_ECUDA, "no current CUDA device");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p) {
      char m[160];
      snprintf(m, sizeof m, "cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
      return set_error(GOCR_ECUDA, m);
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return GOCR_OK;
}

}  // namespace

extern "C" {

int gocr_op_linear_static(int dtype, const void* x, const void* w, float* y, int T, int N, int K, void* stream) {
  if (dtype != GOCR_DTYPE_F32 && dtype != GOCR_DTYPE_BF16) return set_error(GOCR_EINVAL, "bad dtype");
  if (!x || !w || !y) return set_error(GOCR_EINVAL, "null pointer");
  if (T < 1 || N < 1 || K < 8 || K % 8) return set_error(GOCR_EINVAL, "bad shape");
  const size_t need = gocr_op_linear_workspace(T, N, K);
  if (need > STATIC_SCRATCH_BYTES) {
    char m[200];
    snprintf(m, sizeof m, "shape T=%d N=%d K=%d needs %zu bytes of scratch, the static array holds %zu", T, N, K,
             need, STATIC_SCRATCH_BYTES);
    return set_error(GOCR_ECAPACITY, m);
  }
  cudaStream_t s = (cudaStream_t)stream;
  // the scratch address below is the current device's: the stream must belong to it
  int cur = 0, sdev = 0;
  if (cudaGetDevice(&cur) != cudaSuccess || cudaStreamGetDevice(s, &sdev) != cudaSuccess)
    return set_error(GOCR_ECUDA, "cannot read the current or the stream's device");
  if (cur != sdev) return set_error(GOCR_EINVAL, "the stream belongs to another device than the current one");
  void* scratch = nullptr;
  int rc = scratch_on_current_device(&scratch);
  if (rc != GOCR_OK) return rc;
  // the array keeps the previous call's contents: the tile counters must start at zero
  const size_t ctr = ((size_t)gemm_counter_ints(T, N) * 4 + 255) & ~(size_t)255;
  if (cudaMemsetAsync(scratch, 0, ctr, s) != cudaSuccess) return set_error(GOCR_ECUDA, "cudaMemsetAsync failed");
  GemmArgs a{};
  a.x = x; a.x_lo = nullptr; a.ldx = K; a.w = w; a.T = T; a.N = N; a.K = K;
  a.kchunk = gemm_kchunk(N, K);
  a.splits = gemm_splits(N, K);
  a.kgroup = gemm_kgroup(N, K, false);
  a.counters = (int*)scratch;
  a.ws = (float*)((char*)scratch + ctr);
  a.epi = EPI_STORE;
  a.e.y = y;
  a.e.ldy = N;
  if (!launch_gemm(dtype, a, s, false)) return set_error(GOCR_ECUDA, "kernel launch configuration rejected");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    char m[160];
    snprintf(m, sizeof m, "launch failed: %s", cudaGetErrorString(e));
    return set_error(GOCR_ECUDA, m);
  }
  return GOCR_OK;
}

}  // extern "C"
