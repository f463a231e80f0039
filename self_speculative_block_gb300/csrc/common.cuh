// Shared device-side definitions of the decoder kernels.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace gocr {

typedef __nv_bfloat16 bf16;

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<bf16>(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
// round to nearest even
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

// Token codes in a forward's row table.
constexpr int TOK_MASK = -1;      // the [M] embedding row
// prefix row j of the staged prefix embeddings is encoded as -2 - j
__host__ __device__ __forceinline__ int tok_prefix(int j) { return -2 - j; }

// Device error word values (first error wins).
enum DevErr : int {
  DERR_NONE = 0,
  DERR_NAN_LOGITS = 1,
  DERR_CAPACITY = 2,
  DERR_ROUND_LIMIT = 3,
  DERR_BAD_TOKEN = 4,
  DERR_TIMEOUT = 5,     // a bounded wait inside a kernel gave up
};

constexpr int MAX_REQ = 64;       // request slots per handle (host check)
constexpr int NTILE = 128;        // GEMM rows of W per CTA tile
// SMs of a GB300.  Work splits that change results (GEMM split-K counts,
// attention ranks) are sized against this constant rather than the device's
// SM count, so that a result's bits are the same on every device.
constexpr int SM_COUNT = 152;
constexpr int SWIGLU_GROUP = 64;  // gate/up interleave granularity (rows)

// Per-request decode state, resident on the device for the whole decode.
struct ReqState {
  int cache_len;       // p: positions 0..p-1 hold causal state; x0 sits at p
  int x0;              // boundary token (committed, not yet in the cache)
  int committed;       // tokens in out[], the prefill token included
  int max_new;         // stop when committed >= max_new
  int done;
  int error;           // DevErr
  int round;           // rounds (or AR steps) run in this decode
  int max_rounds;      // device-side loop bound
  int eos_id;          // -1 = none
  int n_ref;           // forced-acceptance reference length (0 = off)
  int n_sched;
  int pad_;
  long long st_rounds, st_forwards, st_committed, st_accepted;
  int hist[65];
  // block-step decodes (direct block diffusion, refined drafts): one forward
  // per loop iteration, its kind chosen from `phase`
  int phase;           // PHASE_STEP, PHASE_WRITE (diffusion) or PHASE_VERIFY (refined)
  int steps;           // denoising steps run in the current block or draft
  int n_steps;         // refined drafts: draft forwards per round at most
  float tau;           // confidence threshold (tau_c, or the draft-side tau_d)
  int blk[64];         // slot tokens of the window, -1 = [M] (slot s at position cache_len + 1 + s)
  int win[65];         // refined drafts: the verify window [a0, d1..dB] of the last draft step
  // sampling decodes: softmax temperature and the random-number seed
  float temp;
  unsigned long long seed;
};
enum BlockPhase : int { PHASE_STEP = 0, PHASE_WRITE = 1, PHASE_VERIFY = 2 };

// Row table of one forward (built on the device from ReqState by plan kernels).
struct Plan {
  int n_rows;             // rows in this forward (fixed per launch configuration)
  int n_slots;            // requests in this forward
  int n_logit_rows;       // rows that go through the LM head
  int max_keys;           // max over rows of lim + 1
  int slot_req[MAX_REQ];  // request index of each slot
  int slot_row0[MAX_REQ]; // first row of the slot
  int slot_nrows[MAX_REQ];
  int slot_maxlim[MAX_REQ];
};

}  // namespace gocr
