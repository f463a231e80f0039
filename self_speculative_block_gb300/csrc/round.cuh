// Round bookkeeping shared by the decode loops' commit kernels.
#pragma once
#include "kernels.cuh"

namespace gocr {

// Commits n_commit tokens (cut at max_new and after the first eos), moves the
// cache length and the boundary token, counts the round, and ends the request
// on an error, at max_new, at eos or at the loop bound.
__device__ inline void finish_round(ReqState& q, int* out_row, const int* commit, int n_commit, int A,
                             int new_cache_len, int new_x0, int forwards, const int* err) {
  const int room = q.max_new - q.committed;
  int n = n_commit < room ? n_commit : room;
  bool eos = false;
  if (q.eos_id >= 0) {
    for (int i = 0; i < n; ++i)
      if (commit[i] == q.eos_id) { n = i + 1; eos = true; break; }
  }
  for (int i = 0; i < n; ++i) out_row[q.committed + i] = commit[i];
  q.committed += n;
  q.cache_len = new_cache_len;
  q.x0 = new_x0;
  q.st_rounds += 1;
  q.st_forwards += forwards;
  q.st_committed += n;
  q.st_accepted += A;
  if (A >= 0 && A <= 64) q.hist[A] += 1;
  q.round += 1;
  if (err && *err) { q.error = *err; q.done = 1; }
  if (q.committed >= q.max_new || eos) q.done = 1;
  if (!q.done && q.round >= q.max_rounds) { q.error = DERR_ROUND_LIMIT; q.done = 1; }
}

// Keeps the device-side while loop running while any request is not done.
__device__ inline void set_loop_condition(ReqState* st, const int* slot_req, int n_slots,
                                   unsigned long long cond, int use_cond) {
  if (!use_cond) return;
  int any = 0;
  for (int s = 0; s < n_slots; ++s) any |= !st[slot_req[s]].done;
  cudaGraphSetConditional((cudaGraphConditionalHandle)cond, any ? 1u : 0u);
}

}  // namespace gocr
