// Row-table, embedding and round-control kernels.
//
// Round control follows GravityOCR's decode round (review §3.2 and
// Appendix B.2; velog review, inference section):
//   * the cache holds the causal state of every committed token but the
//     boundary token x0, which sits at position p = cache_len;
//   * draft rows [x0, M x B] sit at p..p+B; verify rows [a0, d1..dB] at
//     p+1..p+B+1;
//   * A = longest prefix with d_j == a_j; the round commits a0, d1..dA and
//     a_(A+1) (at most max_new - committed, cut after eos), keeps cache
//     positions 0..p+A+1 and makes a_(A+1) the next boundary.
#include "epilogue.cuh"
#include "round.cuh"

#include <mutex>
#include <map>
#include <set>
#include <utility>

namespace gocr {

void prefer_shared(const void* fn) {
  static std::mutex mu;
  static std::set<std::pair<int, const void*>> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return;
  std::lock_guard<std::mutex> lk(mu);
  if (!done.insert({dev, fn}).second) return;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
      cudaSuccess)
    cudaGetLastError();  // a hint only: the launch still works without it
}

bool kernel_smem_at_least(const void* fn, size_t bytes, bool nonportable_cluster) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = done.find({dev, fn});
    if (it == done.end() || it->second < bytes) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
        return false;
      if (nonportable_cluster &&
          cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return false;
      done[{dev, fn}] = bytes;
    }
  }
  prefer_shared(fn);
  return true;
}

// ---------------------------------------------------------------- embedding rows
// resid[t] = E[tok] | [M] | prefix row;  X[t] = resid[t] * g0 as GEMM-input
// planes;  ssq[t][i] = sum of squares of columns [128 i, 128 i + 128).
// One CTA per row; warp w takes 128-column groups w, w + 8, ...
template <typename T>
__global__ void __launch_bounds__(256) embed_kernel(const T* embed, const T* mask_embed, const T* prefix,
                                                   float* resid, const float* g0, void* pl_hi, void* pl_lo,
                                                   float* ssq, Rows r, int H, int vocab, int* err) {
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t = blockIdx.x;
  if (t >= r.plan->n_rows) return;
  const int tok = r.row_tok[t];
  const T* src;
  if (tok >= 0) {
    if (tok >= vocab) {
      if (threadIdx.x == 0) set_err(err, DERR_BAD_TOKEN);
      return;
    }
    src = embed + (size_t)tok * H;
  } else if (tok == TOK_MASK) {
    src = mask_embed;
  } else {
    src = prefix + (size_t)(-2 - tok) * H;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int bf = sizeof(T) == 2;
  for (int grp = warp; grp < H / NTILE; grp += 8) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = grp * NTILE + lane + 32 * j;
      const float x = to_f32<T>(src[c]);
      resid[(size_t)t * H + c] = x;
      put_plane(pl_hi, pl_lo, bf, (size_t)t * H + c, x * g0[c]);
      ss = fmaf(x, x, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) ssq[(size_t)t * (H / NTILE) + grp] = ss;
  }
}

void launch_embed(int dtype, const void* embed, const void* mask_embed, const void* prefix,
                  float* resid, const float* g0, void* pl_hi, void* pl_lo, float* ssq, const Rows& r,
                  int T, int H, int vocab, int* err, cudaStream_t s, bool pdl) {
  if (dtype == 1)
    launch_k(embed_kernel<bf16>, dim3(T), dim3(256), 0, s, pdl, (const bf16*)embed, (const bf16*)mask_embed,
             (const bf16*)prefix, resid, g0, pl_hi, pl_lo, ssq, r, H, vocab, err);
  else
    launch_k(embed_kernel<float>, dim3(T), dim3(256), 0, s, pdl, (const float*)embed, (const float*)mask_embed,
             (const float*)prefix, resid, g0, pl_hi, pl_lo, ssq, r, H, vocab, err);
}

// ---------------------------------------------------------------- rotary table
// cos/sin of pos * theta^(-2i/d), evaluated in double and rounded once.
__global__ void rope_table_kernel(float2* tab, int cap, int d, double theta) {
  const int half = d / 2;
  size_t n = (size_t)cap * half;
  for (size_t x = blockIdx.x * (size_t)blockDim.x + threadIdx.x; x < n; x += (size_t)gridDim.x * blockDim.x) {
    int pos = (int)(x / half), i = (int)(x % half);
    double inv = pow(theta, -2.0 * i / d);
    double ang = (double)pos * inv;
    tab[x] = make_float2((float)cos(ang), (float)sin(ang));
  }
}

void launch_rope_table(float2* tab, int cap, int d, float theta, cudaStream_t s) {
  rope_table_kernel<<<256, 256, 0, s>>>(tab, cap, d, (double)theta);
}

// ---------------------------------------------------------------- row tables
// Slot layout: slot s owns rows [s*w, (s+1)*w) with w = 1 (AR), B+1 (draft,
// verify) or P (prefill, one slot).
__global__ void plan_kernel(int kind, Rows r, ReqState* st, const int* slot_req, int n_slots, int B,
                            int prefill_len, const int* dbuf, const int* toks, int cap) {
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int w = kind == PLAN_AR ? 1 : (kind == PLAN_PREFILL ? prefill_len : B + 1);
  const int n_rows = w * n_slots;
  Plan* pl = r.plan;
  for (int t = threadIdx.x; t < n_rows; t += blockDim.x) {
    const int s = t / w, j = t % w;
    const int req = slot_req[s];
    const int p = kind == PLAN_PREFILL ? 0 : st[req].cache_len;
    int pos, lim, tok;
    switch (kind) {
      case PLAN_AR:
        pos = p; lim = p; tok = toks ? toks[t] : st[req].x0;
        break;
      case PLAN_DRAFT:
        pos = p + j; lim = j == 0 ? p : p + B;
        tok = j == 0 ? (toks ? toks[s * w] : st[req].x0) : TOK_MASK;
        break;
      case PLAN_VERIFY:
        pos = p + 1 + j; lim = pos; tok = toks ? toks[t] : dbuf[t];
        break;
      case PLAN_BLOCK: {
        const ReqState& q = st[req];
        if (q.phase == PHASE_STEP) {          // [x0, slots] under the draft mask
          pos = p + j; lim = j == 0 ? p : p + B;
          tok = j == 0 ? q.x0 : (q.blk[j - 1] >= 0 ? q.blk[j - 1] : TOK_MASK);
        } else if (q.phase == PHASE_WRITE) {  // [x0, y_1..y_B], token-causal
          pos = p + j; lim = pos;
          tok = j == 0 ? q.x0 : q.blk[j - 1];
        } else {                              // PHASE_VERIFY: [a0, d_1..d_B] at p+1.., token-causal
          pos = p + 1 + j; lim = pos; tok = q.win[j];
        }
        break;
      }
      default:  // PLAN_PREFILL
        pos = j; lim = j; tok = tok_prefix(j);
        break;
    }
    if (pos >= cap) { pos = cap - 1; lim = min(lim, cap - 1); }
    r.row_slot[t] = s;
    r.row_pos[t] = pos;
    r.row_lim[t] = lim;
    r.row_tok[t] = tok;
    r.logit_row[t] = kind == PLAN_PREFILL ? (s + 1) * w - 1 : t;
  }
  if (threadIdx.x < n_slots) {
    const int s = threadIdx.x;
    const int req = slot_req[s];
    const int p = kind == PLAN_PREFILL ? 0 : st[req].cache_len;
    pl->slot_req[s] = req;
    pl->slot_row0[s] = s * w;
    pl->slot_nrows[s] = w;
    int ml = kind == PLAN_PREFILL ? w - 1 : (kind == PLAN_AR ? p : (kind == PLAN_DRAFT ? p + B : p + B + 1));
    if (kind == PLAN_BLOCK) ml = st[req].phase == PHASE_VERIFY ? p + B + 1 : p + B;
    pl->slot_maxlim[s] = ml;
    if (kind != PLAN_PREFILL && p + (kind == PLAN_AR ? 0 : B + 1) >= cap) {
      st[req].error = DERR_CAPACITY;
      st[req].done = 1;
    }
  }
  if (threadIdx.x == 0) {
    pl->n_rows = n_rows;
    pl->n_slots = n_slots;
    pl->n_logit_rows = kind == PLAN_PREFILL ? n_slots : n_rows;
  }
}

void launch_plan(int kind, const Rows& r, ReqState* st, const int* slot_req, int n_slots, int B,
                 int prefill_len, const int* dbuf, const int* toks, int cap, cudaStream_t s, bool pdl) {
  launch_k(plan_kernel, dim3(1), dim3(1024), 0, s, pdl, kind, r, st, slot_req, n_slots, B, prefill_len, dbuf,
           toks, cap);
}

// One thread per slot, one CTA: updates every request, then sets the loop flag.
__global__ void accept_kernel(ReqState* st, const int* slot_req, int n_slots, int B, const int* dbuf,
                              const int* vbuf, int* out, int out_stride, const int* err,
                              unsigned long long cond, int use_cond) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int s = threadIdx.x;
  if (s < n_slots) {
    const int req = slot_req[s];
    ReqState& q = st[req];
    if (!q.done) {
      const int* d = dbuf + s * (B + 1);   // d[0] = a0, d[j] = d_j
      const int* v = vbuf + s * (B + 1);   // v[j-1] = a_j
      int A = 0;
      while (A < B && d[A + 1] == v[A]) ++A;
      int commit[66];
      commit[0] = d[0];
      for (int j = 1; j <= A + 1; ++j) commit[j] = v[j - 1];
      const int p = q.cache_len;
      finish_round(q, out + (size_t)req * out_stride, commit, A + 2, A, p + A + 2, v[A], 2, err);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) set_loop_condition(st, slot_req, n_slots, cond, use_cond);
}

void launch_accept(ReqState* st, const int* slot_req, int n_slots, int B, const int* dbuf,
                   const int* vbuf, int* out, int out_stride, const int* err,
                   unsigned long long cond, int use_cond, cudaStream_t s, bool pdl) {
  launch_k(accept_kernel, dim3(1), dim3(64), 0, s, pdl, st, slot_req, n_slots, B, dbuf, vbuf, out, out_stride,
           err, cond, use_cond);
}

__global__ void ar_commit_kernel(ReqState* st, const int* slot_req, int n_slots, const int* abuf,
                                 int* out, int out_stride, const int* err,
                                 unsigned long long cond, int use_cond) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int s = threadIdx.x;
  if (s < n_slots) {
    const int req = slot_req[s];
    ReqState& q = st[req];
    if (!q.done) {
      int tok = abuf[s];
      finish_round(q, out + (size_t)req * out_stride, &tok, 1, 0, q.cache_len + 1, tok, 1, err);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) set_loop_condition(st, slot_req, n_slots, cond, use_cond);
}

void launch_ar_commit(ReqState* st, const int* slot_req, int n_slots, const int* abuf, int* out,
                      int out_stride, const int* err, unsigned long long cond, int use_cond,
                      cudaStream_t s, bool pdl) {
  launch_k(ar_commit_kernel, dim3(1), dim3(64), 0, s, pdl, st, slot_req, n_slots, abuf, out, out_stride, err,
           cond, use_cond);
}

// Forced-acceptance hook: between draft and verify, per slot.
__global__ void override_kernel(ReqState* st, const int* slot_req, int n_slots, int B, int* dbuf,
                                const int* ref, int ref_stride, const int* sched, int sched_stride,
                                int vocab) {
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int s = threadIdx.x;
  if (s >= n_slots) return;
  const int req = slot_req[s];
  const ReqState& q = st[req];
  if (q.n_ref <= 0 || q.done) return;
  const int* rr = ref + (size_t)req * ref_stride;
  const int G = q.round < q.n_sched ? sched[(size_t)req * sched_stride + q.round] : 0;
  const int c = q.committed;
  int* d = dbuf + s * (B + 1);
  for (int j = 1; j <= B && j <= G; ++j)
    if (c + j < q.n_ref) d[j] = rr[c + j];
  if (G < B && c + G + 1 < q.n_ref) d[G + 1] = (rr[c + G + 1] + 1) % vocab;
}

void launch_override(ReqState* st, const int* slot_req, int n_slots, int B, int* dbuf,
                     const int* ref, int ref_stride, const int* sched, int sched_stride,
                     int vocab, cudaStream_t s, bool pdl) {
  launch_k(override_kernel, dim3(1), dim3(64), 0, s, pdl, st, slot_req, n_slots, B, dbuf, ref, ref_stride, sched,
           sched_stride, vocab);
}

// ---------------------------------------------------------------- block-step decodes
// Confidence of one LM-head row from its per-tile partials (tile max m_k,
// sum of exp(l - m_k) over the tile): 1 / sum_k s_k exp(m_k - m), m = max_k m_k.
// Lane l folds tiles l, l + 32, ... in order, then the lanes combine in a
// fixed butterfly; lane 0's value is the result.
__device__ float row_confidence(const float2* part, int n_tiles) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY, s = 0.f;
  for (int k = lane; k < n_tiles; k += 32) {
    const float2 pk = part[k];
    if (pk.x > m) {
      s = s * expf(m - pk.x) + pk.y;
      m = pk.x;
    } else {
      s += pk.y * expf(pk.x - m);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const float os = __shfl_xor_sync(0xffffffffu, s, o);
    const float mm = fmaxf(m, om);
    s = (m == -INFINITY ? 0.f : s * expf(m - mm)) + (om == -INFINITY ? 0.f : os * expf(om - mm));
    m = mm;
  }
  return 1.f / s;
}

// Confidences of every still-masked slot's row (slot r is predicted by row r
// of the request's window), one warp per row, into conf[slot][64].
__device__ void masked_slot_confidences(const ReqState* st, const int* slot_req, int n_slots, int B,
                                        const float2* conf_part, int n_tiles, float* conf) {
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int x = warp; x < n_slots * B; x += nw) {
    const int i = x / B, r = x % B;
    const ReqState& q = st[slot_req[i]];
    if (q.done || q.phase != PHASE_STEP || q.blk[r] >= 0) continue;
    const float c = row_confidence(conf_part + (size_t)(i * (B + 1) + r) * n_tiles, n_tiles);
    if ((threadIdx.x & 31) == 0) conf[i * 64 + r] = c;
  }
}

// One denoising step's threshold rule (GravityOCR review, Appendix B.1): every
// masked slot whose confidence reaches tau gets its row's argmax; if none
// does, the most confident masked slot alone (the lowest slot among equals).
// Returns whether every slot is fixed.
__device__ bool fix_slots(ReqState& q, const float* conf, const int* pred, int B) {
  int n_pass = 0, best = -1;
  float bc = 0.f;
  for (int r = 0; r < B; ++r) {
    if (q.blk[r] >= 0) continue;
    if (conf[r] >= q.tau) ++n_pass;
    if (best < 0 || conf[r] > bc) { best = r; bc = conf[r]; }
  }
  bool all = true;
  for (int r = 0; r < B; ++r) {
    if (q.blk[r] >= 0) continue;
    if (n_pass ? conf[r] >= q.tau : r == best) q.blk[r] = pred[r];
    else all = false;
  }
  return all;
}

__device__ void end_iteration(ReqState& q, const int* err) {
  if (err && *err) { q.error = *err; q.done = 1; }
  if (!q.done && q.round >= q.max_rounds) { q.error = DERR_ROUND_LIMIT; q.done = 1; }
}

// Direct block-diffusion decoding, one forward per loop iteration.
//   PHASE_STEP: fix slots by the threshold rule; a finished block commits
//   y_1..y_B (cut at max_new and after the first EOS) and, unless decoding
//   stops, moves to PHASE_WRITE.
//   PHASE_WRITE (the causal cache-write forward has run): positions
//   p..p+B-1 now hold causal state, y_B becomes the boundary, a new block of
//   masks starts.
// Stats: rounds = blocks, forwards = steps + cache writes, hist[steps of a block].
__global__ void diffusion_step_kernel(ReqState* st, const int* slot_req, int n_slots, int B, const int* am,
                                      const float2* conf_part, int n_tiles, int* out, int out_stride,
                                      const int* err, unsigned long long cond, int use_cond) {
  __shared__ float conf[MAX_REQ * 64];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  masked_slot_confidences(st, slot_req, n_slots, B, conf_part, n_tiles, conf);
  __syncthreads();
  const int i = threadIdx.x;
  if (i < n_slots) {
    const int req = slot_req[i];
    ReqState& q = st[req];
    if (!q.done) {
      q.round += 1;
      q.st_forwards += 1;
      if (q.phase == PHASE_STEP) {
        q.steps += 1;
        if (fix_slots(q, conf + i * 64, am + i * (B + 1), B)) {
          const int room = q.max_new - q.committed;
          int n = B < room ? B : room;
          bool eos = false;
          if (q.eos_id >= 0)
            for (int r = 0; r < n; ++r)
              if (q.blk[r] == q.eos_id) { n = r + 1; eos = true; break; }
          int* o = out + (size_t)req * out_stride;
          for (int r = 0; r < n; ++r) o[q.committed + r] = q.blk[r];
          q.committed += n;
          q.st_committed += n;
          q.st_rounds += 1;
          q.hist[q.steps < 64 ? q.steps : 64] += 1;
          if (q.committed >= q.max_new || eos) q.done = 1;
          else q.phase = PHASE_WRITE;
        }
      } else {
        q.cache_len += B;
        q.x0 = q.blk[B - 1];
        for (int r = 0; r < B; ++r) q.blk[r] = -1;
        q.steps = 0;
        q.phase = PHASE_STEP;
      }
      end_iteration(q, err);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) set_loop_condition(st, slot_req, n_slots, cond, use_cond);
}

// Self-speculative rounds with a refined draft (GravityOCR review, Appendix D),
// one forward per loop iteration.
//   PHASE_STEP: a draft forward; fix slots by the draft-side threshold; the
//   verify window becomes [slot 1..B (fixed, else this step's prediction),
//   row B's prediction]; after n_steps draft forwards, or when every slot is
//   fixed, move to PHASE_VERIFY.
//   PHASE_VERIFY: accept, commit and roll back as the one-shot round does.
__global__ void refine_step_kernel(ReqState* st, const int* slot_req, int n_slots, int B, const int* am,
                                   const float2* conf_part, int n_tiles, int* out, int out_stride,
                                   const int* err, unsigned long long cond, int use_cond) {
  __shared__ float conf[MAX_REQ * 64];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  masked_slot_confidences(st, slot_req, n_slots, B, conf_part, n_tiles, conf);
  __syncthreads();
  const int i = threadIdx.x;
  if (i < n_slots) {
    const int req = slot_req[i];
    ReqState& q = st[req];
    if (!q.done) {
      const int* a = am + i * (B + 1);
      if (q.phase == PHASE_STEP) {
        q.round += 1;
        q.st_forwards += 1;
        q.steps += 1;
        const bool all = fix_slots(q, conf + i * 64, a, B);
        for (int r = 0; r < B; ++r) q.win[r] = q.blk[r] >= 0 ? q.blk[r] : a[r];
        q.win[B] = a[B];
        if (all || q.steps >= q.n_steps) q.phase = PHASE_VERIFY;
        end_iteration(q, err);
      } else {
        // a holds a_1..a_(B+1); the drafts d_j = win[j]
        int A = 0;
        while (A < B && q.win[A + 1] == a[A]) ++A;
        int commit[66];
        commit[0] = q.win[0];
        for (int j = 1; j <= A + 1; ++j) commit[j] = a[j - 1];
        const int p = q.cache_len;
        finish_round(q, out + (size_t)req * out_stride, commit, A + 2, A, p + A + 2, a[A], 1, err);
        for (int r = 0; r < B; ++r) q.blk[r] = -1;
        q.steps = 0;
        q.phase = PHASE_STEP;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) set_loop_condition(st, slot_req, n_slots, cond, use_cond);
}

void launch_block_step(int refined, ReqState* st, const int* slot_req, int n_slots, int B, const int* am,
                       const float2* conf_part, int n_tiles, int* out, int out_stride, const int* err,
                       unsigned long long cond, int use_cond, cudaStream_t s, bool pdl) {
  launch_k(refined ? refine_step_kernel : diffusion_step_kernel, dim3(1), dim3(1024), 0, s, pdl, st, slot_req,
           n_slots, B, am, conf_part, n_tiles, out, out_stride, err, cond, use_cond);
}

__global__ void prefill_finish_kernel(ReqState* st, int req, int P, const int* am, int* out,
                                      int out_stride) {
  ReqState& q = st[req];
  const int t0 = am[0];
  q.cache_len = P;
  q.x0 = t0;
  q.committed = 1;
  q.done = 0;
  q.error = 0;
  q.round = 0;
  q.st_rounds = q.st_forwards = q.st_committed = q.st_accepted = 0;
  for (int i = 0; i < 65; ++i) q.hist[i] = 0;
  out[(size_t)req * out_stride] = t0;
}

void launch_prefill_finish(ReqState* st, int req, int P, const int* am, int* out, int out_stride,
                           cudaStream_t s) {
  prefill_finish_kernel<<<1, 1, 0, s>>>(st, req, P, am, out, out_stride);
}

__global__ void begin_decode_kernel(ReqState* st, const int* slot_req, int n_slots,
                                    const int* max_new, int max_rounds, int eos_id, float tau, int n_steps,
                                    float temp, unsigned long long seed) {
  const int s = threadIdx.x;
  if (s >= n_slots) return;
  ReqState& q = st[slot_req[s]];
  q.max_new = max_new[s];
  q.max_rounds = max_rounds;
  q.eos_id = eos_id;
  q.round = 0;
  q.error = 0;
  q.done = q.committed >= q.max_new;
  q.st_rounds = q.st_forwards = q.st_committed = q.st_accepted = 0;
  for (int i = 0; i < 65; ++i) q.hist[i] = 0;
  q.phase = PHASE_STEP;
  q.steps = 0;
  q.n_steps = n_steps;
  q.tau = tau;
  for (int i = 0; i < 64; ++i) q.blk[i] = -1;
  for (int i = 0; i < 65; ++i) q.win[i] = q.x0;
  q.temp = temp;
  q.seed = seed;
}

void launch_begin_decode(ReqState* st, const int* slot_req, int n_slots, const int* max_new,
                         int max_rounds, int eos_id, float tau, int n_steps, float temp, unsigned long long seed,
                         cudaStream_t s) {
  begin_decode_kernel<<<1, 64, 0, s>>>(st, slot_req, n_slots, max_new, max_rounds, eos_id, tau, n_steps, temp,
                                       seed);
}

__global__ void set_override_kernel(ReqState* st, int req, int n_ref, int n_sched) {
  st[req].n_ref = n_ref;
  st[req].n_sched = n_sched;
}

void launch_set_override(ReqState* st, int req, int n_ref, int n_sched, cudaStream_t s) {
  set_override_kernel<<<1, 1, 0, s>>>(st, req, n_ref, n_sched);
}

}  // namespace gocr
