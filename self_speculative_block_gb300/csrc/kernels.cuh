// Kernel interfaces shared by the host orchestration and the kernel files.
//
// Data flow of one decoder forward (T rows):
//   embed:  resid = E[tok] | [M] | prefix row;  X0 = resid * g_attn[0];  ssq
//   per layer:
//     qkv    = rstd * (X W_qkv^T)  -> RoPE; q planes, k/v planes into the KV cache
//     attn   = softmax(q K^T / sqrt(d), row key limits) V   -> A planes
//     resid += A W_o^T             -> X = resid * g_mlp;  ssq
//     h      = silu(g) * u, [g|u] = rstd * (X W_gu^T)        -> H planes
//     resid += H W_d^T             -> X = resid * g_next; ssq
//   logits  = rstd * (X W_lm^T)    -> argmax (lowest index on ties)
// where rstd = 1/sqrt(mean(resid^2) + eps) is rebuilt by each consumer from
// per-128-column sums of squares (ssq) in a fixed order, so RMSNorm needs no
// kernel of its own.  "Planes" are GEMM inputs: for bf16 models two bf16
// arrays hi + lo with hi = bf16(v), lo = bf16(v - hi) (about 16 significant
// bits, both fed to the tensor cores); for fp32 models one fp32 array.
#pragma once
#include "common.cuh"

namespace gocr {

// ---------------------------------------------------------------- row table
struct Rows {
  Plan* plan;       // device
  int* row_slot;    // [T] slot index of each row
  int* row_pos;     // [T] absolute position
  int* row_lim;     // [T] last key position the row may read
  int* row_tok;     // [T] token id, TOK_MASK, or tok_prefix(j)
  int* logit_row;   // [T] rows that go through the LM head
};

// ---------------------------------------------------------------- GEMM
enum EpiKind : int { EPI_STORE = 0, EPI_RESID = 1, EPI_QKV = 2, EPI_SWIGLU = 3, EPI_ARGMAX = 4 };

struct EpiArgs {
  // input normalisation: y *= rstd[row], rstd from ssq_in[row][0..n_ssq)
  const float* ssq_in; int n_ssq; int norm_H; float eps;
  const int* in_rows;            // row of ssq_in for output row t (NULL = t)
  // STORE: fp32 [T, ldy]
  float* y; int ldy;
  // RESID: resid[T, H] += y; planes of resid * g_next; ssq_out[T][H/128]
  float* resid; int H;
  const float* g_next;
  float* ssq_out;
  // planes written by RESID and SWIGLU: bf16 hi/lo (plane_bf16) or one fp32 array in pl_hi
  void* pl_hi; void* pl_lo; int ld_pl; int plane_bf16;
  // QKV: q -> planes [T, q_dim]; k, v -> cache planes of the row's request at its position
  // (bf16 hi/lo planes for bf16 models, one fp32 plane for fp32 models)
  void* q_hi; void* q_lo;
  void* k_hi; void* k_lo; void* v_hi; void* v_lo;  // cache planes of request 0 at this layer
  long long req_stride;          // elements between two requests' caches
  int q_dim, kv_dim, head_dim, cap;
  const float2* rope;            // [cap][head_dim/2] (cos, sin)
  const int* row_pos; const int* row_slot; const Plan* plan;
  // ARGMAX: lowest index among equal maxima via 64-bit atomicMax of
  // (order-preserving value bits << 32 | ~index); the last CTA publishes.
  float* logits; int ld_logits;  // optional full logits (fp32 [T, N])
  // optional per-(row, 128-column tile) softmax partials (tile max m, sum of
  // exp(l - m) over the tile's columns), [T][N / 128]: the confidence of a
  // row is 1 / sum_tiles s exp(m - max m), combined in tile order
  float2* conf_part;
  unsigned long long* amax;      // [T], zero between launches
  int* am_out;                   // [T]
  int* grid_ctr;                 // zero between launches
  int* err;                      // device error word
};

struct alignas(16) GemmArgs {  // 16-byte aligned: tables of them are copied by 16-byte loads
  const void* x; const void* x_lo; int ldx;  // [T, K] planes (x_lo NULL: single plane)
  const void* w;                 // [N, K] dtype
  int T, N, K;
  int splits, kchunk;            // K = splits chunks of kchunk (last may be short)
  int kgroup;                    // tcgen05 kernels: chunks per reduction group (gemm_kgroup)
  float* ws;                     // CUDA-core path: [splits][T][N] fp32 partials
  int* counters;                 // CUDA-core path: tile counters, zero between launches
  int epi;
  EpiArgs e;
  // weights of the forward's next GEMM: the launch's CTAs bring pf_bytes of
  // them into L2 at their start (NULL = none), so that the next kernel's
  // weight loads hit L2 (the forward is a fixed sequence of matrices)
  const void* pf_next;
  size_t pf_bytes;
  // optional launch timeline record (4 words: first CTA start, first and last
  // release from the dependency wait, last CTA end; globaltimer ns)
  unsigned long long* trace;
  int trace_cta;                 // 1: `trace` holds one record per CTA (TRACE_CTA_SLOTS of them)
};

// Split-K GEMM with fused epilogue (bf16: tcgen05 + TMA, split-K reduced
// across a thread-block cluster; fp32: CUDA cores).  pdl: launch with
// programmatic dependent launch.  Returns false when a TMA descriptor cannot
// be encoded or the launch configuration is rejected.
bool launch_gemm(int dtype, const GemmArgs& a, cudaStream_t s, bool pdl);
bool launch_gemm_tc(const GemmArgs& a, cudaStream_t s, bool pdl);
int gemm_splits(int N, int K);
int gemm_kgroup(int N, int K, bool two_groups);
// 128-byte-swizzled TMA descriptor (CUtensorMap, 128 bytes at `out`) of a
// row-major bf16 matrix [rows, cols] with boxes of 64 columns x box_rows.
bool encode_tmap_bf16(void* out, const void* ptr, int rows, int cols, int box_rows);
int gemm_kchunk(int N, int K);
size_t gemm_ws_floats(int T, int N, int K);
int gemm_counter_ints(int T, int N);

// ---------------------------------------------------------------- attention
struct alignas(16) AttnArgs {
  // q [T, Hq, d] and the KV cache [Hkv][cap][d] of request 0 at this layer, as
  // planes: bf16 hi + lo (bf16 models) or fp32 in *_hi (fp32 models)
  const void* q_hi; const void* q_lo;
  const void* k_hi; const void* k_lo; const void* v_hi; const void* v_lo;
  long long req_stride;    // elements between requests' caches
  void* o_hi; void* o_lo;  // output planes [T, Hq*d] (bf16 hi/lo, or fp32 in o_hi)
  int out_bf16;            // output planes are bf16 (1) or fp32 (0)
  const int* row_lim;      // [T]
  // optional second key interval per row (the joint-training mask): row t
  // also reads keys row_lo2[t]..row_hi2[t] (empty when hi2 < lo2); NULL = none
  const int* row_lo2; const int* row_hi2;
  const Plan* plan;        // slot layout; NULL = one slot of T rows, request 0
  // decode launches: the slot table and request states, constant during a
  // forward, let CTAs fetch committed cache chunks before the dependency wait
  const int* slot_req; const ReqState* st; int rows_per_slot;
  int T, Hq, Hkv, d, cap;
  float scale;
  // tensor-core path: partial rows of the ranks, [slot][kv head x row group][rank][64][d + 4] fp32
  float* part;
  int* part_chunks;           // [slot][kv head x row group] chunks the group's rows read
  int ranks;                  // key-chunk ranks R (attention_ranks); 0: attention_ranks(cap, 1)
  // mma.sync kernel: host copy of the four cache planes' TMA maps (attn::KvMaps:
  // rows of d values, AC-row x 64-value boxes, 128-byte swizzle), and the map
  // row of key 0 of (request 0, this layer, kv head 0) and the rows per request
  const void* kv_maps;
  long long kv_row0, kv_req_rows;
  int kind;                   // bf16 models: ATTN_TCGEN05 or ATTN_MMA_SYNC
  int* err;                   // device error word (bounded waits), or NULL
  unsigned long long* trace;  // launch timeline record, as GemmArgs::trace
  int trace_cta;              // as GemmArgs::trace_cta (merge CTAs from slot TRACE_MERGE_SLOT)
};
// Tensor-core attention kernels of bf16 models.  ATTN_MMA_SYNC: 64-row tiles
// on mma.sync.  ATTN_TCGEN05:
// 128-row tiles, both contractions on tcgen05 with accumulators in tensor
// memory.  The two give different bits; a handle fixes one at creation (by
// the chunks per rank at full capacity, or GOCR_ATTN).
enum { ATTN_TCGEN05 = 0, ATTN_MMA_SYNC = 1 };
// Key-chunk ranks of the tensor-core attention: rank r reads chunks r, r + R, ...
// R = attention_ranks(cap, n_req): ATTN_RANKS for one request, fewer (at
// least ATTN_RANKS_MIN) when a forward carries up to n_req requests, so that
// a full batch keeps about as many partial tiles as one request and each
// tile reads more chunks; never more than a KV capacity of cap keys has chunks
// of 32.  A handle fixes R at creation, so every forward of a handle (one row
// or B + 1, one request or a batch) splits a row's keys the same way.
// Measured on the 16-request page batch (tcgen05 attention, round us): 3, 4,
// 5, 6, 7, 8, 10, 12 ranks: 7,241, 7,209, 7,105, 7,026, 7,171, 7,245, 7,690,
// 7,821.
constexpr int ATTN_RANKS = 48;
constexpr int ATTN_RANKS_MIN = 6;
inline int attention_ranks(int cap, int n_req) {
  const int c = (cap + 31) / 32;
  int r = ATTN_RANKS / (n_req < 1 ? 1 : n_req);
  if (r < ATTN_RANKS_MIN) r = ATTN_RANKS_MIN;
  return c < 1 ? 1 : (c < r ? c : r);
}
// fp32 words of the tensor-core attention's partial rows for n_slots slots of up to max_rows rows, R ranks
// (enough for either kind)
size_t attention_part_floats(int n_slots, int max_rows, int Hq, int Hkv, int d, int R);
// dtype 1: tensor-core cluster kernel; 0: CUDA-core kernel.
bool launch_attention(int dtype, const AttnArgs& a, int n_slots, int max_rows_per_slot, cudaStream_t s,
                      bool pdl);

// ---------------------------------------------------------------- small kernels
void launch_embed(int dtype, const void* embed, const void* mask_embed, const void* prefix,
                  float* resid, const float* g0, void* pl_hi, void* pl_lo, float* ssq, const Rows& r,
                  int T, int H, int vocab, int* err, cudaStream_t s, bool pdl);
void launch_rope_table(float2* tab, int cap, int d, float theta, cudaStream_t s);

// PLAN_BLOCK: block-step decodes; each slot's rows follow its ReqState::phase
// (the draft window with the slots' tokens, the causal cache write, or the
// refined round's verify window), B + 1 rows per slot.
enum PlanKind : int { PLAN_AR = 0, PLAN_DRAFT = 1, PLAN_VERIFY = 2, PLAN_PREFILL = 3, PLAN_BLOCK = 4 };
// Decode plans read ReqState; `toks` (optional) overrides the row tokens (debug forwards).
void launch_plan(int kind, const Rows& r, ReqState* st, const int* slot_req, int n_slots, int B,
                 int prefill_len, const int* dbuf, const int* toks, int cap, cudaStream_t s, bool pdl);
void launch_accept(ReqState* st, const int* slot_req, int n_slots, int B, const int* dbuf,
                   const int* vbuf, int* out, int out_stride, const int* err,
                   unsigned long long cond, int use_cond, cudaStream_t s, bool pdl);
void launch_ar_commit(ReqState* st, const int* slot_req, int n_slots, const int* abuf, int* out,
                      int out_stride, const int* err, unsigned long long cond, int use_cond,
                      cudaStream_t s, bool pdl);
void launch_override(ReqState* st, const int* slot_req, int n_slots, int B, int* dbuf,
                     const int* ref, int ref_stride, const int* sched, int sched_stride,
                     int vocab, cudaStream_t s, bool pdl);
void launch_prefill_finish(ReqState* st, int req, int P, const int* am, int* out, int out_stride,
                           cudaStream_t s);
// Arms request slots for a decode call: max_new, the loop bound, eos, stats
// reset, and the block-step state (threshold, draft steps, masked slots).
void launch_begin_decode(ReqState* st, const int* slot_req, int n_slots, const int* max_new,
                         int max_rounds, int eos_id, float tau, int n_steps, float temp, unsigned long long seed,
                         cudaStream_t s);
// Sampling decodes (sampling.cu): Gumbel-max draws of AR or draft rows from
// the forward's logits [n_slots * rows_per_slot, V]; the acceptance-rejection
// commit of a sampling round (then the device-loop condition).
void launch_sample_rows(const ReqState* st, const int* slot_req, int n_slots, int rows_per_slot, const float* logits,
                        int V, int* out, cudaStream_t s, bool pdl);
void launch_accept_sample(ReqState* st, const int* slot_req, int n_slots, int B, const int* dbuf, const float* ld,
                          const float* lv, int V, int* out, int out_stride, const int* err, unsigned long long cond,
                          int use_cond, cudaStream_t s, bool pdl);
// The step kernel of a block-step decode (refined = 0: direct block
// diffusion; 1: self-speculative rounds with refined drafts), after the
// forward whose LM head wrote argmaxes `am` and confidence partials.
void launch_block_step(int refined, ReqState* st, const int* slot_req, int n_slots, int B, const int* am,
                       const float2* conf_part, int n_tiles, int* out, int out_stride, const int* err,
                       unsigned long long cond, int use_cond, cudaStream_t s, bool pdl);
void launch_set_override(ReqState* st, int req, int n_ref, int n_sched, cudaStream_t s);

// Launch timeline records (GemmArgs::trace, TRACE_WORDS words): word 0 min of
// CTA start times, 1 and 2 min / max of dependency-release times, 3 max of
// CTA end times; GEMMs also 4 max of mainloop-done times, 5 max of split-K
// exchange-done times, 6 max of cluster-barrier-passed times, 7 max of
// accumulator-drained times; attention 4 max of first-chunk-ready times, 5 max of
// chunk-loop-done times, 6 max of merge-exchange-done times.
constexpr int TRACE_WORDS = 8;
__device__ __forceinline__ unsigned long long trace_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void trace_mark(unsigned long long* r, int word) {
  if (!r) return;
  const unsigned long long t = trace_now();
  if (word == 0 || word == 1) atomicMin(r + word, t);
  else atomicMax(r + word, t);
  if (word == 1) atomicMax(r + 2, t);
}
// Per-CTA timelines (GOCR_OP_TRACE=2): each launch has TRACE_CTA_SLOTS
// records of TRACE_WORDS words; CTA c of a kernel writes record c (the
// attention merge kernel from TRACE_MERGE_SLOT on) with plain stores: word
// 0 start, 1 release from the dependency wait, then the kernel's own marks
// (GEMMs: 4 mainloop done, 7 accumulator drained, 6 cluster barrier passed,
// 5 split-K exchange done, 2 epilogue start; attention: 4 first chunk
// ready, 5 chunk loop done, 6 merge start), 3 end.
constexpr int TRACE_CTA_SLOTS = 2048;
constexpr int TRACE_MERGE_SLOT = 1024;
template <class Args>
__device__ __forceinline__ void trace_at(const Args& a, int word, int slot0 = 0) {
  if (!a.trace) return;
  if (a.trace_cta) {
    const unsigned cta = slot0 + blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    if (cta < (unsigned)TRACE_CTA_SLOTS) a.trace[(size_t)cta * TRACE_WORDS + word] = trace_now();
  } else if (word != 2) {
    trace_mark(a.trace, word);
  }
}

// Library-level error message returned by gocr_last_error(NULL).
void set_lib_error(const char* msg);

// Ask for the largest shared-memory carveout for kernel `fn` on the current
// device (once).  Every kernel of the decode path runs with the same SM
// configuration, so a kernel launched early under programmatic dependent
// launch can share SMs with the one before it, and two 104 KB CTAs fit on an
// SM.
void prefer_shared(const void* fn);
// Raises kernel fn's dynamic shared-memory limit on the current device to at
// least `bytes` (and allows non-portable cluster sizes when asked), then
// prefer_shared(fn).  Kept per (device, kernel) under a lock, so handles on
// several devices or threads each configure their device.  False when the
// runtime rejects the attribute.
bool kernel_smem_at_least(const void* fn, size_t bytes, bool nonportable_cluster = false);

// Launch helper: plain launch, or with the programmatic-dependent-launch attribute.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            bool pdl, Args... args) {
  prefer_shared(reinterpret_cast<const void*>(k));
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}

}  // namespace gocr
