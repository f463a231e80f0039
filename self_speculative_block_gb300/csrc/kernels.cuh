// Kernel interfaces shared by the host orchestration and the kernel files.
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
  float* y;  int ldy;            // STORE: fp32 [T, N];  RESID: fp32 [T, ldy] +=
  void* hbuf; int ldh;           // SWIGLU: dtype [T, F]
  // QKV: q -> qbuf [T, q_dim]; k, v -> cache of the row's request at its position
  void* qbuf;
  void* kc; void* vc;            // cache of request 0 at this layer
  long long req_stride;          // elements between two requests' caches
  int q_dim, kv_dim, head_dim, cap;
  const float2* rope;            // [cap][head_dim/2] (cos, sin)
  const int* row_pos; const int* row_slot; const Plan* plan;
  // ARGMAX: lowest index among equal maxima
  float* logits; int ld_logits;  // optional full logits (fp32 [T, N])
  float* pmax; int* pidx;        // [n_tiles][T] per-tile partial maxima
  int* am_out;                   // [T]
  int* err;                      // device error word
};

struct GemmArgs {
  const void* x; int ldx;        // [T, K] dtype
  const void* w;                 // [N, K] dtype
  int T, N, K;
  int splits, kchunk;            // K = splits chunks of kchunk (last may be short)
  float* ws;                     // [splits][T][N] fp32 partials
  int* counters;                 // [n_tslices * n_tiles + 1], zero between launches
  int epi;
  EpiArgs e;
};

// Launch of the split-K GEMM with fused epilogue (bf16: tcgen05 + TMA; fp32:
// CUDA cores).  Returns false when a TMA descriptor cannot be encoded.
bool launch_gemm(int dtype, const GemmArgs& a, cudaStream_t s);
bool launch_gemm_tc(const GemmArgs& a, cudaStream_t s);
int gemm_splits(int N, int K);
int gemm_kchunk(int N, int K);
size_t gemm_ws_floats(int T, int N, int K, bool single_split);
int gemm_counter_ints(int T, int N);

// ---------------------------------------------------------------- attention
struct AttnArgs {
  const void* q;           // [T, Hq, d]
  const void* kc; const void* vc;   // request 0's cache at this layer: [Hkv][cap][d]
  long long req_stride;    // elements between requests' caches
  void* o;                 // [T, Hq, d]
  const int* row_lim;      // [T]
  const Plan* plan;        // slot layout; NULL = one slot of T rows, request 0
  int T, Hq, Hkv, d, cap;
  float scale;
};
void launch_attention(int dtype, const AttnArgs& a, int n_slots, int max_rows_per_slot, cudaStream_t s);

// ---------------------------------------------------------------- small kernels
void launch_rmsnorm(int dtype, const float* x, int ldx, const float* g, void* y, int ldy,
                    int T, int H, float eps, const int* gather, const Plan* plan, int which_count,
                    cudaStream_t s);
void launch_embed(int dtype, const void* embed, const void* mask_embed, const void* prefix,
                  float* resid, const Rows& r, int T, int H, int vocab, int* err, cudaStream_t s);
void launch_rope_table(float2* tab, int cap, int d, float theta, cudaStream_t s);

enum PlanKind : int { PLAN_AR = 0, PLAN_DRAFT = 1, PLAN_VERIFY = 2, PLAN_PREFILL = 3 };
// Decode plans read ReqState; `toks` (optional) overrides the row tokens (debug forwards).
void launch_plan(int kind, const Rows& r, ReqState* st, const int* slot_req, int n_slots, int B,
                 int prefill_len, const int* dbuf, const int* toks, int cap, cudaStream_t s);
void launch_accept(ReqState* st, const int* slot_req, int n_slots, int B, const int* dbuf,
                   const int* vbuf, int* out, int out_stride, const int* err,
                   unsigned long long cond, int use_cond, cudaStream_t s);
void launch_ar_commit(ReqState* st, const int* slot_req, int n_slots, const int* abuf, int* out,
                      int out_stride, const int* err, unsigned long long cond, int use_cond,
                      cudaStream_t s);
void launch_override(ReqState* st, const int* slot_req, int n_slots, int B, int* dbuf,
                     const int* ref, int ref_stride, const int* sched, int sched_stride,
                     int vocab, cudaStream_t s);
void launch_prefill_finish(ReqState* st, int req, int P, const int* am, int* out, int out_stride,
                           cudaStream_t s);
// Arms request slots for a decode call: max_new, the round bound, eos, stats reset.
void launch_begin_decode(ReqState* st, const int* slot_req, int n_slots, const int* max_new,
                         int max_rounds, int eos_id, cudaStream_t s);
void launch_set_override(ReqState* st, int req, int n_ref, int n_sched, cudaStream_t s);

}  // namespace gocr
