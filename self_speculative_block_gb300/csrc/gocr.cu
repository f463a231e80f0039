// C ABI and round orchestration of the self-speculative block decoder.
//
// One handle owns, on one GPU: re-packed projection weights, a contiguous KV
// cache per request slot ([layer][kv head][position][head_dim]), activation
// buffers sized for the largest forward, device-resident request state, and a
// cache of instantiated CUDA graphs.  A decode call launches one graph whose
// body is a whole round (draft forward, optional forced-acceptance override,
// verify forward, accept/commit/rollback) inside a device-side while loop; the
// accept kernel clears the loop condition when every request is done, so no
// host synchronisation happens between rounds.
#include "../../include/gocr.h"
#include "kernels.cuh"

#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

using namespace gocr;

namespace {

thread_local std::string g_lib_error;

struct GraphEntry {
  int mode, B, n_slots;
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  bool host_loop;  // body only, no device-side while node
};

// Every kernel argument of one decoder forward: per layer the QKV, O,
// gate/up and down GEMMs, then the LM head; per layer the attention.
struct FwdArgs {
  int T = 0;
  std::vector<GemmArgs> g;
  std::vector<AttnArgs> at;
};

}  // namespace

void gocr::set_lib_error(const char* msg) { g_lib_error = msg; }

struct gocr_handle {
  gocr_config cfg{};
  int es = 4;  // element size of dtype
  int dtype = 0;
  cudaStream_t hs = nullptr;
  cudaStream_t user = nullptr;
  cudaEvent_t ev0 = nullptr, ev1 = nullptr, evu = nullptr;
  gocr_alloc_fn af = nullptr;
  gocr_free_fn ff = nullptr;
  void* au = nullptr;
  std::vector<void*> allocs;

  const void* embed = nullptr;
  const void* mask = nullptr;
  const void* lm = nullptr;
  const float* gfin = nullptr;
  std::vector<void*> wqkv, wgu;
  std::vector<const void*> wo, wd;
  std::vector<const float*> gattn, gmlp;

  int q_dim = 0, kv_dim = 0, qkv_n = 0, gu_n = 0;
  int cap = 0, T_max = 0, T_dec = 0, sched_cap = 0;
  int attn_ranks = 1;  // key-chunk ranks of the tensor-core attention, fixed for the handle
  int attn_kind = ATTN_MMA_SYNC;  // tensor-core attention kernels, fixed for the handle
  bool two_groups = false;        // split-K sums of narrow matrices in two groups (gemm_kgroup)
  long long layer_stride = 0, req_stride = 0;

  // KV cache [req][layer][kv head][position][head_dim]: bf16 hi/lo planes for
  // bf16 models, fp32 (in *_hi) for fp32 models; keys are stored rotated
  void* kc_hi = nullptr;
  void* kc_lo = nullptr;
  void* vc_hi = nullptr;
  void* vc_lo = nullptr;
  float* resid = nullptr;     // residual stream fp32 [T][H]
  void* xg_hi = nullptr;      // GEMM-input planes of resid * g (next norm's gain) [T][H]
  void* xg_lo = nullptr;
  void* at_hi = nullptr;      // attention output planes [T][q_dim]
  void* at_lo = nullptr;
  void* hb_hi = nullptr;      // SwiGLU output planes [T][F]
  void* hb_lo = nullptr;
  float* ssq = nullptr;       // per-128-column sums of squares of resid [T][H/128]
  void* q_hi = nullptr;       // rotated query planes [T][q_dim]
  void* q_lo = nullptr;
  float* logits = nullptr;     // [T_dec][vocab]: debug forwards, and the draft (or AR) rows of sampling decodes
  float* logits_v = nullptr;   // [T_dec][vocab]: the verify rows of sampling rounds (allocated on first use)
  float2* conf_part = nullptr;  // LM-head softmax partials [T_dec][vocab / 128] (block-step decodes)
  float* att_part = nullptr;  // attention partial rows of the key-chunk ranks (bf16 models)
  int* att_chunks = nullptr;  // chunks per (slot, kv head x row group) of the last attention
  unsigned long long* amax = nullptr;
  int* grid_ctr = nullptr;
  bool pdl = true;            // programmatic dependent launch between forward kernels
  bool l2_prefetch = false;   // GEMMs prefetch the next GEMM's weights into L2 (GOCR_L2_PREFETCH=1: on)
  // TMA maps of the KV-cache planes (K hi, K lo, V hi, V lo; bf16 models), 128 bytes each
  alignas(64) unsigned char kv_maps[4][128] = {};
  bool host_loop = false;     // GOCR_HOST_LOOP=1: per-round graphs driven by the host
  int* dbuf = nullptr;
  int* vbuf = nullptr;
  int* abuf = nullptr;
  int* am = nullptr;
  Rows rows{};
  int* slot_req = nullptr;    // decode slot table
  int* slot_one = nullptr;    // one-slot table for prefill / debug
  int* max_new_dev = nullptr;
  ReqState* st = nullptr;
  int* out = nullptr;
  int* ref = nullptr;
  int* sched = nullptr;
  int* err = nullptr;
  int* dbg_toks = nullptr;
  float2* rope = nullptr;
  float* ws = nullptr;
  size_t ws_floats = 0;
  int* counters = nullptr;
  float* pmax = nullptr;
  int* pidx = nullptr;
  void* prefix_stage = nullptr;

  // per-launch timeline of debug forwards run with one kernel per operation
  unsigned long long* op_trace = nullptr;
  bool op_trace_cta = false;  // GOCR_OP_TRACE=2: one record per CTA
  bool op_trace_next = false;

  bool prefilled[MAX_REQ] = {};
  std::vector<GraphEntry> graphs;
  std::string msg;
};

namespace {

// Words of the kernel timelines: one record per launch, or per CTA of a launch.
size_t op_trace_words(const gocr_handle* h) {
  return (size_t)TRACE_WORDS * (h->op_trace_cta ? TRACE_CTA_SLOTS : 1) * (5 * h->cfg.n_layers + 1);
}

int fail(gocr_handle* h, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (h) h->msg = buf; else g_lib_error = buf;
  return code;
}

#define CK(call)                                                                      \
  do {                                                                                \
    cudaError_t e_ = (call);                                                          \
    if (e_ != cudaSuccess)                                                            \
      return fail(h, GOCR_ECUDA, "%s failed: %s", #call, cudaGetErrorString(e_));     \
  } while (0)

void* dev_alloc(gocr_handle* h, size_t bytes) {
  if (bytes == 0) bytes = 256;
  bytes = (bytes + 255) & ~(size_t)255;
  void* p = nullptr;
  if (h->af) {
    p = h->af(bytes, h->au);
  } else if (cudaMalloc(&p, bytes) != cudaSuccess) {
    p = nullptr;
  }
  if (p) {
    h->allocs.push_back(p);
    cudaMemsetAsync(p, 0, bytes, h->hs);
  }
  return p;
}

int n_rows_of(int kind, int n_slots, int B, int P) {
  if (kind == PLAN_AR) return n_slots;
  if (kind == PLAN_PREFILL) return P;
  return n_slots * (B + 1);
}

GemmArgs gemm_base(gocr_handle* h, const void* xh, const void* xl, int ldx, const void* w, int T, int N,
                   int K) {
  GemmArgs a{};
  a.x = xh;
  a.x_lo = h->dtype == GOCR_DTYPE_BF16 ? xl : nullptr;
  a.ldx = ldx; a.w = w; a.T = T; a.N = N; a.K = K;
  a.kchunk = gemm_kchunk(N, K);
  a.splits = gemm_splits(N, K);
  a.kgroup = gemm_kgroup(N, K, h->two_groups);
  a.ws = h->ws;
  a.counters = h->counters;
  a.e.err = h->err;
  a.e.plane_bf16 = h->dtype == GOCR_DTYPE_BF16;
  return a;
}

void set_norm_in(gocr_handle* h, GemmArgs& a) {
  a.e.ssq_in = h->ssq;
  a.e.n_ssq = h->cfg.hidden / NTILE;
  a.e.norm_H = h->cfg.hidden;
  a.e.eps = h->cfg.rms_eps;
}

// Kernel arguments of one decoder forward over the rows the plan kernel lays
// out.  RMSNorm is folded into the GEMMs: producers write resid * g (the next
// norm's gain) as planes plus per-tile sums of squares; consumers scale by rstd.
void forward_args(gocr_handle* h, int kind, int n_slots, int B, int P, int* am_out, float* logits,
                  const int* slot_tab, FwdArgs& f, float2* conf_part = nullptr) {
  const gocr_config& c = h->cfg;
  const int T = n_rows_of(kind, n_slots, B, P);
  const int H = c.hidden;
  f.T = T;
  f.g.clear();
  f.at.clear();
  const size_t kv_es = h->dtype == GOCR_DTYPE_BF16 ? 2 : 4;
  auto lay = [&](void* base, int l) -> void* {
    return base ? (char*)base + (size_t)l * h->layer_stride * kv_es : nullptr;
  };
  for (int l = 0; l < c.n_layers; ++l) {
    // QKV projection (input norm), RoPE, KV-cache write at each row's position
    GemmArgs g = gemm_base(h, h->xg_hi, h->xg_lo, H, h->wqkv[l], T, h->qkv_n, H);
    set_norm_in(h, g);
    g.epi = EPI_QKV;
    g.e.q_hi = h->q_hi; g.e.q_lo = h->q_lo;
    g.e.k_hi = lay(h->kc_hi, l); g.e.k_lo = lay(h->kc_lo, l);
    g.e.v_hi = lay(h->vc_hi, l); g.e.v_lo = lay(h->vc_lo, l);
    g.e.req_stride = h->req_stride;
    g.e.q_dim = h->q_dim; g.e.kv_dim = h->kv_dim; g.e.head_dim = c.head_dim; g.e.cap = h->cap;
    g.e.rope = h->rope;
    g.e.row_pos = h->rows.row_pos; g.e.row_slot = h->rows.row_slot; g.e.plan = h->rows.plan;
    f.g.push_back(g);
    // attention with the row key limits of this forward's mask
    AttnArgs at{};
    at.q_hi = h->q_hi; at.q_lo = h->q_lo;
    at.k_hi = g.e.k_hi; at.k_lo = g.e.k_lo; at.v_hi = g.e.v_hi; at.v_lo = g.e.v_lo;
    at.req_stride = h->req_stride;
    at.o_hi = h->at_hi; at.o_lo = h->at_lo; at.out_bf16 = h->dtype == GOCR_DTYPE_BF16;
    at.row_lim = h->rows.row_lim; at.plan = h->rows.plan;
    // slot geometry is static for a forward; outside prefill (which rewrites the
    // cache from position 0) committed cache chunks may be fetched before the wait
    at.slot_req = slot_tab;
    at.rows_per_slot = kind == PLAN_PREFILL ? P : T / n_slots;
    if (kind != PLAN_PREFILL) at.st = h->st;
    at.T = T; at.Hq = c.n_q_heads; at.Hkv = c.n_kv_heads; at.d = c.head_dim; at.cap = h->cap;
    at.scale = 1.0f / sqrtf((float)c.head_dim);
    at.part = h->att_part;
    at.part_chunks = h->att_chunks;
    at.ranks = h->attn_ranks;
    at.kind = h->attn_kind;
    at.kv_maps = h->kv_maps;
    at.kv_row0 = (long long)l * c.n_kv_heads * h->cap;
    at.kv_req_rows = (long long)c.n_layers * c.n_kv_heads * h->cap;
    at.err = h->err;
    f.at.push_back(at);
    // O projection + residual; planes of resid * g_mlp for the MLP
    GemmArgs go = gemm_base(h, h->at_hi, h->at_lo, h->q_dim, h->wo[l], T, H, h->q_dim);
    go.epi = EPI_RESID;
    go.e.resid = h->resid; go.e.H = H; go.e.g_next = h->gmlp[l]; go.e.ssq_out = h->ssq;
    go.e.pl_hi = h->xg_hi; go.e.pl_lo = h->xg_lo; go.e.ld_pl = H;
    f.g.push_back(go);
    // gate/up (interleaved, input norm) + SwiGLU
    GemmArgs gg = gemm_base(h, h->xg_hi, h->xg_lo, H, h->wgu[l], T, h->gu_n, H);
    set_norm_in(h, gg);
    gg.epi = EPI_SWIGLU;
    gg.e.pl_hi = h->hb_hi; gg.e.pl_lo = h->hb_lo; gg.e.ld_pl = c.ffn;
    f.g.push_back(gg);
    // down + residual; planes of resid * (next layer's g_attn, or the final gain)
    GemmArgs gd = gemm_base(h, h->hb_hi, h->hb_lo, c.ffn, h->wd[l], T, H, c.ffn);
    gd.epi = EPI_RESID;
    gd.e.resid = h->resid; gd.e.H = H; gd.e.ssq_out = h->ssq;
    gd.e.g_next = l + 1 < c.n_layers ? h->gattn[l + 1] : h->gfin;
    gd.e.pl_hi = h->xg_hi; gd.e.pl_lo = h->xg_lo; gd.e.ld_pl = H;
    f.g.push_back(gd);
  }
  // LM head (input norm) + argmax over the rows that need logits
  const int n_logit = kind == PLAN_PREFILL ? n_slots : T;
  const size_t off = kind == PLAN_PREFILL ? (size_t)(P - 1) * H * h->es : 0;
  GemmArgs gl = gemm_base(h, (char*)h->xg_hi + off, h->xg_lo ? (char*)h->xg_lo + off : nullptr, H, h->lm,
                          n_logit, c.vocab, H);
  set_norm_in(h, gl);
  gl.e.in_rows = kind == PLAN_PREFILL ? h->rows.logit_row : nullptr;
  gl.epi = EPI_ARGMAX;
  gl.e.logits = logits; gl.e.ld_logits = c.vocab;
  gl.e.conf_part = conf_part;
  gl.e.amax = h->amax; gl.e.am_out = am_out; gl.e.grid_ctr = h->grid_ctr;
  f.g.push_back(gl);
  // GOCR_L2_PREFETCH=1: each GEMM brings the next GEMM's weights into L2 (at most 48 MB of them)
  if (h->l2_prefetch)
    for (size_t i = 0; i + 1 < f.g.size(); ++i) {
      const GemmArgs& nx = f.g[i + 1];
      const size_t bytes = (size_t)nx.N * nx.K * h->es;
      f.g[i].pf_next = nx.w;
      f.g[i].pf_bytes = bytes < ((size_t)48 << 20) ? bytes : ((size_t)48 << 20);
    }
}

// Enqueue one decoder forward over the rows the plan kernel has laid out:
// the embedding rows, then one kernel per operation.
bool enqueue_forward(gocr_handle* h, int kind, int n_slots, int B, int P, int* am_out,
                     float* logits, const int* slot_tab, float2* conf_part = nullptr) {
  const gocr_config& c = h->cfg;
  const int T = n_rows_of(kind, n_slots, B, P);
  const int H = c.hidden;
  const bool pdl = h->pdl;
  bool ok = true;
  launch_embed(h->dtype, h->embed, h->mask, h->prefix_stage, h->resid, h->gattn[0], h->xg_hi, h->xg_lo,
               h->ssq, h->rows, T, H, c.vocab, h->err, h->hs, pdl);
  FwdArgs f;
  forward_args(h, kind, n_slots, B, P, am_out, logits, slot_tab, f, conf_part);
  if (h->op_trace_next) {
    // launch records in forward order: per layer QKV, attention, O, gate/up, down; then the LM head
    const size_t rec = (size_t)TRACE_WORDS * (h->op_trace_cta ? TRACE_CTA_SLOTS : 1);
    for (int l = 0; l < c.n_layers; ++l) {
      for (int k = 0; k < 4; ++k) {
        f.g[(size_t)l * 4 + k].trace = h->op_trace + rec * (5 * l + (k == 0 ? 0 : k + 1));
        f.g[(size_t)l * 4 + k].trace_cta = h->op_trace_cta;
      }
      f.at[l].trace = h->op_trace + rec * (5 * l + 1);
      f.at[l].trace_cta = h->op_trace_cta;
    }
    f.g[(size_t)c.n_layers * 4].trace = h->op_trace + rec * (5 * c.n_layers);
    f.g[(size_t)c.n_layers * 4].trace_cta = h->op_trace_cta;
  }
  for (int l = 0; l < c.n_layers; ++l) {
    ok &= launch_gemm(h->dtype, f.g[(size_t)l * 4 + 0], h->hs, pdl);
    ok &= launch_attention(h->dtype, f.at[l], kind == PLAN_PREFILL ? 1 : n_slots,
                           kind == PLAN_PREFILL ? P : T / n_slots, h->hs, pdl);
    ok &= launch_gemm(h->dtype, f.g[(size_t)l * 4 + 1], h->hs, pdl);
    ok &= launch_gemm(h->dtype, f.g[(size_t)l * 4 + 2], h->hs, pdl);
    ok &= launch_gemm(h->dtype, f.g[(size_t)l * 4 + 3], h->hs, pdl);
  }
  ok &= launch_gemm(h->dtype, f.g[(size_t)c.n_layers * 4], h->hs, pdl);
  return ok;
}

// Graph-cache modes of the sampling decodes (AR / SELFSPEC with a temperature).
constexpr int MODE_AR_SAMPLE = 16 + GOCR_MODE_AR, MODE_SELFSPEC_SAMPLE = 16 + GOCR_MODE_SELFSPEC;

// One round (or one AR step) of the decode loop.
bool enqueue_round(gocr_handle* h, int mode, int B, int n_slots, unsigned long long cond,
                   int use_cond) {
  bool ok = true;
  const int cap = h->cap;
  const int out_stride = cap;
  const int V = h->cfg.vocab;
  if (mode == MODE_AR_SAMPLE) {
    launch_plan(PLAN_AR, h->rows, h->st, h->slot_req, n_slots, 0, 0, nullptr, nullptr, cap, h->hs, h->pdl);
    ok &= enqueue_forward(h, PLAN_AR, n_slots, 0, 0, h->am, h->logits, h->slot_req);
    launch_sample_rows(h->st, h->slot_req, n_slots, 1, h->logits, V, h->abuf, h->hs, h->pdl);
    launch_ar_commit(h->st, h->slot_req, n_slots, h->abuf, h->out, out_stride, h->err, cond, use_cond, h->hs,
                     h->pdl);
    return ok;
  }
  if (mode == MODE_SELFSPEC_SAMPLE) {
    launch_plan(PLAN_DRAFT, h->rows, h->st, h->slot_req, n_slots, B, 0, nullptr, nullptr, cap, h->hs, h->pdl);
    ok &= enqueue_forward(h, PLAN_DRAFT, n_slots, B, 0, h->am, h->logits, h->slot_req);
    launch_sample_rows(h->st, h->slot_req, n_slots, B + 1, h->logits, V, h->dbuf, h->hs, h->pdl);
    launch_plan(PLAN_VERIFY, h->rows, h->st, h->slot_req, n_slots, B, 0, h->dbuf, nullptr, cap, h->hs, h->pdl);
    ok &= enqueue_forward(h, PLAN_VERIFY, n_slots, B, 0, h->vbuf, h->logits_v, h->slot_req);
    launch_accept_sample(h->st, h->slot_req, n_slots, B, h->dbuf, h->logits, h->logits_v, V, h->out, out_stride,
                         h->err, cond, use_cond, h->hs, h->pdl);
    return ok;
  }
  if (mode == GOCR_MODE_DIFFUSION || mode == GOCR_MODE_REFINED) {
    // one forward per iteration; its rows follow each request's phase
    launch_plan(PLAN_BLOCK, h->rows, h->st, h->slot_req, n_slots, B, 0, nullptr, nullptr, cap, h->hs, h->pdl);
    ok &= enqueue_forward(h, PLAN_DRAFT, n_slots, B, 0, h->dbuf, nullptr, h->slot_req, h->conf_part);
    launch_block_step(mode == GOCR_MODE_REFINED, h->st, h->slot_req, n_slots, B, h->dbuf, h->conf_part,
                      h->cfg.vocab / NTILE, h->out, out_stride, h->err, cond, use_cond, h->hs, h->pdl);
    return ok;
  }
  if (mode == GOCR_MODE_AR) {
    launch_plan(PLAN_AR, h->rows, h->st, h->slot_req, n_slots, 0, 0, nullptr, nullptr, cap, h->hs, h->pdl);
    ok &= enqueue_forward(h, PLAN_AR, n_slots, 0, 0, h->abuf, nullptr, h->slot_req);
    launch_ar_commit(h->st, h->slot_req, n_slots, h->abuf, h->out, out_stride, h->err, cond,
                     use_cond, h->hs, h->pdl);
    return ok;
  }
  launch_plan(PLAN_DRAFT, h->rows, h->st, h->slot_req, n_slots, B, 0, nullptr, nullptr, cap, h->hs, h->pdl);
  ok &= enqueue_forward(h, PLAN_DRAFT, n_slots, B, 0, h->dbuf, nullptr, h->slot_req);
  launch_override(h->st, h->slot_req, n_slots, B, h->dbuf, h->ref, cap, h->sched, h->sched_cap,
                  h->cfg.vocab, h->hs, h->pdl);
  launch_plan(PLAN_VERIFY, h->rows, h->st, h->slot_req, n_slots, B, 0, h->dbuf, nullptr, cap, h->hs, h->pdl);
  ok &= enqueue_forward(h, PLAN_VERIFY, n_slots, B, 0, h->vbuf, nullptr, h->slot_req);
  launch_accept(h->st, h->slot_req, n_slots, B, h->dbuf, h->vbuf, h->out, out_stride, h->err, cond,
                use_cond, h->hs, h->pdl);
  return ok;
}

int build_graph(gocr_handle* h, GraphEntry& e) {
  CK(cudaGraphCreate(&e.graph, 0));
  cudaGraph_t body = e.graph;
  cudaGraphConditionalHandle ch = 0;
  if (!e.host_loop) {
    CK(cudaGraphConditionalHandleCreate(&ch, e.graph, 1, cudaGraphCondAssignDefault));
    cudaGraphNodeParams np{};
    np.type = cudaGraphNodeTypeConditional;
    np.conditional.handle = ch;
    np.conditional.type = cudaGraphCondTypeWhile;
    np.conditional.size = 1;
    cudaGraphNode_t node;
    CK(cudaGraphAddNode(&node, e.graph, nullptr, nullptr, 0, &np));
    body = np.conditional.phGraph_out[0];
  }
  CK(cudaStreamBeginCaptureToGraph(h->hs, body, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal));
  bool enq = enqueue_round(h, e.mode, e.B, e.n_slots, (unsigned long long)ch, e.host_loop ? 0 : 1);
  cudaError_t le = cudaGetLastError();
  cudaGraph_t captured = nullptr;
  cudaError_t ce = cudaStreamEndCapture(h->hs, &captured);
  if (!enq) return fail(h, GOCR_ECUDA, "kernel launch configuration rejected during capture");
  if (le != cudaSuccess) return fail(h, GOCR_ECUDA, "launch during capture: %s", cudaGetErrorString(le));
  if (ce != cudaSuccess) return fail(h, GOCR_ECUDA, "cudaStreamEndCapture: %s", cudaGetErrorString(ce));
  CK(cudaGraphInstantiate(&e.exec, e.graph, 0));
  return GOCR_OK;
}

int get_graph(gocr_handle* h, int mode, int B, int n_slots, cudaGraphExec_t* exec) {
  for (auto& g : h->graphs)
    if (g.mode == mode && g.B == B && g.n_slots == n_slots) { *exec = g.exec; return GOCR_OK; }
  GraphEntry e{mode, B, n_slots, nullptr, nullptr, h->host_loop};
  int rc = build_graph(h, e);
  if (rc != GOCR_OK && h->pdl) {
    // fall back to plain stream order inside the loop body
    if (e.graph) cudaGraphDestroy(e.graph);
    e.graph = nullptr;
    cudaGetLastError();
    h->pdl = false;
    rc = build_graph(h, e);
  }
  if (rc != GOCR_OK) return rc;
  h->graphs.push_back(e);
  *exec = e.exec;
  return GOCR_OK;
}

int check_req(gocr_handle* h, int req) {
  if (!h) return fail(nullptr, GOCR_EINVAL, "null handle");
  if (req < 0 || req >= h->cfg.max_requests) return fail(h, GOCR_EINVAL, "request slot %d out of range", req);
  return GOCR_OK;
}

// Order the handle's private stream after the caller's stream (NULL = the legacy
// default stream), so inputs the caller produced there are complete.
int sync_user(gocr_handle* h) {
  CK(cudaEventRecord(h->evu, h->user));
  CK(cudaStreamWaitEvent(h->hs, h->evu, 0));
  return GOCR_OK;
}

int read_state(gocr_handle* h, int req, ReqState* out) {
  CK(cudaMemcpyAsync(out, h->st + req, sizeof(ReqState), cudaMemcpyDeviceToHost, h->hs));
  CK(cudaStreamSynchronize(h->hs));
  return GOCR_OK;
}

int dev_err_code(int e) {
  if (e == DERR_ROUND_LIMIT) return GOCR_ETIMEOUT;
  if (e == DERR_CAPACITY) return GOCR_ECAPACITY;
  return GOCR_EDEVICE;
}

const char* dev_err_name(int e) {
  switch (e) {
    case DERR_NAN_LOGITS: return "NaN in logits";
    case DERR_CAPACITY: return "KV capacity exceeded on the device";
    case DERR_ROUND_LIMIT: return "round limit reached";
    case DERR_BAD_TOKEN: return "token id out of range";
    case DERR_TIMEOUT: return "a bounded wait inside a kernel timed out";
    default: return "device error";
  }
}

int run_decode(gocr_handle* h, int n, const int* reqs, int mode, int B, const int* max_new,
               int32_t* const* out_tokens, gocr_stats* stats, float tau = 0.f, int draft_steps = 1,
               float temperature = 0.f, unsigned long long seed = 0) {
  const gocr_config& c = h->cfg;
  if (mode != GOCR_MODE_AR && mode != GOCR_MODE_SELFSPEC && mode != GOCR_MODE_DIFFUSION &&
      mode != GOCR_MODE_REFINED)
    return fail(h, GOCR_EINVAL, "bad mode %d", mode);
  if (n < 1 || n > c.max_requests) return fail(h, GOCR_EINVAL, "bad request count %d", n);
  if (mode != GOCR_MODE_AR && (B < 1 || B > c.max_block))
    return fail(h, GOCR_ECAPACITY, "block size %d outside 1..%d", B, c.max_block);
  if (!(temperature >= 0.f) || temperature > 1e30f) return fail(h, GOCR_EINVAL, "bad temperature");
  const bool sampling = temperature > 0.f;
  if (sampling && mode != GOCR_MODE_AR && mode != GOCR_MODE_SELFSPEC)
    return fail(h, GOCR_EINVAL, "sampling applies to the AR and self-speculative modes");
  if (mode == GOCR_MODE_DIFFUSION || mode == GOCR_MODE_REFINED) {
    if (!(tau == tau)) return fail(h, GOCR_EINVAL, "threshold is NaN");
    if (mode == GOCR_MODE_REFINED && (draft_steps < 1 || draft_steps > GOCR_MAX_BLOCK))
      return fail(h, GOCR_EINVAL, "draft steps %d outside 1..%d", draft_steps, GOCR_MAX_BLOCK);
  }
  if (mode == GOCR_MODE_AR) B = 0;
  int rows = mode == GOCR_MODE_AR ? n : n * (B + 1);
  if (rows > h->T_dec) return fail(h, GOCR_ECAPACITY, "%d rows per forward exceed %d", rows, h->T_dec);
  int bound = 0;
  for (int i = 0; i < n; ++i) {
    int r = check_req(h, reqs[i]);
    if (r) return r;
    for (int j = 0; j < i; ++j)
      if (reqs[j] == reqs[i]) return fail(h, GOCR_EINVAL, "request %d listed twice", reqs[i]);
    if (!h->prefilled[reqs[i]]) return fail(h, GOCR_ESTATE, "request %d has no prefill", reqs[i]);
    if (!out_tokens || !out_tokens[i]) return fail(h, GOCR_EINVAL, "null out_tokens");
    if (max_new[i] < 1 || max_new[i] > h->cap) return fail(h, GOCR_EINVAL, "bad max_new %d", max_new[i]);
    ReqState s;
    int rc = read_state(h, reqs[i], &s);
    if (rc) return rc;
    // prefix length P = cache_len - committed + 1; the last round writes up to P + max_new + B
    int need = (s.cache_len - s.committed + 1) + max_new[i] + B + 2;
    if (need > h->cap)
      return fail(h, GOCR_ECAPACITY, "request %d needs %d KV positions, capacity %d", reqs[i], need, h->cap);
    if (max_new[i] > bound) bound = max_new[i];
  }
  CK(cudaMemcpyAsync(h->slot_req, reqs, sizeof(int) * n, cudaMemcpyHostToDevice, h->hs));
  CK(cudaMemcpyAsync(h->max_new_dev, max_new, sizeof(int) * n, cudaMemcpyHostToDevice, h->hs));
  CK(cudaMemsetAsync(h->err, 0, sizeof(int), h->hs));
  // device-side loop bound: rounds (AR steps) for the two-forward loops;
  // loop iterations (one forward each) for the block-step decodes: at most
  // B denoising steps and one cache write per block of B tokens, or
  // draft_steps draft forwards and one verify per round
  long long iters = bound + 2;
  if (mode == GOCR_MODE_DIFFUSION) iters = (long long)(B + 1) * ((bound + B - 1) / B) + 2;
  if (mode == GOCR_MODE_REFINED) iters = (long long)(draft_steps + 1) * (bound + 2);
  if (iters > (1 << 30)) iters = 1 << 30;
  if (sampling && mode == GOCR_MODE_SELFSPEC && !h->logits_v) {
    h->logits_v = (float*)dev_alloc(h, (size_t)h->T_dec * c.vocab * 4);
    if (!h->logits_v) return fail(h, GOCR_ENOMEM, "device allocation failed");
  }
  launch_begin_decode(h->st, h->slot_req, n, h->max_new_dev, (int)iters, c.eos_id, tau,
                      mode == GOCR_MODE_REFINED ? draft_steps : 1, temperature, seed, h->hs);
  CK(cudaGetLastError());
  cudaGraphExec_t exec;
  int rc = get_graph(h, sampling ? 16 + mode : mode, B, n, &exec);
  if (rc) return rc;
  CK(cudaEventRecord(h->ev0, h->hs));
  if (!h->host_loop) {
    CK(cudaGraphLaunch(exec, h->hs));
  } else {
    // one graph per round; the host polls the done flags after every round
    for (long long round = 0; round < iters; ++round) {
      CK(cudaGraphLaunch(exec, h->hs));
      bool all_done = true;
      for (int i = 0; i < n; ++i) {
        int dn = 0;
        CK(cudaMemcpyAsync(&dn, &h->st[reqs[i]].done, sizeof(int), cudaMemcpyDeviceToHost, h->hs));
        CK(cudaStreamSynchronize(h->hs));
        all_done &= dn != 0;
      }
      if (all_done) break;
    }
  }
  CK(cudaEventRecord(h->ev1, h->hs));
  std::vector<ReqState> sts(n);
  for (int i = 0; i < n; ++i) {
    CK(cudaMemcpyAsync(&sts[i], h->st + reqs[i], sizeof(ReqState), cudaMemcpyDeviceToHost, h->hs));
    CK(cudaMemcpyAsync(out_tokens[i], h->out + (size_t)reqs[i] * h->cap, sizeof(int) * max_new[i],
                       cudaMemcpyDeviceToHost, h->hs));
  }
  CK(cudaStreamSynchronize(h->hs));
  float ms = 0.f;
  CK(cudaEventElapsedTime(&ms, h->ev0, h->ev1));
  int ret = GOCR_OK;
  for (int i = 0; i < n; ++i) {
    const ReqState& s = sts[i];
    if (stats) {
      gocr_stats& o = stats[i];
      o.rounds = s.st_rounds; o.forwards = s.st_forwards; o.committed = s.st_committed;
      o.accepted_drafts = s.st_accepted;
      for (int k = 0; k <= GOCR_MAX_BLOCK; ++k) o.accept_hist[k] = s.hist[k];
      o.device_ms = ms;
    }
    if (s.error && ret == GOCR_OK)
      ret = fail(h, dev_err_code(s.error), "request %d: %s", reqs[i], dev_err_name(s.error));
  }
  return ret;
}

}  // namespace

extern "C" {

int gocr_create(const gocr_config* cfg, const gocr_weights* w, void* stream, gocr_alloc_fn alloc,
                gocr_free_fn free_fn, void* alloc_user, gocr_handle** out) {
  gocr_handle* h = nullptr;
  if (!cfg || !w || !out) return fail(nullptr, GOCR_EINVAL, "null argument");
  *out = nullptr;
  const gocr_config c = *cfg;
  const int q_dim = c.n_q_heads * c.head_dim, kv_dim = c.n_kv_heads * c.head_dim;
  if (c.n_layers < 1 || c.hidden < 128 || c.hidden % 128 || c.hidden > 4096 || c.vocab < 128 || c.vocab % 128 ||
      (c.head_dim != 64 && c.head_dim != 128) || c.n_kv_heads < 1 || c.n_q_heads % c.n_kv_heads ||
      q_dim % 128 || kv_dim % 128 || c.ffn < 64 || c.ffn % 64 ||
      (c.dtype != GOCR_DTYPE_F32 && c.dtype != GOCR_DTYPE_BF16))
    return fail(nullptr, GOCR_EINVAL, "unsupported model shape");
  if (c.max_block < 1 || c.max_block > GOCR_MAX_BLOCK || c.max_requests < 1 || c.max_requests > MAX_REQ ||
      c.max_ctx < c.max_block + 4 || c.max_ctx > (1 << 20) || c.eos_id >= c.vocab)
    return fail(nullptr, GOCR_EINVAL, "bad capacity settings");
  {
    // attention rows (token, q head) of one forward are indexed below 2^20 with at most 64 q heads per kv head
    const long long rows = c.max_ctx > c.max_requests * (c.max_block + 1) ? c.max_ctx : c.max_requests * (c.max_block + 1);
    if (c.n_q_heads / c.n_kv_heads > 64 || rows * (c.n_q_heads / c.n_kv_heads) > (1 << 20))
      return fail(nullptr, GOCR_EINVAL, "more attention rows than supported (q heads per kv head x rows > 2^20)");
  }
  if (!w->embed || !w->mask_embed || !w->lm_head || !w->g_final || !w->layer)
    return fail(nullptr, GOCR_EINVAL, "null weight pointer");
  for (int i = 0; i < c.n_layers * GOCR_LAYER_TENSORS; ++i)
    if (!w->layer[i]) return fail(nullptr, GOCR_EINVAL, "null layer tensor %d", i);
  if ((alloc == nullptr) != (free_fn == nullptr)) return fail(nullptr, GOCR_EINVAL, "alloc and free come together");

  h = new gocr_handle();
  h->cfg = c;
  h->dtype = c.dtype;
  h->es = c.dtype == GOCR_DTYPE_BF16 ? 2 : 4;
  h->af = alloc; h->ff = free_fn; h->au = alloc_user;
  h->user = (cudaStream_t)stream;
  h->q_dim = q_dim; h->kv_dim = kv_dim;
  h->qkv_n = q_dim + 2 * kv_dim;
  h->gu_n = 2 * c.ffn;
  h->cap = c.max_ctx;
  h->T_dec = c.max_requests * (c.max_block + 1);
  h->T_max = h->T_dec > c.max_ctx ? h->T_dec : c.max_ctx;
  h->sched_cap = c.max_ctx;
  h->layer_stride = (long long)c.n_kv_heads * h->cap * c.head_dim;
  h->req_stride = h->layer_stride * c.n_layers;
  *out = h;  // freed by gocr_free on any later failure
#define CKC(call)                                                                  \
  do {                                                                             \
    cudaError_t e_ = (call);                                                       \
    if (e_ != cudaSuccess) {                                                       \
      int r_ = fail(h, GOCR_ECUDA, "%s failed: %s", #call, cudaGetErrorString(e_)); \
      g_lib_error = h->msg; gocr_free(h); *out = nullptr; return r_;               \
    }                                                                              \
  } while (0)
  {
    const char* hl = getenv("GOCR_HOST_LOOP");
    h->host_loop = hl && hl[0] == '1';
    const char* lp = getenv("GOCR_L2_PREFETCH");
    h->l2_prefetch = lp && lp[0] == '1';  // off: measured faster at the decode shapes
    // key-chunk ranks by the rule; GOCR_ATTN_RANKS=<n> replaces the rule's count
    h->attn_ranks = attention_ranks(h->cap, c.max_requests);
    // handles that batch requests run their batched GEMMs on the many-slice
    // kernel, which splits narrow matrices over two CTAs per slice
    h->two_groups = c.max_requests > 1;
    // attention kernels: tcgen05 when a rank averages at least four chunks at
    // full capacity (its heavier tile setup is then amortised: measured 2.8%
    // faster on the 16-request batch), mma.sync otherwise (faster at one or
    // two chunks per rank); GOCR_ATTN=tc | mma overrides
    h->attn_kind = (h->cap + 31) / 32 >= 4 * h->attn_ranks ? ATTN_TCGEN05 : ATTN_MMA_SYNC;
    const char* ak = getenv("GOCR_ATTN");
    if (ak && strcmp(ak, "tc") == 0) h->attn_kind = ATTN_TCGEN05;
    if (ak && strcmp(ak, "mma") == 0) h->attn_kind = ATTN_MMA_SYNC;
    if (c.max_requests <= 1 && h->attn_kind == ATTN_MMA_SYNC) {
      // one request on the mma.sync kernel (64-row tiles, two CTAs per SM):
      // no more ranks than fill two CTAs per SM in one wave for the (kv head,
      // 64-row group) tiles of the handle's largest forward (max_block + 1
      // rows); measured on the table region (2,992 positions, B = 32): 38
      // ranks 1,641 us per round against 48 ranks 1,785 us; on a 65-row draft
      // forward after 2,048 positions: 19 ranks 1,072 us against 38 ranks
      // 1,165 us
      const int fw_rows = c.max_block + 1;
      const int fw_groups = c.n_kv_heads * ((fw_rows * (c.n_q_heads / c.n_kv_heads) + 63) / 64);
      const int wave = 2 * SM_COUNT / (fw_groups > 0 ? fw_groups : 1);
      const int cap_r = wave < ATTN_RANKS_MIN ? ATTN_RANKS_MIN : wave;
      if (h->attn_ranks > cap_r) h->attn_ranks = cap_r;
    }
    const char* ar = getenv("GOCR_ATTN_RANKS");
    if (ar && atoi(ar) >= 1 && atoi(ar) <= 64) h->attn_ranks = atoi(ar) < (h->cap + 31) / 32 ? atoi(ar) : (h->cap + 31) / 32;
  }
  CKC(cudaStreamCreateWithFlags(&h->hs, cudaStreamNonBlocking));
  CKC(cudaEventCreate(&h->ev0));
  CKC(cudaEventCreate(&h->ev1));
  CKC(cudaEventCreateWithFlags(&h->evu, cudaEventDisableTiming));
  CKC(cudaEventRecord(h->evu, h->user));
  CKC(cudaStreamWaitEvent(h->hs, h->evu, 0));

  const int H = c.hidden, R = c.max_requests, T = h->T_max;
  const size_t es = h->es;
  bool ok = true;
  auto A = [&](size_t bytes) { void* p = dev_alloc(h, bytes); if (!p) ok = false; return p; };
  h->embed = w->embed; h->mask = w->mask_embed; h->lm = w->lm_head; h->gfin = w->g_final;
  for (int l = 0; l < c.n_layers; ++l) {
    const void* const* L = w->layer + (size_t)l * GOCR_LAYER_TENSORS;
    void* qkv = A((size_t)h->qkv_n * H * es);
    void* gu = A((size_t)h->gu_n * H * es);
    if (!ok) break;
    CKC(cudaMemcpyAsync(qkv, L[0], (size_t)q_dim * H * es, cudaMemcpyDeviceToDevice, h->hs));
    CKC(cudaMemcpyAsync((char*)qkv + (size_t)q_dim * H * es, L[1], (size_t)kv_dim * H * es,
                        cudaMemcpyDeviceToDevice, h->hs));
    CKC(cudaMemcpyAsync((char*)qkv + (size_t)(q_dim + kv_dim) * H * es, L[2], (size_t)kv_dim * H * es,
                        cudaMemcpyDeviceToDevice, h->hs));
    // gate/up interleaved in groups of 64 rows: [g 64 rows][u 64 rows] ...
    const size_t grp = (size_t)SWIGLU_GROUP * H * es;
    CKC(cudaMemcpy2DAsync(gu, 2 * grp, L[4], grp, grp, c.ffn / SWIGLU_GROUP, cudaMemcpyDeviceToDevice, h->hs));
    CKC(cudaMemcpy2DAsync((char*)gu + grp, 2 * grp, L[5], grp, grp, c.ffn / SWIGLU_GROUP,
                          cudaMemcpyDeviceToDevice, h->hs));
    h->wqkv.push_back(qkv); h->wgu.push_back(gu);
    h->wo.push_back(L[3]); h->wd.push_back(L[6]);
    h->gattn.push_back((const float*)L[7]); h->gmlp.push_back((const float*)L[8]);
  }
  const size_t kv_elems = (size_t)h->req_stride * R;
  const size_t kv_es = h->dtype == GOCR_DTYPE_BF16 ? 2 : 4;
  h->kc_hi = A(kv_elems * kv_es);
  h->vc_hi = A(kv_elems * kv_es);
  h->q_hi = A((size_t)T * q_dim * kv_es);
  if (h->dtype == GOCR_DTYPE_BF16) {
    h->kc_lo = A(kv_elems * kv_es);
    h->vc_lo = A(kv_elems * kv_es);
    h->q_lo = A((size_t)T * q_dim * kv_es);
  }
  if (ok && h->dtype == GOCR_DTYPE_BF16) {
    // the attention's TMA maps over each cache plane: every request, layer and kv head, rows of head_dim values
    const long long rows = (long long)R * c.n_layers * c.n_kv_heads * h->cap;
    const void* planes[4] = {h->kc_hi, h->kc_lo, h->vc_hi, h->vc_lo};
    for (int i = 0; i < 4 && ok; ++i)
      if (rows > 0x7FFFFFFFLL || !encode_tmap_bf16(h->kv_maps[i], planes[i], (int)rows, c.head_dim, 32)) {
        int r_ = fail(h, GOCR_EINVAL, "KV cache too large for the attention's tensor maps");
        g_lib_error = h->msg; gocr_free(h); *out = nullptr; return r_;
      }
  }
  h->resid = (float*)A((size_t)T * H * 4);
  h->xg_hi = A((size_t)T * H * es);
  h->at_hi = A((size_t)T * q_dim * es);
  h->hb_hi = A((size_t)T * c.ffn * es);
  if (h->dtype == GOCR_DTYPE_BF16) {
    h->xg_lo = A((size_t)T * H * es);
    h->at_lo = A((size_t)T * q_dim * es);
    h->hb_lo = A((size_t)T * c.ffn * es);
  }
  h->ssq = (float*)A((size_t)T * (H / NTILE) * 4);
  h->logits = (float*)A((size_t)h->T_dec * c.vocab * 4);
  h->conf_part = (float2*)A((size_t)h->T_dec * (c.vocab / NTILE) * sizeof(float2));
  if (h->dtype == GOCR_DTYPE_BF16) {
    // partial rows of the attention ranks: a prefill (one slot of up to
    // max_ctx rows) or a decode forward (max_requests slots of max_block + 1 rows)
    const int AR = h->attn_ranks;
    const size_t pf = attention_part_floats(1, c.max_ctx, c.n_q_heads, c.n_kv_heads, c.head_dim, AR);
    const size_t df = attention_part_floats(R, c.max_block + 1, c.n_q_heads, c.n_kv_heads, c.head_dim, AR);
    h->att_part = (float*)A((pf > df ? pf : df) * 4);
    const size_t pg = (size_t)c.n_kv_heads * ((c.max_ctx * (c.n_q_heads / c.n_kv_heads) + 63) / 64);
    const size_t dg = (size_t)R * c.n_kv_heads * (((c.max_block + 1) * (c.n_q_heads / c.n_kv_heads) + 63) / 64);
    h->att_chunks = (int*)A((pg > dg ? pg : dg) * 4);
  }
  h->amax = (unsigned long long*)A((size_t)T * 8);
  h->grid_ctr = (int*)A(256);
  h->dbuf = (int*)A((size_t)h->T_dec * 4);
  h->vbuf = (int*)A((size_t)h->T_dec * 4);
  h->abuf = (int*)A((size_t)h->T_dec * 4);
  h->am = (int*)A((size_t)h->T_dec * 4);
  h->rows.plan = (Plan*)A(sizeof(Plan));
  h->rows.row_slot = (int*)A((size_t)T * 4);
  h->rows.row_pos = (int*)A((size_t)T * 4);
  h->rows.row_lim = (int*)A((size_t)T * 4);
  h->rows.row_tok = (int*)A((size_t)T * 4);
  h->rows.logit_row = (int*)A((size_t)T * 4);
  h->slot_req = (int*)A(MAX_REQ * 4);
  h->slot_one = (int*)A(MAX_REQ * 4);
  h->max_new_dev = (int*)A(MAX_REQ * 4);
  h->st = (ReqState*)A(sizeof(ReqState) * R);
  h->out = (int*)A((size_t)R * h->cap * 4);
  h->ref = (int*)A((size_t)R * h->cap * 4);
  h->sched = (int*)A((size_t)R * h->sched_cap * 4);
  h->err = (int*)A(256);
  h->dbg_toks = (int*)A((size_t)h->T_dec * 4);
  h->rope = (float2*)A((size_t)h->cap * (c.head_dim / 2) * sizeof(float2));
  h->prefix_stage = A((size_t)c.max_ctx * H * es);
  // the CUDA-core GEMM of fp32 models reduces its split-K partials through global memory
  if (h->dtype == GOCR_DTYPE_F32) {
    size_t wsf = 0;
    int ctr = 0;
    const int shapes[5][2] = {{h->qkv_n, H}, {H, q_dim}, {h->gu_n, H}, {H, c.ffn}, {c.vocab, H}};
    for (auto& sh : shapes) {
      size_t a = gemm_ws_floats(T, sh[0], sh[1]);
      if (a > wsf) wsf = a;
      int ci = gemm_counter_ints(T, sh[0]);
      if (ci > ctr) ctr = ci;
    }
    h->ws_floats = wsf;
    h->ws = (float*)A(wsf * 4);
    h->counters = (int*)A((size_t)ctr * 4);
  }
  if (h->dtype == GOCR_DTYPE_BF16) {
    const char* ot = getenv("GOCR_OP_TRACE");
    if (ot && (ot[0] == '1' || ot[0] == '2')) {
      h->op_trace_cta = ot[0] == '2';
      h->op_trace = (unsigned long long*)A(op_trace_words(h) * 8);
    }
  }
  if (!ok) {
    int r = fail(h, GOCR_ENOMEM, "device allocation failed");
    g_lib_error = h->msg;
    gocr_free(h);
    *out = nullptr;
    return r;
  }
  launch_rope_table(h->rope, h->cap, c.head_dim, c.rope_theta, h->hs);
  CKC(cudaGetLastError());
  CKC(cudaStreamSynchronize(h->hs));
#undef CKC
  return GOCR_OK;
}

int gocr_prefill(gocr_handle* h, int req, const void* prefix_embeds, int P) {
  int r = check_req(h, req);
  if (r) return r;
  if (!prefix_embeds) return fail(h, GOCR_EINVAL, "null prefix");
  if (P < 1) return fail(h, GOCR_EINVAL, "prefix length %d", P);
  if (P + 1 > h->cap) return fail(h, GOCR_ECAPACITY, "prefix %d exceeds capacity %d", P, h->cap);
  if ((r = sync_user(h))) return r;
  CK(cudaMemcpyAsync(h->prefix_stage, prefix_embeds, (size_t)P * h->cfg.hidden * h->es,
                     cudaMemcpyDefault, h->hs));
  CK(cudaMemcpyAsync(h->slot_one, &req, sizeof(int), cudaMemcpyHostToDevice, h->hs));
  CK(cudaMemsetAsync(h->err, 0, sizeof(int), h->hs));
  launch_plan(PLAN_PREFILL, h->rows, h->st, h->slot_one, 1, 0, P, nullptr, nullptr, h->cap, h->hs, false);
  if (!enqueue_forward(h, PLAN_PREFILL, 1, 0, P, h->am, nullptr, h->slot_one))
    return fail(h, GOCR_ECUDA, "kernel launch configuration rejected");
  launch_prefill_finish(h->st, req, P, h->am, h->out, h->cap, h->hs);
  CK(cudaGetLastError());
  int e = 0;
  CK(cudaMemcpyAsync(&e, h->err, sizeof(int), cudaMemcpyDeviceToHost, h->hs));
  CK(cudaStreamSynchronize(h->hs));
  if (e) return fail(h, dev_err_code(e), "prefill: %s", dev_err_name(e));
  h->prefilled[req] = true;
  return GOCR_OK;
}

int gocr_decode(gocr_handle* h, int req, int mode, int B, int max_new, int32_t* out_tokens,
                gocr_stats* stats) {
  int r = check_req(h, req);
  if (r) return r;
  if ((r = sync_user(h))) return r;
  int32_t* outs[1] = {out_tokens};
  return run_decode(h, 1, &req, mode, B, &max_new, outs, stats);
}

int gocr_decode_batch(gocr_handle* h, int n_req, const int32_t* reqs, int mode, int B,
                      const int32_t* max_new, int32_t* const* out_tokens, gocr_stats* stats) {
  if (!h) return fail(nullptr, GOCR_EINVAL, "null handle");
  if (!reqs || !max_new || !out_tokens) return fail(h, GOCR_EINVAL, "null argument");
  int r = sync_user(h);
  if (r) return r;
  return run_decode(h, n_req, reqs, mode, B, max_new, out_tokens, stats);
}

int gocr_decode_ex(gocr_handle* h, int n_req, const int32_t* reqs, int mode, int B, const gocr_decode_opts* opts,
                   const int32_t* max_new, int32_t* const* out_tokens, gocr_stats* stats) {
  if (!h) return fail(nullptr, GOCR_EINVAL, "null handle");
  if (!reqs || !max_new || !out_tokens) return fail(h, GOCR_EINVAL, "null argument");
  if ((mode == GOCR_MODE_DIFFUSION || mode == GOCR_MODE_REFINED) && !opts)
    return fail(h, GOCR_EINVAL, "mode %d needs options", mode);
  int r = sync_user(h);
  if (r) return r;
  return run_decode(h, n_req, reqs, mode, B, max_new, out_tokens, stats, opts ? opts->tau : 0.f,
                    opts ? opts->draft_steps : 1, opts ? opts->temperature : 0.f, opts ? opts->seed : 0ull);
}

int gocr_set_draft_override(gocr_handle* h, int req, const int32_t* ref_tokens, int n_ref,
                            const int32_t* schedule, int n_rounds) {
  int r = check_req(h, req);
  if (r) return r;
  if (n_ref < 0 || n_ref > h->cap || n_rounds < 0 || n_rounds > h->sched_cap)
    return fail(h, GOCR_ECAPACITY, "override sizes out of range");
  if (n_ref > 0 && (!ref_tokens || (n_rounds > 0 && !schedule)))
    return fail(h, GOCR_EINVAL, "null override array");
  for (int i = 0; i < n_ref; ++i)
    if (ref_tokens[i] < 0 || ref_tokens[i] >= h->cfg.vocab) return fail(h, GOCR_EINVAL, "reference token out of range");
  for (int i = 0; i < n_rounds; ++i)
    if (schedule[i] < 0) return fail(h, GOCR_EINVAL, "negative schedule entry");
  if (n_ref > 0) {
    CK(cudaMemcpyAsync(h->ref + (size_t)req * h->cap, ref_tokens, sizeof(int) * n_ref,
                       cudaMemcpyHostToDevice, h->hs));
    if (n_rounds > 0)
      CK(cudaMemcpyAsync(h->sched + (size_t)req * h->sched_cap, schedule, sizeof(int) * n_rounds,
                         cudaMemcpyHostToDevice, h->hs));
  }
  launch_set_override(h->st, req, n_ref, n_ref > 0 ? n_rounds : 0, h->hs);
  CK(cudaGetLastError());
  CK(cudaStreamSynchronize(h->hs));
  return GOCR_OK;
}

int gocr_debug_forward(gocr_handle* h, int req, int kind, const int32_t* tokens, int n,
                       float* logits_out) {
  return gocr_debug_forward_batch(h, 1, &req, kind, tokens, n, logits_out);
}

int gocr_debug_forward_batch(gocr_handle* h, int n_req, const int32_t* reqs, int kind, const int32_t* tokens,
                             int n, float* logits_out) {
  if (!h) return fail(nullptr, GOCR_EINVAL, "null handle");
  if (!reqs || !tokens) return fail(h, GOCR_EINVAL, "null argument");
  if (n_req < 1 || n_req > h->cfg.max_requests) return fail(h, GOCR_EINVAL, "bad request count %d", n_req);
  int pk, B = 0;
  if (kind == GOCR_FWD_AR) {
    if (n != 1) return fail(h, GOCR_EINVAL, "AR forward takes one token");
    pk = PLAN_AR;
  } else if (kind == GOCR_FWD_DRAFT || kind == GOCR_FWD_VERIFY) {
    B = n - 1;
    if (B < 1 || B > h->cfg.max_block) return fail(h, GOCR_ECAPACITY, "block %d out of range", B);
    pk = kind == GOCR_FWD_DRAFT ? PLAN_DRAFT : PLAN_VERIFY;
  } else {
    return fail(h, GOCR_EINVAL, "bad forward kind %d", kind);
  }
  for (int i = 0; i < n * n_req; ++i)
    if (tokens[i] < 0 || tokens[i] >= h->cfg.vocab) return fail(h, GOCR_EINVAL, "token out of range");
  int r = GOCR_OK;
  for (int i = 0; i < n_req; ++i) {
    if ((r = check_req(h, reqs[i]))) return r;
    for (int j = 0; j < i; ++j)
      if (reqs[j] == reqs[i]) return fail(h, GOCR_EINVAL, "request %d listed twice", reqs[i]);
    if (!h->prefilled[reqs[i]]) return fail(h, GOCR_ESTATE, "request %d has no prefill", reqs[i]);
    ReqState s;
    if ((r = read_state(h, reqs[i], &s))) return r;
    if (s.cache_len + n + 1 > h->cap) return fail(h, GOCR_ECAPACITY, "window exceeds capacity");
  }
  const int n_slots = n_req;
  CK(cudaMemcpyAsync(h->dbg_toks, tokens, sizeof(int) * n * n_req, cudaMemcpyHostToDevice, h->hs));
  CK(cudaMemcpyAsync(h->slot_one, reqs, sizeof(int) * n_req, cudaMemcpyHostToDevice, h->hs));
  CK(cudaMemsetAsync(h->err, 0, sizeof(int), h->hs));
  if (h->op_trace) {
    // aggregate records start at (max, max, 0, ...) for their atomic min / max; per-CTA records at zero
    std::vector<unsigned long long> init(op_trace_words(h));
    for (size_t i = 0; i < init.size(); ++i) init[i] = !h->op_trace_cta && (i % TRACE_WORDS) < 2 ? ~0ull : 0ull;
    CK(cudaMemcpy(h->op_trace, init.data(), init.size() * 8, cudaMemcpyHostToDevice));
    h->op_trace_next = true;
  }
  // GOCR_DEBUG_GRAPH=1: run the forward from a captured graph, as a decode
  // round runs it (a profiling aid: launch timing differs from eager launches)
  const char* dg = getenv("GOCR_DEBUG_GRAPH");
  const bool as_graph = dg && dg[0] == '1';
  cudaGraph_t graph = nullptr;
  if (as_graph) CK(cudaStreamBeginCapture(h->hs, cudaStreamCaptureModeThreadLocal));
  launch_plan(pk, h->rows, h->st, h->slot_one, n_slots, B, 0, nullptr, h->dbg_toks, h->cap, h->hs, false);
  const bool enq = enqueue_forward(h, pk, n_slots, B, 0, h->am, h->logits, h->slot_one);
  h->op_trace_next = false;
  if (as_graph) {
    const cudaError_t ce = cudaStreamEndCapture(h->hs, &graph);
    if (!enq || ce != cudaSuccess) {
      if (graph) cudaGraphDestroy(graph);
      return fail(h, GOCR_ECUDA, "debug forward capture failed");
    }
    cudaGraphExec_t ge = nullptr;
    const cudaError_t ie = cudaGraphInstantiate(&ge, graph, 0);
    cudaGraphDestroy(graph);
    if (ie != cudaSuccess) return fail(h, GOCR_ECUDA, "cudaGraphInstantiate: %s", cudaGetErrorString(ie));
    const cudaError_t le = cudaGraphLaunch(ge, h->hs);
    cudaStreamSynchronize(h->hs);
    cudaGraphExecDestroy(ge);
    if (le != cudaSuccess) return fail(h, GOCR_ECUDA, "cudaGraphLaunch: %s", cudaGetErrorString(le));
  }
  if (!enq) return fail(h, GOCR_ECUDA, "kernel launch configuration rejected");
  CK(cudaGetLastError());
  if (logits_out)
    CK(cudaMemcpyAsync(logits_out, h->logits, sizeof(float) * n * n_req * h->cfg.vocab, cudaMemcpyDeviceToHost,
                       h->hs));
  int e = 0;
  CK(cudaMemcpyAsync(&e, h->err, sizeof(int), cudaMemcpyDeviceToHost, h->hs));
  CK(cudaStreamSynchronize(h->hs));
  if (e) return fail(h, dev_err_code(e), "debug forward: %s", dev_err_name(e));
  return GOCR_OK;
}

int gocr_read_kv(gocr_handle* h, int req, int layer, int pos0, int n, float* k_out, float* v_out) {
  int r = check_req(h, req);
  if (r) return r;
  const gocr_config& c = h->cfg;
  if (layer < 0 || layer >= c.n_layers || pos0 < 0 || n < 0 || pos0 + n > h->cap || !k_out || !v_out)
    return fail(h, GOCR_EINVAL, "bad KV range");
  const size_t d = c.head_dim, Hkv = c.n_kv_heads;
  const bool bf = h->dtype == GOCR_DTYPE_BF16;
  const size_t es = bf ? 2 : 4;
  std::vector<unsigned char> hi(n * Hkv * d * es), lo(bf ? n * Hkv * d * es : 0);
  void* planes[2][2] = {{h->kc_hi, h->kc_lo}, {h->vc_hi, h->vc_lo}};
  float* outs[2] = {k_out, v_out};
  for (int kv = 0; kv < 2; ++kv) {
    for (int p = 0; p < (bf ? 2 : 1); ++p) {
      unsigned char* dst = p ? lo.data() : hi.data();
      for (size_t kvh = 0; kvh < Hkv; ++kvh) {
        size_t off = (size_t)req * h->req_stride + (size_t)layer * h->layer_stride + (kvh * h->cap + pos0) * d;
        CK(cudaMemcpy2DAsync(dst + kvh * d * es, Hkv * d * es, (char*)planes[kv][p] + off * es, d * es, d * es, n,
                             cudaMemcpyDeviceToHost, h->hs));
      }
    }
    CK(cudaStreamSynchronize(h->hs));
    const size_t m = (size_t)n * Hkv * d;
    if (bf) {
      const uint16_t* a = reinterpret_cast<const uint16_t*>(hi.data());
      const uint16_t* b = reinterpret_cast<const uint16_t*>(lo.data());
      for (size_t i = 0; i < m; ++i) {
        uint32_t ua = (uint32_t)a[i] << 16, ub = (uint32_t)b[i] << 16;
        float fa, fb;
        memcpy(&fa, &ua, 4);
        memcpy(&fb, &ub, 4);
        outs[kv][i] = fa + fb;
      }
    } else {
      memcpy(outs[kv], hi.data(), m * 4);
    }
  }
  return GOCR_OK;
}

int gocr_get_state(gocr_handle* h, int req, int32_t* cache_len, int32_t* x0) {
  int r = check_req(h, req);
  if (r) return r;
  ReqState s;
  if ((r = read_state(h, req, &s))) return r;
  if (cache_len) *cache_len = s.cache_len;
  if (x0) *x0 = s.x0;
  return GOCR_OK;
}

int gocr_get_option(const gocr_handle* h, int option, int* value) {
  if (!h || !value) return fail(nullptr, GOCR_EINVAL, "null argument");
  if (option == GOCR_OPT_ATTENTION) {
    *value = h->attn_kind == ATTN_MMA_SYNC ? GOCR_ATTN_MMA_SYNC : GOCR_ATTN_TCGEN05;
    return GOCR_OK;
  }
  if (option == GOCR_OPT_ATTN_RANKS) {
    *value = h->attn_ranks;
    return GOCR_OK;
  }
  return GOCR_EINVAL;
}

int gocr_read_trace(gocr_handle* h, int which, uint64_t* out, size_t n_words) {
  if (!h || !out) return fail(h, GOCR_EINVAL, "null argument");
  if (which != GOCR_TRACE_KERNELS && which != GOCR_TRACE_CTAS) return fail(h, GOCR_EINVAL, "bad trace kind %d", which);
  if (!h->op_trace || h->op_trace_cta != (which == GOCR_TRACE_CTAS))
    return fail(h, GOCR_ESTATE, "this kernel trace is off (GOCR_OP_TRACE=1 or 2 at create)");
  const size_t words = op_trace_words(h);
  if (n_words < words) return fail(h, GOCR_ECAPACITY, "trace needs %zu words", words);
  CK(cudaStreamSynchronize(h->hs));
  CK(cudaMemcpy(out, h->op_trace, words * 8, cudaMemcpyDeviceToHost));
  return GOCR_OK;
}

const char* gocr_last_error(const gocr_handle* h) {
  return h ? h->msg.c_str() : g_lib_error.c_str();
}

void gocr_free(gocr_handle* h) {
  if (!h) return;
  if (h->hs) cudaStreamSynchronize(h->hs);
  for (auto& g : h->graphs) {
    if (g.exec) cudaGraphExecDestroy(g.exec);
    if (g.graph) cudaGraphDestroy(g.graph);
  }
  for (void* p : h->allocs) {
    if (h->ff) h->ff(p, h->au); else cudaFree(p);
  }
  if (h->ev0) cudaEventDestroy(h->ev0);
  if (h->ev1) cudaEventDestroy(h->ev1);
  if (h->evu) cudaEventDestroy(h->evu);
  if (h->hs) cudaStreamDestroy(h->hs);
  delete h;
}

// ---------------------------------------------------------------- single kernels

size_t gocr_op_linear_workspace(int T, int N, int K) {
  if (T < 1 || N < 1 || K < 1) return 0;
  size_t ctr = ((size_t)gemm_counter_ints(T, N) * 4 + 255) & ~(size_t)255;
  return ctr + gemm_ws_floats(T, N, K) * 4 + 256 + (((size_t)T * 8 + 255) & ~(size_t)255);
}

int gocr_op_linear(int dtype, const void* x, const void* w, float* y, int T, int N, int K,
                   void* workspace, size_t workspace_bytes, void* stream) {
  gocr_handle* h = nullptr;
  if (dtype != GOCR_DTYPE_F32 && dtype != GOCR_DTYPE_BF16) return fail(h, GOCR_EINVAL, "bad dtype");
  if (!x || !w || !y || !workspace) return fail(h, GOCR_EINVAL, "null pointer");
  if (T < 1 || N < 1 || K < 8 || K % 8) return fail(h, GOCR_EINVAL, "bad shape T=%d N=%d K=%d", T, N, K);
  if (workspace_bytes < gocr_op_linear_workspace(T, N, K)) return fail(h, GOCR_ECAPACITY, "workspace too small");
  GemmArgs a{};
  a.x = x; a.x_lo = nullptr; a.ldx = K; a.w = w; a.T = T; a.N = N; a.K = K;
  a.kchunk = gemm_kchunk(N, K); a.splits = gemm_splits(N, K); a.kgroup = gemm_kgroup(N, K, false);
  a.counters = (int*)workspace;
  size_t ctr = ((size_t)gemm_counter_ints(T, N) * 4 + 255) & ~(size_t)255;
  a.ws = (float*)((char*)workspace + ctr);
  a.epi = EPI_STORE;
  a.e.y = y; a.e.ldy = N;
  if (!launch_gemm(dtype, a, (cudaStream_t)stream, false))
    return fail(h, GOCR_ECUDA, "kernel launch configuration rejected");
  CK(cudaGetLastError());
  return GOCR_OK;
}

int gocr_op_linear_planes(const void* x_hi, const void* x_lo, const void* w, float* y, int T, int N, int K,
                          void* workspace, size_t workspace_bytes, unsigned flags, void* stream) {
  gocr_handle* h = nullptr;
  if (!x_hi || !x_lo || !w || !y || !workspace) return fail(h, GOCR_EINVAL, "null pointer");
  if (flags & ~GOCR_OP_OVERLAP) return fail(h, GOCR_EINVAL, "unknown flags 0x%x", flags);
  if (T < 1 || N < 1 || K < 8 || K % 8) return fail(h, GOCR_EINVAL, "bad shape T=%d N=%d K=%d", T, N, K);
  if (((uintptr_t)x_hi | (uintptr_t)x_lo | (uintptr_t)w) & 15) return fail(h, GOCR_EINVAL, "operand not 16-byte aligned");
  if (workspace_bytes < gocr_op_linear_workspace(T, N, K)) return fail(h, GOCR_ECAPACITY, "workspace too small");
  GemmArgs a{};
  a.x = x_hi; a.x_lo = x_lo; a.ldx = K; a.w = w; a.T = T; a.N = N; a.K = K;
  a.kchunk = gemm_kchunk(N, K); a.splits = gemm_splits(N, K); a.kgroup = gemm_kgroup(N, K, false);
  a.counters = (int*)workspace;
  size_t ctr = ((size_t)gemm_counter_ints(T, N) * 4 + 255) & ~(size_t)255;
  a.ws = (float*)((char*)workspace + ctr);
  a.epi = EPI_STORE;
  a.e.y = y; a.e.ldy = N;
  if (!launch_gemm(GOCR_DTYPE_BF16, a, (cudaStream_t)stream, (flags & GOCR_OP_OVERLAP) != 0))
    return fail(h, GOCR_ECUDA, "kernel launch configuration rejected");
  CK(cudaGetLastError());
  return GOCR_OK;
}

int gocr_op_attention(int dtype, const void* q_hi, const void* q_lo, const void* k_hi, const void* k_lo,
                      const void* v_hi, const void* v_lo, float* o, const int32_t* lim, int T, int Hq, int Hkv,
                      int d, int cap, void* stream) {
  return gocr_op_attention_ranges(dtype, q_hi, q_lo, k_hi, k_lo, v_hi, v_lo, o, lim, nullptr, nullptr, T, Hq, Hkv,
                                  d, cap, stream);
}

int gocr_three_stream_ranges(int P, int N, int B, int32_t* lim, int32_t* lo2, int32_t* hi2, int32_t* pos) {
  if (P < 0 || N < 0 || B < 1 || (long long)P + 3LL * N > (1 << 28)) return fail(nullptr, GOCR_EINVAL, "bad sizes");
  if (!lim || !lo2 || !hi2) return fail(nullptr, GOCR_EINVAL, "null argument");
  for (int r = 0; r < P + 3 * N; ++r) {
    int l, a = 1, b = 0, p;
    if (r < P) {                     // image + prompt prefix: causal
      l = r;
      p = r;
    } else if (r < P + N) {          // clean response stream: causal over prefix and clean tokens
      l = r;
      p = r;
    } else {                         // corrupted stream s, response token i of block blk
      const int s = (r - P) / N, i = (r - P) % N, blk = i / B;
      l = P + blk * B - 1;           // the prefix and the clean blocks before this one
      a = P + s * N + blk * B;       // its own corrupted block, bidirectionally
      b = P + s * N + (N < (blk + 1) * B ? N : (blk + 1) * B) - 1;
      p = P + i;
    }
    lim[r] = l;
    lo2[r] = a;
    hi2[r] = b;
    if (pos) pos[r] = p;
  }
  return GOCR_OK;
}

// waves of resident attention CTAs that the rank count of a second-interval call fills
static constexpr int OP_R2_WAVES = 2;

int gocr_op_attention_ranges(int dtype, const void* q_hi, const void* q_lo, const void* k_hi, const void* k_lo,
                             const void* v_hi, const void* v_lo, float* o, const int32_t* lim, const int32_t* lo2,
                             const int32_t* hi2, int T, int Hq, int Hkv, int d, int cap, void* stream) {
  gocr_handle* h = nullptr;
  if ((lo2 == nullptr) != (hi2 == nullptr)) return fail(h, GOCR_EINVAL, "lo2 and hi2 come together");
  if (dtype != GOCR_DTYPE_F32 && dtype != GOCR_DTYPE_BF16) return fail(h, GOCR_EINVAL, "bad dtype");
  if (!q_hi || !k_hi || !v_hi || !o || !lim) return fail(h, GOCR_EINVAL, "null pointer");
  if (dtype == GOCR_DTYPE_BF16 && (!q_lo || !k_lo || !v_lo)) return fail(h, GOCR_EINVAL, "missing lo plane");
  if (T < 1 || Hkv < 1 || Hq % Hkv || Hq / Hkv > 64 || (long long)T * (Hq / Hkv) > (1 << 20) || (d != 64 && d != 128) ||
      cap < 1)
    return fail(h, GOCR_EINVAL, "bad shape");
  AttnArgs a{};
  a.q_hi = q_hi; a.q_lo = q_lo; a.k_hi = k_hi; a.k_lo = k_lo; a.v_hi = v_hi; a.v_lo = v_lo;
  a.req_stride = 0; a.o_hi = o; a.o_lo = nullptr; a.out_bf16 = 0;
  a.row_lim = lim; a.plan = nullptr;
  a.row_lo2 = lo2; a.row_hi2 = hi2;
  a.T = T; a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.cap = cap; a.scale = 1.0f / sqrtf((float)d);
  {
    // kernel and key-chunk ranks.  Plain calls: the mma.sync kernel (GOCR_ATTN=tc:
    // tcgen05) over the rule's ranks, which keeps every row's bits the same
    // whatever the number of rows in the call.  Rows with a second key
    // interval (joint-training forwards, one call over the whole packed
    // sequence) take instead no more ranks than fill OP_R2_WAVES waves of the
    // kernel's resident CTAs over its (kv head, row tile) groups (many tiles
    // need few ranks, and each rank costs a partial row set and its merge),
    // and the tcgen05 kernel when its ranks average at least four chunks.
    // GOCR_ATTN=tc / mma forces the kernel; GOCR_ATTN_RANKS=<n> replaces the
    // count (1 .. the rule's).
    const char* ak = getenv("GOCR_ATTN");
    const bool force_tc = ak && strcmp(ak, "tc") == 0, force_mma = ak && strcmp(ak, "mma") == 0;
    const int rule = attention_ranks(cap, 1);
    const int G = Hq / Hkv, n_chunk = (cap + 31) / 32;
    auto r2_ranks = [&](int tile_rows, int per_sm) {
      const long long groups = (long long)Hkv * (((long long)T * G + tile_rows - 1) / tile_rows);
      const long long fill = (OP_R2_WAVES * (long long)per_sm * SM_COUNT + groups - 1) / groups;
      return fill < rule ? (int)fill : rule;
    };
    int R = rule;
    a.kind = force_tc ? ATTN_TCGEN05 : ATTN_MMA_SYNC;
    if (lo2) {
      const int r_tc = r2_ranks(128, 1);
      const bool tc = force_tc || (!force_mma && n_chunk >= 4 * r_tc);
      a.kind = tc ? ATTN_TCGEN05 : ATTN_MMA_SYNC;
      R = tc ? r_tc : r2_ranks(64, 2);
    }
    const char* ar = getenv("GOCR_ATTN_RANKS");
    if (ar && atoi(ar) >= 1) R = atoi(ar) < rule ? atoi(ar) : rule;
    a.ranks = R < 1 ? 1 : R;
  }
  alignas(64) unsigned char maps[4][128];
  if (dtype == GOCR_DTYPE_BF16) {
    // TMA maps over the K and V planes: rows of d values, [Hkv * cap] rows
    const void* planes[4] = {k_hi, k_lo, v_hi, v_lo};
    if ((long long)Hkv * cap > 0x7FFFFFFFLL) return fail(h, GOCR_EINVAL, "bad shape");
    for (int i = 0; i < 4; ++i)
      if (!encode_tmap_bf16(maps[i], planes[i], Hkv * cap, d, 32))
        return fail(h, GOCR_EINVAL, "K/V planes not usable by TMA (16-byte aligned device memory required)");
    a.kv_maps = maps;
    a.kv_row0 = 0;
    a.kv_req_rows = 0;
  }
  if (dtype == GOCR_DTYPE_BF16) {
    // partial rows of the attention ranks: a process-wide scratch buffer per
    // device, grown on demand (calls must not overlap on the GPU)
    static std::mutex mu;
    static std::vector<std::pair<void*, size_t>> bufs(64, {nullptr, 0});
    int dev = 0;
    CK(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return fail(h, GOCR_ECUDA, "device index %d", dev);
    const size_t groups = (size_t)Hkv * ((T * (Hq / Hkv) + 63) / 64);
    const size_t part_bytes =
        (attention_part_floats(1, T, Hq, Hkv, d, attention_ranks(cap, 1)) * 4 + 255) & ~(size_t)255;
    const size_t need = part_bytes + groups * 4;
    std::lock_guard<std::mutex> lk(mu);
    if (bufs[dev].second < need) {
      if (bufs[dev].first) {
        CK(cudaStreamSynchronize((cudaStream_t)stream));
        cudaFree(bufs[dev].first);
      }
      bufs[dev] = {nullptr, 0};
      void* p = nullptr;
      if (cudaMalloc(&p, need) != cudaSuccess) return fail(h, GOCR_ENOMEM, "attention scratch allocation failed");
      bufs[dev] = {p, need};
    }
    a.part = (float*)bufs[dev].first;
    a.part_chunks = (int*)((char*)bufs[dev].first + part_bytes);
  }
  if (!launch_attention(dtype, a, 1, T, (cudaStream_t)stream, false))
    return fail(h, GOCR_ECUDA, "kernel launch configuration rejected");
  CK(cudaGetLastError());
  return GOCR_OK;
}

}  // extern "C"
