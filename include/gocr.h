/*
 * gocr.h - C ABI of the GB300 self-speculative block decoder.
 *
 * The library runs the decode round of a decoder trained for both AR and
 * block-diffusion decoding (GravityOCR, "Diffusion Drafts, AR Verifies"):
 *
 *   draft   one forward of [x0, M x B]: the boundary token x0 reads the cache
 *           causally and yields a0; the B [M] rows read the cache and the whole
 *           window bidirectionally and yield drafts d1..dB
 *           (GravityOCR review, §3.2 "Self-Speculative Decoding");
 *   verify  one token-causal forward of [a0, d1..dB] yields a1..a(B+1) and
 *           overwrites the draft's KV slots with causal state in place
 *           (review, Appendix B.2 "Self-Speculative Decoding and KV-Cache Update");
 *   accept  A = longest prefix with d_j == a_j; commit a0, d1..dA, a(A+1);
 *           the rejected suffix is rolled back (velog review, inference section).
 *
 * Everything runs on one GPU in hand-written sm_103a kernels.  All entry points
 * return GOCR_OK (0) or a negative GOCR_E* code; nothing throws across the ABI.
 * A handle is not thread-safe: calls on one handle must not overlap.
 *
 * Layouts: every matrix is row-major [out, in] (y = x W^T), elements in the
 * handle's dtype (fp32, or bf16 as uint16 bit patterns).  Norm gains are fp32.
 */
#ifndef GOCR_H
#define GOCR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define GOCR_OK          0
#define GOCR_EINVAL     (-1) /* bad argument: null pointer, size out of range   */
#define GOCR_ECAPACITY  (-2) /* KV capacity, rows or block size over the limit  */
#define GOCR_ECUDA      (-3) /* a CUDA runtime call failed (see gocr_last_error) */
#define GOCR_EDEVICE    (-4) /* a kernel raised its error word (NaN logits ...)  */
#define GOCR_ETIMEOUT   (-5) /* the on-device round loop hit its round limit     */
#define GOCR_ENOMEM     (-6) /* allocation failed                                */
#define GOCR_ESTATE     (-7) /* call order: decode before prefill, and the like  */

enum { GOCR_DTYPE_F32 = 0, GOCR_DTYPE_BF16 = 1 };
/* decode modes: AR greedy (one token per forward), self-speculative rounds,
 * and (gocr_decode_ex) direct block diffusion and self-speculative rounds
 * with a refined draft */
enum { GOCR_MODE_AR = 0, GOCR_MODE_SELFSPEC = 1, GOCR_MODE_DIFFUSION = 2, GOCR_MODE_REFINED = 3 };
/* single-forward kinds for gocr_debug_forward */
enum { GOCR_FWD_AR = 0, GOCR_FWD_DRAFT = 1, GOCR_FWD_VERIFY = 2 };

#define GOCR_MAX_BLOCK 64      /* largest block size B */
#define GOCR_LAYER_TENSORS 9   /* wq wk wv wo wg wu wd g_attn g_mlp */

/* Model and capacity.  q_dim = n_q_heads*head_dim and kv_dim =
 * n_kv_heads*head_dim must be multiples of 128, head_dim 64 or 128, ffn a
 * multiple of 64, hidden and vocab multiples of 128, n_q_heads a multiple of
 * n_kv_heads. */
typedef struct gocr_config {
  int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
  int32_t dtype;          /* GOCR_DTYPE_F32 | GOCR_DTYPE_BF16 */
  float rms_eps;          /* RMSNorm epsilon (1e-6) */
  float rope_theta;       /* rotary base (1e4) */
  int32_t max_ctx;        /* KV positions per request: >= P + max_new + B + 2 */
  int32_t max_block;      /* largest B the handle will be asked for (<= 64) */
  int32_t max_requests;   /* request slots (KV caches) */
  int32_t eos_id;         /* stop token, -1 = none */
} gocr_config;

/* Device pointers to the weights.  The caller owns them and keeps them alive
 * until gocr_free; the handle copies the projections it re-packs (QKV fused,
 * gate/up interleaved) at create time and reads the others in place. */
typedef struct gocr_weights {
  const void* embed;        /* [vocab, hidden] dtype */
  const void* mask_embed;   /* [hidden] dtype: the single [M] row */
  const void* lm_head;      /* [vocab, hidden] dtype (untied) */
  const float* g_final;     /* [hidden] fp32 */
  /* host array of n_layers * GOCR_LAYER_TENSORS device pointers, per layer:
   * wq [Hq*d, h], wk [Hkv*d, h], wv [Hkv*d, h], wo [h, Hq*d], wg [F, h],
   * wu [F, h], wd [h, F] (dtype), g_attn [h], g_mlp [h] (fp32) */
  const void* const* layer;
} gocr_weights;

/* Decode statistics (review §4.1 eq. 5: TPF = committed / forwards, the
 * prefill excluded; a round with A accepted drafts commits A + 2 tokens). */
typedef struct gocr_stats {
  int64_t rounds;           /* self-spec rounds, or AR steps                  */
  int64_t forwards;         /* draft + verify forwards (AR: one per token)    */
  int64_t committed;        /* decode-committed tokens (prefill token not in) */
  int64_t accepted_drafts;  /* sum of A over rounds                          */
  int32_t accept_hist[GOCR_MAX_BLOCK + 1]; /* rounds per accepted count A    */
  double device_ms;         /* device time of the decode call (CUDA events)  */
} gocr_stats;

/* Optional device allocator (for example backed by PyTorch's caching
 * allocator).  Must return 256-byte-aligned device memory or NULL. */
typedef void* (*gocr_alloc_fn)(size_t bytes, void* user);
typedef void (*gocr_free_fn)(void* ptr, void* user);

typedef struct gocr_handle gocr_handle;

/* Create a decoder on the current CUDA device.
 *   stream      cudaStream_t every launch goes to (NULL = legacy default).
 *   alloc/free  device allocator; both NULL = cudaMalloc/cudaFree.
 * Returns GOCR_EINVAL for an unsupported shape (including more than 64 q
 * heads per kv head, or more than 2^20 attention rows (token, q head) in one
 * forward: max(max_ctx, max_requests x (max_block + 1)) x q heads per kv
 * head), GOCR_ENOMEM, GOCR_ECUDA. */
int gocr_create(const gocr_config* cfg, const gocr_weights* w, void* stream,
                gocr_alloc_fn alloc, gocr_free_fn free_fn, void* alloc_user,
                gocr_handle** out);

/* Causal prefill of request slot `req` from P prefix embeddings (the image +
 * prompt prefix, [P, hidden] in dtype; host or device pointer, copied before
 * the call returns).  Resets the slot: the argmax of the last row becomes
 * out[0] and the boundary token x0; the cache holds positions 0..P-1.
 * GOCR_ECAPACITY if P + 1 > max_ctx. */
int gocr_prefill(gocr_handle* h, int req, const void* prefix_embeds, int P);

/* Decode request `req` until max_new tokens are in out (out[0], the prefill
 * token, counts) or eos.  mode GOCR_MODE_AR commits one token per forward;
 * GOCR_MODE_SELFSPEC runs draft/verify/accept rounds of block size B.  The
 * whole loop runs on the device (a CUDA graph with a device-side while loop,
 * no host synchronisation between rounds); the call blocks until it ends and
 * then copies out_tokens (host, caller-owned, >= max_new entries) and stats
 * (may be NULL).  GOCR_ECAPACITY if P + max_new + B + 2 > max_ctx. */
int gocr_decode(gocr_handle* h, int req, int mode, int B, int max_new,
                int32_t* out_tokens, gocr_stats* stats);

/* Batched decode of n_req prefilled request slots in one round loop: every
 * forward concatenates the requests' windows (ragged caches, one position
 * sequence per request).  max_new[i] per request; out_tokens[i] host buffers;
 * stats: array of n_req or NULL.  Finished requests stop committing while
 * the others continue. */
int gocr_decode_batch(gocr_handle* h, int n_req, const int32_t* reqs, int mode, int B,
                      const int32_t* max_new, int32_t* const* out_tokens, gocr_stats* stats);

/* Options of the block-step decodes. */
typedef struct gocr_decode_opts {
  float tau;            /* DIFFUSION: the confidence threshold tau_c; REFINED: the
                           draft-side threshold.  Confidence = the largest softmax
                           probability of a row; a value equal to tau passes. */
  int32_t draft_steps;  /* REFINED: draft forwards per round at most, 1..64 */
  float temperature;    /* AR, SELFSPEC: 0 = greedy; > 0 = sampling from
                           softmax(logits / temperature) (see below) */
  uint32_t reserved;    /* 0 */
  uint64_t seed;        /* sampling: key of the random numbers */
} gocr_decode_opts;

/* gocr_decode_batch with every mode, one forward per device-loop iteration
 * for the two block-step modes (opts required for them, ignored otherwise):
 *
 *   GOCR_MODE_DIFFUSION  direct block-diffusion decoding (GravityOCR review,
 *     §2 "Block Diffusion" and Appendix B.1 "Direct Block-Diffusion
 *     Decoding"): a block of B slots at positions p+1..p+B starts as [M];
 *     each denoising step forwards the draft window [x0, slots] (x0 causal,
 *     the slots reading the cache and the whole window) and fixes every masked
 *     slot whose confidence reaches tau (slot s takes the argmax of the row at
 *     position p+s-1, the shift-by-one convention), or else the single most
 *     confident masked slot (the lowest slot among equals).  A finished block
 *     commits its B tokens (cut at max_new and after the first eos); unless
 *     decoding stops there, a token-causal cache-write forward of [x0,
 *     y_1..y_B] at p..p+B follows, the cache keeps positions 0..p+B-1 and
 *     y_B becomes the boundary.  Stats: rounds = blocks, forwards = denoising
 *     steps + cache writes, accept_hist[k] = blocks finished in k steps,
 *     accepted_drafts = 0.
 *   GOCR_MODE_REFINED  self-speculative rounds whose draft runs up to
 *     draft_steps denoising forwards (review Appendix D, "Draft Schedule"):
 *     each step fixes slots by the rule above with the draft-side threshold;
 *     after the last step (or when every slot is fixed) the verify window is
 *     [slot 1..slot B, the last step's prediction at position p+B+1], unfixed
 *     slots taking the last step's predictions; verify, accept and rollback
 *     are those of GOCR_MODE_SELFSPEC, so the output equals AR greedy.
 *     draft_steps = 1 is the one-shot round (the same tokens, stats and bits
 *     as GOCR_MODE_SELFSPEC).  Stats: forwards = draft steps + verifies.
 *
 *   Sampling (GOCR_MODE_AR or GOCR_MODE_SELFSPEC with temperature > 0): the
 *     decode tokens are drawn from softmax(logits / temperature) (the
 *     prefill token stays the greedy argmax).  Self-speculative rounds then
 *     use the speculative acceptance-rejection rule (review §2 "Speculative
 *     Decoding"; the blog: the rule preserves the AR distribution): a0 is
 *     drawn from the boundary row, d_j from [M] row j (draft distribution
 *     q_j); verify row j - 1 gives the target p_j; d_j is accepted when a
 *     uniform u_j < min(1, p_j(d_j) / q_j(d_j)); the first rejection draws
 *     the replacement from max(0, p_j - q_j) renormalised, B acceptances
 *     draw the bonus from verify row B; commit and rollback as in the greedy
 *     round.  Random numbers: Philox4x32-10 (Salmon et al., SC 2011), key
 *     (seed low word, seed high word), counter (v / 4, position, purpose,
 *     request slot), lane v % 4, uniform ((x >> 9) + 0.5) / 2^23; a draw is
 *     a Gumbel-max, argmax of score_v - log(-log u_v) with the lowest index
 *     among equals; purposes 0 a target token at its position (AR steps, a0,
 *     the bonus), 1 a draft token, 2 an acceptance uniform (v = 0), 3 a
 *     replacement; the token at absolute position t uses position t.
 *
 * No forced-acceptance override applies to the block-step modes or to
 * sampling.  Errors as gocr_decode_batch; GOCR_EINVAL for a NaN threshold,
 * draft_steps out of range, a negative or NaN temperature, or a temperature
 * with the block-step modes. */
int gocr_decode_ex(gocr_handle* h, int n_req, const int32_t* reqs, int mode, int B, const gocr_decode_opts* opts,
                   const int32_t* max_new, int32_t* const* out_tokens, gocr_stats* stats);

/* Forced-acceptance hook for request `req` (host arrays, copied):  in round r
 * with c tokens committed, drafts become d_j = ref[c+j] for j <= G_r and
 * d_(G_r+1) = (ref[c+G_r+1] + 1) mod vocab, G_r = schedule[r] (rounds past
 * n_rounds use G = 0; positions past n_ref keep the model's draft).
 * n_ref = 0 removes the hook.  Applied between draft and verify. */
int gocr_set_draft_override(gocr_handle* h, int req, const int32_t* ref_tokens, int n_ref,
                            const int32_t* schedule, int n_rounds);

/* One forward at the request's current state, for parity checks; nothing is
 * committed and cache_len is unchanged (KV slots at and after cache_len are
 * written).  kind AR: tokens = [x], n = 1, at position cache_len.  DRAFT:
 * tokens[0] = x0 and n = B + 1 (rows 1..B are [M]), positions cache_len.. .
 * VERIFY: tokens = [a0, d1..dB], n = B + 1, positions cache_len+1.. (call it
 * after a DRAFT at the same state, which wrote x0's slot).  logits_out: host
 * [n, vocab] fp32, or NULL. */
int gocr_debug_forward(gocr_handle* h, int req, int kind, const int32_t* tokens, int n,
                       float* logits_out);

/* gocr_debug_forward over n_req prefilled request slots in one batched
 * forward, as gocr_decode_batch runs its rounds: request i's window is rows
 * [i n, (i + 1) n) with tokens[i n .. (i + 1) n) (same per-kind meaning as
 * above, each at its own request's cache length), and logits_out (host, or
 * NULL) receives [n_req n, vocab] fp32 in that row order.  The requests are
 * distinct; GOCR_ECAPACITY when a window does not fit its cache. */
int gocr_debug_forward_batch(gocr_handle* h, int n_req, const int32_t* reqs, int kind, const int32_t* tokens,
                             int n, float* logits_out);

/* Copy n cached positions from pos0 of layer `layer` to host buffers
 * k_out/v_out, each [n, n_kv_heads, head_dim] fp32 (keys are stored rotated;
 * bf16 models keep the cache as bf16 hi + lo planes, returned as their sum). */
int gocr_read_kv(gocr_handle* h, int req, int layer, int pos0, int n, float* k_out, float* v_out);

/* Current cache length (position of the boundary token) and boundary token. */
int gocr_get_state(gocr_handle* h, int req, int32_t* cache_len, int32_t* x0);

/* Read-only handle properties.
 *   GOCR_OPT_ATTENTION  the tensor-core attention kernels of a bf16 handle,
 *                     fixed at create time:
 *     GOCR_ATTN_MMA_SYNC  64-row tiles on mma.sync;
 *     GOCR_ATTN_TCGEN05  128-row tiles with both contractions on tcgen05 and
 *       their accumulators in tensor memory.
 *   A handle takes TCGEN05 when its key-chunk ranks average at least four
 *   32-key chunks at full capacity (batched handles), MMA_SYNC otherwise;
 *   GOCR_ATTN=tc or GOCR_ATTN=mma in the environment at create time
 *   overrides (gocr_op_attention reads it per call; MMA_SYNC by default).
 *   The two round differently; each is bit-consistent across its own
 *   forwards.
 *   GOCR_OPT_ATTN_RANKS  key-chunk ranks of the handle's attention (the
 *                     split of a row's keys, fixed at create time).
 * GOCR_EINVAL for an unknown option. */
enum { GOCR_OPT_ATTENTION = 5, GOCR_OPT_ATTN_RANKS = 6 };
enum { GOCR_ATTN_TCGEN05 = 0, GOCR_ATTN_MMA_SYNC = 1 };
int gocr_get_option(const gocr_handle* h, int option, int* value);

/* Timeline of the last debug forward (a profiling aid; GOCR_ESTATE when the
 * trace is off).  out: host, at least n_words words.
 *   GOCR_TRACE_KERNELS  one record per launch of a debug forward (on with
 *     GOCR_OP_TRACE=1 in the environment at create time): n_words >=
 *     8 * (5 * n_layers + 1), laid out [launch][8] in forward order (per
 *     layer QKV, attention, O, gate/up, down; then the LM head); a record is
 *     (first CTA start, first and last release from the dependency wait,
 *     last CTA end, last mainloop end, last split-K exchange end, 0, 0),
 *     globaltimer ns (the last two marks for GEMMs only). */
/*   GOCR_TRACE_CTAS  the same launches with one record per CTA (on with
 *     GOCR_OP_TRACE=2): n_words >= 8 * 2048 * (5 * n_layers + 1), laid out
 *     [launch][CTA slot][8]; CTA c of a kernel (linear block index) fills slot
 *     c, the attention merge kernel's CTAs slots 1024 + c; a record is (start,
 *     release from the dependency wait, GEMM epilogue start, end, then as the
 *     launch records: mainloop end, split-K exchange end, cluster barrier
 *     passed, accumulator drained; attention: first chunk ready, chunk loop
 *     done, merge start), zero where a CTA did not reach a mark. */
enum { GOCR_TRACE_KERNELS = 1, GOCR_TRACE_CTAS = 2 };
int gocr_read_trace(gocr_handle* h, int which, uint64_t* out, size_t n_words);

/* Last error message of the handle (or of the library when h is NULL). */
const char* gocr_last_error(const gocr_handle* h);

void gocr_free(gocr_handle* h);

/* ---- single-kernel entry points (parity tests, device pointers) --------- */

/* y[T, N] (fp32) = x[T, K] w[N, K]^T, the decoder's weight-streaming GEMM with
 * its fixed split-K reduction (the split count depends on N and K only, so a
 * row's result does not depend on T).  x and w in dtype, K % 8 == 0.
 * workspace: device, >= gocr_op_linear_workspace(T, N, K) bytes, all zero
 * before the first call (the kernel leaves it ready for the next call). */
size_t gocr_op_linear_workspace(int T, int N, int K);
int gocr_op_linear(int dtype, const void* x, const void* w, float* y, int T, int N, int K,
                   void* workspace, size_t workspace_bytes, void* stream);

/* y[T, N] (fp32) = (x_hi + x_lo)[T, K] w[N, K]^T with bf16 planes x_hi,
 * x_lo and bf16 w: the decoder's GEMM on the hi + lo activation planes its
 * epilogues write (each K chunk takes the hi and the lo products as separate
 * tensor-core accumulators, adds them, and the chunk sums are added in chunk
 * order).  Up to two 128-row token slices split each tile's K chunks over a
 * thread-block cluster; more rows run them in one CTA per 64-token slice.
 * Either way a row's bits depend on neither T nor the kernel that ran it.  K % 8 == 0; x_hi, x_lo,
 * w 16-byte aligned.  workspace: as gocr_op_linear.
 * flags: 0, or GOCR_OP_OVERLAP: launched as the decoder launches it, with
 * programmatic dependent launch, so that it may start while the stream's
 * previous kernel finishes.  It then fetches w before that kernel has
 * completed (x_hi, x_lo and y only after): w must not be written by it.
 * Errors: GOCR_EINVAL (null pointer, shape, flags), GOCR_ECAPACITY
 * (workspace), GOCR_ECUDA (launch). */
#define GOCR_OP_OVERLAP 1u
int gocr_op_linear_planes(const void* x_hi, const void* x_lo, const void* w, float* y, int T, int N, int K,
                          void* workspace, size_t workspace_bytes, unsigned flags, void* stream);

/* Grouped-query attention of one request window against a KV cache, the
 * decoder's kernel for that dtype.  Operands are planes, as the decoder keeps
 * them: for GOCR_DTYPE_BF16, bf16 hi and lo arrays with v = hi + lo (tensor
 * cores, about 16 significant bits); for GOCR_DTYPE_F32, fp32 arrays in *_hi
 * with the lo pointers NULL.  q [T, Hq, d], k and v [Hkv, cap, d] (device);
 * o [T, Hq, d] fp32 (device); lim: device int32[T], row t reads keys
 * 0..lim[t] (draft: row 0 = p, rows 1..B = p+B; verify/AR: the row's own
 * position).  d in {64, 128}; Hq / Hkv <= 64 and T x Hq / Hkv <= 2^20
 * (GOCR_EINVAL otherwise).  GOCR_DTYPE_BF16 reads K and V by TMA: the four
 * K/V planes must be 16-byte aligned (GOCR_EINVAL otherwise).  GOCR_DTYPE_BF16 keeps its partial rows in a
 * device scratch buffer of the library (one per device, allocated or grown
 * by the first call that needs more): calls that overlap on the GPU race. */
int gocr_op_attention(int dtype, const void* q_hi, const void* q_lo, const void* k_hi, const void* k_lo,
                      const void* v_hi, const void* v_lo, float* o, const int32_t* lim, int T, int Hq, int Hkv,
                      int d, int cap, void* stream);

/* gocr_op_attention with a second key interval per row: row t reads keys
 * 0..lim[t] and lo2[t]..hi2[t] (none when hi2[t] < lo2[t]); lo2, hi2:
 * device int32[T], both NULL = the plain call.  With lo2/hi2 given, the
 * bf16 path splits each row tile's keys over fewer ranks as T grows (at most
 * two waves of the kernel's resident CTAs) and runs the tcgen05 kernel when
 * its ranks average at least four 32-key chunks, else the mma.sync kernel
 * (GOCR_ATTN=tc / mma forces one): a row's result then depends on T in its
 * last bits (the plain call's does not).  Key chunks masked for every row of
 * a tile are skipped, which changes no bits. */
int gocr_op_attention_ranges(int dtype, const void* q_hi, const void* q_lo, const void* k_hi, const void* k_lo,
                             const void* v_hi, const void* v_lo, float* o, const int32_t* lim, const int32_t* lo2,
                             const int32_t* hi2, int T, int Hq, int Hkv, int d, int cap, void* stream);

/* Row key intervals of the joint AR / block-diffusion training attention
 * (GravityOCR review §3.1 "Joint AR-Diffusion Training"; the Trillion Labs
 * blog's three-stream figure): one forward over the packed sequence
 * [prefix (P), clean response (N), corrupted stream 1 (N), corrupted stream
 * 2 (N)], responses cut into blocks of B tokens.  The prefix (image and
 * prompt, never corrupted) and the clean stream are causal; a token of block
 * b of a corrupted stream reads the prefix, the clean blocks before b and
 * the whole of its own corrupted block b (bidirectional), and nothing of the
 * other corrupted stream, of its own stream's other blocks, or of clean
 * block b and later.  Host outputs, [P + 3 N] each: lim, lo2, hi2 as
 * gocr_op_attention_ranges reads them, and pos (or NULL) the rotary
 * position of each row (a stream's response token i sits at P + i).
 * GOCR_EINVAL for negative sizes, B < 1, or a null output. */
int gocr_three_stream_ranges(int P, int N, int B, int32_t* lim, int32_t* lo2, int32_t* hi2, int32_t* pos);

/* ---- allocation-free GEMM ------------------------------------------------ */

/* Bytes of the device scratch array behind gocr_op_linear_static (per GPU). */
#define GOCR_STATIC_SCRATCH_BYTES (16u << 20)

/* gocr_op_linear for callers that cannot allocate device memory: a plug-in
 * whose host application owns every allocation, a real-time loop that may not
 * enter the allocator, a sandbox that forbids cudaMalloc.  Same arguments,
 * layouts and results as gocr_op_linear, but no workspace: the split-K partial
 * sums and tile counters live in one file-scope device array of
 * GOCR_STATIC_SCRATCH_BYTES that every GPU loading this library keeps until
 * the process exits.  GravityOCR has no counterpart: this is a deployment
 * convenience of this library.
 *   - Calls nothing that allocates (no cudaMalloc/cudaFree, no library
 *     allocator): it clears the counters with cudaMemsetAsync and launches.
 *   - GOCR_ECAPACITY when gocr_op_linear_workspace(T, N, K) exceeds
 *     GOCR_STATIC_SCRATCH_BYTES (message in gocr_last_error(NULL)).
 *   - The first call on a device looks up the array's device address with
 *     that device current and caches it; make that first call before any
 *     stream capture.  Under lazy module loading (the CUDA default) that
 *     first call is also where the driver reserves the array on the device,
 *     and it fails with GOCR_ECUDA if the device has no room for it; from
 *     the second call on, nothing is reserved.
 *   - `stream` must belong to the current device (GOCR_EINVAL otherwise).
 *   - All calls on a device share the array and it keeps the last call's
 *     contents: calls that overlap on the GPU (other streams, other threads)
 *     race; order them on one stream. */
int gocr_op_linear_static(int dtype, const void* x, const void* w, float* y, int T, int N, int K,
                          void* stream);

#ifdef __cplusplus
}
#endif
#endif /* GOCR_H */
