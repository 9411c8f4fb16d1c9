/*
 * slm_attn.h -- C ABI of the GB300 (sm_103a) attention hot path for bounded
 * generation: packed variable-length causal GQA prefill, shared-prefix beam
 * decode attention with parent-index suffix reorder, and two-stage beam
 * candidate selection.
 *
 * The operations are those of the article "SLM 生成式高并发推理引擎：延迟约束下的
 * 有效吞吐优化": section 3.1 (packed prefill), section 3.2 (request-internal
 * shared-prefix K/V layout), section 3.3 (beam candidates and state reorder).
 *
 * Conventions (all entry points):
 *   - bf16 is IEEE bfloat16; fp32 is IEEE binary32.  Dense layouts are
 *     row-major and contiguous in the order written, e.g. [T, Hq, D].
 *   - Every tensor pointer is DEVICE memory owned by the caller, 16-byte
 *     aligned.  The library never allocates, frees or keeps a pointer after
 *     the call returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronise, except slm_check_status.
 *     Stream order holds as usual; most kernels are launched as programmatic
 *     dependents of the kernel before them, so their set-up (barriers,
 *     tensor memory) may overlap it, but none reads or writes global memory
 *     before everything earlier on the stream has completed.
 *   - Arguments that can be checked on the host are; a bad one returns a
 *     status other than SLM_OK, sets a thread-local message readable with
 *     slm_last_error(), and enqueues nothing.  No call throws, aborts or traps.
 *   - Conditions only the device can see (a malformed sequence boundary, an
 *     out-of-range parent index, a stuck pipeline) make the kernel skip or
 *     finish early and OR a bit into *dev_status (when non-NULL); the affected
 *     outputs are then undefined.
 *   - Query head h reads KV head h / (Hq / Hkv): contiguous head groups.
 *   - Supported: head_dim 64 or 128; Hq % Hkv == 0; Hq / Hkv <= 128.
 */
#ifndef SLM_ATTN_H_
#define SLM_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SLM_OK = 0,
  SLM_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, aliasing, bad host boundary */
  SLM_ERR_UNSUPPORTED = 2,   /* valid request outside what the kernels implement */
  SLM_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed (message has the CUDA error) */
  SLM_ERR_WORKSPACE = 4,     /* workspace missing or smaller than the *_workspace_size query */
  SLM_ERR_DEVICE_CHECK = 5   /* slm_check_status found device-side error bits */
} slm_status;

/* Device status bits (OR-ed into *dev_status by kernels). */
#define SLM_DEV_BAD_SEQLENS 1        /* cu_seqlens not non-decreasing from 0 to total_tokens */
#define SLM_DEV_BAD_PARENT 2         /* a parent index outside [0, W) */
#define SLM_DEV_PIPELINE_TIMEOUT 4   /* an in-kernel bounded wait ran out (kernel ended early) */
#define SLM_DEV_BOUNDS 8             /* debug-bounds builds only (-DSLM_DEBUG_BOUNDS): an index a
                                        kernel computed lay outside its buffer; the access was skipped */

/* Thread-local description of the last failure on this thread ("" if none). */
const char* slm_last_error(void);

/* ABI version of this header (incremented on incompatible changes). */
int32_t slm_abi_version(void);

/*
 * Packed variable-length causal GQA prefill attention (article section 3.1).
 *
 *   q  bf16 [T, Hq, D], k / v bf16 [T, Hkv, D]: the valid tokens of all
 *      sequences packed back to back (no padding);
 *   cu_seqlens int32 [num_seqs + 1] (device): sequence boundary, prefix sums
 *      of the lengths, cu_seqlens[0] = 0, cu_seqlens[num_seqs] = T =
 *      total_tokens; equal neighbours are allowed (empty sequences);
 *   cu_seqlens_host (nullable): host copy of the same; when given it is
 *      validated on the host (monotone, ends at T, lengths <= max_seqlen);
 *   max_seqlen >= every length (sizes the schedule);
 *   softmax_scale > 0 multiplies q.k before the softmax (1/sqrt(D) usually).
 *
 *   o   bf16 [T, Hq, D] (may not alias q, k, v):
 *       o[t, h] = sum_j softmax_j(scale * q[t,h] . k[j, h/G]) v[j, h/G]
 *       over the tokens j of t's own sequence with j <= t (block-diagonal
 *       causal mask); fp32 accumulation and fp32 online softmax.
 *   lse (nullable) fp32 [Hq, T]: natural-log log-sum-exp of the scaled scores.
 *
 *   workspace: device scratch of at least slm_prefill_workspace_size(...)
 *   bytes (the schedule of query tiles).  dev_status: nullable device int32.
 */
slm_status slm_packed_prefill_attn(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                                   const int32_t* cu_seqlens_host, int32_t num_seqs, int32_t total_tokens,
                                   int32_t max_seqlen, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                   float softmax_scale, void* o, float* lse, void* workspace, size_t workspace_bytes,
                                   int32_t* dev_status, void* stream);

/* Workspace bytes slm_packed_prefill_attn needs for these sizes (0 = unsupported). */
size_t slm_prefill_workspace_size(int32_t num_seqs, int32_t total_tokens, int32_t max_seqlen, int32_t n_q_heads,
                                  int32_t n_kv_heads);

/*
 * Shared-prefix beam decode attention with parent-index suffix reorder
 * (article sections 3.2 and 3.3).
 *
 *   q      bf16 [W, Hq, D]: one query token per beam, in the NEW beam order;
 *   kp, vp bf16 [Lp, Hkv, D]: the prompt K/V, one copy shared by all beams
 *          (nullable when Lp == 0);
 *   ks, vs bf16 [W, Smax, Hkv, D]: suffix K/V of the previous step, rows
 *          s < L_prev valid, in the PREVIOUS beam order;
 *   k_new, v_new bf16 [W, Hkv, D] (nullable together): K/V of each beam's
 *          new token, new order; when NULL nothing is appended;
 *   parent_idx int32 [W] (device, nullable = identity): new beam b continues
 *          previous beam parent_idx[b], 0 <= parent_idx[b] < W.
 *
 *   ks_out, vs_out bf16 [W, Smax, Hkv, D] (must not alias ks/vs): reordered
 *          suffix, ks_out[b, s] = ks[parent_idx[b], s] for s < L_prev and
 *          ks_out[b, L_prev] = k_new[b]; rows s >= L_s are not written.
 *   o      bf16 [W, Hq, D]: o[b, h] = Attention(q[b, h],
 *          [kp[:, h/G]; ks_out[b, :L_s, h/G]], [vp ...; vs_out ...]) with
 *          L_s = L_prev + (k_new != NULL); the concatenation is never built:
 *          prefix and suffix contributions meet in one fp32 online-softmax
 *          state.  The prompt K/V is never reordered or copied.
 *   lse    (nullable) fp32 [W, Hq].
 *
 *   workspace (nullable): device scratch, 16-byte aligned, of
 *          workspace_bytes bytes, ZERO-FILLED before its first use.  With at
 *          least slm_shared_prefix_decode_workspace_size(...) bytes the
 *          prompt's key blocks may be split over several CTAs (their partial
 *          softmax states merged before the suffix); with less, or NULL, they
 *          are not split.  The result is the same up to fp32 summation order.
 *          A call that completes leaves the workspace fit for the next call,
 *          of any sizes (its tickets back at zero); after a call whose
 *          dev_status reports a pipeline timeout, zero it again (a unit that
 *          gave up never takes its ticket).  The caller owns the memory and
 *          must not share it between calls in flight at the same time.
 *   dev_status: nullable device int32 (bad parent index, pipeline timeout).
 *
 * Requires Lp + L_s >= 1 and L_s <= Smax.
 */
slm_status slm_shared_prefix_decode_attn(const void* q, const void* kp, const void* vp, const void* ks,
                                         const void* vs, const void* k_new, const void* v_new,
                                         const int32_t* parent_idx, int32_t W, int32_t Lp, int32_t L_prev,
                                         int32_t Smax, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                         float softmax_scale, void* ks_out, void* vs_out, void* o, float* lse,
                                         int32_t* dev_status, void* workspace, size_t workspace_bytes,
                                         void* stream);

/* Workspace bytes that let slm_shared_prefix_decode_attn split the prompt's
 * key blocks for these sizes (0 = it never splits them: Lp <= 128 or
 * unsupported sizes). */
size_t slm_shared_prefix_decode_workspace_size(int32_t W, int32_t Lp, int32_t n_q_heads, int32_t n_kv_heads,
                                               int32_t head_dim);

/*
 * Two-stage beam candidate selection (article section 3.3).
 *
 *   logits bf16 [W_in, V]: next-token logits of the W_in current beams
 *          (W_in = 1 at the first step, else the beam width);
 *   cum_scores fp32 [W_in]: cumulative beam scores;
 *   W: beams to keep, 1 <= W and 2W <= V.
 *
 *   Per beam the 2W largest logits (ties: lower token id) give the token
 *   ids; their scores are read from the FP32 log-softmax over the full
 *   vocabulary, lp = fl32(x - lse_b) with lse_b the fp32 log-sum-exp of the
 *   row, plus the beam's cumulative score, score = fl32(cum_b + lp).  The
 *   W_in x 2W candidates are flattened and the global 2W best kept in order:
 *   higher score first, equal scores by lower flat index (lower parent, then
 *   the beam's own order).
 *
 *   out_token / out_parent int32 [W], out_score fp32 [W]: the first W (the
 *   next beams; parent = source beam of each);
 *   out_cand_token / out_cand_parent int32 [2W], out_cand_score fp32 [2W]
 *   (each nullable): all 2W global candidates, for setting finished beams
 *   aside;  out_lse (nullable) fp32 [W_in]: lse_b.
 *
 *   workspace: at least slm_beam_select_workspace_size(W_in, V, W) bytes.
 */
slm_status slm_beam_select(const void* logits, const float* cum_scores, int32_t W_in, int32_t V, int32_t W,
                           int32_t* out_token, int32_t* out_parent, float* out_score, int32_t* out_cand_token,
                           int32_t* out_cand_parent, float* out_cand_score, float* out_lse, void* workspace,
                           size_t workspace_bytes, void* stream);

/* Workspace bytes slm_beam_select needs (0 = unsupported sizes). */
size_t slm_beam_select_workspace_size(int32_t W_in, int32_t V, int32_t W);

/*
 * Fused SwiGLU and per-token dynamic E4M3 re-quantisation (article section
 * 3.4, the MLP data path between the FP8 Gate/Up and Down GEMMs): one pass
 * per token row, without a BF16 SwiGLU intermediate.
 *
 *   gate_up bf16 [T, 2*I]: row t holds gate_t [I] then up_t [I] (the Gate/Up
 *           GEMM output);
 *   q       E4M3 (OCP FP8, one byte per element) [T, I]: codes of
 *           h_t * (448 / amax_t), rounded to nearest even and saturated to
 *           +-448, where h_t = SiLU(gate_t) * up_t in FP32 and amax_t =
 *           max |h_t|;
 *   scale   fp32 [T]: amax_t / 448 (so h_t ~= code * scale); a row with
 *           amax_t = 0 gets scale 1 and all-zero codes.
 *
 * Requires I % 8 == 0.  No workspace.
 */
slm_status slm_swiglu_quant_e4m3(const void* gate_up, int32_t T, int32_t I, void* q, float* scale, void* stream);

/*
 * Last-valid-token extraction and label scoring for Prefill-Only models
 * (article sections 1.1 and 3.1): the same sequence boundary as the packed
 * prefill selects each sequence's last row of hidden states; its next-token
 * logits are computed for the label tokens only, and a softmax over the
 * labels gives the scores.
 *
 *   hidden     bf16 [total_tokens, d_model]: final hidden states, packed;
 *   cu_seqlens int32 [num_seqs + 1] (device): sequence boundaries;
 *   w_label    bf16 [n_labels, d_model]: the label tokens' rows of the
 *              prediction head;
 *   logits     fp32 [num_seqs, n_labels]: z_bk = sum_j h_b[j] * w_k[j], FP32
 *              accumulation, h_b = hidden[cu_seqlens[b+1] - 1];
 *   probs      fp32 [num_seqs, n_labels] (nullable): softmax of z_b over k.
 *
 * A sequence of length 0 gets NaN logits and probs.  A malformed boundary
 * (decreasing, or outside [0, total_tokens]) gives NaN for that sequence and
 * sets SLM_DEV_BAD_SEQLENS in *dev_status (nullable).  Requires
 * 1 <= n_labels <= 32 and d_model % 8 == 0.
 */
slm_status slm_label_scores(const void* hidden, const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                            int32_t d_model, const void* w_label, int32_t n_labels, float* logits, float* probs,
                            int32_t* dev_status, void* stream);

/*
 * Finished-beam handling with the 2W global candidates (article section
 * 3.3: the intermediate step keeps 2W global candidates so that sequences
 * that produced the stop token can be set aside while W active beams go on).
 *
 *   cand_token / cand_parent int32 [2W], cand_score fp32 [2W]: the global
 *              candidates in order, as slm_beam_select writes them;
 *   out_token / out_parent int32 [W], out_score fp32 [W]: the first W
 *              candidates whose token is not stop_id, in order -- the next
 *              active beams;
 *   fin_token / fin_parent int32 [W], fin_score fp32 [W]: the candidates
 *              ranked among the first W whose token is stop_id, in order --
 *              the hypotheses finished at this step; fin_count int32 [1]:
 *              how many.
 *
 * Each beam's row holds the stop token once, so at most W_in <= W
 * candidates are stops and W active beams always remain.  Requires
 * 1 <= W <= 1024.
 */
slm_status slm_beam_split_finished(const int32_t* cand_token, const int32_t* cand_parent, const float* cand_score,
                                   int32_t W, int32_t stop_id, int32_t* out_token, int32_t* out_parent,
                                   float* out_score, int32_t* fin_token, int32_t* fin_parent, float* fin_score,
                                   int32_t* fin_count, void* stream);

/*
 * Token-history reorder of fixed-depth beam search (article section 2.3: the
 * generated token sequence is one of the states the parent index reorders
 * each step).
 *
 *   hist_in  int32 [W_in, max_len]: tokens of the current beams, columns
 *            0..t-1 valid (may be NULL when t == 0);
 *   parent_idx int32 [W] (device; NULL = identity): source beam of each new
 *            beam, in [0, W_in);
 *   token    int32 [W]: the new beams' tokens;
 *   hist_out int32 [W, max_len]: hist_out[b, s] = hist_in[parent[b], s] for
 *            s < t and hist_out[b, t] = token[b]; must not alias hist_in.
 *
 * When t > 0, a parent outside [0, W_in) reads row 0 and sets
 * SLM_DEV_BAD_PARENT in *dev_status (nullable); at t = 0 no row is read and
 * the parent index is ignored.  Requires 0 <= t < max_len.
 */
slm_status slm_beam_reorder_history(const int32_t* hist_in, const int32_t* parent_idx, const int32_t* token,
                                    int32_t W, int32_t W_in, int32_t t, int32_t max_len, int32_t* hist_out,
                                    int32_t* dev_status, void* stream);

/*
 * slm_packed_prefill_attn without a workspace argument.  The article has no
 * counterpart; this entry point exists for callers that cannot allocate
 * device memory where they run attention (a frozen ahead-of-time compiled
 * graph with a fixed memory plan, a host that owns all allocation, a hot path
 * on which allocation is forbidden).
 *
 * Arguments and results are those of slm_packed_prefill_attn.  The tile
 * schedule is kept in a 192 KiB array of this library's own device memory
 * that every GPU which loads the library holds until the process exits.
 *   - Limit: total_tokens / (2 * (128 / (n_q_heads / n_kv_heads))) +
 *     num_seqs + 1 <= 16383 work items (e.g. 130,000 tokens in 240 sequences
 *     with 16 query / 8 KV heads use about 1,260); larger requests return
 *     SLM_ERR_UNSUPPORTED and enqueue nothing.
 *   - The first call on each device looks up the array's device address (no
 *     allocation); make that first call before any stream capture.
 *   - All calls share the one array and each overwrites it: calls that can
 *     overlap on the GPU (different streams without ordering) race and give
 *     wrong results.  Nothing needs clearing between calls.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.
 */
slm_status slm_packed_prefill_attn_noalloc(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                                           const int32_t* cu_seqlens_host, int32_t num_seqs, int32_t total_tokens,
                                           int32_t max_seqlen, int32_t n_q_heads, int32_t n_kv_heads,
                                           int32_t head_dim, float softmax_scale, void* o, float* lse,
                                           int32_t* dev_status, void* stream);

/*
 * Test/debug helper: synchronises `stream`, reads *dev_status and returns
 * SLM_ERR_DEVICE_CHECK (message lists the bits) if it is non-zero, else
 * SLM_OK.  Does not clear the word.
 */
slm_status slm_check_status(const int32_t* dev_status, void* stream);

/*
 * Test and diagnostic variants with an fp32 output (article section 3.1:
 * FP32 online softmax; section 3.2 for decode).  Arguments, validation,
 * kernels and results are those of slm_packed_prefill_attn and
 * slm_shared_prefix_decode_attn, except that o is fp32 with the same layout
 * ([T, Hq, D] and [W, Hq, D]) and receives each row's fp32 result before any
 * bf16 rounding.  They exist so that an accuracy bound can be checked on the
 * attention arithmetic itself, without the output's bf16 rounding; prefill
 * writes rows with plain stores here instead of TMA stores.
 */
slm_status slm_packed_prefill_attn_f32(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                                       const int32_t* cu_seqlens_host, int32_t num_seqs, int32_t total_tokens,
                                       int32_t max_seqlen, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                       float softmax_scale, float* o, float* lse, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_status, void* stream);
slm_status slm_shared_prefix_decode_attn_f32(const void* q, const void* kp, const void* vp, const void* ks,
                                             const void* vs, const void* k_new, const void* v_new,
                                             const int32_t* parent_idx, int32_t W, int32_t Lp, int32_t L_prev,
                                             int32_t Smax, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                             float softmax_scale, void* ks_out, void* vs_out, float* o, float* lse,
                                             int32_t* dev_status, void* workspace, size_t workspace_bytes,
                                             void* stream);

/*
 * Test and diagnostic control of the attention kernels' bounded waits (the
 * failure detection that article section 2.5 asks of the serving path: bounded
 * waiting rather than a hang).  Every wait of a pipeline stage inside the
 * prefill and decode attention kernels gives up after `ns` nanoseconds; the
 * kernel then drains the copies and tensor-core work it issued, frees its
 * tensor memory, ends early and sets SLM_DEV_PIPELINE_TIMEOUT (outputs
 * undefined).  The default is 1 s.  ns = 0 makes every wait that is not
 * already complete give up at once, which forces that path in a test.
 * Process-wide; read when a call is enqueued (a captured CUDA graph keeps the
 * value of its capture).  Returns the previous value.  Draining itself always
 * allows 1 s.
 */
uint64_t slm_set_wait_timeout_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* SLM_ATTN_H_ */
