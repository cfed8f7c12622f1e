/*
 * tokengate.h -- C ABI of libtokengate.so, the TokenGate pruned-prefill hot
 * path on NVIDIA B300 (sm_103a).
 *
 * TokenGate (MarkTechPost article "Researchers from Stanford and UC Berkeley
 * introduce TokenGate", section "How does TokenGate's learned token pruning
 * work?") splits the prefill forward pass in three phases: the layers below
 * the gate layer L run on all N tokens; at layer L a small MLP scores every
 * token from its post-attention residual and a top-K selector keeps the
 * highest-scoring ones (only the document is prunable, the question is never
 * pruned); the layers above L run on the kept tokens only and create no KV
 * entries for the pruned ones.  Section "What is token-gated attention?": the
 * kept token's score becomes a bias on the attention logits above the gate,
 * refined by a learnable per-head gain and a learnable temperature.
 *
 * The calls below are the steps of that path, in order:
 *   tg_gate_score -> tg_topk_select -> tg_gather_kept -> (per layer)
 *   tg_qkv_rope_bf16 (the Q/K/V projection with RoPE fused into it) ->
 *   tg_gated_attention_rotated -> [tg_linear_bf16 for the output projection
 *   with the residual add].
 * When q, k and v come from elsewhere, tg_gated_attention_fwd (=
 * tg_rope_qk -> tg_gated_attention_rotated) rotates them itself.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument is DEVICE memory, allocated and owned by the
 *   caller, unless stated otherwise.  The library allocates no device memory
 *   on any compute call; scratch space is passed in as `workspace`.
 * - bf16 tensors are dense row-major arrays of 16-bit bfloat16 values; base
 *   pointers of bf16 matrices must be 16-byte aligned.
 * - Packed (varlen) layout: the rows of the `batch` sequences are
 *   concatenated; sequence b owns rows [cu_seqlens[b], cu_seqlens[b+1]).  Each
 *   sequence is its document (the first n_doc[b] rows) followed by its
 *   question (the remaining rows).
 * - Calls are asynchronous on `stream` and never synchronise.  Arguments are
 *   validated on the host before anything is launched: an invalid argument
 *   returns an error status and launches nothing.  Conditions that only the
 *   device can see (an index out of range, a device-side wait that timed out)
 *   are recorded in a device status word, read by tg_check_device_status().
 * - Thread safety: calls may be issued from several host threads; the last
 *   error string is per thread.
 */
#ifndef TOKENGATE_H_
#define TOKENGATE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define TG_API __attribute__((visibility("default")))
#else
#define TG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TG_OK = 0,
  TG_ERR_INVALID_ARG = 1,   /* bad pointer, size, shape or alignment        */
  TG_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head_dim 96) */
  TG_ERR_WORKSPACE = 3,     /* workspace missing or too small               */
  TG_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed            */
  TG_ERR_TIMEOUT = 5,       /* a device-side wait exceeded its cycle limit  */
  TG_ERR_DEVICE_INDEX = 6   /* a device-side index/size check failed        */
} tg_status;

/*
 * Gate MLP scores (gate module, "How does TokenGate's learned token pruning
 * work?", second phase; the spec fixes the algebra).  For every DOCUMENT row j:
 *     z_j = w2 . GELU(W1 x_j + b1) + b2,   s_j = logsigmoid(z_j)
 * with the exact-erf GELU; for every QUESTION row s_j = +0.0.
 *
 *   x_bf16     [n_rows, d] bf16, the gate-layer residuals (packed layout)
 *   n_rows     total rows; must equal cu_seqlens[batch]
 *   d          hidden size, multiple of 64, 64 <= d <= 65536
 *   cu_seqlens [batch+1] int32, device
 *   n_doc      [batch] int32, device; 0 <= n_doc[b] <= seqlen_b
 *   w1_bf16    [h, d] bf16 (nn.Linear layout)
 *   b1         [h] fp32 or NULL (zero)
 *   w2_bf16    [h] bf16
 *   b2         scalar
 *   h          hidden width, multiple of 16, 16 <= h <= 256
 *   s_out      [n_rows] fp32 output
 *   topk_ws    NULL, or the workspace of the tg_topk_select call that will
 *              read these scores (tg_topk_workspace_size(batch) bytes,
 *              16-byte aligned, batch <= 65535): the gate's epilogue then
 *              also counts each sequence's scores into the histograms that
 *              give the top-K its first two radix digits
 *   topk_ws_bytes  its size
 * Bf16 inputs, fp32 accumulation on the tensor cores, fp32 epilogue.
 * Device-side errors: n_doc out of range -> TG_ERR_DEVICE_INDEX (those rows
 * are then left unwritten).
 */
TG_API tg_status tg_gate_score(const void* x_bf16, int64_t n_rows, int32_t d,
                        const int32_t* cu_seqlens, const int32_t* n_doc, int32_t batch,
                        const void* w1_bf16, const float* b1, const void* w2_bf16, float b2,
                        int32_t h, float* s_out, void* topk_ws, size_t topk_ws_bytes,
                        cudaStream_t stream);

/*
 * Bytes of the top-K workspace for `batch` sequences (0 for batch outside
 * [1, 65535]): per sequence, counts of the scores' top 8 and top 16 bits of
 * their order key (1 KB + 256 KB).  Host-only, no CUDA call.
 */
TG_API size_t tg_topk_workspace_size(int32_t batch);

/*
 * Top-K selection (same section: "a top-K selector keeps the tokens with the
 * highest score"; "only the document part of the prompt is prunable, the
 * question is never pruned").  For each sequence b with K_b = min(k[b],
 * n_doc[b]): the K_b document rows with the largest s (ties broken towards the
 * lower row index; -0.0 equals +0.0; NaN ranks below every number), written
 * in ascending row order, followed by every question row of b in order.
 * Row ids are global (packed) row numbers.  k[b] > n_doc[b] keeps the whole
 * document; k[b] = 0 keeps the question only.
 *
 *   s           [n_rows] fp32 scores
 *   cu_seqlens  [batch+1] int32, n_doc [batch] int32, k [batch] int32 (device)
 *   max_n_doc   host-side upper bound on every n_doc[b] (sizes the launch);
 *               a larger n_doc[b] on the device -> TG_ERR_DEVICE_INDEX
 *   kept_idx    [sum_b T_b] int32 output, T_b = min(k[b], n_doc[b]) + n_q[b]
 *   cu_kept     [batch+1] int32 output, prefix sums of T_b
 *   workspace   NULL, or tg_topk_workspace_size(batch) bytes (16-byte
 *               aligned, batch <= 65535) that held zeros when first
 *               allocated.  When the tg_gate_score call that produced s was
 *               given the same workspace (and s is unchanged since), its
 *               score histograms give the selection its first two radix
 *               digits and it runs two passes instead of four.  The call
 *               zeroes the histograms of every
 *               sequence it completes, ready for the next gate call.  Counts
 *               that do not match n_doc (a gate call whose histograms no
 *               top-K consumed, or none at all) select with the four passes;
 *               the result is the same either way.  Calls that share one
 *               workspace must not overlap on the GPU.
 *   ws_bytes    its size
 * Exact integer result: bit-identical to the definition for any input.
 * The kernel is launched early behind the previous kernel in the stream
 * (programmatic dependent launch) and waits for it before touching memory.
 */
TG_API tg_status tg_topk_select(const float* s, int64_t n_rows, const int32_t* cu_seqlens,
                         const int32_t* n_doc, const int32_t* k, int32_t batch,
                         int32_t max_n_doc, int32_t* kept_idx, int32_t* cu_kept,
                         void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * General prunable spans (the prompt template marks the prunable text; with
 * several marked spans, the document need not be a prefix).  A per-row mask
 * replaces n_doc: prunable [n_rows] uint8, nonzero = prunable.  The reading
 * taken: the gate scores the prunable rows (0 on every other row), a
 * sequence's budget k[b] goes to its prunable rows, and every other row is
 * kept; with the mask equal to the document prefix both calls give exactly
 * the results of tg_gate_score and tg_topk_select.
 *
 * tg_gate_score_masked: as tg_gate_score, with s = 0 on rows outside the
 *   mask.  The sequence arguments serve only the top-K workspace: with
 *   topk_ws (tg_topk_workspace_size(batch) bytes, zero on entry, as for
 *   tg_gate_score) the gate also counts each sequence's prunable scores for
 *   the masked top-K's first two radix digits, and needs cu_seqlens [batch+1]
 *   and batch >= 1; with topk_ws NULL both are ignored.
 *
 * tg_topk_select_masked: per sequence b, the min(k[b], n_prunable[b])
 *   prunable rows with the largest score (ties: lower row first) together with
 *   every row outside the mask, in ascending row order; cu_kept as in
 *   tg_topk_select.
 *   max_len        host upper bound on every sequence's length (sizes the launch)
 *   kept_capacity  length of kept_idx; a sequence whose kept rows would end
 *                  past it writes nothing and sets TG_ERR_DEVICE_INDEX
 *   n_prunable     [batch] int32 output: prunable rows per sequence (also the
 *                  call's scratch: written by a counting kernel, then read)
 *   workspace      NULL, or the top-K workspace a tg_gate_score_masked call
 *                  with the same cu_seqlens filled (its first two digits come
 *                  from there; cleared again for the next gate call)
 *   The total kept count is cu_kept[batch] = sum_b min(k[b], n_prunable[b]) +
 *   (length_b - n_prunable[b]); a caller that does not know the mask on the
 *   host can size kept_idx by n_rows.
 */
TG_API tg_status tg_gate_score_masked(const void* x_bf16, int64_t n_rows, int32_t d,
                               const uint8_t* prunable, const void* w1_bf16,
                               const float* b1, const void* w2_bf16, float b2, int32_t h,
                               float* s_out, const int32_t* cu_seqlens, int32_t batch, void* topk_ws,
                               size_t topk_ws_bytes, cudaStream_t stream);
TG_API tg_status tg_topk_select_masked(const float* s, int64_t n_rows, const int32_t* cu_seqlens,
                                const uint8_t* prunable, const int32_t* k, int32_t batch,
                                int32_t max_len, int64_t kept_capacity, int32_t* kept_idx,
                                int32_t* cu_kept, int32_t* n_prunable, void* workspace,
                                size_t ws_bytes, cudaStream_t stream);

/*
 * Gather of the kept rows (third phase: the layers above L run on the kept
 * tokens only).  For kept slot i of sequence b:
 *     x_kept[i] = X[kept_idx[i]],  pos_kept[i] = kept_idx[i] - cu_seqlens[b],
 *     s_kept[i] = s[kept_idx[i]]
 *
 *   x_bf16 [n_rows, d] bf16; s [n_rows] fp32; cu_seqlens [batch+1];
 *   n_rows  rows of x and s (kept ids at or beyond it are flagged, not read)
 *   kept_idx [n_kept], cu_kept [batch+1] as written by tg_topk_select
 *   n_kept  host-side total kept rows (= cu_kept[batch])
 *   x_kept_bf16 [n_kept, d] bf16, pos_kept [n_kept] int32, s_kept [n_kept]
 *   fp32 outputs; any of the three may be NULL to skip it.
 * d is a multiple of 8 and x_bf16, x_kept_bf16 are 16-byte aligned (rows
 * are moved by the bulk-copy engine through shared memory); otherwise
 * TG_ERR_INVALID_ARG.
 * A kept index outside its sequence -> TG_ERR_DEVICE_INDEX, row skipped.
 * The kernel is launched early behind the previous kernel in the stream
 * (programmatic dependent launch) and waits for it before reading anything.
 */
TG_API tg_status tg_gather_kept(const void* x_bf16, int64_t n_rows, int32_t d, const float* s,
                         const int32_t* cu_seqlens, const int32_t* kept_idx,
                         const int32_t* cu_kept, int32_t batch, int64_t n_kept,
                         void* x_kept_bf16, int32_t* pos_kept, float* s_kept,
                         cudaStream_t stream);

/*
 * Token-gated causal attention over the kept tokens ("What is token-gated
 * attention?"; the spec fixes the algebra).  For kept row i of sequence b and
 * query head h, with G = hq / hkv and g = floor(h / G):
 *   logit_ij = (q'_i,h . k'_j,g) / (sqrt(head_dim) * tau) + gain[h] * s_kept[j]
 * over the kept rows j of b with pos_kept[j] <= pos_kept[i];
 *   o_i,h = sum_j softmax_j(logit_ij) v_j,g,   lse[h, i] = ln sum_j exp(logit_ij)
 * where q' and k' are q and k rotated by rotate-half RoPE at the ORIGINAL
 * positions pos_kept with base rope_theta (1e6 for Qwen3).
 *
 *   q  [n_kept, hq, head_dim] bf16;  k, v [n_kept, hkv, head_dim] bf16
 *   pos_kept [n_kept] int32, STRICTLY increasing within each sequence (as
 *            tg_gather_kept writes it); otherwise TG_ERR_DEVICE_INDEX
 *   s_kept [n_kept] fp32;  gain [hq] fp32;  tau > 0;  rope_theta > 0
 *   cu_kept [batch+1] int32 (device);  max_kept: host upper bound on every
 *            sequence's kept length (sizes the launch)
 *   hq % hkv == 0, hq / hkv even or 1; head_dim in {64, 128}
 *   o      [n_kept, hq, head_dim] bf16 output
 *   lse    [hq, n_kept] fp32 output (natural log), or NULL
 *   k_cache [n_kept, hkv, head_dim] bf16 output: the rotated keys k' (the
 *            kept-only KV cache), or NULL (then kept in the workspace)
 *   workspace of at least tg_attention_workspace_size(...) bytes, 256-byte
 *            aligned; holds q' (and k' when k_cache is NULL)
 * Rounding: q', k' and the softmax probabilities are rounded to bf16 before
 * the tensor-core products; accumulation and softmax are fp32.
 */
TG_API tg_status tg_gated_attention_fwd(const void* q, const void* k, const void* v,
                                 const int32_t* pos_kept, const float* s_kept,
                                 const float* gain, float tau, float rope_theta,
                                 const int32_t* cu_kept, int32_t batch, int64_t n_kept,
                                 int32_t max_kept, int32_t hq, int32_t hkv, int32_t head_dim,
                                 void* o, float* lse, void* k_cache,
                                 void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/*
 * The two steps of tg_gated_attention_fwd as separate calls, for a caller
 * that keeps the rotated keys (a kept-only KV cache) or times the steps.
 *
 * tg_rope_qk: q' and k', q and k rotated by rotate-half RoPE at the ORIGINAL
 * positions pos_kept with base rope_theta (the angle pos * theta^(-2i/D) is
 * formed and reduced in fp64, its sine and cosine taken in fp32), rounded to
 * bf16.  Also checks that pos_kept is non-negative and strictly increasing
 * within each sequence; otherwise TG_ERR_DEVICE_INDEX.
 *   q [n_kept, hq, head_dim], k [n_kept, hkv, head_dim] bf16 inputs;
 *   q_out, k_out of the same shapes, bf16 outputs (must not alias the inputs);
 *   cu_kept [batch+1] int32 (device); head_dim in {64, 128}.
 */
TG_API tg_status tg_rope_qk(const void* q, const void* k, const int32_t* pos_kept, float rope_theta,
                     const int32_t* cu_kept, int32_t batch, int64_t n_kept, int32_t hq,
                     int32_t hkv, int32_t head_dim, void* q_out, void* k_out,
                     cudaStream_t stream);

/*
 * tg_gated_attention_rotated: the attention of tg_gated_attention_fwd on
 * inputs already rotated by tg_rope_qk (q_rot [n_kept, hq, head_dim], k_rot
 * [n_kept, hkv, head_dim] bf16); every other argument as there.  Needs no
 * workspace.  The kernel also checks that pos_kept strictly increases within
 * each sequence (its causal tile skipping relies on it); otherwise
 * TG_ERR_DEVICE_INDEX.
 */
TG_API tg_status tg_gated_attention_rotated(const void* q_rot, const void* k_rot, const void* v,
                                     const int32_t* pos_kept, const float* s_kept,
                                     const float* gain, float tau, const int32_t* cu_kept,
                                     int32_t batch, int64_t n_kept, int32_t max_kept,
                                     int32_t hq, int32_t hkv, int32_t head_dim, void* o,
                                     float* lse, cudaStream_t stream);

/* Bytes of workspace tg_gated_attention_fwd needs (q' and, if no k_cache is
 * given, k').  Host-only, no CUDA call. */
TG_API size_t tg_attention_workspace_size(int64_t n_kept, int32_t hq, int32_t hkv,
                                   int32_t head_dim, int32_t has_k_cache);

/*
 * Backward of token-gated attention with respect to the score-side parameters
 * (the gradient path from the attention loss back to the gate: section "What
 * is token-gated attention?" makes the kept score a bias g_h s_j on the
 * logits, with a learnable gain per head and a learnable temperature).  For
 * the loss L = sum_{i,h} dO[i,h,:] . o[i,h,:] it writes
 *   d_s[j]    = dL/ds_j  = sum_h gain_h sum_i dl_ij
 *   d_gain[h] = dL/dg_h  = sum_{i,j} s_j dl_ij
 *   d_tau[0]  = dL/dtau  = -sum_{h,i,j} dl_ij (q'_i . k'_j) / (sqrt(D) tau^2)
 * with P = softmax of the forward's logits, dP_ij = dO_i . v_j, D_i = dO_i . o_i
 * and dl_ij = P_ij (dP_ij - D_i).  dq, dk and dv are not computed.  A key
 * whose score is -inf has P = 0 and adds nothing to d_gain.
 *
 *   q_rot [n_kept, hq, head_dim], k_rot [n_kept, hkv, head_dim] bf16: the
 *            rotated q' and k' the forward used (tg_rope_qk's outputs; k_rot
 *            is the kept-only K cache)
 *   v [n_kept, hkv, head_dim] bf16;  o [n_kept, hq, head_dim] bf16 and
 *   lse [hq, n_kept] fp32: the forward's outputs (tg_gated_attention_rotated)
 *   d_o [n_kept, hq, head_dim] bf16: the upstream gradient dL/do
 *   pos_kept, s_kept, gain, tau, cu_kept, batch, n_kept, max_kept, hq, hkv,
 *            head_dim: as for the forward; hq / hkv <= 8, hq <= 256; positions strictly
 *            increasing within each sequence (the forward checks it)
 *   d_s [n_kept], d_gain [hq], d_tau [1]: fp32 device outputs (d_s is 0 for
 *            rows outside every sequence)
 *   workspace of at least tg_attention_bwd_workspace_size(n_kept, hq) bytes,
 *            256-byte aligned
 * All pointers are caller-owned device memory; q_rot, k_rot, v, o and d_o
 * 16-byte aligned.  A sequence longer than max_kept sets TG_ERR_DEVICE_INDEX.
 * The result is deterministic (fixed reduction order).  Precision: P is
 * recomputed in fp32 from the bf16 q', k' (as in the forward); D_i uses the
 * bf16 o; all sums are fp32.
 */
TG_API tg_status tg_gated_attention_bwd(const void* q_rot, const void* k_rot, const void* v,
                                 const void* o, const float* lse, const void* d_o,
                                 const int32_t* pos_kept, const float* s_kept,
                                 const float* gain, float tau, const int32_t* cu_kept,
                                 int32_t batch, int64_t n_kept, int32_t max_kept,
                                 int32_t hq, int32_t hkv, int32_t head_dim,
                                 float* d_s, float* d_gain, float* d_tau,
                                 void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/* Bytes of workspace tg_gated_attention_bwd needs.  Host-only, no CUDA call. */
TG_API size_t tg_attention_bwd_workspace_size(int64_t n_kept, int32_t hq);

/*
 * Pruned Gated DeltaNet scan.  TokenGate prunes the Gated DeltaNet layers of
 * the hybrid Qwen3.5 model as well as its attention layers (MarkTechPost
 * article, section "Does it work on hybrid attention models?", and the
 * DeltaNet row of its table "TokenGate vs FastKV, SlimInfer, GemFilter and
 * DASH"); above the gate such a layer runs its recurrence
 * over the kept tokens only, and a pruned token never updates the state.  The
 * layer's recurrence is the gated delta rule (Gated DeltaNet).  Per sequence b
 * and value head h, from S = initial_state[b, h] (zero when initial_state is
 * NULL), over the kept tokens of b in order:
 *     k^ = k / sqrt(|k|^2 + 1e-6),   q^ = scale q / sqrt(|q|^2 + 1e-6)
 *     S  = exp(g) (S - beta (S k^) k^T) + beta v k^T,    o = S q^
 * with S of shape [dv, dk]; value head h reads q/k head h / (hv / hk).
 *
 *   q, k   [n_kept, hk, dk] bf16, dk in {64, 128}
 *   v      [n_kept, hv, dv] bf16, hv a multiple of hk, dv a multiple of 16
 *          in [16, 1024]
 *   g      [n_kept, hv] fp32 log-decays (exp(g) in (0, 1] for g <= 0)
 *   beta   [n_kept, hv] fp32 write strengths
 *   cu_kept [batch+1] int32 (device), sequences of kept tokens
 *   scale  positive (1/sqrt(dk) in the layer)
 *   initial_state [batch, hv, dv, dk] fp32 or NULL
 *   o      [n_kept, hv, dv] bf16 output
 *   final_state   [batch, hv, dv, dk] fp32 output, or NULL
 *   workspace     NULL, or tg_gated_delta_scan_workspace_size(...) bytes,
 *                 256-byte aligned: the chunked form on the tensor cores
 *                 (chunks of 64 tokens; per-chunk products in parallel, the
 *                 state carried from chunk to chunk; tf32 MMAs on fp32
 *                 operands).  With batch * hv up to half the SMs (and batch
 *                 <= 96) both run in one cooperative launch, the state
 *                 carries on some SMs consuming chunks as the others finish
 *                 them; otherwise in two launches.  The results are the same
 *                 bit for bit.  Contents on entry do not matter; the call
 *                 overwrites them (one call at a time per workspace).  Needs
 *                 dv <= 128; with a larger dv, or NULL, the scan runs token
 *                 by token on the CUDA cores (fp32) and the workspace is not
 *                 touched.
 * Every other pointer 16-byte aligned.  fp32 state and accumulation; o
 * rounded once to bf16.
 * Errors: a workspace smaller than the size -> TG_ERR_WORKSPACE.
 * Device-side errors: cu_kept out of range -> TG_ERR_DEVICE_INDEX; a chunked
 * kernel's wait past the watchdog -> TG_ERR_TIMEOUT.
 */
TG_API tg_status tg_gated_delta_scan(const void* q, const void* k, const void* v,
                              const float* g, const float* beta, const int32_t* cu_kept,
                              int32_t batch, int64_t n_kept, int32_t hk, int32_t hv,
                              int32_t dk, int32_t dv, float scale,
                              const float* initial_state, void* o, float* final_state,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Bytes of the chunked scan's workspace: 0 when the shape does not take the
 * chunked form (dk not 64 or 128, dv not a multiple of 16 in [16, 128], or
 * batch < 1).  Host-only, no CUDA call. */
TG_API size_t tg_gated_delta_scan_workspace_size(int64_t n_kept, int32_t batch, int32_t hv, int32_t dk,
                                                 int32_t dv);

/*
 * The layer around the pruned path, for the whole pruned prefill and its
 * first decode step (the three phases of "How does TokenGate's learned token
 * pruning work?"; the model is Qwen3, "How does TokenGate perform on the
 * benchmarks?").  Not part of the pruned path itself.
 *
 * tg_rms_norm: y = x / sqrt(mean(x^2) + eps) * w for each of `rows` rows of
 *   length d (x, y [rows, d] bf16, w [d] bf16; 16-byte aligned; d a multiple
 *   of 8).  With rows = T * heads and d = head_dim it is the per-head
 *   QK-norm.  fp32 arithmetic, one rounding to bf16.
 *
 * tg_swiglu: y = SiLU(a) * b with a = gate_up[:, :f], b = gate_up[:, f:]
 *   (gate_up [rows, 2f] bf16, the fused gate/up projection; y [rows, f]
 *   bf16; f a multiple of 8; 16-byte aligned).
 *
 * tg_decode_attention: one new query per sequence (the first decode step).
 *   Sequence b's new token attends the rows [cache_cu[b], cache_cu[b+1]) of
 *   the cache and its own key, with logits (q' . k'_j) / (sqrt(D) tau) +
 *   gain_h s_j (the new token's own score is 0; s_cache and gain NULL: no
 *   bias, as in the layers at or below the gate).  q_rot [B, hq, D],
 *   k_new_rot and v_new [B, hkv, D], k_cache (rotated) and v_cache
 *   [cache_rows, hkv, D], all bf16; s_cache [cache_rows] fp32; gain [hq]
 *   fp32; o [B, hq, D] bf16 output.  max_cache_len: host bound on every
 *   sequence's cache length (sizes the split of the cache over CTAs).
 *   hq / hkv <= 8, head_dim 64 or 128.  Workspace of
 *   tg_decode_workspace_size(...) bytes, 16-byte aligned.  fp32 arithmetic.
 */
TG_API tg_status tg_rms_norm(const void* x, const void* w, int64_t rows, int32_t d, float eps,
                      void* y, cudaStream_t stream);
TG_API tg_status tg_swiglu(const void* gate_up, int64_t rows, int32_t f, void* y,
                    cudaStream_t stream);
TG_API size_t tg_decode_workspace_size(int32_t batch, int32_t hq, int32_t head_dim,
                                int32_t max_cache_len);
TG_API tg_status tg_decode_attention(const void* q_rot, const void* k_new_rot, const void* v_new,
                              const void* k_cache, const void* v_cache,
                              const int32_t* cache_cu, int32_t batch, int64_t cache_rows,
                              int32_t max_cache_len, const float* s_cache, const float* gain,
                              float tau, int32_t hq, int32_t hkv, int32_t head_dim, void* o,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Dense projection for the layers above the gate (long-context workload: a
 * stack of token-gated attention layers, each with its own Q/K/V/O
 * projections):  out[m, n] = sum_k a[m, k] * w[n, k]  (+ residual[m, n])
 *
 *   a [m, kdim] bf16, w [n, kdim] bf16 (nn.Linear layout), residual [m, n]
 *   bf16 or NULL, out [m, n] bf16 (may alias residual).
 *   kdim multiple of 64; n multiple of 16.  fp32 accumulation, one rounding.
 */
TG_API tg_status tg_linear_bf16(const void* a, const void* w, const void* residual, void* out,
                         int64_t m, int32_t n, int32_t kdim, cudaStream_t stream);

/*
 * The Q/K/V projection of a layer above the gate with RoPE fused into it
 * (the same long-context stack; MarkTechPost article, "What is token-gated
 * attention?": the kept tokens keep their original positions, and the
 * rotated keys are the kept-only KV cache, "How does TokenGate's learned
 * token pruning work?").  One GEMM against the stacked weight
 *   w_qkv [(hq + 2 hkv) * head_dim, kdim] (rows: W_q, then W_k, then W_v),
 * whose fp32 result is split into heads of head_dim columns:
 *   q_out[m, hq, D]  = RoPE(x W_q^T)  at pos[m]    (the queries q')
 *   k_out[m, hkv, D] = RoPE(x W_k^T)  at pos[m]    (the K cache k')
 *   v_out[m, hkv, D] = x W_v^T
 * RoPE as tg_rope_qk (rotate-half, rate rope_theta^(-2i/D) per position),
 * applied to the fp32 accumulators and rounded once to bf16, so q' and k'
 * are within one bf16 rounding of the exact rotation of the exact product.
 * tg_gated_attention_rotated then takes q_out, k_out and v_out directly.
 *   x [m, kdim] bf16 (kdim a multiple of 64), pos [m] int32 (the rows'
 *   original positions, not checked here: the attention kernel checks them),
 *   head_dim 64 or 128; all buffers device memory, 16-byte aligned, owned by
 *   the caller; outputs must not overlap x or w_qkv.
 * Errors: invalid sizes or pointers return TG_ERR_INVALID_ARG /
 * TG_ERR_UNSUPPORTED before any launch.
 */
TG_API tg_status tg_qkv_rope_bf16(const void* x, const void* w_qkv, int64_t m, int32_t kdim,
                           int32_t hq, int32_t hkv, int32_t head_dim, const int32_t* pos,
                           float rope_theta, void* q_out, void* k_out, void* v_out,
                           cudaStream_t stream);

/*
 * Token-gated attention with no workspace argument.  The TokenGate articles
 * have no counterpart of this call: it computes exactly what
 * tg_gated_attention_fwd computes, with the same arguments minus `workspace`
 * and `workspace_bytes`, for callers that cannot allocate device memory when
 * they call -- an engine that plans all of its device memory at start-up and
 * forbids allocation afterwards, a plugin running under a host runtime that
 * owns the allocator, or a plain C program that does not want to manage a
 * scratch buffer.
 *
 * Scratch space (the rotated queries, and the rotated keys when k_cache is
 * NULL) comes from a fixed array of tg_attention_static_scratch_bytes()
 * bytes (64 MiB) inside the library, which every device that loads the
 * library holds until the process exits.  A call needs
 * tg_attention_workspace_size(n_kept, hq, hkv, head_dim, k_cache != NULL)
 * bytes of it; a larger problem returns TG_ERR_WORKSPACE and launches
 * nothing.  The library allocates no memory on this path.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current): make that first call before any stream
 * capture.  The address is cached per device ordinal and belongs to the
 * device's primary context (the one the CUDA runtime uses); a caller that
 * drives the library from another driver context, or resets the device and
 * starts a new context, must not use this call afterwards in that process.  All calls share the one array and it keeps the last call's
 * contents; nothing in it needs to start at zero, since each call overwrites
 * what it reads.  Calls whose kernels overlap on the GPU (different streams
 * or host threads) race on the array: serialise them.
 */
TG_API tg_status tg_gated_attention_fwd_noalloc(const void* q, const void* k, const void* v,
                                                const int32_t* pos_kept, const float* s_kept,
                                                const float* gain, float tau, float rope_theta,
                                                const int32_t* cu_kept, int32_t batch, int64_t n_kept,
                                                int32_t max_kept, int32_t hq, int32_t hkv, int32_t head_dim,
                                                void* o, float* lse, void* k_cache, cudaStream_t stream);

/* Size in bytes of the fixed scratch array used by
 * tg_gated_attention_fwd_noalloc.  Host-only, no CUDA call. */
TG_API size_t tg_attention_static_scratch_bytes(void);

/* Synchronises `stream`, then reads and clears the device status word of the
 * current device: TG_OK, TG_ERR_TIMEOUT or TG_ERR_DEVICE_INDEX. */
TG_API tg_status tg_check_device_status(cudaStream_t stream);

/* Cycle limit of every device-side wait (default 2^31 SM cycles, about one
 * second).  A wait that runs out records TG_ERR_TIMEOUT and its kernel
 * returns.  0 restores the default. */
TG_API void tg_set_watchdog_cycles(long long cycles);

/* Message of the last error returned on this host thread ("" if none). */
TG_API const char* tg_last_error_string(void);

/* Library version string. */
TG_API const char* tg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TOKENGATE_H_ */
