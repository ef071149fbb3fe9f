/*
 * dg.h -- C ABI of libdg, the GB300 (sm_103a) structured-slot-read denoise step.
 *
 * The calls follow the prefill / denoise / commit split of the DiffusionGemma
 * sampler (24-ai.news, "DiffusionGemma integrated into vLLM", section
 * "Integration into vLLM infrastructure") and the structured-read extension
 * that seeds the canvas and reads decision slots after one denoise forward
 * (tau-home.com, "DiffusionGemma like Jev", section "Refusing JSON token
 * generation").
 *
 * Conventions shared by every call
 * --------------------------------
 *  - bf16 tensors are passed as `const uint16_t*` (raw bfloat16 bit patterns).
 *  - Every tensor pointer is a DEVICE pointer unless its comment says "host".
 *    Tensors are dense and row-major in the layout given; device pointers of
 *    bf16 matrices read by TMA must be 16-byte aligned and their row length
 *    (in bytes) a multiple of 16.
 *  - Ownership: the caller allocates and frees every buffer, including the
 *    workspace (size from dg_workspace_bytes).  The library never allocates,
 *    frees or synchronises; every compute call only enqueues work on `stream`
 *    (a cudaStream_t, NULL = legacy default stream) and returns.
 *  - Return value: DG_OK, or a negative DG_ERR_* found by synchronous argument
 *    validation BEFORE anything is launched (nothing was enqueued), or
 *    DG_ERR_CUDA if a launch failed.  Conditions found on the device (a wait
 *    that timed out, an out-of-range page or label id met by a kernel) set
 *    bits in the library's device status word, read with dg_get_status; the
 *    kernel skips the offending access instead of faulting.
 */
#ifndef DG_H_
#define DG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
#define DG_OK 0
#define DG_ERR_ARG (-1)             /* null pointer, non-positive size, misalignment */
#define DG_ERR_TOO_MANY_LABELS (-2) /* a slot with more than 26 labels (A..Z)        */
#define DG_ERR_LABEL (-3)           /* duplicate label id, or id outside [0, V)      */
#define DG_ERR_SHAPE (-4)           /* unsupported or inconsistent dimensions        */
#define DG_ERR_CUDA (-5)            /* a CUDA runtime call or launch failed          */
#define DG_ERR_WORKSPACE (-6)       /* workspace null or smaller than required       */

/* bits of the device status word */
#define DG_DEV_TIMEOUT 1    /* a bounded wait inside a kernel gave up        */
#define DG_DEV_BAD_PAGE 2   /* a page-table entry outside the page pool      */
#define DG_DEV_BAD_LABEL 4  /* a label id or label count out of range        */
#define DG_DEV_BAD_INDEX 8  /* a slot row / token id outside its tensor      */
#define DG_DEV_RANGE 16     /* reserved: no call of this version raises it    */

#define DG_MAX_LABELS 26 /* sotaaz.com, "The server accepts at most 26 alternatives per question" */
#define DG_MAX_WIDE_LABELS 256 /* label table stride limit of dg_slot_read_wide */

/* workspace kinds for dg_workspace_bytes */
#define DG_WS_ATTN 1
#define DG_WS_LMHEAD 2
#define DG_WS_SLOT_READ 3
#define DG_WS_SELFCOND 4
#define DG_WS_HEADS 5
#define DG_WS_PROBS_EMBED 6
#define DG_WS_PREFILL 7
#define DG_WS_PROBS_EMBED8 8
#define DG_WS_LMHEAD_NVFP4_MMA 9

/* Problem dimensions.  B requests, C canvas tokens each, P_max the longest
 * prompt (encoder KV) length, Hq/Hkv query/KV heads (GQA, Hq % Hkv == 0),
 * d_head in {64, 512}, W the +-W canvas window, d_model, V the vocabulary.
 * sm_share: the number of SMs an attention call (dg_attn_decode,
 * dg_prefill_attn, dg_attn_mixed) plans its grid for, when other work on
 * another stream holds the rest of the device: fewer SMs mean fewer key
 * splits (longer CTAs, less combine work), as long as no CTA gets more than
 * 40 key tiles of 128 keys; longer key ranges are split as for the whole
 * device.  0 (or <= 0, or more than the device has) plans for all SMs.  The attention workspace size depends on it:
 * size and call with the same dims.  Other calls ignore it. */
typedef struct {
  int B, C, P_max, Hq, Hkv, d_head, W, d_model, V;
  int sm_share;
} dg_dims;

/* ---- a1: decoder-mode attention ----------------------------------------
 * 24-ai.news, "How does diffusion text generation differ?": decoder mode is
 * bidirectional attention inside a +-W sliding window over the canvas;
 * thakicloud.com, "What is DiffusionGemma": decoder mode reads the causal
 * encoder KV of the prompt.  Row i of request b, query head h, attends to all
 * prompt_len[b] prompt keys and to canvas keys j with |i - j| <= W, one joint
 * softmax, scale 1/sqrt(d_head); query head h reads KV head h / (Hq/Hkv).
 *   q      [B, C, Hq, d]  bf16        kc, vc [B, C, Hkv, d] bf16
 *   contiguous prompt KV (page_table == NULL): kenc, venc [B, P_max, Hkv, d]
 *   paged prompt KV: kenc, venc are page pools [n_pages, page_size, Hkv, d],
 *     page_table [B, pages_per_req] int32 (key j of request b lives at
 *     pool[page_table[b][j / page_size]][j % page_size]); entries outside
 *     [0, n_pages) set DG_DEV_BAD_PAGE and are read as masked keys.
 *   prompt_len [B] int32, each in [0, P_max]
 *   out [B, C, Hq, d] bf16;  lse [B, Hq, C] fp32 (natural log)
 *   workspace: dg_workspace_bytes(dims, DG_WS_ATTN, 0) bytes.
 * d_head = 512 runs on the tensor-core kernel, which takes pages of 8, 16, 32,
 * 64 or 128 keys; another page size returns DG_ERR_SHAPE (nothing launched). */
int dg_attn_decode(const dg_dims* dims, const uint16_t* q, const uint16_t* kc,
                   const uint16_t* vc, const uint16_t* kenc, const uint16_t* venc,
                   const int32_t* page_table, int pages_per_req, int n_pages,
                   int page_size, const int32_t* prompt_len, uint16_t* out,
                   float* lse, void* workspace, size_t workspace_bytes,
                   void* stream);

/* ---- a2: lm-head -> log-softmax -> entropy -> label gather ---------------
 * tau-home.com, "Refusing JSON token generation": one denoise forward gives
 * the logprobs and entropy that the read uses, and the logprobs of the allowed
 * label ids at the answer slots; 24-ai.news, "Token commit mechanism":
 * per-token confidence for the commit.  For each of the M rows,
 * z = (h_i . w_v) * inv_t[i] over the whole vocabulary, and
 *   lse[i] = log sum_v exp z_v, entropy[i] = lse - sum_v p_v z_v (nats),
 *   maxz[i] = max_v z_v, argmax[i] = lowest v attaining it;
 * for each of the S slots (S = 0: none), at row i = slot_row[s],
 *   label_lp[s][k] = z_i[label_ids[s][k]] - lse[i]   (k < n_labels[s]),
 * taken from the accumulators in the pass's epilogue.  The [M, V] logits are
 * never written to memory.
 *   h [M, d_model] bf16;  w [V, d_model] bf16;  inv_t [M] fp32 (> 0)
 *   slot_row [S] int32 (distinct rows in [0, M));  label_ids [S, 26] int32;
 *   n_labels [S] int32 (0..26);  label_lp [S, 26] fp32 (entries past
 *   n_labels[s] untouched)
 *   lse, entropy, maxz [M] fp32;  argmax [M] int32
 *   workspace: dg_workspace_bytes(dims, DG_WS_LMHEAD, M) bytes.
 * S > M returns DG_ERR_SHAPE; S > 0 with a NULL slot argument DG_ERR_ARG.  A
 * label id outside [0, V) sets DG_DEV_BAD_LABEL (its label_lp is -inf); a slot
 * row outside [0, M) or shared by two slots sets DG_DEV_BAD_INDEX.
 * dg_validate_slots checks the tables on the host before upload. */
int dg_lmhead_logsoftmax_entropy(const dg_dims* dims, const uint16_t* h, int M,
                                 const uint16_t* w, const float* inv_t,
                                 const int32_t* slot_row, const int32_t* label_ids,
                                 const int32_t* n_labels, int S, float* lse,
                                 float* entropy, float* maxz, int32_t* argmax,
                                 float* label_lp, void* workspace, size_t workspace_bytes,
                                 void* stream);

/* ---- a0: noise draws for the slot reads --------------------------------
 * sotaaz.com, "The server accepts at most 26 alternatives per question": the
 * answer slot is left as noise and re-read with fresh noise draws.  For slot s
 * and draw r: token n = Philox4x32-10(key = seed, counter = (slot_req[s],
 * step, r, s)) word 0, top log2(V) bits (V must be a power of two); the row
 * rows_out[s*R + r] = bf16(h[slot_row[s]] + e[n]) (fp32 add, round to nearest
 * even), inv_t_out[s*R + r] = inv_t[slot_row[s]].
 *   h [M, d_model] bf16 (M = rows of h);  e [V, d_model] bf16;  inv_t [M] fp32
 *   slot_row, slot_req [S] int32;  rows_out [S*R, d_model] bf16
 *   inv_t_out [S*R] fp32;  noise_tok_out [S, R] int32 (may be NULL)
 * h, e and rows_out must be 16-byte aligned (DG_ERR_ARG otherwise). */
int dg_slot_noise(const dg_dims* dims, const uint16_t* h, int M, const uint16_t* e,
                  const float* inv_t, const int32_t* slot_row,
                  const int32_t* slot_req, int S, int R, uint64_t seed, int step,
                  uint16_t* rows_out, float* inv_t_out, int32_t* noise_tok_out,
                  void* stream);

/* ---- a3: slot read with the entropy-gated resample ---------------------
 * tau-home.com, "Refusing JSON token generation" and sotaaz.com, "The server
 * accepts at most 26 alternatives per question".  dg_slot_finish takes the
 * S*R noised draw rows (dg_slot_noise) and their full-vocabulary lse
 * (dg_lmhead_logsoftmax_entropy over those rows).  Per slot and draw:
 *   z_k = (row . w[label_k]) * inv_t_row, lp[s][r][k] = z_k - lse_row,
 *   q^(r) = softmax over the slot's n_labels[s] label logits, H^(r) = entropy.
 * If samples > 1 and H^(0) > gate: q_avg = mean of q^(0..samples-1),
 * n_reads = samples, resampled = 1; else q_avg = q^(0), n_reads = 1.
 * chosen = argmax q_avg (lowest label index on ties), h_slot = entropy of q_avg.
 *   label_ids [S, 26] int32 (first n_labels[s] used);  n_labels [S] int32
 *   q_avg [S, 26] fp32 (zero past n_labels);  h_slot [S] fp32;  chosen [S] int32
 *   lp_draws [S, R, 26] fp32;  resampled [S] uint8;  n_reads [S] int32
 * R is the number of draw rows per slot; 1 <= samples <= R <= 8.  A slot with
 * n_labels[s] == 0 is a question that was not asked (see dg_ask_if_select): it
 * is not read; chosen = -1, n_reads = 0 and its outputs are zero.
 * rows == NULL (w and inv_t_rows then unused): lp_draws already holds every
 * z_k of every draw, as the label gather of dg_denoise_heads writes them, and
 * the call turns them into lp in place; otherwise the z_k are computed here as
 * the dot products above (labels known only after the pass, as in a second
 * ask_if stage). */
int dg_slot_finish(const dg_dims* dims, const uint16_t* rows, const float* inv_t_rows,
                   const float* lse_rows, const uint16_t* w, const int32_t* label_ids,
                   const int32_t* n_labels, int S, int R, int samples, float gate,
                   float* q_avg, float* h_slot, int32_t* chosen, float* lp_draws,
                   uint8_t* resampled, int32_t* n_reads, void* stream);

/* Read-only structured read (the `diffusion_read_only` mode of tau-home.com,
 * "Refusing JSON token generation"): dg_slot_noise, then one lm-head pass over
 * all S*R draw rows (W streamed once) that also gathers every draw's label
 * logits from its accumulators, then dg_slot_finish on them (rows = NULL).  Arguments as in
 * those calls; R = samples draws are always computed (the gate only selects).
 *   workspace: dg_workspace_bytes(dims, DG_WS_SLOT_READ, S*samples) bytes. */
int dg_slot_read(const dg_dims* dims, const uint16_t* h, int M, const uint16_t* w,
                 const uint16_t* e, const float* inv_t, const int32_t* slot_row,
                 const int32_t* slot_req, const int32_t* label_ids,
                 const int32_t* n_labels, int S, uint64_t seed, int step,
                 int samples, float gate, float* q_avg, float* h_slot,
                 int32_t* chosen, float* lp_draws, uint8_t* resampled,
                 int32_t* n_reads, int32_t* noise_tok_out, void* workspace,
                 size_t workspace_bytes, void* stream);

/* ---- next: encoder-mode prefill writing the paged prompt KV -------------
 * thakicloud.com, "What is DiffusionGemma": one backbone runs in two modes; the
 * encoder mode reads the prompt causally and keeps its KV cache, which the
 * decoder mode (dg_attn_decode) then reads.  24-ai.news, "How does diffusion
 * text generation differ?": the encoder mode is causal.  For every request b
 * and prompt row i < prompt_len[b]:
 *   out[b, i, h] = softmax_{j <= i}(q_i . k_j / sqrt(d)) v_j   (query head h reads
 *   KV head h / (Hq/Hkv)), lse[b, h, i] its log-normaliser (natural log);
 * rows i >= prompt_len[b] are not written.  With a page table, the first
 * prompt_len[b] rows of k and v are also copied into the page pools
 * (pool[page_table[b, i / page_size], i % page_size] = row i), the layout
 * dg_attn_decode reads.  dims: B, P_max (rows of q/k/v per request), Hq, Hkv,
 * d_head = 512 (Hq/Hkv dividing 128); the other fields are ignored.
 *   q, out [B, P_max, Hq, 512] bf16;  k, v [B, P_max, Hkv, 512] bf16;
 *   prompt_len [B] int32 (clamped to [0, P_max]);  lse [B, Hq, P_max] fp32;
 *   page_table [B, pages_per_req] int32 or NULL;  pool_k, pool_v
 *   [n_pages, page_size, Hkv, 512] bf16 (16-byte aligned, like q, k, v, out);
 *   workspace: dg_workspace_bytes(dims, DG_WS_PREFILL, 0) bytes.
 * A page index outside [0, n_pages) sets DG_DEV_BAD_PAGE and skips that row. */
int dg_prefill_attn(const dg_dims* dims, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const int32_t* prompt_len, uint16_t* out, float* lse,
                    const int32_t* page_table, int pages_per_req, int n_pages, int page_size,
                    uint16_t* pool_k, uint16_t* pool_v, void* workspace, size_t workspace_bytes,
                    void* stream);

/* ---- next: decoder and encoder requests in one attention launch ---------
 * 24-ai.news, "DiffusionGemma integrated into vLLM" ("Integration into the
 * vLLM infrastructure"): causal attention switched per sequence lets
 * encoder-mode and decoder-mode requests share one batch.  One launch of the
 * 512-wide-head kernel over a batch whose request b is
 *   mode[b] = 0, decoder: rows i < rows_len[b] attend to the prompt keys
 *     (prompt_len[b] of kenc/venc, contiguous or paged as in dg_attn_decode)
 *     and to the rows j < rows_len[b] with |i - j| <= W (dg_attn_decode with a
 *     canvas of rows_len[b] rows);
 *   mode[b] = 1, encoder: rows i < rows_len[b] attend to rows j <= i of the
 *     same request (dg_prefill_attn without the page write); prompt_len[b] is
 *     not read.
 * dims: B, C = rows per request in q/kc/vc/out, P_max, Hq, Hkv, d_head = 512, W.
 *   mode, rows_len [B] int32;  q, out [B, C, Hq, 512];  kc, vc [B, C, Hkv, 512];
 *   kenc, venc, page_table, prompt_len, lse and the workspace (DG_WS_ATTN) as in
 *   dg_attn_decode.  Rows at or past rows_len[b] are not written.  Page sizes
 *   the tensor-core kernel cannot take (not a divisor of 128 or below 8) return
 *   DG_ERR_SHAPE. */
int dg_attn_mixed(const dg_dims* dims, const int32_t* mode, const int32_t* rows_len,
                  const uint16_t* q, const uint16_t* kc, const uint16_t* vc, const uint16_t* kenc,
                  const uint16_t* venc, const int32_t* page_table, int pages_per_req,
                  int n_pages, int page_size, const int32_t* prompt_len, uint16_t* out,
                  float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* ---- next: the lm-head pass on 8-bit operands ---------------------------
 * tau-home.com, "DiffusionGemma like Jev" ("Running NVFP4 locally with a
 * Jev-compatible System One endpoint") and 24-ai.news, "DiffusionGemma
 * integrated into vLLM" ("Measured performance": an FP8 checkpoint with
 * dynamic activation scaling) run the model on 8- and 4-bit weights.  Here W
 * and the hidden rows are e4m3 with one fp32 scale per row (the rows' scales
 * computed per call), so the W stream of the HBM-bound pass halves.  dg_quantize_rows_e4m3: scale[r] = max_k |x[r, k]| / 448 (1 for a
 * zero row), q[r, k] = e4m3(x[r, k] / scale[r]) (fp32 division, round to
 * nearest even, saturating).  x [rows, cols] bf16;  q [rows, cols] uint8;
 * scale [rows] fp32. */
int dg_quantize_rows_e4m3(const uint16_t* x, int rows, int cols, uint8_t* q, float* scale,
                          void* stream);

/* dg_lmhead_logsoftmax_entropy on quantised operands: the row statistics of
 * softmax(z_i / T_i) with z_iv = (sum_k h8[i, k] w8[v, k]) * h_scale[i] * w_scale[v]
 * (e4m3 products accumulated in fp32 by the tensor cores).  Label gather,
 * outputs, workspace (DG_WS_LMHEAD) and errors as dg_lmhead_logsoftmax_entropy;
 * d_model must be a multiple of 16; h8, w8 and w_scale 16-byte aligned.
 *   h8 [M, d_model], w8 [V, d_model] uint8 (e4m3);  h_scale [M], w_scale [V] fp32 */
int dg_lmhead_logsoftmax_entropy_fp8(const dg_dims* dims, const uint8_t* h8, const float* h_scale,
                                     int M, const uint8_t* w8, const float* w_scale,
                                     const float* inv_t, const int32_t* slot_row,
                                     const int32_t* label_ids, const int32_t* n_labels, int S,
                                     float* lse, float* entropy, float* maxz, int32_t* argmax,
                                     float* label_lp, void* workspace, size_t workspace_bytes,
                                     void* stream);

/* ---- next: the self-conditioning P . E on 8-bit operands -----------------
 * The same deployments (8-bit weights and activations) applied to the second
 * GEMM of the step, e_i = sum_v p_iv E[v] (24-ai.news, "Token commit
 * mechanism").  The scale of E must sit outside the sum over the vocabulary,
 * so E is quantised per d_model column and stored transposed:
 * dg_quantize_cols_e4m3: scale[c] = max_r |x[r, c]| / 448 (1 for a zero
 * column), qt[c, r] = e4m3(x[r, c] / scale[c]) (fp32 division, round to nearest
 * even, saturating).  x [rows, cols] bf16;  qt [cols, rows] uint8;  scale [cols]
 * fp32 (also used as scratch during the call).  A one-time preparation of E. */
int dg_quantize_cols_e4m3(const uint16_t* x, int rows, int cols, uint8_t* qt, float* scale,
                          void* stream);

/* out[i, c] = row_scale[i] * p_scale[i] * e_scale[c] * sum_v p8[i, v] e8t[c, v]
 * (e4m3 products accumulated in fp32 by the tensor cores, split over the
 * vocabulary and summed in a fixed order).  With p8/p_scale the per-row e4m3
 * quantisation of dg_denoise_heads' probabilities (dg_quantize_rows_e4m3),
 * row_scale its prob_scale, and e8t/e_scale from dg_quantize_cols_e4m3(e), out
 * is the expected embedding on 8-bit operands.
 *   p8 [M, V] uint8;  p_scale [M] fp32;  row_scale [M] fp32 or NULL (1);
 *   e8t [d_model, V] uint8;  e_scale [d_model] fp32;  out [M, d_model] fp32.
 * V must be a multiple of 16 and d_model of 4; p8, e8t, e_scale and out
 * 16-byte aligned (else DG_ERR_SHAPE / DG_ERR_ARG).
 *   workspace: dg_workspace_bytes(dims, DG_WS_PROBS_EMBED8, M) bytes. */
int dg_selfcond_from_probs8(const dg_dims* dims, const uint8_t* p8, const float* p_scale,
                            const float* row_scale, int M, const uint8_t* e8t,
                            const float* e_scale, float* out, void* workspace,
                            size_t workspace_bytes, void* stream);

/* ---- next: the lm-head pass against NVFP4 weights -------------------------
 * tau-home.com, "DiffusionGemma like Jev" ("Running NVFP4 locally with a
 * Jev-compatible System One endpoint") and agentlenshq.com, "4x faster via
 * parallel diffusion" ("Architecture": NVFP4 kernels for Hopper and Blackwell)
 * run the model on NVFP4 weights: e2m1 elements, one e4m3 scale per 16
 * elements of a row, one fp32 scale per tensor.  dg_quantize_nvfp4 (a one-time
 * preparation of W): g = amax|x| / (6 * 448) (1 for an all-zero tensor);
 * per block of 16 of a row s = e4m3((amax_block / 6) / g) (round to nearest
 * even, saturating); codes e2m1(x / (s * g)) (round to nearest, ties to the
 * even mantissa, saturating at 6; 0 for a block whose scale is 0), fp32
 * arithmetic throughout.  Layout, K-block-major (the layout the pass copies
 * whole): codes [cols/64][rows][32] bytes (element 64 kb + j of row v is the
 * low nibble of byte j / 2 for even j, the high nibble for odd j), scales
 * [cols/64][rows][4] e4m3 bytes (byte q: elements 64 kb + 16 q ..), *g (device).
 * cols must be a multiple of 64; x and codes 16-byte aligned. */
int dg_quantize_nvfp4(const uint16_t* x, int rows, int cols, uint8_t* codes, uint8_t* scales,
                      float* g, void* stream);

/* dg_lmhead_logsoftmax_entropy against NVFP4 weights: the row statistics of
 * softmax(z_i / T_i) with z_iv = (h_i . (e2m1 * s)_v) * g, the rows times the
 * weights widened on chip (exact: e2m1 times an e4m3 scale fits bf16 and f16),
 * fp32 accumulation on the tensor cores.  Up to 16 rows take f16 operands: each
 * row is divided by a power of two that keeps it below 2^15 and converted to
 * f16 (exact for elements of magnitude 2^-14 or more after the division; the
 * power of two is multiplied back into the logits); more rows stay bf16.  Operands from
 * dg_quantize_nvfp4(w, V, d_model, ..); label gather, outputs, workspace
 * (DG_WS_LMHEAD) and errors as dg_lmhead_logsoftmax_entropy; d_model a multiple
 * of 64 and V of 4 (else DG_ERR_SHAPE); h, codes and scales 16-byte aligned. */
int dg_lmhead_logsoftmax_entropy_nvfp4(const dg_dims* dims, const uint16_t* h, int M,
                                       const uint8_t* codes, const uint8_t* scales,
                                       const float* g, const float* inv_t,
                                       const int32_t* slot_row, const int32_t* label_ids,
                                       const int32_t* n_labels, int S, float* lse,
                                       float* entropy, float* maxz, int32_t* argmax,
                                       float* label_lp, void* workspace, size_t workspace_bytes,
                                       void* stream);

/* The same pass with the rows in NVFP4 too (the pages' checkpoint quantises
 * weights and activations), on the block-scaled tensor-core kind
 * (kind::mxf4nvf4, one e4m3 scale per 16 values of both operands):
 * z_iv = (sum_k e2m1(h)_ik s(h)_ik e2m1(w)_vk s(w)_vk) * g_h * g_w, fp32
 * accumulation; the rows are quantised inside the call by the recipe of
 * dg_quantize_nvfp4 with their own tensor scale g_h.  Any M: up to 16 rows (the
 * slot reads' draw rows) stay resident in one pass with the vocabulary on the
 * tensor-memory lanes (d_model at most 3072 there), more rows go through the
 * GEMM form; d_model a multiple of 64, else DG_ERR_SHAPE.
 * codes and sf from dg_quantize_nvfp4_mma(w, V, d_model, ..), g its tensor scale;
 * label gather and outputs as dg_lmhead_logsoftmax_entropy; workspace:
 * dg_workspace_bytes(dims, DG_WS_LMHEAD_NVFP4_MMA, M) bytes (256-byte aligned).
 * h, codes and sf 16-byte aligned. */
int dg_lmhead_logsoftmax_entropy_nvfp4_mma(const dg_dims* dims, const uint16_t* h, int M,
                                           const uint8_t* codes, const uint8_t* sf,
                                           const float* g, const float* inv_t,
                                           const int32_t* slot_row, const int32_t* label_ids,
                                           const int32_t* n_labels, int S, float* lse,
                                           float* entropy, float* maxz, int32_t* argmax,
                                           float* label_lp, void* workspace,
                                           size_t workspace_bytes, void* stream);

/* NVFP4 quantisation (the recipe of dg_quantize_nvfp4) in the layout the
 * block-scaled pass reads.  Codes in 16 KB blocks, one per (128-row tile,
 * 256-value K block), [ceil(rows/128)][ceil(cols/256)][128][128] bytes: element
 * k of row v sits in byte (k % 256) / 2 of row v % 128 of block
 * (v / 128, k / 256), the low nibble for even k; rows past `rows` and values
 * past cols in the last block are zero codes.  dg_nvfp4_mma_codes_bytes(rows,
 * cols) gives the size (0 for rows < 1 or cols not a positive multiple of 64).
 * Every TMA box of the pass is one block or two consecutive tiles' blocks, a
 * contiguous run, where row-major codes made it 128 rows of 128 bytes cols/2
 * bytes apart.  Scales as 512-byte atoms, one per
 * 128-row tile and 64-value K-step, atoms [ceil(rows/128)][cols/64]: row 32 j + l
 * of the tile has its four e4m3 scales (values 16 q .. 16 q + 15 of the step in
 * byte q) at bytes 16 l + 4 j .. 16 l + 4 j + 3 of the atom; rows of the last tile
 * past `rows` have scale 0.  *g the fp32 tensor scale (device).  sf holds
 * ceil(rows/128) * (cols/64) * 512 bytes.  cols a multiple of 64 (else
 * DG_ERR_SHAPE); x and codes 16-byte aligned, sf 4-byte aligned. */
int dg_quantize_nvfp4_mma(const uint16_t* x, int rows, int cols, uint8_t* codes, uint8_t* sf,
                          float* g, void* stream);
size_t dg_nvfp4_mma_codes_bytes(int rows, int cols);

/* ---- next: one wide read in place of the two-stage path -----------------
 * sotaaz.com, "The server accepts at most 26 alternatives per question": the
 * example server letters a question's alternatives A-Z, so 77 intents are read
 * as a 9-way group question and then the chosen group's items; the same page
 * ("Same model, same groups, a 14-point gap") reports a follow-up in which all
 * 77 intents are read in one read and the two-stage path loses.  This is
 * dg_slot_read with label tables of row stride L (1 <= L <= 256): slot s has
 * n_labels[s] <= L labels at label_ids[s*L ..].  The arithmetic is that of
 * dg_slot_read (renormalise over the slot's labels, entropy gate, mean of the
 * reads, argmax with ties to the lowest index).
 *   label_ids [S, L] int32;  q_avg [S, L] fp32;  lp_draws [S, R, L] fp32; the
 *   other arguments, the workspace (DG_WS_SLOT_READ with rows = S * samples)
 *   and the errors are those of dg_slot_read; L > 256 returns
 *   DG_ERR_TOO_MANY_LABELS. */
int dg_slot_read_wide(const dg_dims* dims, const uint16_t* h, int M, const uint16_t* w,
                      const uint16_t* e, const float* inv_t, const int32_t* slot_row,
                      const int32_t* slot_req, const int32_t* label_ids, const int32_t* n_labels,
                      int S, int L, uint64_t seed, int step, int samples, float gate,
                      float* q_avg, float* h_slot, int32_t* chosen, float* lp_draws,
                      uint8_t* resampled, int32_t* n_reads, int32_t* noise_tok_out,
                      void* workspace, size_t workspace_bytes, void* stream);

/* ---- a7: ask_if gating of a second read stage --------------------------
 * sotaaz.com, "The server accepts at most 26 alternatives per question": a
 * question carrying ask_if is read only when the earlier answer matches (77
 * intents read as a 9-way group question, then the chosen group's items).
 * Question q depends on stage-1 slot cond_slot[q] and fires when
 * chosen1[cond_slot[q]] == cond_value[q]; it fills stage-2 slot q_owner[q].
 * Each stage-2 slot j receives the labels of the first fired question that
 * owns it, or n_labels2[j] = 0 (not asked, skipped by dg_slot_finish).  The
 * decision stays on the device: no host round trip between the stages.
 *   chosen1 [S1] int32 (dg_slot_read / dg_slot_finish output)
 *   cond_slot, cond_value, q_owner [Q] int32;  q_label_ids [Q, 26] int32
 *   q_n_labels [Q] int32;  label_ids2 [S2, 26] int32 (-1 padded);
 *   n_labels2 [S2] int32;  fired [Q] uint8 (may be NULL).
 * A cond_slot outside [0, S1) sets DG_DEV_BAD_INDEX and never fires. */
int dg_ask_if_select(const int32_t* chosen1, int S1, const int32_t* cond_slot,
                     const int32_t* cond_value, const int32_t* q_owner,
                     const int32_t* q_label_ids, const int32_t* q_n_labels, int Q, int S2,
                     int32_t* label_ids2, int32_t* n_labels2, uint8_t* fired, void* stream);

/* ---- a4: entropy-ordered commit ----------------------------------------
 * 24-ai.news, "Token commit mechanism": accept the most confident tokens first
 * until the cumulative entropy exceeds a preset threshold; committed tokens are
 * fixed and leave later steps' candidate sets.  Per request b, the candidates
 * are positions with cand != 0 and (if committed_state is given) not yet
 * committed; they are ordered by entropy ascending (ties: lower position); the
 * first is always accepted, the k-th while the sum of the first k entropies is
 * <= gamma[b].
 *   entropy [B, C] fp32;  argmax [B, C] int32;  cand [B, C] uint8;  gamma [B] fp32
 *   committed_state [B, C] uint8, in/out, may be NULL: |= the accepted mask
 *   token_state [B, C] int32, in/out, may be NULL: argmax written where accepted
 *   commit [B, C] uint8 (1 = accepted now);  tokens [B, C] int32 (argmax where
 *   accepted now, -1 elsewhere);  n_commit [B] int32.  C <= 1024. */
int dg_commit(const dg_dims* dims, const float* entropy, const int32_t* argmax,
              const uint8_t* cand, const float* gamma, uint8_t* committed_state,
              int32_t* token_state, uint8_t* commit, int32_t* tokens, int32_t* n_commit,
              void* stream);

/* ---- a5: self-conditioning expected embedding ---------------------------
 * 24-ai.news, "Token commit mechanism": the previous step's full softmax
 * becomes a probability-weighted average of embeddings fed back as input.
 * out[i] = sum_v p_iv e[v] with p_i = softmax(z_i), z as in the lm-head call;
 * lse must be that call's output for the same rows.
 *   h [M, d_model] bf16;  w, e [V, d_model] bf16 (the same row-major layout
 *   every call uses);  inv_t, lse [M] fp32;  out [M, d_model] fp32
 *   workspace: dg_workspace_bytes(dims, DG_WS_SELFCOND, M) bytes. */
int dg_selfcond_embed(const dg_dims* dims, const uint16_t* h, int M,
                      const uint16_t* w, const uint16_t* e, const float* inv_t,
                      const float* lse, float* out, void* workspace,
                      size_t workspace_bytes, void* stream);

/* ---- a2 + a3 + a5 fused: one stream of W per denoise step ----------------
 * The lm-head pass of dg_lmhead_logsoftmax_entropy over the M canvas rows,
 * plus, from the same W tiles:
 *  - the full-vocabulary log-normaliser of n_draw <= 16 slot draw rows
 *    (dg_slot_noise output), for dg_slot_finish (sotaaz.com, "The server
 *    accepts at most 26 alternatives per question");
 *  - the self-conditioning probabilities of the canvas rows (24-ai.news,
 *    "Token commit mechanism") as unnormalised bf16 values
 *    probs[i][v] = 2^(z_iv log2(e) - r_i), r_i a per-row reference (from the
 *    first 8 vocabulary entries, raised by whole powers of two wherever a logit
 *    lies far above it), and prob_scale[i] = 1 / sum_v probs[i][v], so
 *    p_iv = probs[i][v] * prob_scale[i].
 *  - the label gather of the draw rows (tau-home.com, "Refusing JSON token
 *    generation"): draw j is draw j % draw_R of slot j / draw_R, and
 *    draw_label_z[j][k] = z_j[draw_label_ids[j / draw_R][k]] (k <
 *    draw_n_labels[j / draw_R]), the label logits dg_slot_finish takes with
 *    rows = NULL.
 * The statistics and the probabilities are exact (no clamped or overflowing
 * exponent) while every scaled logit z_iv log2(e) lies less than 2^13 above the
 * largest of the row's first eight.
 *   h [M, d_model] bf16;  draw_rows [n_draw, d_model] bf16 (NULL if n_draw = 0)
 *   w [V, d_model] bf16;  inv_t [M], inv_t_draw [n_draw] fp32
 *   w_tiled: NULL, or dg_heads_weights_tile's copy of the same w (16-byte
 *   aligned; DG_ERR_ARG when d_model is not a multiple of 64).  With draw rows
 *   the pass streams W from it (the same values, read in contiguous blocks);
 *   without draw rows it reads w.  The caller keeps it in step with w.
 *   lse, entropy, maxz [M] fp32;  argmax [M] int32;  lse_draw [n_draw] fp32
 *   draw_label_ids [n_draw / draw_R, 26] int32;  draw_n_labels [n_draw / draw_R]
 *   int32;  draw_label_z [n_draw, 26] fp32 (NULL: no gather; else n_draw a
 *   multiple of draw_R >= 1, DG_ERR_ARG otherwise; a label id outside [0, V)
 *   sets DG_DEV_BAD_LABEL and gets -inf)
 *   prob_scale [M] fp32;  probs [M, probs_ld] bf16 (probs_ld >= V, multiple of
 *   64; 32-byte aligned; NULL to skip the probabilities)
 *   workspace: dg_workspace_bytes(dims, DG_WS_HEADS, M) bytes. */
int dg_denoise_heads(const dg_dims* dims, const uint16_t* h, int M,
                     const uint16_t* draw_rows, int n_draw, const uint16_t* w,
                     const uint16_t* w_tiled, const float* inv_t, const float* inv_t_draw, float* lse,
                     float* entropy, float* maxz, int32_t* argmax, float* lse_draw,
                     const int32_t* draw_label_ids, const int32_t* draw_n_labels,
                     int draw_R, float* draw_label_z, float* prob_scale, uint16_t* probs,
                     size_t probs_ld, void* workspace, size_t workspace_bytes,
                     void* stream);

/* The fused pass on e4m3 operands (tau-home.com, "Running NVFP4 locally with a
 * Jev-compatible System One endpoint"; 24-ai.news, "Measured performance": the
 * FP8 checkpoint): the canvas rows, the draw rows and W each quantised to e4m3
 * with one fp32 scale per row (dg_quantize_rows_e4m3), and
 * z_iv = (sum_k h8_ik w8_vk) h_scale_i w_scale_v, likewise for the draw rows
 * with draw_scale.  Everything else (statistics, draw-row normalisers, label
 * gather, probabilities, the exactness range, workspace DG_WS_HEADS) as
 * dg_denoise_heads, on those logits: the statistics of the dequantised
 * operands.  The per-row reference comes from the dequantised first eight W
 * rows.  d_model a multiple of 16 (else DG_ERR_SHAPE).
 *   h8 [M, d_model], draw8 [n_draw, d_model], w8 [V, d_model] e4m3 bytes
 *   (16-byte aligned); h_scale [M], draw_scale [n_draw], w_scale [V] fp32
 *   (w_scale 16-byte aligned); the rest as dg_denoise_heads. */
int dg_denoise_heads_fp8(const dg_dims* dims, const uint8_t* h8, const float* h_scale,
                         int M, const uint8_t* draw8, const float* draw_scale, int n_draw,
                         const uint8_t* w8, const float* w_scale, const float* inv_t,
                         const float* inv_t_draw, float* lse, float* entropy, float* maxz,
                         int32_t* argmax, float* lse_draw, const int32_t* draw_label_ids,
                         const int32_t* draw_n_labels, int draw_R, float* draw_label_z,
                         float* prob_scale, uint16_t* probs, size_t probs_ld, void* workspace,
                         size_t workspace_bytes, void* stream);

/* W in the tiled layout dg_denoise_heads streams (a layout of the lm-head
 * weights of tau-home.com, "Refusing JSON token generation", no arithmetic):
 * tiles of 224 vocabulary rows, each cut into blocks of 64 columns, block
 * (t, kb) one contiguous run of 224 x 64 bf16:
 *   w_tiled[((t * (d_model / 64) + kb) * 224 + r) * 64 + c] = w[224 t + r][64 kb + c]
 * and zero for rows 224 t + r >= V.  dg_heads_weights_bytes gives its size,
 * ceil(V / 224) * 224 * d_model * 2 bytes (0 when d_model is not a multiple of
 * 64 or the dims are invalid); dg_heads_weights_tile writes it on the stream
 * (DG_ERR_SHAPE for such dims; w and w_tiled 16-byte aligned, DG_ERR_ARG
 * otherwise).  Written once per weight matrix, beside the row-major w that
 * the other calls read. */
size_t dg_heads_weights_bytes(const dg_dims* dims);
int dg_heads_weights_tile(const dg_dims* dims, const uint16_t* w, uint16_t* w_tiled,
                          void* stream);

/* Expected embedding from dg_denoise_heads' probabilities:
 * out[i] = prob_scale[i] * sum_v probs[i][v] e[v] (24-ai.news, "Token commit
 * mechanism").  probs [M, probs_ld] bf16;  prob_scale [M] fp32;
 * e [V, d_model] bf16;  out [M, d_model] fp32.
 *   workspace: dg_workspace_bytes(dims, DG_WS_PROBS_EMBED, M) bytes. */
int dg_selfcond_from_probs(const dg_dims* dims, const uint16_t* probs, size_t probs_ld,
                           const float* prob_scale, int M, const uint16_t* e,
                           float* out, void* workspace, size_t workspace_bytes,
                           void* stream);

/* ---- a6: next-step canvas input ----------------------------------------
 * 24-ai.news, "Token commit mechanism" (self-conditioning is an extra input)
 * read additively: h_out[i] = bf16(h0[i] + e_sc[i]) for open rows and
 * bf16(h0[i] + emb[tokens[i]]) where committed[i] != 0.
 *   h0 [M, d_model] bf16;  e_sc [M, d_model] fp32;  emb [V, d_model] bf16
 *   tokens [M] int32;  committed [M] uint8;  h_out [M, d_model] bf16 */
int dg_canvas_update(const dg_dims* dims, const uint16_t* h0, const float* e_sc,
                     const uint16_t* emb, const int32_t* tokens,
                     const uint8_t* committed, int M, uint16_t* h_out, void* stream);

/* ---- test hook: raw Philox4x32-10 --------------------------------------
 * out4[i] = Philox4x32-10(counter = ctr4[i], key = seed); n counters. */
int dg_philox_fill(uint64_t seed, const uint32_t* ctr4, int n, uint32_t* out4,
                   void* stream);

/* ---- housekeeping ------------------------------------------------------ */
/* Synchronous check of a slot table held in HOST memory (the 422 "at most 26
 * alternatives" rejection of sotaaz.com happens here): n_labels in [1, 26],
 * label ids distinct and in [0, V), slot_row in [0, M).  No GPU work. */
int dg_validate_slots(const dg_dims* dims, const int32_t* slot_row_host,
                      const int32_t* label_ids_host, const int32_t* n_labels_host,
                      int S, int M);
/* The same check for the label tables of dg_slot_read_wide (row stride L,
 * 1 <= L <= 256): n_labels in [1, L] (DG_ERR_TOO_MANY_LABELS above L or for
 * L outside [1, 256]), label ids distinct and in [0, V), slot_row in [0, M).
 * No GPU work.  dg_validate_slots is this check with L = 26. */
int dg_validate_slots_wide(const dg_dims* dims, const int32_t* slot_row_host,
                           const int32_t* label_ids_host, const int32_t* n_labels_host,
                           int S, int L, int M);
/* Bytes of device workspace a call needs (rows = M for DG_WS_LMHEAD,
 * DG_WS_SELFCOND, DG_WS_HEADS and DG_WS_PROBS_EMBED, S*samples for
 * DG_WS_SLOT_READ, ignored for DG_WS_ATTN); 0 for an invalid request. */
size_t dg_workspace_bytes(const dg_dims* dims, int which, int rows);
/* Row length (elements) of the probability buffer dg_denoise_heads writes for
 * a vocabulary of V: V rounded up to a multiple of 64; 0 if V < 1. */
size_t dg_probs_ld(int V);
/* Diagnostic of the device status path: one warp waits on a shared-memory
 * barrier that nothing arrives on, under the same kind of bound as every wait
 * inside the library's kernels, here limit_ns of wall time (1 ns .. 1 s).
 * When the bound passes the kernel sets DG_DEV_TIMEOUT in the status word and
 * returns, leaving the context usable; *waited_us (device memory) receives the
 * time it waited.  No counterpart on the pages: it exists so that the timeout
 * path can be exercised without a fault. */
int dg_check_wait_timeout(int64_t limit_ns, int32_t* waited_us, void* stream);

/* Copy the device status word into *status_out (host) after the work already
 * on `stream` finishes; this call synchronises that stream. */
int dg_get_status(void* stream, int32_t* status_out);
/* Zero the device status word (enqueued on `stream`). */
int dg_clear_status(void* stream);
/* Static description of a DG_ERR_* code. */
const char* dg_strerror(int code);
/* Number of SMs the library sizes its persistent grids for (device 0 query,
 * cached); -1 if no device is visible. */
int dg_num_sms(void);

/* ---- lm-head pass without a caller-provided workspace -------------------
 * The pages describe nothing like this call; it exists for callers that cannot
 * allocate device memory or pass the library a buffer of their own -- a
 * serving runtime whose allocator is locked after start-up, or a plugin that
 * only receives the tensors it works on.  It computes exactly what
 * dg_lmhead_logsoftmax_entropy computes, with the same arguments minus the
 * workspace: the per-CTA partial statistics live in a fixed array of 2.5 MiB
 * compiled into the library (held on every GPU that loads it until the
 * process exits).
 *  - M may be at most DG_NOALLOC_MAX_ROWS; larger M returns DG_ERR_SHAPE.
 *  - The first call on a device looks up the array's device address (a
 *    runtime query, no allocation); make that first call before any stream
 *    capture.  Later calls on that device reuse the address, unless the
 *    device's context has been created anew since (after cudaDeviceReset),
 *    in which case the call looks it up again.
 *  - The array is shared by every call on a device and keeps the last call's
 *    contents (each launch overwrites all of it that it reads, so nothing needs
 *    clearing).  Calls whose work overlaps on the GPU, e.g. on two streams
 *    without ordering between them, race on it: order them on one stream. */
#define DG_NOALLOC_MAX_ROWS 512
int dg_lmhead_logsoftmax_entropy_noalloc(const dg_dims* dims, const uint16_t* h, int M,
                                         const uint16_t* w, const float* inv_t, float* lse,
                                         float* entropy, float* maxz, int32_t* argmax,
                                         void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DG_H_ */
