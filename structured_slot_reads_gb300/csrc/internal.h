// internal.h -- declarations shared between the C-ABI layer and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace dgi {

// Identity of the CUDA context current on this thread (0 if none): a context
// created again (e.g. after cudaDeviceReset) gets a new identity.
uint64_t context_id();
// Device address of one of this library's __device__ variables on the current
// device.  The address is cached per device together with the context it was
// looked up in, and looked up again (cudaGetSymbolAddress: no allocation) when
// the current context differs.  `symbol` is the host-side stand-in of the
// variable, which must never reach a kernel itself.
enum SymbolSlot { SYM_STATUS = 0, SYM_NOALLOC_SCRATCH = 1, SYM_COUNT = 2 };
void* device_symbol(const void* symbol, int slot);
// Device address of the library's status word on the current device.
int* status_ptr();
// Shapes every lm-head entry point accepts: d_model a positive multiple of 8
// (16-byte rows for TMA), a non-empty vocabulary.
inline bool lm_dims_ok(int d_model, int V) { return d_model >= 8 && d_model % 8 == 0 && V >= 1; }
int num_sms();
// SMs a launch plans its grid for: the caller's share when it is in (0, num_sms()),
// else the whole device.
int plan_sms(int share);
// Build a 2-D TMA map over a row-major bf16 matrix [outer, inner] whose rows are
// row_bytes apart, with a (box_inner x box_outer) box and 128-byte swizzle.
// Returns false on failure.
bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                       uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);
// 2-D tensor map of 8-bit elements (e4m3 operands), 128-byte swizzle.
bool make_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);
// 4-D tensor map of 8-bit elements (dims innermost first; strides of dims 1..3 in
// bytes), 128-byte swizzle.
bool make_tmap_u8_4d(CUtensorMap* map, const void* base, const uint64_t (&dims)[4],
                     const uint64_t (&stride_bytes)[3], const uint32_t (&box)[4]);
// 3-D tensor map (dims innermost first; strides of dims 1 and 2 in bytes), 128-byte swizzle.
bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, const uint64_t (&dims)[3],
                       const uint64_t (&stride_bytes)[2], const uint32_t (&box)[3]);

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---- tcgen05 GEMM family (gemm_tc.cu) ------------------------------------
struct RowStats {
  float* lse;
  float* entropy;
  float* maxz;
  int32_t* argmax;
};
// Label gather of an lm-head pass: for every row g that is a slot row, the
// logits z/T of its slot's labels (z - lse with sub_lse), taken from the
// accumulators in the pass's epilogue and written at out[o * L + k].  R > 0:
// row g < S R is draw g % R of slot g / R and o = g.  R == 0: slot s sits at
// row slot_row[s] and o = s; row_slot [M] is scratch the call fills (the slot
// of each row, or -1).  A label id outside [0, V) sets DG_DEV_BAD_LABEL and
// gets -inf; a slot row outside [0, M) or shared by two slots sets
// DG_DEV_BAD_INDEX.
struct LabelGather {
  const int32_t* label_ids;  // [S][L]
  const int32_t* n_labels;   // [S] (clamped to [0, L])
  const int32_t* slot_row;   // R == 0: [S]
  int32_t* row_slot;         // R == 0: [M] scratch
  float* out;                // null: no gather
  int L, S, R;
  int sub_lse;
};
size_t lmhead_ws_bytes(int M, int V);
cudaError_t lmhead_stats(const uint16_t* h, int M, const uint16_t* w, int V, int D,
                         const float* inv_t, RowStats out, void* ws, cudaStream_t st,
                         const LabelGather* gather = nullptr);
// lm-head statistics from e4m3 operands with per-row scales:
// z[i, v] = (h8_i . w8_v) * h_scale[i] * w_scale[v] / T_i.  Workspace: lmhead_ws_bytes.
cudaError_t lmhead_stats_fp8(const uint8_t* h8, const float* h_scale, int M, const uint8_t* w8,
                             const float* w_scale, int V, int D, const float* inv_t, RowStats out,
                             void* ws, cudaStream_t st, const LabelGather* gather = nullptr);
// Per-row e4m3 quantisation: scale = amax / 448 (1 for a zero row), q = e4m3(x / scale).
cudaError_t quantize_rows_e4m3(const uint16_t* x, int rows, int cols, uint8_t* q, float* scale,
                               cudaStream_t st);
cudaError_t quantize_cols_e4m3(const uint16_t* x, int rows, int cols, uint8_t* qt, float* scale,
                               cudaStream_t st);
// NVFP4 weights, K-block-major: codes [cols/64][rows][32] bytes, scales
// [cols/64][rows][4] e4m3, *g the fp32 tensor scale (cols a multiple of 64).
cudaError_t quantize_nvfp4(const uint16_t* x, int rows, int cols, uint8_t* codes,
                           uint8_t* scales, float* g, cudaStream_t st);
// lm-head statistics of bf16 rows against NVFP4 weights: z = (h . (e2m1 * s)) * g / T.
cudaError_t lmhead_stats_nvfp4(const uint16_t* h, int M, const uint8_t* codes,
                               const uint8_t* scales, const float* g, int V, int D,
                               const float* inv_t, RowStats out, void* ws, cudaStream_t st,
                               const LabelGather* gather = nullptr);
// NVFP4 in the layout of the block-scaled MMA pass: codes row-major [rows][cols/2],
// scales as 512-byte atoms [ceil(rows/128)][cols/64] (row 32 j + l of a 128-row
// tile at byte 16 l + 4 j of its atom), *g the fp32 tensor scale.
cudaError_t quantize_nvfp4_mma(const uint16_t* x, int rows, int cols, uint8_t* codes, uint8_t* sf,
                               float* g, cudaStream_t st);
// The same for at most 16 rows in one launch: codes [16][cols/2] (rows >= M zero),
// scale atoms [cols/64][512] (one tile), *g.
cudaError_t quantize_rows_nvfp4_mma(const uint16_t* x, int M, int cols, uint8_t* codes,
                                    uint8_t* sf, float* g, cudaStream_t st);
// The same for any number of rows: the largest magnitude into *amax (scratch),
// then one thread per (padded row, block of 16); *g written.
cudaError_t quantize_many_rows_nvfp4_mma(const uint16_t* x, int rows, int cols, uint8_t* codes,
                                         uint8_t* sf, float* g, unsigned int* amax,
                                         cudaStream_t st);
// lm-head statistics with both operands in NVFP4 on the block-scaled tensor-core kind:
// z = (sum_k e2m1_h s_h e2m1_w s_w) * g_h * g_w / T, at most 16 rows (quantised in the
// call).  Workspace: lmhead_nvfp4_mma_ws_bytes.
size_t lmhead_nvfp4_mma_ws_bytes(int M, int V, int D);
bool lmhead_nvfp4_mma_ok(int M, int D);
cudaError_t lmhead_stats_nvfp4_mma(const uint16_t* h, int M, const uint8_t* codes,
                                   const uint8_t* sf, const float* g, int V, int D,
                                   const float* inv_t, RowStats out, void* ws, cudaStream_t st,
                                   const LabelGather* gather = nullptr);
size_t probs_embed8_ws_bytes(int M, int V, int D);
cudaError_t probs_embed8(const uint8_t* p8, const float* p_scale, const float* row_scale, int M,
                         const uint8_t* e8t, const float* e_scale, int V, int D, float* out,
                         void* ws, cudaStream_t st);
size_t selfcond_ws_bytes(int M, int V, int D);
cudaError_t selfcond(const uint16_t* h, int M, const uint16_t* w, const uint16_t* e, int V,
                     int D, const float* inv_t, const float* lse, float* out, void* ws,
                     cudaStream_t st);

// P . E from bf16 probabilities (optionally unnormalised, times row_scale).
size_t probs_embed_ws_bytes(int M, int V, int D);
// e is the embedding table [V, D] row-major (read as an MN-major B operand).
cudaError_t probs_embed(const uint16_t* probs, size_t ldp, const float* row_scale, int M,
                        const uint16_t* e, int V, int D, float* out, void* ws,
                        cudaStream_t st);

// ---- fused lm-head pass of a step (heads_tc.cu) ------------------------------
size_t heads_ws_bytes(int M, int V, int n_draw);
size_t heads_probs_ld(int V);
// W's tiled copy for the pass with draw rows (224-row tiles x 64-column blocks,
// each block contiguous); 0 bytes when d_model is not a multiple of 64.
size_t heads_tiled_bytes(int V, int D);
cudaError_t heads_tile_weights(const uint16_t* w, int V, int D, uint16_t* out, cudaStream_t st);
// w_tiled (or null): the tiled copy of w, streamed instead of w when there are draw rows
cudaError_t denoise_heads(const uint16_t* h, int M, const uint16_t* draw_rows, int n_draw,
                          const uint16_t* w, const uint16_t* w_tiled, int V, int D,
                          const float* inv_t,
                          const float* inv_t_draw, RowStats out, float* lse_draw,
                          float* prob_scale, uint16_t* probs, size_t probs_ld, void* ws,
                          cudaStream_t st, const LabelGather* gather = nullptr);

// The fused pass on e4m3 operands (per-row scales h_scale [M], d_scale [n_draw],
// w_scale [V]); d_model a multiple of 16.
cudaError_t denoise_heads_fp8(const uint8_t* h8, const float* h_scale, int M,
                              const uint8_t* d8, const float* d_scale, int n_draw,
                              const uint8_t* w8, const float* w_scale, int V, int D,
                              const float* inv_t, const float* inv_t_draw, RowStats out,
                              float* lse_draw, float* prob_scale, uint16_t* probs,
                              size_t probs_ld, void* ws, cudaStream_t st,
                              const LabelGather* gather = nullptr);

// ---- attention (attn.cu) ---------------------------------------------------
struct AttnArgs {
  int B, C, Pmax, Hq, Hkv, d, W;
  const uint16_t *q, *kc, *vc, *kenc, *venc;
  const int32_t* page_table;
  int pages_per_req, n_pages, page_size;
  const int32_t* prompt_len;
  uint16_t* out;
  float* lse;
  int causal = 0;                     // encoder prefill (d = 512 tensor-core kernel only)
  const int32_t* seq_len = nullptr;   // causal: rows per request (q/k/v are [B, C, H, d])
  const int32_t* mode = nullptr;      // mixed batch: per request 1 = causal, 0 = decoder
  const int32_t* rows_len = nullptr;  // mixed batch: valid rows per request
  int sms = 0;                        // SMs to plan the grid for (0: all of the device)
};
size_t attn_ws_bytes(int B, int C, int Pmax, int Hq, int Hkv, int d, int W, int sms);
cudaError_t attn_decode(const AttnArgs& a, void* ws, cudaStream_t st);
// Merge split-KV partials ([splits][B][C][Hq][d] fp32 O, [splits][B][Hq][C] (m, l));
// with seq_len, rows at or past seq_len[b] are left untouched.
cudaError_t attn_combine(int B, int C, int Hq, int d, int splits, float* ws_o, float* ws_ml,
                         uint16_t* out, float* lse, cudaStream_t st,
                         const int32_t* seq_len = nullptr);
// d = 512 on tcgen05 (attn_tc.cu): 128 query rows x 256 output columns per CTA.
bool attn_tc_supported(const AttnArgs& a);
size_t attn_tc_ws_bytes(int B, int C, int Pmax, int Hq, int Hkv, int W, int sms);
cudaError_t attn_decode_tc(const AttnArgs& a, void* ws, cudaStream_t st);
// Copy the first seq_len[b] rows of k, v [B, P, Hkv, d] into the page pools
// [n_pages, page_size, Hkv, d] through page_table [B, pages_per_req].
cudaError_t kv_page_write(const uint16_t* k, const uint16_t* v, int B, int P, int Hkv, int d,
                          const int32_t* seq_len, const int32_t* page_table, int pages_per_req,
                          int n_pages, int page_size, uint16_t* pool_k, uint16_t* pool_v,
                          cudaStream_t st);

// ---- small kernels (slot.cu) -----------------------------------------------
cudaError_t philox_fill(uint64_t seed, const uint32_t* ctr4, int n, uint32_t* out4,
                        cudaStream_t st);
cudaError_t slot_noise(const uint16_t* h, int M, const uint16_t* e, int V, int D,
                       const float* inv_t, const int32_t* slot_row, const int32_t* slot_req,
                       int S, int R, uint64_t seed, int step, uint16_t* rows_out,
                       float* inv_t_out, int32_t* tok_out, cudaStream_t st);
cudaError_t slot_finish(const uint16_t* rows, const float* inv_t_rows, const float* lse_rows,
                        const uint16_t* w, int V, int D, const int32_t* label_ids,
                        const int32_t* n_labels, int S, int R, int samples, float gate,
                        float* q_avg, float* h_slot, int32_t* chosen, float* lp_draws,
                        uint8_t* resampled, int32_t* n_reads, cudaStream_t st);
// The same with label tables of row stride L <= 256 (wide-label reads).
cudaError_t slot_finish_wide(const uint16_t* rows, const float* inv_t_rows, const float* lse_rows,
                             const uint16_t* w, int V, int D, const int32_t* label_ids,
                             const int32_t* n_labels, int L, int S, int R, int samples,
                             float gate, float* q_avg, float* h_slot, int32_t* chosen,
                             float* lp_draws, uint8_t* resampled, int32_t* n_reads,
                             cudaStream_t st);
// Diagnostic of the bounded-wait path (see dg_check_wait_timeout).
cudaError_t check_wait_timeout(uint64_t limit_ns, int* waited_us, cudaStream_t st);
cudaError_t ask_if_select(const int32_t* chosen1, int S1, const int32_t* cond_slot,
                          const int32_t* cond_value, const int32_t* q_owner,
                          const int32_t* q_label_ids, const int32_t* q_n_labels, int Q, int S2,
                          int32_t* label_ids2, int32_t* n_labels2, uint8_t* fired,
                          cudaStream_t st);
cudaError_t commit(int B, int C, const float* entropy, const int32_t* argmax,
                   const uint8_t* cand, const float* gamma, uint8_t* committed_state,
                   int32_t* token_state, uint8_t* commit_out, int32_t* tokens,
                   int32_t* n_commit, cudaStream_t st);
cudaError_t canvas_update(const uint16_t* h0, const float* e_sc, const uint16_t* emb, int V,
                          const int32_t* tokens, const uint8_t* committed, int M, int D,
                          uint16_t* h_out, cudaStream_t st);

}  // namespace dgi
