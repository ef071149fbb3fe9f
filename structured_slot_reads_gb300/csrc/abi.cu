// abi.cu -- the extern "C" entry points of libdg (declared in include/dg.h):
// synchronous argument validation, workspace sizing, the device status word,
// TMA descriptor creation and dispatch to the kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <set>

#include "dg.h"
#include "internal.h"

namespace {

__device__ int g_status;  // bits DG_DEV_*, sticky until dg_clear_status

constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {};
std::mutex g_mu;
// device addresses of this library's __device__ variables, per device, with the
// context they were looked up in
void* g_sym_addr[dgi::SYM_COUNT][kMaxDevices] = {};
uint64_t g_sym_ctx[dgi::SYM_COUNT][kMaxDevices] = {};

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return (dev >= 0 && dev < kMaxDevices) ? dev : -1;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool dims_lm(const dg_dims* d) { return d && dgi::lm_dims_ok(d->d_model, d->V); }

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

int launch_result(cudaError_t e) { return e == cudaSuccess ? DG_OK : DG_ERR_CUDA; }

}  // namespace

namespace dgi {

uint64_t context_id() {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_cur || !get_id) return 0;
  CUcontext c = nullptr;
  if (get_cur(&c) != CUDA_SUCCESS || !c) return 0;
  unsigned long long id = 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return (uint64_t)id + 1;  // 0 stands for "no context"
}

void* device_symbol(const void* symbol, int slot) {
  const int dev = current_device();
  if (dev < 0 || slot < 0 || slot >= SYM_COUNT) return nullptr;
  uint64_t ctx = context_id();
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sym_addr[slot][dev] && ctx != 0 && g_sym_ctx[slot][dev] == ctx)
    return g_sym_addr[slot][dev];
  // first use on this device, or a new context (after cudaDeviceReset the old
  // address belongs to a module that no longer exists): look it up again
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess || !p) return nullptr;
  if (ctx == 0) ctx = context_id();  // the lookup made the primary context current
  g_sym_addr[slot][dev] = p;
  g_sym_ctx[slot][dev] = ctx;
  return p;
}

int* status_ptr() { return static_cast<int*>(device_symbol(&g_status, SYM_STATUS)); }

int num_sms() {
  const int dev = current_device();
  if (dev < 0) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

int plan_sms(int share) {
  const int n = num_sms();
  return (share > 0 && share < n) ? share : n;
}

bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                       uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_u8_4d(CUtensorMap* map, const void* base, const uint64_t (&dims)[4],
                     const uint64_t (&stride_bytes)[3], const uint32_t (&box)[4]) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  const cuuint64_t st[3] = {stride_bytes[0], stride_bytes[1], stride_bytes[2]};
  const cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), d, st, bx, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, const uint64_t (&dims)[3],
                       const uint64_t (&stride_bytes)[2], const uint32_t (&box)[3]) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t st[2] = {stride_bytes[0], stride_bytes[1]};
  const cuuint32_t bx[3] = {box[0], box[1], box[2]};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), d, st, bx, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace dgi

namespace {

size_t slot_read_ws(const dg_dims* d, int rows) {
  using dgi::align_up;
  const size_t r = (size_t)rows;
  return align_up(r * d->d_model * 2, 256) + 5 * align_up(r * 4, 256) +
         dgi::lmhead_ws_bytes(rows, d->V);
}

// Workspace of the lm-head passes: the per-CTA partial statistics, then the
// row -> slot map of a label gather ([M] int32).
size_t lmhead_ws(const dg_dims* d, int M) {
  return dgi::lmhead_ws_bytes(M, d->V) + dgi::align_up((size_t)M * 4, 256);
}

// The label gather of an lm-head pass (slot s at row slot_row[s], label table
// of stride 26, label_lp [S][26] = z - lse): none when S == 0, else every
// pointer is required.  Call after the workspace has been checked.
int lm_gather(const dg_dims* d, int M, const int32_t* slot_row, const int32_t* label_ids,
              const int32_t* n_labels, int S, float* label_lp, void* workspace,
              dgi::LabelGather* g) {
  *g = dgi::LabelGather{};
  if (S < 0) return DG_ERR_ARG;
  if (S == 0) return DG_OK;
  if (!slot_row || !label_ids || !n_labels || !label_lp) return DG_ERR_ARG;
  if (S > M) return DG_ERR_SHAPE;
  g->label_ids = label_ids;
  g->n_labels = n_labels;
  g->slot_row = slot_row;
  g->row_slot = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) +
                                           dgi::lmhead_ws_bytes(M, d->V));
  g->out = label_lp;
  g->L = DG_MAX_LABELS;
  g->S = S;
  g->R = 0;
  g->sub_lse = 1;
  return DG_OK;
}

bool prefill_dims_ok(const dg_dims* d) {
  if (!d || d->B < 1 || d->P_max < 1 || d->Hq < 1 || d->Hkv < 1 || d->Hq % d->Hkv) return false;
  return d->d_head == 512 && 128 % (d->Hq / d->Hkv) == 0;
}

bool attn_dims_ok(const dg_dims* d) {
  if (!d || d->B < 1 || d->C < 1 || d->Hq < 1 || d->Hkv < 1 || d->P_max < 0 || d->W < 0)
    return false;
  if (d->Hq % d->Hkv) return false;
  const int g = d->Hq / d->Hkv;
  if (64 % g) return false;
  return d->d_head == 64 || d->d_head == 512;
}

// The slot read with label tables of row stride L (26 for dg_slot_read).
int slot_read_impl(const dg_dims* d, const uint16_t* h, int M, const uint16_t* w, const uint16_t* e,
                   const float* inv_t, const int32_t* slot_row, const int32_t* slot_req,
                   const int32_t* label_ids, const int32_t* n_labels, int S, int L, uint64_t seed,
                 int step, int samples, float gate, float* q_avg, float* h_slot, int32_t* chosen,
                 float* lp_draws, uint8_t* resampled, int32_t* n_reads, int32_t* noise_tok_out,
                 void* workspace, size_t workspace_bytes, void* stream) {
  if (!d || S < 0 || samples < 1 || samples > 8 || M < 1) return DG_ERR_ARG;
  if (!dims_lm(d) || !pow2(d->V)) return DG_ERR_SHAPE;
  if (S == 0) return DG_OK;
  if (!h || !w || !e || !inv_t || !slot_row || !slot_req || !label_ids || !n_labels || !q_avg ||
      !h_slot || !chosen || !lp_draws || !resampled || !n_reads)
    return DG_ERR_ARG;
  if (!aligned(h, 16) || !aligned(w, 16) || !aligned(e, 16)) return DG_ERR_ARG;
  const int R = samples;
  const int rows = S * R;
  const size_t need = slot_read_ws(d, rows);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return DG_ERR_WORKSPACE;
  using dgi::align_up;
  uint8_t* p = static_cast<uint8_t*>(workspace);
  uint16_t* draw_rows = reinterpret_cast<uint16_t*>(p);
  p += align_up((size_t)rows * d->d_model * 2, 256);
  float* inv_rows = reinterpret_cast<float*>(p);
  p += align_up((size_t)rows * 4, 256);
  float* lse_rows = reinterpret_cast<float*>(p);
  p += align_up((size_t)rows * 4, 256);
  float* ent_rows = reinterpret_cast<float*>(p);
  p += align_up((size_t)rows * 4, 256);
  float* maxz_rows = reinterpret_cast<float*>(p);
  p += align_up((size_t)rows * 4, 256);
  int32_t* arg_rows = reinterpret_cast<int32_t*>(p);
  p += align_up((size_t)rows * 4, 256);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t err = dgi::slot_noise(h, M, e, d->V, d->d_model, inv_t, slot_row, slot_req, S, R,
                                    seed, step, draw_rows, inv_rows, noise_tok_out, st);
  if (err != cudaSuccess) return DG_ERR_CUDA;
  // the pass gathers every draw's label logits z/T into lp_draws from its
  // accumulators; the finish then works from them alone
  dgi::LabelGather g{};
  g.label_ids = label_ids;
  g.n_labels = n_labels;
  g.out = lp_draws;
  g.L = L;
  g.S = S;
  g.R = R;
  err = dgi::lmhead_stats(draw_rows, rows, w, d->V, d->d_model, inv_rows,
                          dgi::RowStats{lse_rows, ent_rows, maxz_rows, arg_rows}, p, st, &g);
  if (err != cudaSuccess) return DG_ERR_CUDA;
  err = (L == DG_MAX_LABELS)
            ? dgi::slot_finish(nullptr, inv_rows, lse_rows, nullptr, d->V, d->d_model, label_ids,
                               n_labels, S, R, samples, gate, q_avg, h_slot, chosen, lp_draws,
                               resampled, n_reads, st)
            : dgi::slot_finish_wide(nullptr, inv_rows, lse_rows, nullptr, d->V, d->d_model,
                                    label_ids, n_labels, L, S, R, samples, gate, q_avg, h_slot,
                                    chosen, lp_draws, resampled, n_reads, st);
  return launch_result(err);
}

}  // namespace

extern "C" {

const char* dg_strerror(int code) {
  switch (code) {
    case DG_OK: return "ok";
    case DG_ERR_ARG: return "invalid argument (null pointer, size or alignment)";
    case DG_ERR_TOO_MANY_LABELS: return "at most 26 alternatives per slot";
    case DG_ERR_LABEL: return "duplicate label id or label id outside the vocabulary";
    case DG_ERR_SHAPE: return "unsupported or inconsistent dimensions";
    case DG_ERR_CUDA: return "CUDA launch or runtime error";
    case DG_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown dg status";
  }
}

int dg_num_sms(void) {
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n == 0) return -1;
  return dgi::num_sms();
}

size_t dg_workspace_bytes(const dg_dims* d, int which, int rows) {
  if (!d) return 0;
  switch (which) {
    case DG_WS_ATTN:
      if (!attn_dims_ok(d)) return 0;
      return dgi::attn_ws_bytes(d->B, d->C, d->P_max, d->Hq, d->Hkv, d->d_head,
                                d->W > d->C ? d->C : d->W, d->sm_share);
    case DG_WS_LMHEAD:
      if (!dims_lm(d) || rows < 1) return 0;
      return lmhead_ws(d, rows);
    case DG_WS_SLOT_READ:
      if (!dims_lm(d) || rows < 1) return 0;
      return slot_read_ws(d, rows);
    case DG_WS_SELFCOND:
      if (!dims_lm(d) || rows < 1) return 0;
      return dgi::selfcond_ws_bytes(rows, d->V, d->d_model);
    case DG_WS_HEADS: {
      if (!dims_lm(d) || rows < 1) return 0;
      const size_t a = dgi::heads_ws_bytes(rows, d->V, 0);
      const size_t b = dgi::heads_ws_bytes(rows, d->V, 1);
      return a > b ? a : b;
    }
    case DG_WS_PROBS_EMBED:
      if (!dims_lm(d) || rows < 1) return 0;
      return dgi::probs_embed_ws_bytes(rows, d->V, d->d_model);
    case DG_WS_PROBS_EMBED8:
      if (!dims_lm(d) || rows < 1) return 0;
      return dgi::probs_embed8_ws_bytes(rows, d->V, d->d_model);
    case DG_WS_LMHEAD_NVFP4_MMA:
      if (!dims_lm(d) || !dgi::lmhead_nvfp4_mma_ok(rows, d->d_model)) return 0;
      return dgi::lmhead_nvfp4_mma_ws_bytes(rows, d->V, d->d_model);
    case DG_WS_PREFILL:
      if (!prefill_dims_ok(d)) return 0;
      return dgi::attn_tc_ws_bytes(d->B, d->P_max, 0, d->Hq, d->Hkv, d->P_max, d->sm_share);
    default:
      return 0;
  }
}

size_t dg_probs_ld(int V) { return V < 1 ? 0 : dgi::heads_probs_ld(V); }

size_t dg_heads_weights_bytes(const dg_dims* d) {
  if (!d || !dims_lm(d)) return 0;
  return dgi::heads_tiled_bytes(d->V, d->d_model);
}

int dg_heads_weights_tile(const dg_dims* d, const uint16_t* w, uint16_t* w_tiled, void* stream) {
  if (!d) return DG_ERR_ARG;
  if (!dims_lm(d) || !dgi::heads_tiled_bytes(d->V, d->d_model)) return DG_ERR_SHAPE;
  if (!w || !w_tiled || !aligned(w, 16) || !aligned(w_tiled, 16)) return DG_ERR_ARG;
  return launch_result(dgi::heads_tile_weights(w, d->V, d->d_model, w_tiled,
                                               static_cast<cudaStream_t>(stream)));
}

int dg_denoise_heads(const dg_dims* d, const uint16_t* h, int M, const uint16_t* draw_rows,
                     int n_draw, const uint16_t* w, const uint16_t* w_tiled,
                     const float* inv_t, const float* inv_t_draw,
                     float* lse, float* entropy, float* maxz, int32_t* argmax, float* lse_draw,
                     const int32_t* draw_label_ids, const int32_t* draw_n_labels, int draw_R,
                     float* draw_label_z, float* prob_scale, uint16_t* probs, size_t probs_ld,
                     void* workspace, size_t workspace_bytes, void* stream) {
  if (!d || M < 1 || n_draw < 0 || n_draw > 16) return DG_ERR_ARG;
  if (!dims_lm(d)) return DG_ERR_SHAPE;
  if (!h || !w || !inv_t || !lse || !entropy || !maxz || !argmax || !prob_scale)
    return DG_ERR_ARG;
  if (n_draw > 0 && (!draw_rows || !inv_t_draw || !lse_draw)) return DG_ERR_ARG;
  if (!aligned(h, 16) || !aligned(w, 16) || (n_draw > 0 && !aligned(draw_rows, 16)))
    return DG_ERR_ARG;
  if (w_tiled && (!aligned(w_tiled, 16) || !dgi::heads_tiled_bytes(d->V, d->d_model)))
    return DG_ERR_ARG;
  if (probs && (probs_ld < (size_t)d->V || probs_ld % 64 || !aligned(probs, 32)))
    return DG_ERR_ARG;
  dgi::LabelGather g{};
  if (draw_label_z && n_draw > 0) {
    // draw j is draw j % draw_R of slot j / draw_R
    if (!draw_label_ids || !draw_n_labels || draw_R < 1 || n_draw % draw_R) return DG_ERR_ARG;
    g.label_ids = draw_label_ids;
    g.n_labels = draw_n_labels;
    g.out = draw_label_z;
    g.L = DG_MAX_LABELS;
    g.S = n_draw / draw_R;
    g.R = draw_R;
  }
  const size_t need = dg_workspace_bytes(d, DG_WS_HEADS, M);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return DG_ERR_WORKSPACE;
  return launch_result(dgi::denoise_heads(h, M, draw_rows, n_draw, w, w_tiled, d->V, d->d_model,
                                          inv_t, inv_t_draw,
                                          dgi::RowStats{lse, entropy, maxz, argmax},
                                          lse_draw, prob_scale, probs, probs_ld, workspace,
                                          static_cast<cudaStream_t>(stream), &g));
}

int dg_denoise_heads_fp8(const dg_dims* d, const uint8_t* h8, const float* h_scale, int M,
                         const uint8_t* draw8, const float* draw_scale, int n_draw,
                         const uint8_t* w8, const float* w_scale, const float* inv_t,
                         const float* inv_t_draw, float* lse, float* entropy, float* maxz,
                         int32_t* argmax, float* lse_draw, const int32_t* draw_label_ids,
                         const int32_t* draw_n_labels, int draw_R, float* draw_label_z,
                         float* prob_scale, uint16_t* probs, size_t probs_ld, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (!d || M < 1 || n_draw < 0 || n_draw > 16) return DG_ERR_ARG;
  if (!dims_lm(d) || d->d_model % 16) return DG_ERR_SHAPE;
  if (!h8 || !h_scale || !w8 || !w_scale || !inv_t || !lse || !entropy || !maxz || !argmax ||
      !prob_scale)
    return DG_ERR_ARG;
  if (n_draw > 0 && (!draw8 || !draw_scale || !inv_t_draw || !lse_draw)) return DG_ERR_ARG;
  if (!aligned(h8, 16) || !aligned(w8, 16) || !aligned(w_scale, 16) ||
      (n_draw > 0 && !aligned(draw8, 16)))
    return DG_ERR_ARG;
  if (probs && (probs_ld < (size_t)d->V || probs_ld % 64 || !aligned(probs, 32)))
    return DG_ERR_ARG;
  dgi::LabelGather g{};
  if (draw_label_z && n_draw > 0) {
    if (!draw_label_ids || !draw_n_labels || draw_R < 1 || n_draw % draw_R) return DG_ERR_ARG;
    g.label_ids = draw_label_ids;
    g.n_labels = draw_n_labels;
    g.out = draw_label_z;
    g.L = DG_MAX_LABELS;
    g.S = n_draw / draw_R;
    g.R = draw_R;
  }
  const size_t need = dg_workspace_bytes(d, DG_WS_HEADS, M);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return DG_ERR_WORKSPACE;
  return launch_result(dgi::denoise_heads_fp8(
      h8, h_scale, M, draw8, draw_scale, n_draw, w8, w_scale, d->V, d->d_model, inv_t, inv_t_draw,
      dgi::RowStats{lse, entropy, maxz, argmax}, lse_draw, prob_scale, probs, probs_ld, workspace,
      static_cast<cudaStream_t>(stream), &g));
}

int dg_selfcond_from_probs(const dg_dims* d, const uint16_t* probs, size_t probs_ld,
                           const float* prob_scale, int M, const uint16_t* e, float* out,
                           void* workspace, size_t workspace_bytes, void* stream) {
  if (!d || M < 1) return DG_ERR_ARG;
  if (!dims_lm(d) || d->V % 8) return DG_ERR_SHAPE;
  if (!probs || !prob_scale || !e || !out) return DG_ERR_ARG;
  if (probs_ld < (size_t)d->V || probs_ld % 8 || !aligned(probs, 16) || !aligned(e, 16) ||
      !aligned(out, 16))
    return DG_ERR_ARG;
  const size_t need = dg_workspace_bytes(d, DG_WS_PROBS_EMBED, M);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return DG_ERR_WORKSPACE;
  return launch_result(dgi::probs_embed(probs, probs_ld, prob_scale, M, e, d->V, d->d_model,
                                        out, workspace, static_cast<cudaStream_t>(stream)));
}

int dg_validate_slots_wide(const dg_dims* d, const int32_t* slot_row, const int32_t* label_ids,
                           const int32_t* n_labels, int S, int L, int M) {
  if (!d || S < 0 || M < 0) return DG_ERR_ARG;
  if (L < 1 || L > DG_MAX_WIDE_LABELS) return DG_ERR_TOO_MANY_LABELS;
  if (S > 0 && (!slot_row || !label_ids || !n_labels)) return DG_ERR_ARG;
  for (int s = 0; s < S; ++s) {
    const int n = n_labels[s];
    if (n > L) return DG_ERR_TOO_MANY_LABELS;
    if (n < 1) return DG_ERR_LABEL;
    if (slot_row[s] < 0 || slot_row[s] >= M) return DG_ERR_SHAPE;
    std::set<int32_t> seen;
    for (int k = 0; k < n; ++k) {
      const int32_t id = label_ids[(long long)s * L + k];
      if (id < 0 || id >= d->V) return DG_ERR_LABEL;
      if (!seen.insert(id).second) return DG_ERR_LABEL;
    }
  }
  return DG_OK;
}

int dg_validate_slots(const dg_dims* d, const int32_t* slot_row, const int32_t* label_ids,
                      const int32_t* n_labels, int S, int M) {
  return dg_validate_slots_wide(d, slot_row, label_ids, n_labels, S, DG_MAX_LABELS, M);
}

int dg_get_status(void* stream, int32_t* status_out) {
  if (!status_out) return DG_ERR_ARG;
  int* p = dgi::status_ptr();
  if (!p) return DG_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, p, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return DG_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return DG_ERR_CUDA;
  *status_out = v;
  return DG_OK;
}

int dg_clear_status(void* stream) {
  int* p = dgi::status_ptr();
  if (!p) return DG_ERR_CUDA;
  return launch_result(cudaMemsetAsync(p, 0, sizeof(int), static_cast<cudaStream_t>(stream)));
}

int dg_philox_fill(uint64_t seed, const uint32_t* ctr4, int n, uint32_t* out4, void* stream) {
  if (n < 0 || (n > 0 && (!ctr4 || !out4))) return DG_ERR_ARG;
  if (!aligned(ctr4, 16) || !aligned(out4, 16)) return DG_ERR_ARG;
  return launch_result(dgi::philox_fill(seed, ctr4, n, out4, static_cast<cudaStream_t>(stream)));
}

int dg_attn_decode(const dg_dims* d, const uint16_t* q, const uint16_t* kc, const uint16_t* vc,
                   const uint16_t* kenc, const uint16_t* venc, const int32_t* page_table,
                   int pages_per_req, int n_pages, int page_size, const int32_t* prompt_len,
                   uint16_t* out, float* lse, void* workspace, size_t workspace_bytes,
                   void* stream) {
  if (!d) return DG_ERR_ARG;
  if (!attn_dims_ok(d)) return DG_ERR_SHAPE;
  if (!q || !kc || !vc || !prompt_len || !out || !lse) return DG_ERR_ARG;
  if (d->P_max > 0 && (!kenc || !venc)) return DG_ERR_ARG;
  for (const void* p : {(const void*)q, (const void*)kc, (const void*)vc, (const void*)kenc,
                        (const void*)venc, (const void*)out})
    if (!aligned(p, 16)) return DG_ERR_ARG;
  if (page_table) {
    if (page_size < 1 || n_pages < 1 ||
        (long long)pages_per_req * page_size < (long long)d->P_max)
      return DG_ERR_SHAPE;
  }
  const size_t need = dg_workspace_bytes(d, DG_WS_ATTN, 0);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return DG_ERR_WORKSPACE;
  dgi::AttnArgs a{};
  a.sms = d->sm_share;
  a.B = d->B;
  a.C = d->C;
  a.Pmax = d->P_max;
  a.Hq = d->Hq;
  a.Hkv = d->Hkv;
  a.d = d->d_head;
  a.W = d->W;
  a.q = q;
  a.kc = kc;
  a.vc = vc;
  a.kenc = kenc ? kenc : kc;
  a.venc = venc ? venc : vc;
  a.page_table = page_table;
  a.pages_per_req = pages_per_req;
  a.n_pages = n_pages;
  a.page_size = page_size;
  a.prompt_len = prompt_len;
  a.out = out;
  a.lse = lse;
  // 512-wide heads run only on the tensor-core kernel: page sizes it cannot
  // take are rejected here rather than run on another kernel
  if (a.d == 512 && !dgi::attn_tc_supported(a)) return DG_ERR_SHAPE;
  return launch_result(dgi::attn_decode(a, workspace, static_cast<cudaStream_t>(stream)));
}

int dg_lmhead_logsoftmax_entropy(const dg_dims* d, const uint16_t* h, int M, const uint16_t* w,
                                 const float* inv_t, const int32_t* slot_row,
                                 const int32_t* label_ids, const int32_t* n_labels, int S,
                                 float* lse, float* entropy, float* maxz, int32_t* argmax,
                                 float* label_lp, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  if (!d || M < 1 || S < 0) return DG_ERR_ARG;
  if (!dims_lm(d)) return DG_ERR_SHAPE;
  if (!h || !w || !inv_t || !lse || !entropy || !maxz || !argmax) return DG_ERR_ARG;
  if (!aligned(h, 16) || !aligned(w, 16)) return DG_ERR_ARG;
  const size_t need = lmhead_ws(d, M);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return DG_ERR_WORKSPACE;
  dgi::LabelGather g;
  if (int rc = lm_gather(d, M, slot_row, label_ids, n_labels, S, label_lp, workspace, &g))
    return rc;
  return launch_result(dgi::lmhead_stats(h, M, w, d->V, d->d_model, inv_t,
                                         dgi::RowStats{lse, entropy, maxz, argmax}, workspace,
                                         static_cast<cudaStream_t>(stream), &g));
}

int dg_slot_noise(const dg_dims* d, const uint16_t* h, int M, const uint16_t* e,
                  const float* inv_t, const int32_t* slot_row, const int32_t* slot_req, int S,
                  int R, uint64_t seed, int step, uint16_t* rows_out, float* inv_t_out,
                  int32_t* noise_tok_out, void* stream) {
  if (!d || S < 0 || R < 1 || R > 8 || M < 1) return DG_ERR_ARG;
  if (!dims_lm(d) || !pow2(d->V)) return DG_ERR_SHAPE;
  if (S > 0 && (!h || !e || !inv_t || !slot_row || !slot_req || !rows_out || !inv_t_out))
    return DG_ERR_ARG;
  if (!aligned(h, 16) || !aligned(e, 16) || !aligned(rows_out, 16)) return DG_ERR_ARG;
  return launch_result(dgi::slot_noise(h, M, e, d->V, d->d_model, inv_t, slot_row, slot_req, S,
                                       R, seed, step, rows_out, inv_t_out, noise_tok_out,
                                       static_cast<cudaStream_t>(stream)));
}

int dg_slot_finish(const dg_dims* d, const uint16_t* rows, const float* inv_t_rows,
                   const float* lse_rows, const uint16_t* w, const int32_t* label_ids,
                   const int32_t* n_labels, int S, int R, int samples, float gate, float* q_avg,
                   float* h_slot, int32_t* chosen, float* lp_draws, uint8_t* resampled,
                   int32_t* n_reads, void* stream) {
  if (!d || S < 0 || R < 1 || R > 8 || samples < 1 || samples > R) return DG_ERR_ARG;
  if (!dims_lm(d)) return DG_ERR_SHAPE;
  if (S > 0 && (!lse_rows || !label_ids || !n_labels || !q_avg || !h_slot || !chosen ||
                !lp_draws || !resampled || !n_reads))
    return DG_ERR_ARG;
  // rows == null: lp_draws already holds the gathered label logits
  if (S > 0 && rows && (!inv_t_rows || !w)) return DG_ERR_ARG;
  if (!aligned(rows, 4) || !aligned(w, 4)) return DG_ERR_ARG;
  return launch_result(dgi::slot_finish(rows, inv_t_rows, lse_rows, w, d->V, d->d_model,
                                        label_ids, n_labels, S, R, samples, gate, q_avg, h_slot,
                                        chosen, lp_draws, resampled, n_reads,
                                        static_cast<cudaStream_t>(stream)));
}

int dg_slot_read(const dg_dims* d, const uint16_t* h, int M, const uint16_t* w, const uint16_t* e,
                 const float* inv_t, const int32_t* slot_row, const int32_t* slot_req,
                 const int32_t* label_ids, const int32_t* n_labels, int S, uint64_t seed,
                 int step, int samples, float gate, float* q_avg, float* h_slot, int32_t* chosen,
                 float* lp_draws, uint8_t* resampled, int32_t* n_reads, int32_t* noise_tok_out,
                 void* workspace, size_t workspace_bytes, void* stream) {
  return slot_read_impl(d, h, M, w, e, inv_t, slot_row, slot_req, label_ids, n_labels, S,
                        DG_MAX_LABELS, seed, step, samples, gate, q_avg, h_slot, chosen, lp_draws,
                        resampled, n_reads, noise_tok_out, workspace, workspace_bytes, stream);
}

int dg_slot_read_wide(const dg_dims* d, const uint16_t* h, int M, const uint16_t* w,
                      const uint16_t* e, const float* inv_t, const int32_t* slot_row,
                      const int32_t* slot_req, const int32_t* label_ids, const int32_t* n_labels,
                      int S, int L, uint64_t seed, int step, int samples, float gate,
                      float* q_avg, float* h_slot, int32_t* chosen, float* lp_draws,
                      uint8_t* resampled, int32_t* n_reads, int32_t* noise_tok_out,
                      void* workspace, size_t workspace_bytes, void* stream) {
  if (L < 1 || L > DG_MAX_WIDE_LABELS) return DG_ERR_TOO_MANY_LABELS;
  return slot_read_impl(d, h, M, w, e, inv_t, slot_row, slot_req, label_ids, n_labels, S, L,
                        seed, step, samples, gate, q_avg, h_slot, chosen, lp_draws, resampled,
                        n_reads, noise_tok_out, workspace, workspace_bytes, stream);
}

int dg_prefill_attn(const dg_dims* d, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const int32_t* prompt_len, uint16_t* out, float* lse,
                    const int32_t* page_table, int pages_per_req, int n_pages, int page_size,
                    uint16_t* pool_k, uint16_t* pool_v, void* workspace, size_t workspace_bytes,
                    void* stream) {
  if (!d) return DG_ERR_ARG;
  if (!prefill_dims_ok(d)) return DG_ERR_SHAPE;
  if (!q || !k || !v || !prompt_len || !out || !lse) return DG_ERR_ARG;
  for (const void* p : {(const void*)q, (const void*)k, (const void*)v, (const void*)out})
    if (!aligned(p, 16)) return DG_ERR_ARG;
  if (page_table) {
    if (!pool_k || !pool_v || !aligned(pool_k, 16) || !aligned(pool_v, 16)) return DG_ERR_ARG;
    if (page_size < 1 || n_pages < 1 ||
        (long long)pages_per_req * page_size < (long long)d->P_max)
      return DG_ERR_SHAPE;
  }
  const size_t need = dg_workspace_bytes(d, DG_WS_PREFILL, 0);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return DG_ERR_WORKSPACE;
  dgi::AttnArgs a{};
  a.sms = d->sm_share;
  a.B = d->B;
  a.C = d->P_max;
  a.Pmax = 0;
  a.Hq = d->Hq;
  a.Hkv = d->Hkv;
  a.d = d->d_head;
  a.W = d->P_max;
  a.q = q;
  a.kc = k;
  a.vc = v;
  a.prompt_len = prompt_len;
  a.out = out;
  a.lse = lse;
  a.causal = 1;
  a.seq_len = prompt_len;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t err = dgi::attn_decode_tc(a, workspace, st);
  if (err == cudaSuccess && page_table)
    err = dgi::kv_page_write(k, v, d->B, d->P_max, d->Hkv, d->d_head, prompt_len, page_table,
                             pages_per_req, n_pages, page_size, pool_k, pool_v, st);
  return launch_result(err);
}

int dg_attn_mixed(const dg_dims* d, const int32_t* mode, const int32_t* rows_len,
                  const uint16_t* q, const uint16_t* kc, const uint16_t* vc, const uint16_t* kenc,
                  const uint16_t* venc, const int32_t* page_table, int pages_per_req,
                  int n_pages, int page_size, const int32_t* prompt_len, uint16_t* out,
                  float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!d) return DG_ERR_ARG;
  if (!attn_dims_ok(d) || d->d_head != 512) return DG_ERR_SHAPE;
  if (!mode || !rows_len || !q || !kc || !vc || !prompt_len || !out || !lse) return DG_ERR_ARG;
  if (d->P_max > 0 && (!kenc || !venc)) return DG_ERR_ARG;
  for (const void* p : {(const void*)q, (const void*)kc, (const void*)vc, (const void*)kenc,
                        (const void*)venc, (const void*)out})
    if (!aligned(p, 16)) return DG_ERR_ARG;
  if (page_table && (page_size < 1 || n_pages < 1 ||
                     (long long)pages_per_req * page_size < (long long)d->P_max))
    return DG_ERR_SHAPE;
  dgi::AttnArgs a{};
  a.sms = d->sm_share;
  a.B = d->B;
  a.C = d->C;
  a.Pmax = d->P_max;
  a.Hq = d->Hq;
  a.Hkv = d->Hkv;
  a.d = d->d_head;
  a.W = d->W;
  a.q = q;
  a.kc = kc;
  a.vc = vc;
  a.kenc = kenc ? kenc : kc;
  a.venc = venc ? venc : vc;
  a.page_table = page_table;
  a.pages_per_req = pages_per_req;
  a.n_pages = n_pages;
  a.page_size = page_size;
  a.prompt_len = prompt_len;
  a.out = out;
  a.lse = lse;
  a.mode = mode;
  a.rows_len = rows_len;
  if (!dgi::attn_tc_supported(a)) return DG_ERR_SHAPE;
  const size_t need = dg_workspace_bytes(d, DG_WS_ATTN, 0);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return DG_ERR_WORKSPACE;
  return launch_result(dgi::attn_decode_tc(a, workspace, static_cast<cudaStream_t>(stream)));
}

int dg_check_wait_timeout(int64_t limit_ns, int32_t* waited_us, void* stream) {
  if (limit_ns < 1 || limit_ns > 1000000000LL || !waited_us) return DG_ERR_ARG;
  return launch_result(dgi::check_wait_timeout((uint64_t)limit_ns, waited_us,
                                               static_cast<cudaStream_t>(stream)));
}

int dg_quantize_rows_e4m3(const uint16_t* x, int rows, int cols, uint8_t* q, float* scale,
                          void* stream) {
  if (rows < 0 || cols < 1) return DG_ERR_ARG;
  if (rows > 0 && (!x || !q || !scale)) return DG_ERR_ARG;
  return launch_result(
      dgi::quantize_rows_e4m3(x, rows, cols, q, scale, static_cast<cudaStream_t>(stream)));
}

int dg_quantize_cols_e4m3(const uint16_t* x, int rows, int cols, uint8_t* qt, float* scale,
                          void* stream) {
  if (rows < 0 || cols < 1) return DG_ERR_ARG;
  if (rows > 0 && (!x || !qt || !scale || !aligned(scale, 4))) return DG_ERR_ARG;
  return launch_result(
      dgi::quantize_cols_e4m3(x, rows, cols, qt, scale, static_cast<cudaStream_t>(stream)));
}

int dg_selfcond_from_probs8(const dg_dims* d, const uint8_t* p8, const float* p_scale,
                            const float* row_scale, int M, const uint8_t* e8t,
                            const float* e_scale, float* out, void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (!d || M < 1) return DG_ERR_ARG;
  if (!dims_lm(d) || d->V % 16 || d->d_model % 4) return DG_ERR_SHAPE;
  if (!p8 || !p_scale || !e8t || !e_scale || !out) return DG_ERR_ARG;
  if (!aligned(p8, 16) || !aligned(e8t, 16) || !aligned(e_scale, 16) || !aligned(out, 16))
    return DG_ERR_ARG;
  const size_t need = dg_workspace_bytes(d, DG_WS_PROBS_EMBED8, M);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return DG_ERR_WORKSPACE;
  return launch_result(dgi::probs_embed8(p8, p_scale, row_scale, M, e8t, e_scale, d->V,
                                         d->d_model, out, workspace,
                                         static_cast<cudaStream_t>(stream)));
}

int dg_lmhead_logsoftmax_entropy_fp8(const dg_dims* d, const uint8_t* h8, const float* h_scale,
                                     int M, const uint8_t* w8, const float* w_scale,
                                     const float* inv_t, const int32_t* slot_row,
                                     const int32_t* label_ids, const int32_t* n_labels, int S,
                                     float* lse, float* entropy, float* maxz, int32_t* argmax,
                                     float* label_lp, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  if (!d || M < 1 || S < 0) return DG_ERR_ARG;
  if (!dims_lm(d) || d->d_model % 16) return DG_ERR_SHAPE;
  if (!h8 || !h_scale || !w8 || !w_scale || !inv_t || !lse || !entropy || !maxz || !argmax)
    return DG_ERR_ARG;
  if (!aligned(h8, 16) || !aligned(w8, 16) || !aligned(w_scale, 16)) return DG_ERR_ARG;
  const size_t need = dg_workspace_bytes(d, DG_WS_LMHEAD, M);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return DG_ERR_WORKSPACE;
  dgi::LabelGather g;
  if (int rc = lm_gather(d, M, slot_row, label_ids, n_labels, S, label_lp, workspace, &g))
    return rc;
  return launch_result(dgi::lmhead_stats_fp8(h8, h_scale, M, w8, w_scale, d->V, d->d_model, inv_t,
                                             dgi::RowStats{lse, entropy, maxz, argmax}, workspace,
                                             static_cast<cudaStream_t>(stream), &g));
}

int dg_quantize_nvfp4(const uint16_t* x, int rows, int cols, uint8_t* codes, uint8_t* scales,
                      float* g, void* stream) {
  if (rows < 0 || cols < 1) return DG_ERR_ARG;
  if (cols % 64) return DG_ERR_SHAPE;
  if (rows > 0 && (!x || !codes || !scales || !g)) return DG_ERR_ARG;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 4) || !aligned(g, 4))
    return DG_ERR_ARG;
  return launch_result(
      dgi::quantize_nvfp4(x, rows, cols, codes, scales, g, static_cast<cudaStream_t>(stream)));
}

int dg_lmhead_logsoftmax_entropy_nvfp4(const dg_dims* d, const uint16_t* h, int M,
                                       const uint8_t* codes, const uint8_t* scales,
                                       const float* g, const float* inv_t,
                                       const int32_t* slot_row, const int32_t* label_ids,
                                       const int32_t* n_labels, int S, float* lse,
                                       float* entropy, float* maxz, int32_t* argmax,
                                       float* label_lp, void* workspace, size_t workspace_bytes,
                                       void* stream) {
  if (!d || M < 1 || S < 0) return DG_ERR_ARG;
  if (!dims_lm(d) || d->d_model % 64 || d->V % 4) return DG_ERR_SHAPE;
  if (!h || !codes || !scales || !g || !inv_t || !lse || !entropy || !maxz || !argmax)
    return DG_ERR_ARG;
  if (!aligned(h, 16) || !aligned(codes, 16) || !aligned(scales, 16) || !aligned(g, 4))
    return DG_ERR_ARG;
  const size_t need = dg_workspace_bytes(d, DG_WS_LMHEAD, M);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return DG_ERR_WORKSPACE;
  dgi::LabelGather lg;
  if (int rc = lm_gather(d, M, slot_row, label_ids, n_labels, S, label_lp, workspace, &lg))
    return rc;
  return launch_result(dgi::lmhead_stats_nvfp4(h, M, codes, scales, g, d->V, d->d_model, inv_t,
                                               dgi::RowStats{lse, entropy, maxz, argmax},
                                               workspace, static_cast<cudaStream_t>(stream),
                                               &lg));
}

size_t dg_nvfp4_mma_codes_bytes(int rows, int cols) {
  if (rows < 1 || cols < 64 || cols % 64) return 0;
  return (size_t)((rows + 127) / 128) * ((cols / 64 + 3) / 4) * 128 * 128;
}

int dg_quantize_nvfp4_mma(const uint16_t* x, int rows, int cols, uint8_t* codes, uint8_t* sf,
                          float* g, void* stream) {
  if (rows < 0 || cols < 1) return DG_ERR_ARG;
  if (cols % 64) return DG_ERR_SHAPE;
  if (rows > 0 && (!x || !codes || !sf || !g)) return DG_ERR_ARG;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(sf, 4) || !aligned(g, 4))
    return DG_ERR_ARG;
  return launch_result(
      dgi::quantize_nvfp4_mma(x, rows, cols, codes, sf, g, static_cast<cudaStream_t>(stream)));
}

int dg_lmhead_logsoftmax_entropy_nvfp4_mma(const dg_dims* d, const uint16_t* h, int M,
                                           const uint8_t* codes, const uint8_t* sf,
                                           const float* g, const float* inv_t,
                                           const int32_t* slot_row, const int32_t* label_ids,
                                           const int32_t* n_labels, int S, float* lse,
                                           float* entropy, float* maxz, int32_t* argmax,
                                           float* label_lp, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  if (!d || M < 1 || S < 0) return DG_ERR_ARG;
  if (!dims_lm(d) || !dgi::lmhead_nvfp4_mma_ok(M, d->d_model)) return DG_ERR_SHAPE;
  if (!h || !codes || !sf || !g || !inv_t || !lse || !entropy || !maxz || !argmax)
    return DG_ERR_ARG;
  if (!aligned(h, 16) || !aligned(codes, 16) || !aligned(sf, 16) || !aligned(g, 4))
    return DG_ERR_ARG;
  const size_t need = dg_workspace_bytes(d, DG_WS_LMHEAD_NVFP4_MMA, M);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return DG_ERR_WORKSPACE;
  dgi::LabelGather lg;
  if (int rc = lm_gather(d, M, slot_row, label_ids, n_labels, S, label_lp, workspace, &lg))
    return rc;
  return launch_result(dgi::lmhead_stats_nvfp4_mma(h, M, codes, sf, g, d->V, d->d_model, inv_t,
                                                   dgi::RowStats{lse, entropy, maxz, argmax},
                                                   workspace, static_cast<cudaStream_t>(stream),
                                                   &lg));
}

int dg_ask_if_select(const int32_t* chosen1, int S1, const int32_t* cond_slot,
                     const int32_t* cond_value, const int32_t* q_owner,
                     const int32_t* q_label_ids, const int32_t* q_n_labels, int Q, int S2,
                     int32_t* label_ids2, int32_t* n_labels2, uint8_t* fired, void* stream) {
  if (S1 < 0 || Q < 0 || S2 < 0) return DG_ERR_ARG;
  if (S2 > 0 && (!label_ids2 || !n_labels2)) return DG_ERR_ARG;
  if (Q > 0 && (!chosen1 || !cond_slot || !cond_value || !q_owner || !q_label_ids ||
                !q_n_labels))
    return DG_ERR_ARG;
  return launch_result(dgi::ask_if_select(chosen1, S1, cond_slot, cond_value, q_owner,
                                          q_label_ids, q_n_labels, Q, S2, label_ids2, n_labels2,
                                          fired, static_cast<cudaStream_t>(stream)));
}

int dg_commit(const dg_dims* d, const float* entropy, const int32_t* argmax, const uint8_t* cand,
              const float* gamma, uint8_t* committed_state, int32_t* token_state,
              uint8_t* commit, int32_t* tokens, int32_t* n_commit, void* stream) {
  if (!d || d->B < 1 || d->C < 1) return DG_ERR_ARG;
  if (d->C > 1024) return DG_ERR_SHAPE;
  if (!entropy || !argmax || !cand || !gamma || !commit || !tokens || !n_commit)
    return DG_ERR_ARG;
  return launch_result(dgi::commit(d->B, d->C, entropy, argmax, cand, gamma, committed_state,
                                   token_state, commit, tokens, n_commit,
                                   static_cast<cudaStream_t>(stream)));
}

int dg_selfcond_embed(const dg_dims* d, const uint16_t* h, int M, const uint16_t* w,
                      const uint16_t* e, const float* inv_t, const float* lse, float* out,
                      void* workspace, size_t workspace_bytes, void* stream) {
  if (!d || M < 1) return DG_ERR_ARG;
  if (!dims_lm(d) || d->V % 8) return DG_ERR_SHAPE;
  if (!h || !w || !e || !inv_t || !lse || !out) return DG_ERR_ARG;
  if (!aligned(h, 16) || !aligned(w, 16) || !aligned(e, 16) || !aligned(out, 16))
    return DG_ERR_ARG;
  const size_t need = dgi::selfcond_ws_bytes(M, d->V, d->d_model);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return DG_ERR_WORKSPACE;
  return launch_result(dgi::selfcond(h, M, w, e, d->V, d->d_model, inv_t, lse, out, workspace,
                                     static_cast<cudaStream_t>(stream)));
}


int dg_canvas_update(const dg_dims* d, const uint16_t* h0, const float* e_sc, const uint16_t* emb,
                     const int32_t* tokens, const uint8_t* committed, int M, uint16_t* h_out,
                     void* stream) {
  if (!d || M < 0 || d->d_model < 2 || d->d_model % 2) return DG_ERR_SHAPE;
  if (M > 0 && (!h0 || !e_sc || !emb || !tokens || !committed || !h_out)) return DG_ERR_ARG;
  if (!aligned(h0, 4) || !aligned(e_sc, 8) || !aligned(emb, 4) || !aligned(h_out, 4))
    return DG_ERR_ARG;
  return launch_result(dgi::canvas_update(h0, e_sc, emb, d->V, tokens, committed, M, d->d_model,
                                          h_out, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
