// noalloc.cu -- a variant of the lm-head pass that needs no caller-allocated
// workspace.
//
// Some callers cannot call cudaMalloc, or cannot hand the library a device
// buffer they own: a host runtime that forbids allocation once serving has
// started (all memory is reserved up front and the allocator is locked), a
// plugin that only sees the tensors it is given, or code running where the
// allocator must not be touched.  dg_lmhead_logsoftmax_entropy_noalloc keeps
// the pass's scratch (the per-CTA partial row statistics that the finalize
// kernel merges) in a fixed array compiled into this library instead of a
// workspace argument.  The array exists once per GPU that loads the library
// and stays allocated until the process exits.
#include <cuda_runtime.h>

#include <cstdint>

#include "dg.h"
#include "internal.h"

namespace {

// Largest scratch the no-allocation pass may use: five fp32 planes of
// [rows][CTAs] partial statistics, 2.5 MiB: DG_NOALLOC_MAX_ROWS rows with up
// to 256 CTAs sharing the vocabulary.
constexpr size_t kScratchBytes = (size_t)5 * 256 * DG_NOALLOC_MAX_ROWS * sizeof(float);
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch array on the current device.  The host-side
// symbol is only a stand-in and must not reach a kernel; the address is looked
// up with cudaGetSymbolAddress (no allocation) the first time on a device and
// again whenever the current context is a different one (after cudaDeviceReset
// the library's module is loaded anew and the old address is stale).
void* scratch_on_current_device() {
  return dgi::device_symbol(g_noalloc_scratch, dgi::SYM_NOALLOC_SCRATCH);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int dg_lmhead_logsoftmax_entropy_noalloc(const dg_dims* d, const uint16_t* h, int M,
                                                    const uint16_t* w, const float* inv_t,
                                                    float* lse, float* entropy, float* maxz,
                                                    int32_t* argmax, void* stream) {
  if (!d || M < 1) return DG_ERR_ARG;
  // the same shape rule as dg_lmhead_logsoftmax_entropy
  if (!dgi::lm_dims_ok(d->d_model, d->V)) return DG_ERR_SHAPE;
  if (M > DG_NOALLOC_MAX_ROWS) return DG_ERR_SHAPE;
  if (!h || !w || !inv_t || !lse || !entropy || !maxz || !argmax) return DG_ERR_ARG;
  if (!aligned16(h) || !aligned16(w)) return DG_ERR_ARG;
  if (dgi::lmhead_ws_bytes(M, d->V) > kScratchBytes) return DG_ERR_SHAPE;
  void* scratch = scratch_on_current_device();
  if (!scratch) return DG_ERR_CUDA;
  // Every partial the finalize kernel reads is written by this launch first, so
  // nothing left over from an earlier call needs clearing.
  const cudaError_t e = dgi::lmhead_stats(h, M, w, d->V, d->d_model, inv_t,
                                          dgi::RowStats{lse, entropy, maxz, argmax}, scratch,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}
