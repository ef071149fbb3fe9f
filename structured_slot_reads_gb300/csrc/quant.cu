// quant.cu -- e4m3 operands for the 8-bit lm-head pass: per-row scales.
//
// A row x (bf16) becomes scale = amax|x| / 448 (the largest finite e4m3
// value; 1 for an all-zero row) and q = e4m3(x / scale), rounded to nearest
// even and saturated.  The lm-head pass multiplies the e4m3 products back by
// the row scales of both operands.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace {

__global__ void quantize_rows_e4m3_kernel(const __nv_bfloat16* x, int cols, uint8_t* q,
                                          float* scale) {
  const int row = blockIdx.x;
  const __nv_bfloat16* xr = x + (long long)row * cols;
  uint8_t* qr = q + (long long)row * cols;
  __shared__ float wmax[32];
  __shared__ float s_scale;
  float m = 0.f;
  for (int i = threadIdx.x; i < cols; i += blockDim.x) m = fmaxf(m, fabsf(__bfloat162float(xr[i])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) a = fmaxf(a, wmax[w]);
    const float sc = a > 0.f ? a / 448.f : 1.f;
    s_scale = sc;
    scale[row] = sc;
  }
  __syncthreads();
  const float sc = s_scale;
  for (int i = threadIdx.x; i < cols; i += blockDim.x)
    qr[i] = __nv_cvt_float_to_fp8(__bfloat162float(xr[i]) / sc, __NV_SATFINITE, __NV_E4M3);
}

}  // namespace

namespace dgi {

cudaError_t quantize_rows_e4m3(const uint16_t* x, int rows, int cols, uint8_t* q, float* scale,
                               cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  quantize_rows_e4m3_kernel<<<rows, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(x), cols,
                                                  q, scale);
  return cudaGetLastError();
}

}  // namespace dgi
