// quant.cu -- e4m3 operands of the 8-bit passes.
//
// A row x (bf16) becomes scale = amax|x| / 448 (the largest finite e4m3
// value; 1 for an all-zero row) and q = e4m3(x / scale), rounded to nearest
// even and saturated.  The lm-head pass multiplies the e4m3 products back by
// the row scales of both operands.  For P . E the embedding table is
// quantised per column instead (its scale must sit outside the sum over the
// vocabulary) and stored transposed, [d_model, V], so that both operands of
// that GEMM have the vocabulary contiguous.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>

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

// Long rows (the unnormalised probabilities, V wide): many blocks per row.
// Block (row, chunk) covers QR_CHUNK values with 16-byte loads; the row maxima
// go to amax_bits[row] (atomicMax on float bits, zero on entry).
constexpr int QR_CHUNK = 8192;  // 256 threads x 4 loads x 8 bf16

__global__ void row_amax_long_kernel(const __nv_bfloat16* x, int cols, unsigned int* amax_bits) {
  const int row = blockIdx.y;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (long long)row * cols);
  const int n8 = cols / 8;
  const int i0 = blockIdx.x * (QR_CHUNK / 8);
  const int i1 = min(n8, i0 + QR_CHUNK / 8);
  float m = 0.f;
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    const uint4 u = xr[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wmax[8];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) a = fmaxf(a, wmax[w]);
    atomicMax(amax_bits + row, __float_as_uint(a));
  }
}

__device__ __forceinline__ float row_scale_of(unsigned int bits) {
  const float a = __uint_as_float(bits);
  return a > 0.f ? a / 448.f : 1.f;
}

__global__ void row_quantize_long_kernel(const __nv_bfloat16* x, int cols,
                                         const unsigned int* amax_bits, uint8_t* q) {
  const int row = blockIdx.y;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (long long)row * cols);
  uint2* qr = reinterpret_cast<uint2*>(q + (long long)row * cols);
  const float sc = row_scale_of(amax_bits[row]);
  const int n8 = cols / 8;
  const int i0 = blockIdx.x * (QR_CHUNK / 8);
  const int i1 = min(n8, i0 + QR_CHUNK / 8);
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    const uint4 u = xr[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t out[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
      const uint32_t b0 = __nv_cvt_float_to_fp8(f.x / sc, __NV_SATFINITE, __NV_E4M3);
      const uint32_t b1 = __nv_cvt_float_to_fp8(f.y / sc, __NV_SATFINITE, __NV_E4M3);
      out[k >> 1] |= (b0 | (b1 << 8)) << (16 * (k & 1));
    }
    qr[i] = make_uint2(out[0], out[1]);
  }
}

__global__ void amax_to_row_scale_kernel(float* scale_io, int rows) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r < rows) scale_io[r] = row_scale_of(reinterpret_cast<const unsigned int*>(scale_io)[r]);
}

// Column maxima of |x| [rows, cols]: block = 64 columns x ROWS_PER_BLOCK rows,
// thread (c, g) takes column c and every 4th row of the block; the block's
// maxima go to amax_bits by atomicMax on the float bits (non-negative floats
// order like their bit patterns).  amax_bits must be zero on entry.
constexpr int QC_ROWS = 1024;

__global__ void col_amax_kernel(const __nv_bfloat16* x, int rows, int cols,
                                unsigned int* amax_bits) {
  const int c = blockIdx.x * 64 + (threadIdx.x & 63);
  const int g = threadIdx.x >> 6;  // 0..3
  const int r0 = blockIdx.y * QC_ROWS;
  const int r1 = min(rows, r0 + QC_ROWS);
  __shared__ float red[4][64];
  float m = 0.f;
  if (c < cols)
    for (int r = r0 + g; r < r1; r += 4)
      m = fmaxf(m, fabsf(__bfloat162float(x[(long long)r * cols + c])));
  red[g][threadIdx.x & 63] = m;
  __syncthreads();
  if (g == 0 && c < cols) {
    const float a = fmaxf(fmaxf(red[0][threadIdx.x], red[1][threadIdx.x]),
                          fmaxf(red[2][threadIdx.x], red[3][threadIdx.x]));
    atomicMax(amax_bits + c, __float_as_uint(a));
  }
}

__device__ __forceinline__ float col_scale_of(unsigned int bits) {
  const float a = __uint_as_float(bits);
  return a > 0.f ? a / 448.f : 1.f;
}

// qt[c, r] = e4m3(x[r, c] / scale[c]): a 64 x 64 tile through shared memory,
// read along the columns of x and written along the rows of qt (16 bytes per
// thread).
__global__ void quantize_transpose_kernel(const __nv_bfloat16* x, int rows, int cols,
                                          const unsigned int* amax_bits, uint8_t* qt) {
  __shared__ __align__(16) uint8_t tile[64][64 + 16];
  const int c0 = blockIdx.x * 64, r0 = blockIdx.y * 64;
  const int tc = threadIdx.x & 63, tr = threadIdx.x >> 6;  // 4 rows per pass
  const int c = c0 + tc;
  const float sc = c < cols ? col_scale_of(amax_bits[c]) : 1.f;
  for (int i = tr; i < 64; i += 4) {
    const int r = r0 + i;
    uint8_t q = 0;
    if (r < rows && c < cols)
      q = __nv_cvt_float_to_fp8(__bfloat162float(x[(long long)r * cols + c]) / sc,
                                __NV_SATFINITE, __NV_E4M3);
    tile[tc][i] = q;
  }
  __syncthreads();
  // thread t writes column (t / 4), rows [16 (t % 4), +16)
  const int oc = c0 + (threadIdx.x >> 2), orr = r0 + (threadIdx.x & 3) * 16;
  if (oc >= cols) return;
  const uint8_t* src = &tile[threadIdx.x >> 2][(threadIdx.x & 3) * 16];
  uint8_t* dst = qt + (long long)oc * rows + orr;
  if (orr + 16 <= rows && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  } else {
    for (int k = 0; k < 16 && orr + k < rows; ++k) dst[k] = src[k];
  }
}

// scale[c] from the column maxima held in the same words.
__global__ void amax_to_scale_kernel(float* scale_io, int cols) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c < cols)
    scale_io[c] = col_scale_of(reinterpret_cast<const unsigned int*>(scale_io)[c]);
}

// ---------------------------------------------------------------------------
// NVFP4 weights (e2m1 elements, one e4m3 scale per 16 elements of a row, one
// fp32 scale per tensor).  Tensor scale g = amax|x| / (6 * 448) (1 for an
// all-zero tensor); block scale s = e4m3((amax_block / 6) / g); element code
// e2m1(x / (s * g)), rounded to nearest with ties to the even mantissa and
// saturated at 6.  Stored K-block-major, the layout the 4-bit lm-head pass
// copies: codes [cols/64][rows][32] bytes (element 64 kb + j of row v in byte
// j / 2, the even element in the low nibble), scales [cols/64][rows][4] bytes.
// ---------------------------------------------------------------------------
__global__ void tensor_amax_kernel(const uint4* x, long long n8, unsigned int* amax_bits) {
  float m = 0.f;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (long long)gridDim.x * blockDim.x) {
    const uint4 u = x[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wmax[8];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) a = fmaxf(a, wmax[w]);
    atomicMax(amax_bits, __float_as_uint(a));
  }
}

__device__ __forceinline__ float nvfp4_tensor_scale(unsigned int amax_bits) {
  const float a = __uint_as_float(amax_bits);
  return a > 0.f ? a / 2688.f : 1.f;
}

// e2m1 code of y: nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6 by magnitude, a tie going to
// the value whose mantissa bit is 0, saturating at 6; the sign bit for a nonzero code
__device__ __forceinline__ uint32_t e2m1_code(float y) {
  const float a = fabsf(y);
  const uint32_t m = a <= 0.25f  ? 0u
                     : a < 0.75f ? 1u
                     : a <= 1.25f ? 2u
                     : a < 1.75f  ? 3u
                     : a <= 2.5f  ? 4u
                     : a < 3.5f   ? 5u
                     : a <= 5.f   ? 6u
                                  : 7u;
  return m | ((m != 0u && signbit(y)) ? 8u : 0u);
}

// NVFP4 codes and block scales of 64 consecutive values of a row (four blocks of
// 16): the 32 code bytes as eight words in cw (element 2i in the low nibble of
// byte i); returns the four e4m3 scale bytes in one word (block q in byte q).
__device__ __forceinline__ uint32_t nvfp4_quant64(const __nv_bfloat16* x64, float g,
                                                  uint32_t (&cw)[8]) {
  const uint4* src = reinterpret_cast<const uint4*>(x64);
  uint32_t sc4 = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float xv[16];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 u = src[2 * q + h];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
        xv[8 * h + 2 * k] = f.x;
        xv[8 * h + 2 * k + 1] = f.y;
      }
    }
    float bm = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) bm = fmaxf(bm, fabsf(xv[j]));
    const __nv_fp8_storage_t sb = __nv_cvt_float_to_fp8((bm / 6.f) / g, __NV_SATFINITE, __NV_E4M3);
    const __half_raw hr = __nv_cvt_fp8_to_halfraw(sb, __NV_E4M3);
    const float den = __half2float(__half(hr)) * g;
    sc4 |= (uint32_t)sb << (8 * q);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      uint32_t word = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float y = xv[8 * i + j];
        const uint32_t c = den > 0.f ? e2m1_code(y / den) : 0u;
        word |= c << (4 * j);
      }
      cw[2 * q + i] = word;
    }
  }
  return sc4;
}

// One thread per (K block of 64, row): consecutive threads take consecutive rows,
// so the code and scale writes of a warp are contiguous.
__global__ void quantize_nvfp4_kernel(const __nv_bfloat16* x, int rows, int cols,
                                      const unsigned int* amax_bits, uint8_t* codes,
                                      uint8_t* scales) {
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int nkb = cols / 64;
  if (t >= (long long)rows * nkb) return;
  const int kb = (int)(t / rows);
  const int v = (int)(t % rows);
  const float g = nvfp4_tensor_scale(*amax_bits);
  uint32_t cw[8];
  const uint32_t sc4 = nvfp4_quant64(x + (long long)v * cols + kb * 64, g, cw);
  uint4* cdst = reinterpret_cast<uint4*>(codes + ((long long)kb * rows + v) * 32);
  cdst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
  cdst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
  *reinterpret_cast<uint32_t*>(scales + ((long long)kb * rows + v) * 4) = sc4;
}

// The layout of the block-scaled MMA pass (tcgen05 kind::mxf4nvf4): codes row-major
// [rows][cols/2]; the scales as one 512-byte atom per 128-row tile and 64-column
// K-step, atoms [ceil(rows/128)][cols/64], row 32 j + l of the tile at byte
// 16 l + 4 j (its four blocks of 16 in the four bytes), the order in which
// tcgen05.cp .32x128b.warpx4 places them in tensor memory.  Rows of the last tile
// past `rows` get scale 0.  One thread per (K-step, padded row).
__device__ __forceinline__ long long nvfp4_atom_offset(int v, int ks, int nks) {
  return ((long long)(v >> 7) * nks + ks) * 512 + (v & 31) * 16 + ((v >> 5) & 3) * 4;
}

// Byte offset of the 32 code bytes of row v, 64-value step ks in the tiled codes:
// 16 KB blocks [ceil(rows/128)][nkb][128 rows][128 bytes], nkb = ceil(cols/256).
__device__ __forceinline__ long long nvfp4_code_offset(int v, int ks, int nkb) {
  return (((long long)(v >> 7) * nkb + (ks >> 2)) * 128 + (v & 127)) * 128 + (ks & 3) * 32;
}

// One thread per (row, 64-value step) of the padded rows x steps, so that the
// padding rows and the steps past cols in the last 256-value block get zero codes.
__global__ void quantize_nvfp4_mma_kernel(const __nv_bfloat16* x, int rows, int cols,
                                          const unsigned int* amax_bits, uint8_t* codes,
                                          uint8_t* sf) {
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int nks = cols / 64;
  const int nkb = (nks + 3) / 4;
  const int rows_pad = (rows + 127) & ~127;
  if (t >= (long long)rows_pad * nkb * 4) return;
  const int ks = (int)(t / rows_pad);
  const int v = (int)(t % rows_pad);
  uint32_t sc4 = 0;
  uint32_t cw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (v < rows && ks < nks)
    sc4 = nvfp4_quant64(x + (long long)v * cols + ks * 64, nvfp4_tensor_scale(*amax_bits), cw);
  uint4* cdst = reinterpret_cast<uint4*>(codes + nvfp4_code_offset(v, ks, nkb));
  cdst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
  cdst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
  if (ks < nks) *reinterpret_cast<uint32_t*>(sf + nvfp4_atom_offset(v, ks, nks)) = sc4;
}

// The rows of a block-scaled pass (at most 16): one thread per (row slot, block of
// 16 values), 16 x cols/16 threads.  Each CTA first takes the tensor scale from the
// largest magnitude of all M rows (every CTA the same value: the maximum is exact in
// any order), then writes its blocks' codes (rows >= M all 0) and e4m3 scales into
// the atoms of one 128-row tile; the atoms' other bytes (rows 16..127) are zeroed by
// the threads in turn.  CTA 0 writes g.
__global__ void __launch_bounds__(256)
    quantize_rows_nvfp4_mma_kernel(const __nv_bfloat16* x, int M, int cols, uint8_t* codes,
                                   uint8_t* sf, float* g_out) {
  __shared__ float wmax[8];
  float m = 0.f;
  const long long n8 = (long long)M * cols / 8;
  for (long long i = threadIdx.x; i < n8; i += blockDim.x) {
    const uint4 u = reinterpret_cast<const uint4*>(x)[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  float a = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) a = fmaxf(a, wmax[w]);
  const float g = nvfp4_tensor_scale(__float_as_uint(a));
  const int nb = cols / 16, nks = cols / 64;
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  // zero the atom words that hold no row < 16 (row l < 16, j = 0 is word 4 l)
  for (int wi = t; wi < nks * 128; wi += gridDim.x * blockDim.x) {
    const int wa = wi & 127;
    if (wa >= 64 || (wa & 3) != 0) reinterpret_cast<uint32_t*>(sf)[wi] = 0u;
  }
  if (t >= 16 * nb) return;
  const int r = t / nb, blk = t % nb;   // consecutive threads: consecutive blocks of a row
  uint32_t c0 = 0u, c1 = 0u;
  uint8_t sb = 0;
  if (r < M) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (long long)r * cols + blk * 16);
    float xv[16];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 u = src[h];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
        xv[8 * h + 2 * k] = f.x;
        xv[8 * h + 2 * k + 1] = f.y;
      }
    }
    float bm = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) bm = fmaxf(bm, fabsf(xv[j]));
    const __nv_fp8_storage_t s8 = __nv_cvt_float_to_fp8((bm / 6.f) / g, __NV_SATFINITE, __NV_E4M3);
    const __half_raw hr = __nv_cvt_fp8_to_halfraw(s8, __NV_E4M3);
    const float den = __half2float(__half(hr)) * g;
    sb = (uint8_t)s8;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c0 |= (den > 0.f ? e2m1_code(xv[j] / den) : 0u) << (4 * j);
      c1 |= (den > 0.f ? e2m1_code(xv[8 + j] / den) : 0u) << (4 * j);
    }
  }
  *reinterpret_cast<uint2*>(codes + (long long)r * (cols / 2) + blk * 8) = make_uint2(c0, c1);
  sf[(long long)(blk >> 2) * 512 + r * 16 + (blk & 3)] = sb;
  if (t == 0) *g_out = g;
}

// The rows of a block-scaled pass, more than 16 of them: one thread per (padded row,
// block of 16 values) after tensor_amax_kernel has left the rows' largest magnitude
// in *amax_bits; codes [rows][cols/2], scale atoms [ceil(rows/128)][cols/64] (rows
// past `rows` scale 0); thread 0 writes g.
__global__ void quantize_blocks_nvfp4_mma_kernel(const __nv_bfloat16* x, int rows, int cols,
                                                 const unsigned int* amax_bits, uint8_t* codes,
                                                 uint8_t* sf, float* g_out) {
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int nb = cols / 16, nks = cols / 64;
  const int rows_pad = (rows + 127) & ~127;
  if (t >= (long long)rows_pad * nb) return;
  const int r = (int)(t / nb), blk = (int)(t % nb);
  const float g = nvfp4_tensor_scale(*amax_bits);
  if (t == 0) *g_out = g;
  uint8_t sb = 0;
  if (r < rows) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (long long)r * cols + blk * 16);
    float xv[16];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 u = src[h];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
        xv[8 * h + 2 * k] = f.x;
        xv[8 * h + 2 * k + 1] = f.y;
      }
    }
    float bm = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) bm = fmaxf(bm, fabsf(xv[j]));
    const __nv_fp8_storage_t s8 = __nv_cvt_float_to_fp8((bm / 6.f) / g, __NV_SATFINITE, __NV_E4M3);
    const __half_raw hr = __nv_cvt_fp8_to_halfraw(s8, __NV_E4M3);
    const float den = __half2float(__half(hr)) * g;
    sb = (uint8_t)s8;
    uint32_t c0 = 0u, c1 = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c0 |= (den > 0.f ? e2m1_code(xv[j] / den) : 0u) << (4 * j);
      c1 |= (den > 0.f ? e2m1_code(xv[8 + j] / den) : 0u) << (4 * j);
    }
    *reinterpret_cast<uint2*>(codes + (long long)r * (cols / 2) + blk * 8) = make_uint2(c0, c1);
  }
  sf[nvfp4_atom_offset(r, blk >> 2, nks) + (blk & 3)] = sb;
}

__global__ void nvfp4_scale_kernel(float* g_io) {
  g_io[0] = nvfp4_tensor_scale(reinterpret_cast<const unsigned int*>(g_io)[0]);
}

}  // namespace

namespace dgi {

cudaError_t quantize_nvfp4(const uint16_t* x, int rows, int cols, uint8_t* codes,
                           uint8_t* scales, float* g, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  // g holds the tensor maximum (as float bits) until the last kernel
  unsigned int* amax = reinterpret_cast<unsigned int*>(g);
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(unsigned int), st);
  if (e != cudaSuccess) return e;
  const long long n8 = (long long)rows * cols / 8;
  tensor_amax_kernel<<<(int)std::min<long long>((n8 + 255) / 256, 4096), 256, 0, st>>>(
      reinterpret_cast<const uint4*>(x), n8, amax);
  const long long items = (long long)rows * (cols / 64);
  quantize_nvfp4_kernel<<<(int)((items + 127) / 128), 128, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(x), rows, cols, amax, codes, scales);
  nvfp4_scale_kernel<<<1, 1, 0, st>>>(g);
  return cudaGetLastError();
}

cudaError_t quantize_nvfp4_mma(const uint16_t* x, int rows, int cols, uint8_t* codes, uint8_t* sf,
                               float* g, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  unsigned int* amax = reinterpret_cast<unsigned int*>(g);
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(unsigned int), st);
  if (e != cudaSuccess) return e;
  const long long n8 = (long long)rows * cols / 8;
  tensor_amax_kernel<<<(int)std::min<long long>((n8 + 255) / 256, 4096), 256, 0, st>>>(
      reinterpret_cast<const uint4*>(x), n8, amax);
  const long long items = (long long)((rows + 127) & ~127) * ((cols / 64 + 3) / 4 * 4);
  quantize_nvfp4_mma_kernel<<<(int)((items + 127) / 128), 128, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(x), rows, cols, amax, codes, sf);
  nvfp4_scale_kernel<<<1, 1, 0, st>>>(g);
  return cudaGetLastError();
}

cudaError_t quantize_many_rows_nvfp4_mma(const uint16_t* x, int rows, int cols, uint8_t* codes,
                                         uint8_t* sf, float* g, unsigned int* amax,
                                         cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(unsigned int), st);
  if (e != cudaSuccess) return e;
  const long long n8 = (long long)rows * cols / 8;
  tensor_amax_kernel<<<(int)std::min<long long>((n8 + 255) / 256, 1024), 256, 0, st>>>(
      reinterpret_cast<const uint4*>(x), n8, amax);
  const long long items = (long long)((rows + 127) & ~127) * (cols / 16);
  quantize_blocks_nvfp4_mma_kernel<<<(int)((items + 255) / 256), 256, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(x), rows, cols, amax, codes, sf, g);
  return cudaGetLastError();
}

cudaError_t quantize_rows_nvfp4_mma(const uint16_t* x, int M, int cols, uint8_t* codes,
                                    uint8_t* sf, float* g, cudaStream_t st) {
  const int threads = 16 * (cols / 16);
  quantize_rows_nvfp4_mma_kernel<<<(threads + 255) / 256, 256, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(x), M, cols, codes, sf, g);
  return cudaGetLastError();
}

cudaError_t quantize_cols_e4m3(const uint16_t* x, int rows, int cols, uint8_t* qt, float* scale,
                               cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  // the scale array holds the column maxima (as float bits) until the last kernel
  unsigned int* amax = reinterpret_cast<unsigned int*>(scale);
  cudaError_t e = cudaMemsetAsync(amax, 0, (size_t)cols * sizeof(unsigned int), st);
  if (e != cudaSuccess) return e;
  const auto* xb = reinterpret_cast<const __nv_bfloat16*>(x);
  col_amax_kernel<<<dim3((cols + 63) / 64, (rows + QC_ROWS - 1) / QC_ROWS), 256, 0, st>>>(
      xb, rows, cols, amax);
  quantize_transpose_kernel<<<dim3((cols + 63) / 64, (rows + 63) / 64), 256, 0, st>>>(
      xb, rows, cols, amax, qt);
  amax_to_scale_kernel<<<(cols + 255) / 256, 256, 0, st>>>(scale, cols);
  return cudaGetLastError();
}

cudaError_t quantize_rows_e4m3(const uint16_t* x, int rows, int cols, uint8_t* q, float* scale,
                               cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const bool vec = cols % 8 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(q) & 7) == 0 &&
                   (reinterpret_cast<uintptr_t>(scale) & 3) == 0;
  if (vec && cols >= 2 * QR_CHUNK && rows <= 65535) {
    // the scale array holds the row maxima (as float bits) until the last kernel
    unsigned int* amax = reinterpret_cast<unsigned int*>(scale);
    cudaError_t e = cudaMemsetAsync(amax, 0, (size_t)rows * sizeof(unsigned int), st);
    if (e != cudaSuccess) return e;
    const dim3 grid((cols + QR_CHUNK - 1) / QR_CHUNK, rows);
    const auto* xb = reinterpret_cast<const __nv_bfloat16*>(x);
    row_amax_long_kernel<<<grid, 256, 0, st>>>(xb, cols, amax);
    row_quantize_long_kernel<<<grid, 256, 0, st>>>(xb, cols, amax, q);
    amax_to_row_scale_kernel<<<(rows + 255) / 256, 256, 0, st>>>(scale, rows);
    return cudaGetLastError();
  }
  quantize_rows_e4m3_kernel<<<rows, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(x), cols,
                                                  q, scale);
  return cudaGetLastError();
}

}  // namespace dgi
