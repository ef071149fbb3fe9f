// heads_tc.cu -- the fused lm-head pass of one denoise step (one stream of W).
//
// For the canvas rows (tau-home.com "Refusing JSON token generation";
// 24-ai.news "Token commit mechanism") the pass computes the row statistics of
// softmax(h W^T / T) and, for self-conditioning, the unnormalised
// probabilities  P~[i, v] = 2^(z_iv log2 e - r_i)  in bf16.  The per-row
// reference r_i (the row's largest scaled logit over the first 8 vocabulary
// entries, plus a fixed headroom) is computed once by ref_kernel before the
// pass and read by every CTA, so the per-CTA sums S_i = sum_v P~ add without
// rescaling and p_iv = P~_iv / S_i exactly; the P.E GEMM applies 1/S_i in its
// reduction.
//
// The pass is exact while every scaled logit lies less than 2^13 log2 units
// above the largest of the row's first 8.  An epilogue thread owns one row of
// its CTA's vocabulary range and sums each 32-entry chunk against its
// reference; if the chunk's largest
// exponent passes RAISE it raises the reference by a whole number k of log2
// units (2^-k is then exact), scales what it summed and wrote before the chunk
// by 2^-k and sums the chunk again.  Each CTA reports the reference of its sums
// and probabilities; the finalize takes the largest, merges the sums against it
// and brings the probabilities of any CTA range with a lower reference to it
// (again by a power of two).  Without a raise (the usual case) every factor is
// 1 and nothing is rewritten.
//
// For the slot-read draw rows (sotaaz.com "The server accepts at most 26
// alternatives per question": noise reads of an answer slot) the same W tiles
// feed a "swapped" MMA: A = the W tile (vocabulary on TMEM lanes), B = the
// <= 16 draw rows (N = 16), so the draw rows' log-normalisers come out of the
// same pass instead of a second stream of W.
//
// Tile geometry: BN vocabulary rows per tile (224 with draw rows, so that
// 2 x 224 canvas columns + 2 x 16 draw columns fit the 512 TMEM columns), 64-
// element K blocks, one shared-memory ring whose stages hold the canvas rows,
// the W tile and the draw rows of a K block (128-byte swizzled by TMA), one
// CTA per SM.
//
// W may come from a tiled copy (heads_tile_weights): tile t, K block kb is one
// contiguous 224 x 64 run, so every TMA box reads 28 KB of consecutive memory
// instead of 224 rows of 128 bytes each one W row apart.  A streaming probe of
// the two layouts on GB300 measured 6.63 TB/s tiled against 6.12 TB/s row-major.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace {

using namespace dgk;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int REF_N = 8;              // vocabulary entries behind the reference
constexpr float REF_HEADROOM = 24.f;  // log2 units added to the reference maximum
constexpr float RAISE = 64.f;         // exponent (log2 units) past which a reference is raised
constexpr float V_CLAMP = 100.f;      // exponent guard while a chunk is first summed
constexpr int DRAW_N = 16;
constexpr int TILED_ROWS = 224;       // vocabulary rows of a tile of W's tiled copy
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void epi_bar(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

struct HeadsParams {
  int M;        // canvas rows
  int n_draw;   // draw rows (0..16)
  int V, K;
  int cpg, n_tiles;
  const float* inv_t;       // [M]
  const float* inv_t_draw;  // [n_draw]
  const float* ref;         // [M] reference r (log2 units)
  float* part;              // canvas: 5 planes of [M][cpg]: s, t, best, idx, reference
  float* part_draw;         // draws: 2 planes of [n_draw][cpg]: m, s
  __nv_bfloat16* probs;     // [M][ldp] or null
  long long ldp;
  dgi::LabelGather gl;      // draws' label logits z/T (R > 0 form; gl.out null: none)
  int* status;
  int w_nkb;                // W from its tiled copy (K blocks per tile), 0: row-major W
  // e4m3 operands (the 8-bit pass): the scale of each canvas row, W row and draw row
  const float* h_scale;
  const float* w_scale;
  const float* d_scale;
};

// Reference of each canvas row: max over the first REF_N vocabulary entries of
// (h . w_v) / T in log2 units, plus headroom.  One CTA per row; warp w takes
// entry w % REF_N over a quarter of d_model (w / REF_N), so each lane has only
// a few 16-byte chunks and the partial sums meet in shared memory.
constexpr int REF_KSPLIT = 4;
__global__ void __launch_bounds__(REF_N * REF_KSPLIT * 32)
    ref_kernel(const __nv_bfloat16* h, const __nv_bfloat16* w, const float* inv_t, int M, int V,
               int D, float* ref) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = warp % REF_N, ks = warp / REF_N;
  const int row = blockIdx.x;
  __shared__ float part[REF_KSPLIT][REF_N];
  const uint4* x = reinterpret_cast<const uint4*>(h + (long long)row * D);
  const uint4* y = reinterpret_cast<const uint4*>(w + (long long)u * D);
  const int n16 = D / 8;
  const int per = (n16 + REF_KSPLIT - 1) / REF_KSPLIT;
  const int i0 = ks * per, i1 = min(n16, i0 + per);
  float acc = 0.f;
  if (u < V) {
#pragma unroll 4
    for (int i = i0 + lane; i < i1; i += 32) {
      const uint4 a = x[i];
      const uint4 b = __ldg(y + i);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 fa = __bfloat1622float2(a2[q]);
        const float2 fb = __bfloat1622float2(b2[q]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) part[ks][u] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    for (int e = 0; e < REF_N && e < V; ++e) {
      float t = 0.f;
      for (int k = 0; k < REF_KSPLIT; ++k) t += part[k][e];
      m = fmaxf(m, t);
    }
    // on a grid of 1/256 log2 units, so that adding whole raises keeps it exact
    ref[row] = rintf((m * inv_t[row] * LOG2E + REF_HEADROOM) * 256.f) * (1.f / 256.f);
  }
}

// The reference of the e4m3 pass: the same definition on the dequantised
// operands, max over the first REF_N entries of (h8 . w8_v) h_scale w_scale_v / T.
// One CTA per row, warp e takes entry e; each lane reads 16 codes at a time.
__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  return __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)byte, __NV_E4M3)));
}

__global__ void __launch_bounds__(REF_N * 32)
    ref8_kernel(const uint8_t* h8, const float* h_scale, const uint8_t* w8, const float* w_scale,
                const float* inv_t, int V, int D, float* ref) {
  const int e = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x;
  __shared__ float part[REF_N];
  float acc = 0.f;
  if (e < V) {
    const uint4* x = reinterpret_cast<const uint4*>(h8 + (long long)row * D);
    const uint4* y = reinterpret_cast<const uint4*>(w8 + (long long)e * D);
    for (int i = lane; i < D / 16; i += 32) {
      const uint4 a = __ldg(x + i), b = __ldg(y + i);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          acc = fmaf(e4m3_to_float((av[q] >> (8 * k)) & 0xFFu),
                     e4m3_to_float((bv[q] >> (8 * k)) & 0xFFu), acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    acc *= __ldg(h_scale + row) * __ldg(w_scale + e);
  }
  if (lane == 0) part[e] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    for (int k = 0; k < REF_N && k < V; ++k) m = fmaxf(m, part[k]);
    ref[row] = rintf((m * inv_t[row] * LOG2E + REF_HEADROOM) * 256.f) * (1.f / 256.f);
  }
}

// The same reference for many rows (batched canvases): one warp per row reads
// the row once and takes all REF_N dot products against W's first REF_N rows
// (which stay in L1), where the kernel above would read each row REF_N times.
constexpr int REF_ROWS_MIN = 1024;   // rows from which the warp-per-row form is used
__global__ void __launch_bounds__(256)
    ref_rows_kernel(const __nv_bfloat16* h, const __nv_bfloat16* w, const float* inv_t, int M,
                    int V, int D, float* ref) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= M) return;
  const uint4* x = reinterpret_cast<const uint4*>(h + (long long)row * D);
  const int n16 = D / 8;
  const int nu = min(REF_N, V);
  float acc[REF_N];
#pragma unroll
  for (int u = 0; u < REF_N; ++u) acc[u] = 0.f;
#pragma unroll 2
  for (int i = lane; i < n16; i += 32) {
    const uint4 a = x[i];
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    float2 fa[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) fa[q] = __bfloat1622float2(a2[q]);
#pragma unroll
    for (int u = 0; u < REF_N; ++u) {
      if (u >= nu) break;
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(w + (long long)u * D) + i);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 fb = __bfloat1622float2(b2[q]);
        acc[u] = fmaf(fa[q].x, fb.x, acc[u]);
        acc[u] = fmaf(fa[q].y, fb.y, acc[u]);
      }
    }
  }
  float m = -INFINITY;
#pragma unroll
  for (int u = 0; u < REF_N; ++u) {
    float a = acc[u];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (u < nu) m = fmaxf(m, a);
  }
  if (lane == 0) ref[row] = rintf((m * inv_t[row] * LOG2E + REF_HEADROOM) * 256.f) * (1.f / 256.f);
}

// F8: e4m3 operands, K blocks of 128 values, so every row of a block is 128
// bytes as in the bf16 pass and the stage geometry is the same.
template <int MT, int BN, bool DRAWS, bool F8 = false>
struct HCfg {
  static constexpr int KBE = F8 ? 2 * BK : BK;            // values of a K block
  static constexpr int A_BYTES = BM * BK * 2;             // one 128-row canvas tile
  static constexpr int A_STAGE = MT * A_BYTES;
  static constexpr int W_SLOT = BN * BK * 2;
  static constexpr int D_BYTES = DRAWS ? DRAW_N * BK * 2 : 0;
  static constexpr int STAGE_BYTES = A_STAGE + W_SLOT + D_BYTES;
  static constexpr int DRAW_COLS = DRAWS ? 2 * DRAW_N : 0;
  static constexpr int ACC_COLS = MT * BN + DRAW_COLS;
  static constexpr int ACC_STAGES = (2 * ACC_COLS <= 512) ? 2 : 1;
  static constexpr int TMEM_COLS = 512;
  static constexpr int EPI_WARPS = 4 * MT;
  static constexpr int THREADS = (EPI_WARPS + 2) * 32;    // + producer + MMA issuer
  static constexpr int GBITS_OFF = 512 + EPI_WARPS * DRAW_N * 8;  // label-gather chunk bits
  static constexpr int GBITS_WORDS = 64;
  static constexpr int BAR_BYTES = GBITS_OFF + GBITS_WORDS * 4;
  static constexpr int NS_FIT = (232448 - 1024 - BAR_BYTES) / STAGE_BYTES;
  static constexpr int NSTAGE = NS_FIT > 8 ? 8 : NS_FIT;
  static constexpr int SMEM_BYTES = 1024 + NSTAGE * STAGE_BYTES + BAR_BYTES;
  static constexpr uint32_t IDESC = F8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN);
  static constexpr uint32_t IDESC_DRAW =
      F8 ? idesc_e4m3_f32(BM, DRAW_N) : idesc_bf16_f32(BM, DRAW_N);
  static constexpr int HALF1_ROW = BN - 128;  // the second swapped MMA reads W rows [BN-128, BN)
  static constexpr uint32_t TX = A_STAGE + W_SLOT;
  static_assert(ACC_COLS <= 512, "accumulators exceed tensor memory");
  static_assert(BN % 32 == 0 && BN <= 256, "BN");
  static_assert(!DRAWS || (BN >= 128 && BN % 8 == 0), "swapped draw MMA geometry");
  static_assert(STAGE_BYTES % 1024 == 0 && W_SLOT % 1024 == 0, "stages stay 1 KB aligned");
  static_assert(NSTAGE >= 2 && SMEM_BYTES <= 232448, "shared memory");
};

// 2^-k for a whole k >= 0, built from its bit pattern (exact); 0 below the
// normal range, as the flush-to-zero exponentials of the pass give there.
__device__ __forceinline__ float pow2_neg(int k) {
  return k > 126 ? 0.f : __int_as_float((127 - k) << 23);
}

// Multiply the bf16 probabilities [v0, v1) of one row by f (a power of two, so
// exact unless a value underflows).  v0, v1 are multiples of 8; rare path.
__device__ __forceinline__ void rescale_probs(__nv_bfloat16* row, int v0, int v1, float f) {
  for (int v = v0; v < v1; v += 8) {
    uint4 u = *reinterpret_cast<const uint4*>(row + v);
    __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 x = __bfloat1622float2(b[q]);
      b[q] = __floats2bfloat162_rn(x.x * f, x.y * f);
    }
    *reinterpret_cast<uint4*>(row + v) = u;
  }
}

template <int MT, int BN, bool DRAWS, bool F8>
__global__ void __launch_bounds__(HCfg<MT, BN, DRAWS, F8>::THREADS, 1)
    heads_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmD, HeadsParams p) {
  using CF = HCfg<MT, BN, DRAWS, F8>;
  constexpr int NSTAGE = CF::NSTAGE;
  constexpr int PRODUCER_WARP = CF::EPI_WARPS;
  constexpr int MMA_WARP = CF::EPI_WARPS + 1;
  constexpr int EPI_THREADS = CF::EPI_WARPS * 32;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  uint8_t* bar_base = smem + NSTAGE * CF::STAGE_BYTES;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(bar_base);
  uint64_t* empty_bar = full_bar + NSTAGE;
  uint64_t* tfull_bar = empty_bar + NSTAGE;
  uint64_t* tempty_bar = tfull_bar + CF::ACC_STAGES;
  uint64_t* drain_bar = tempty_bar + CF::ACC_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* draw_red = reinterpret_cast<float*>(bar_base + 512);
  uint32_t* gbits = reinterpret_cast<uint32_t*>(bar_base + CF::GBITS_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    for (int a = 0; a < CF::ACC_STAGES; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], CF::EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tmem_slot, CF::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == PRODUCER_WARP && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (DRAWS) prefetch_tmap(&tmD);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total_kb = (p.K + CF::KBE - 1) / CF::KBE;
  const int gm = blockIdx.x / p.cpg;
  const int gn = blockIdx.x % p.cpg;
  const int t_begin = (int)((long long)gn * p.n_tiles / p.cpg);
  const int t_end = (int)((long long)(gn + 1) * p.n_tiles / p.cpg);
  const int m_base = gm * MT * BM;
  const bool draws_here = DRAWS && gm == 0 && p.n_draw > 0;

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      const uint64_t pol_keep = policy_evict_last();
      const uint64_t pol_stream = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0, issued_mask = 0, last_phase = 0;
      bool ok = true;
      for (int t = t_begin; t < t_end && ok; ++t) {
        for (int kb = 0; kb < total_kb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* s_a = stages + stage * CF::STAGE_BYTES;
          uint8_t* s_w = s_a + CF::A_STAGE;
          mbar_arrive_expect_tx(&full_bar[stage], CF::TX + (draws_here ? CF::D_BYTES : 0));
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
            tma_load_2d_hint(s_a + mt * CF::A_BYTES, &tmA, &full_bar[stage], kb * CF::KBE,
                             m_base + mt * BM, pol_keep);
          if (p.w_nkb)  // tiled copy: block (t, kb) is one contiguous box
            tma_load_3d_hint(s_w, &tmB, &full_bar[stage], 0, 0, t * p.w_nkb + kb, pol_stream);
          else
            tma_load_2d_hint(s_w, &tmB, &full_bar[stage], kb * CF::KBE, t * BN, pol_stream);
          if (draws_here)
            tma_load_2d_hint(s_w + CF::W_SLOT, &tmD, &full_bar[stage], kb * CF::KBE, 0, pol_keep);
          issued_mask |= 1u << stage;
          last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == NSTAGE) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < NSTAGE; ++s)
          if (issued_mask & (1u << s)) mbar_wait_drain(&full_bar[s], (last_phase >> s) & 1u);
      }
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = t_begin; t < t_end && ok; ++t) {
        if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_base = tmem_base + acc * CF::ACC_COLS;
        for (int kb = 0; kb < total_kb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stages + stage * CF::STAGE_BYTES);
          const uint32_t w_addr = a_addr + CF::A_STAGE;
          const uint32_t d_addr = w_addr + CF::W_SLOT;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t acc_flag = (kb > 0 || kk > 0) ? 1u : 0u;
            const uint64_t bdesc = sw128_kmajor_desc(w_addr + kk * 32);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              const uint64_t adesc = sw128_kmajor_desc(a_addr + mt * CF::A_BYTES + kk * 32);
              if constexpr (F8)
                tc_mma_f8(d_base + mt * BN, adesc, bdesc, CF::IDESC, acc_flag);
              else
                tc_mma_f16(d_base + mt * BN, adesc, bdesc, CF::IDESC, acc_flag);
            }
            if (DRAWS && draws_here) {
              const uint64_t ddesc = sw128_kmajor_desc(d_addr + kk * 32);
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                const uint32_t row0 = half ? CF::HALF1_ROW : 0;
                const uint64_t wdesc = sw128_kmajor_desc(w_addr + row0 * 128 + kk * 32);
                if constexpr (F8)
                  tc_mma_f8(d_base + MT * BN + half * DRAW_N, wdesc, ddesc, CF::IDESC_DRAW,
                            acc_flag);
                else
                  tc_mma_f16(d_base + MT * BN + half * DRAW_N, wdesc, ddesc, CF::IDESC_DRAW,
                             acc_flag);
              }
            }
          }
          tc_commit(&empty_bar[stage]);
          if (++stage == NSTAGE) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&tfull_bar[acc]);
        if (++acc == CF::ACC_STAGES) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      tc_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0);
    }
  } else {
    // ---- epilogue warps -----------------------------------------------------
    const int mt = warp >> 2;
    const int quarter = warp & 3;
    const int row = m_base + mt * BM + quarter * 32 + lane;
    const bool row_ok = row < p.M;
    const float scale = row_ok ? __ldg(p.inv_t + row) * LOG2E : 0.f;
    const float r_ref = row_ok ? __ldg(p.ref + row) : 0.f;
    const float rs8 = (F8 && row_ok) ? __ldg(p.h_scale + row) : 1.f;   // e4m3: the row's scale
    float s_run = 0.f, t_run = 0.f, best = -INFINITY;
    float r_cur = r_ref;  // reference of the sums and probabilities: r_ref + whole raises
    int best_idx = 0x7fffffff;
    // draw-row running statistics: lane = vocabulary row of a half tile
    float dm[DRAW_N], ds[DRAW_N], dscale[DRAW_N];
#pragma unroll
    for (int j = 0; j < DRAW_N; ++j) {
      dm[j] = -INFINITY;
      ds[j] = 0.f;
      dscale[j] = (DRAWS && j < p.n_draw) ? __ldg(p.inv_t_draw + j) * LOG2E : 0.f;
      if (F8 && DRAWS && j < p.n_draw) dscale[j] *= __ldg(p.d_scale + j);
    }
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    // Label gather of the draw rows: one bit per 32 vocabulary rows of this
    // CTA's range that hold a label of some draw (aliased modulo 2048 chunks,
    // which can only add chunks to scan), so a warp scans the label table only
    // for the rare 32-row chunks that hold a label.
    const bool gat = DRAWS && draws_here && p.gl.out != nullptr;
    const int g_lo = t_begin * BN;
    if (gat) {
      for (int i = threadIdx.x; i < CF::GBITS_WORDS; i += EPI_THREADS) gbits[i] = 0;
      epi_bar(EPI_THREADS);
      const int hi = min(t_end * BN, p.V);
      for (int i = threadIdx.x; i < p.gl.S * p.gl.L; i += EPI_THREADS) {
        const int sl = i / p.gl.L;
        if (i % p.gl.L >= min(max(__ldg(p.gl.n_labels + sl), 0), p.gl.L)) continue;
        const int id = __ldg(p.gl.label_ids + i);
        if (id >= g_lo && id < hi) {
          const int c = ((id - g_lo) >> 5) & (CF::GBITS_WORDS * 32 - 1);
          atomicOr(gbits + (c >> 5), 1u << (c & 31));
        }
      }
      epi_bar(EPI_THREADS);
    }
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = t_begin; t < t_end; ++t) {
      if (!mbar_wait(&tfull_bar[acc], acc_phase, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + lane_base + acc * CF::ACC_COLS + mt * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld_32x32b_x32(taddr + c * 32, r);
        tmem_ld_wait();
        const int n0 = t * BN + c * 32;
        if (!row_ok || n0 >= p.V) continue;
        if constexpr (F8) {
          // the logits of e4m3 operands: the sums times the row's and the W rows' scales
          if (n0 + 32 <= p.V) {
            const float4* cs4 = reinterpret_cast<const float4*>(p.w_scale + n0);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 c4 = __ldg(cs4 + q);
              r[4 * q] = __float_as_uint(__uint_as_float(r[4 * q]) * rs8 * c4.x);
              r[4 * q + 1] = __float_as_uint(__uint_as_float(r[4 * q + 1]) * rs8 * c4.y);
              r[4 * q + 2] = __float_as_uint(__uint_as_float(r[4 * q + 2]) * rs8 * c4.z);
              r[4 * q + 3] = __float_as_uint(__uint_as_float(r[4 * q + 3]) * rs8 * c4.w);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n0 + j < p.V)
                r[j] = __float_as_uint(__uint_as_float(r[j]) * rs8 * __ldg(p.w_scale + n0 + j));
          }
        }
        float e[32];
        float cmax = -INFINITY;
        const float s_prev = s_run, t_prev = t_run;
        if (n0 + 32 <= p.V) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float a = __uint_as_float(r[j]);
            cmax = fmaxf(cmax, a);
            e[j] = ex2(fminf(fmaf(a, scale, -r_cur), V_CLAMP));
            s_run += e[j];
            t_run = fmaf(e[j], a, t_run);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float a = __uint_as_float(r[j]);
            const bool ok = n0 + j < p.V;
            if (ok) cmax = fmaxf(cmax, a);
            e[j] = ok ? ex2(fminf(fmaf(a, scale, -r_cur), V_CLAMP)) : 0.f;
            s_run += e[j];
            t_run = fmaf(e[j], a, t_run);
          }
        }
        const float xmax = fmaf(cmax, scale, -r_cur);
        if (xmax > RAISE) {
          // rare: a logit far above this row's reference.  Raise the reference by
          // k whole log2 units, scale what was summed and written before this
          // chunk by 2^-k (exact) and sum the chunk again against the new one.
          const int k = (int)fminf(ceilf(xmax), 8192.f);
          const float f = pow2_neg(k);
          r_cur += (float)k;
          float s_c = 0.f, t_c = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float a = __uint_as_float(r[j]);
            e[j] = (n0 + j < p.V) ? ex2(fmaf(a, scale, -r_cur)) : 0.f;
            s_c += e[j];
            t_c = fmaf(e[j], a, t_c);
          }
          s_run = fmaf(s_prev, f, s_c);
          t_run = fmaf(t_prev, f, t_c);
          if (p.probs) rescale_probs(p.probs + (long long)row * p.ldp, t_begin * BN, n0, f);
        }
        if (cmax > best) {  // columns ascend, so the first occurrence is the lowest id
          int first = 0x7fffffff;
#pragma unroll
          for (int j = 31; j >= 0; --j)
            if (n0 + j < p.V && __uint_as_float(r[j]) == cmax) first = n0 + j;
          best = cmax;
          best_idx = first;
        }
        if (p.probs) {
          __nv_bfloat16* dst = p.probs + (long long)row * p.ldp + n0;
          if (n0 + 32 <= p.V) {
            // two 256-bit stores per lane: whole 32-byte sectors (the row pitch is a
            // multiple of 128 bytes and chunks start on 32-byte boundaries)
#pragma unroll
            for (int j = 0; j < 32; j += 16) {
              uint32_t w[8];
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                __nv_bfloat162 bq = __floats2bfloat162_rn(e[j + 2 * q], e[j + 2 * q + 1]);
                w[q] = *reinterpret_cast<uint32_t*>(&bq);
              }
              asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + j),
                           "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),
                           "r"(w[6]), "r"(w[7])
                           : "memory");
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n0 + j < p.V) dst[j] = __float2bfloat16_rn(e[j]);
          }
        }
      }
      if (DRAWS && draws_here) {
        // warpgroup mt handles half mt (with one M-tile, warpgroup 0 does both)
#pragma unroll
        for (int hh = 0; hh < (MT == 1 ? 2 : 1); ++hh) {
          const int half = (MT == 1) ? hh : mt;
          uint32_t r[DRAW_N];
          __syncwarp();
          tmem_ld_32x32b_x16(tmem_base + lane_base + acc * CF::ACC_COLS + MT * BN + half * DRAW_N,
                             r);
          tmem_ld_wait();
          // row of the W tile on this lane; half 1 starts at row BN-128, so its
          // lanes below row 128 repeat half 0 and are skipped
          const int vl = (half ? CF::HALF1_ROW : 0) + quarter * 32 + lane;
          const int vocab = t * BN + vl;
          const bool lane_ok = (half == 0 || vl >= 128) && vl < BN && vocab < p.V;
          // e4m3: this lane's W row scale (the draw rows' scales are in dscale)
          const float wsv = (F8 && lane_ok) ? __ldg(p.w_scale + vocab) : 1.f;
          if (lane_ok) {
#pragma unroll
            for (int j = 0; j < DRAW_N; ++j) {
              if (j < p.n_draw) {
                const float v = __uint_as_float(r[j]) * wsv * dscale[j];
                const float mn = fmaxf(dm[j], v);
                ds[j] = ds[j] * ex2(dm[j] - mn) + ex2(v - mn);
                dm[j] = mn;
              }
            }
          }
          if (gat) {
            // the warp's 32 vocabulary rows are one chunk (BN and the half-1
            // offset are multiples of 32): a uniform test, then a scan of the
            // label table by the lanes whose row is a label
            const int c = ((t * BN + vl - lane - g_lo) >> 5) & (CF::GBITS_WORDS * 32 - 1);
            if ((gbits[c >> 5] >> (c & 31)) & 1u) {
              for (int sl = 0; sl < p.gl.S && lane_ok; ++sl) {
                const int n = min(max(__ldg(p.gl.n_labels + sl), 0), p.gl.L);
                for (int k = 0; k < n; ++k) {
                  if (__ldg(p.gl.label_ids + sl * p.gl.L + k) != vocab) continue;
                  for (int rr = 0; rr < p.gl.R; ++rr) {
                    const int j = sl * p.gl.R + rr;
                    float z = __uint_as_float(r[0]);
#pragma unroll
                    for (int q = 1; q < DRAW_N; ++q) z = j == q ? __uint_as_float(r[q]) : z;
                    if (F8) z *= wsv * __ldg(p.d_scale + j);
                    p.gl.out[(long long)j * p.gl.L + k] = z * __ldg(p.inv_t_draw + j);
                  }
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc]);
      if (++acc == CF::ACC_STAGES) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (row_ok) {
      const long long o = (long long)row * p.cpg + gn;
      const long long plane = (long long)p.cpg * p.M;
      p.part[o] = s_run;
      p.part[o + plane] = t_run;
      p.part[o + 2 * plane] = best;
      reinterpret_cast<int*>(p.part)[o + 3 * plane] = best_idx;
      p.part[o + 4 * plane] = r_cur;
    }
    if (DRAWS && draws_here) {
      // merge the draw statistics over the lanes, then over the epilogue warps
#pragma unroll
      for (int j = 0; j < DRAW_N; ++j) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float mo = __shfl_xor_sync(0xffffffffu, dm[j], o);
          const float so = __shfl_xor_sync(0xffffffffu, ds[j], o);
          const float mn = fmaxf(dm[j], mo);
          ds[j] = (mn == -INFINITY) ? 0.f : ds[j] * ex2(dm[j] - mn) + so * ex2(mo - mn);
          dm[j] = mn;
        }
      }
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < DRAW_N; ++j) {
          draw_red[(warp * DRAW_N + j) * 2] = dm[j];
          draw_red[(warp * DRAW_N + j) * 2 + 1] = ds[j];
        }
      }
      epi_bar(EPI_THREADS);
      if (warp == 0 && lane < p.n_draw) {
        const int j = lane;
        float m = -INFINITY, s = 0.f;
        for (int w = 0; w < CF::EPI_WARPS; ++w) {
          const float mo = draw_red[(w * DRAW_N + j) * 2];
          const float so = draw_red[(w * DRAW_N + j) * 2 + 1];
          const float mn = fmaxf(m, mo);
          s = (mn == -INFINITY) ? 0.f : s * ex2(m - mn) + so * ex2(mo - mn);
          m = mn;
        }
        const long long o = (long long)j * p.cpg + gn;
        p.part_draw[o] = m;
        p.part_draw[o + (long long)p.n_draw * p.cpg] = s;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == MMA_WARP) tmem_dealloc(tmem_base, CF::TMEM_COLS);
}

// Canvas rows, one warp per row.  Each CTA's sums and probabilities are
// relative to its reference ref[row] + k_g (k_g whole log2 units, 0 unless that
// CTA raised it; the references lie on a 1/256 grid, so the differences are
// exact); they are brought to the largest reference and added (every factor is
// exactly 1 without a raise), with the best logit and its lowest index over the
// CTAs.  The probabilities of a CTA range with a lower reference are scaled to
// the largest (a power of two, exact), so that p = P~ * prob_scale over the row.
__device__ void finalize_row(int row, int lane, const float* part, int cpg, int M,
                             const float* inv_t, float* lse, float* entropy, float* maxz,
                             int32_t* argmax, float* prob_scale, __nv_bfloat16* probs,
                             long long ldp, int n_tiles, int bn, int V) {
  const long long plane = (long long)cpg * M;
  const float* pm = part + (long long)row * cpg;
  float rmax = -INFINITY;
  for (int g = lane; g < cpg; g += 32) rmax = fmaxf(rmax, pm[g + 4 * plane]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, o));
  float s = 0.f, t = 0.f, best = -INFINITY;
  int idx = 0x7fffffff;
  bool lower = false;
  for (int g = lane; g < cpg; g += 32) {
    const float rg = pm[g + 4 * plane];
    const float f = pow2_neg((int)(rmax - rg));
    lower |= rg < rmax;
    s += pm[g] * f;
    t += pm[g + plane] * f;
    const float bg = pm[g + 2 * plane];
    const int ig = reinterpret_cast<const int*>(pm)[g + 3 * plane];
    if (bg > best || (bg == best && ig < idx)) {
      best = bg;
      idx = ig;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    t += __shfl_xor_sync(0xffffffffu, t, o);
    const float bo = __shfl_xor_sync(0xffffffffu, best, o);
    const int io = __shfl_xor_sync(0xffffffffu, idx, o);
    if (bo > best || (bo == best && io < idx)) {
      best = bo;
      idx = io;
    }
  }
  if (lane == 0) {
    const float it = inv_t[row];
    const float l = (rmax + log2f(s)) * LN2;
    lse[row] = l;
    entropy[row] = l - it * (t / s);
    maxz[row] = best * it;
    argmax[row] = idx;
    if (prob_scale) prob_scale[row] = 1.f / s;
  }
  // rare: some CTA of this row raised its reference; bring the others to it
  if (probs && __any_sync(0xffffffffu, lower)) {
    __nv_bfloat16* pr = probs + (long long)row * ldp;
    for (int g = 0; g < cpg; ++g) {
      const float rg = pm[g + 4 * plane];
      if (!(rg < rmax)) continue;
      const float f = pow2_neg((int)(rmax - rg));
      const int v0 = (int)((long long)g * n_tiles / cpg) * bn;
      const int v1 = min(V, (int)((long long)(g + 1) * n_tiles / cpg) * bn);
      for (int v = v0 + 2 * lane; v < v1; v += 64) {
        if (v + 1 < v1) {
          __nv_bfloat162* q = reinterpret_cast<__nv_bfloat162*>(pr + v);
          const float2 x = __bfloat1622float2(*q);
          *q = __floats2bfloat162_rn(x.x * f, x.y * f);
        } else {
          pr[v] = __float2bfloat16_rn(__bfloat162float(pr[v]) * f);
        }
      }
    }
  }
}

// Draw rows: per-CTA (max, sum) pairs merged, one warp per row; the row's
// gathered label logits get their ids checked.
__device__ void finalize_draw(int j, int lane, const float* part_draw, int cpg, int n_draw,
                              float* lse_draw, const dgi::LabelGather& gl, int V, int* status) {
  if (gl.out != nullptr && j < gl.S * gl.R) {
    const int sl = j / gl.R;
    const int n = min(max(gl.n_labels[sl], 0), gl.L);
    for (int k = lane; k < n; k += 32) {
      const int id = gl.label_ids[(long long)sl * gl.L + k];
      if (id < 0 || id >= V) {
        atomicOr(status, 4 /* DG_DEV_BAD_LABEL */);
        gl.out[(long long)j * gl.L + k] = -INFINITY;
      }
    }
  }
  const float* pm = part_draw + (long long)j * cpg;
  const float* ps = part_draw + (long long)n_draw * cpg + (long long)j * cpg;
  float m = -INFINITY;
  for (int g = lane; g < cpg; g += 32) m = fmaxf(m, pm[g]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f;
  for (int g = lane; g < cpg; g += 32)
    if (pm[g] != -INFINITY) s += ps[g] * exp2f(pm[g] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) lse_draw[j] = (m + log2f(s)) * LN2;
}

// Both finalisations in one launch: the first row_blocks blocks take the canvas
// rows, the rest the draw rows (8 rows a block).
__global__ void heads_finalize_kernel(const float* part, int cpg, int M, const float* inv_t,
                                      float* lse, float* entropy, float* maxz,
                                      int32_t* argmax, float* prob_scale, __nv_bfloat16* probs,
                                      long long ldp,
                                      int n_tiles, int bn, int V, const float* part_draw,
                                      int n_draw, float* lse_draw, int row_blocks,
                                      dgi::LabelGather gl, int* status) {
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  if ((int)blockIdx.x < row_blocks) {
    const int row = blockIdx.x * (blockDim.x >> 5) + w;
    if (row < M)
      finalize_row(row, lane, part, cpg, M, inv_t, lse, entropy, maxz, argmax, prob_scale,
                   probs, ldp, n_tiles, bn, V);
  } else {
    const int j = (blockIdx.x - row_blocks) * (blockDim.x >> 5) + w;
    if (j < n_draw) finalize_draw(j, lane, part_draw, cpg, n_draw, lse_draw, gl, V, status);
  }
}

template <int MT, int BN, bool DRAWS, bool F8 = false>
cudaError_t launch_heads(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td,
                         const HeadsParams& p, int grid, cudaStream_t st) {
  using CF = HCfg<MT, BN, DRAWS, F8>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(heads_kernel<MT, BN, DRAWS, F8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         CF::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  heads_kernel<MT, BN, DRAWS, F8><<<grid, CF::THREADS, CF::SMEM_BYTES, st>>>(ta, tb, td, p);
  return cudaGetLastError();
}

int heads_bn(int n_draw) { return n_draw > 0 ? TILED_ROWS : 256; }
int heads_mt(int M) { return M <= BM ? 1 : 2; }

int heads_cpg(int M, int V, int n_draw) {
  const int mt = heads_mt(M);
  const int groups = (M + mt * BM - 1) / (mt * BM);
  const int bn = heads_bn(n_draw);
  const int n_tiles = (V + bn - 1) / bn;
  return std::min(std::max(1, dgi::num_sms() / groups), n_tiles);
}

// W's tiled copy: out[((t nkb + kb) 224 + r) 64 + c] = w[224 t + r][64 kb + c],
// zero for rows past V; one thread per 16 bytes.
__global__ void tile_weights_kernel(const uint4* __restrict__ w, uint4* __restrict__ out, int V,
                                    int D, int nkb, long long n16) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n16) return;
  const int c8 = (int)(i % (BK / 8));
  long long q = i / (BK / 8);
  const int r = (int)(q % TILED_ROWS);
  q /= TILED_ROWS;
  const int kb = (int)(q % nkb);
  const long long row = (q / nkb) * TILED_ROWS + r;
  out[i] = row < V ? w[(row * D + (long long)kb * BK) / 8 + c8] : make_uint4(0, 0, 0, 0);
}

}  // namespace

namespace dgi {

size_t heads_tiled_bytes(int V, int D) {
  if (V < 1 || D < BK || D % BK) return 0;
  return (size_t)((V + TILED_ROWS - 1) / TILED_ROWS) * TILED_ROWS * D * 2;
}

cudaError_t heads_tile_weights(const uint16_t* w, int V, int D, uint16_t* out, cudaStream_t st) {
  const size_t bytes = heads_tiled_bytes(V, D);
  if (!bytes) return cudaErrorInvalidValue;
  const long long n16 = (long long)(bytes / 16);
  tile_weights_kernel<<<(unsigned)((n16 + 255) / 256), 256, 0, st>>>(
      reinterpret_cast<const uint4*>(w), reinterpret_cast<uint4*>(out), V, D, D / BK, n16);
  return cudaGetLastError();
}

size_t heads_ws_bytes(int M, int V, int n_draw) {
  const int cpg = heads_cpg(M, V, n_draw);
  return align_up((size_t)5 * cpg * M * 4, 256) + align_up((size_t)2 * cpg * DRAW_N * 4, 256) +
         align_up((size_t)M * 4, 256);
}

size_t heads_probs_ld(int V) { return align_up((size_t)V, 64); }

cudaError_t denoise_heads(const uint16_t* h, int M, const uint16_t* draw_rows, int n_draw,
                          const uint16_t* w, const uint16_t* w_tiled, int V, int D,
                          const float* inv_t,
                          const float* inv_t_draw, RowStats out, float* lse_draw,
                          float* prob_scale, uint16_t* probs, size_t probs_ld, void* ws,
                          cudaStream_t st, const LabelGather* gather) {
  const int mt = heads_mt(M);
  const int groups = (M + mt * BM - 1) / (mt * BM);
  const int bn = heads_bn(n_draw);
  HeadsParams p{};
  p.M = M;
  p.n_draw = n_draw;
  p.V = V;
  p.K = D;
  p.cpg = heads_cpg(M, V, n_draw);
  p.n_tiles = (V + bn - 1) / bn;
  p.inv_t = inv_t;
  p.inv_t_draw = inv_t_draw;
  uint8_t* wp = static_cast<uint8_t*>(ws);
  p.part = reinterpret_cast<float*>(wp);
  wp += align_up((size_t)5 * p.cpg * M * 4, 256);
  p.part_draw = reinterpret_cast<float*>(wp);
  wp += align_up((size_t)2 * p.cpg * DRAW_N * 4, 256);
  float* ref = reinterpret_cast<float*>(wp);
  p.ref = ref;
  p.probs = reinterpret_cast<__nv_bfloat16*>(probs);
  p.ldp = (long long)probs_ld;
  p.status = status_ptr();
  if (gather && n_draw > 0) p.gl = *gather;
  CUtensorMap ta, tb, td;
  if (!make_tmap_bf16_2d(&ta, h, D, M, (uint64_t)D * 2, BK, BM)) return cudaErrorInvalidValue;
  p.w_nkb = 0;
  if (w_tiled && bn == TILED_ROWS && heads_tiled_bytes(V, D)) {
    // the tiled copy as [tiles x K blocks][224 rows][64 columns]; one box is one block
    const int nkb = D / BK;
    const uint64_t dims[3] = {BK, TILED_ROWS, (uint64_t)p.n_tiles * nkb};
    const uint64_t str[2] = {BK * 2, (uint64_t)TILED_ROWS * BK * 2};
    const uint32_t box[3] = {BK, TILED_ROWS, 1};
    if (!make_tmap_bf16_3d(&tb, w_tiled, dims, str, box)) return cudaErrorInvalidValue;
    p.w_nkb = nkb;
  } else if (!make_tmap_bf16_2d(&tb, w, D, V, (uint64_t)D * 2, BK, bn)) {
    return cudaErrorInvalidValue;
  }
  if (n_draw > 0) {
    if (!make_tmap_bf16_2d(&td, draw_rows, D, n_draw, (uint64_t)D * 2, BK, DRAW_N))
      return cudaErrorInvalidValue;
  } else {
    td = tb;  // unused
  }
  if (M >= REF_ROWS_MIN)
    ref_rows_kernel<<<(M + 7) / 8, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(h),
                                                reinterpret_cast<const __nv_bfloat16*>(w), inv_t,
                                                M, V, D, ref);
  else
    ref_kernel<<<M, REF_N * REF_KSPLIT * 32, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(h),
                                  reinterpret_cast<const __nv_bfloat16*>(w), inv_t, M, V, D, ref);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int grid = groups * p.cpg;
  if (n_draw > 0)
    e = (mt == 1) ? launch_heads<1, 224, true>(ta, tb, td, p, grid, st)
                  : launch_heads<2, 224, true>(ta, tb, td, p, grid, st);
  else
    e = (mt == 1) ? launch_heads<1, 256, false>(ta, tb, td, p, grid, st)
                  : launch_heads<2, 256, false>(ta, tb, td, p, grid, st);
  if (e != cudaSuccess) return e;
  const int row_blocks = (M + 7) / 8, draw_blocks = (n_draw + 7) / 8;
  heads_finalize_kernel<<<row_blocks + draw_blocks, 256, 0, st>>>(
      p.part, p.cpg, M, inv_t, out.lse, out.entropy, out.maxz, out.argmax, prob_scale, p.probs,
      p.ldp, p.n_tiles, bn, V, p.part_draw, n_draw, lse_draw, row_blocks, p.gl, p.status);
  return cudaGetLastError();
}

// The same pass on e4m3 operands (rows, draw rows and W each with one fp32 scale
// per row): 128-value K blocks through 8-bit tensor maps, kind::f8f6f4 MMAs,
// the scales applied to the accumulators in the epilogue.
cudaError_t denoise_heads_fp8(const uint8_t* h8, const float* h_scale, int M,
                              const uint8_t* d8, const float* d_scale, int n_draw,
                              const uint8_t* w8, const float* w_scale, int V, int D,
                              const float* inv_t, const float* inv_t_draw, RowStats out,
                              float* lse_draw, float* prob_scale, uint16_t* probs,
                              size_t probs_ld, void* ws, cudaStream_t st,
                              const LabelGather* gather) {
  const int mt = heads_mt(M);
  const int groups = (M + mt * BM - 1) / (mt * BM);
  const int bn = heads_bn(n_draw);
  HeadsParams p{};
  p.M = M;
  p.n_draw = n_draw;
  p.V = V;
  p.K = D;
  p.cpg = heads_cpg(M, V, n_draw);
  p.n_tiles = (V + bn - 1) / bn;
  p.inv_t = inv_t;
  p.inv_t_draw = inv_t_draw;
  p.h_scale = h_scale;
  p.w_scale = w_scale;
  p.d_scale = d_scale;
  uint8_t* wp = static_cast<uint8_t*>(ws);
  p.part = reinterpret_cast<float*>(wp);
  wp += align_up((size_t)5 * p.cpg * M * 4, 256);
  p.part_draw = reinterpret_cast<float*>(wp);
  wp += align_up((size_t)2 * p.cpg * DRAW_N * 4, 256);
  float* ref = reinterpret_cast<float*>(wp);
  p.ref = ref;
  p.probs = reinterpret_cast<__nv_bfloat16*>(probs);
  p.ldp = (long long)probs_ld;
  p.status = status_ptr();
  if (gather && n_draw > 0) p.gl = *gather;
  CUtensorMap ta, tb, td;
  // one 128-byte row of a box is one 128-value K block of e4m3
  if (!make_tmap_u8_2d(&ta, h8, D, M, (uint64_t)D, 128, BM)) return cudaErrorInvalidValue;
  if (!make_tmap_u8_2d(&tb, w8, D, V, (uint64_t)D, 128, bn)) return cudaErrorInvalidValue;
  if (n_draw > 0) {
    if (!make_tmap_u8_2d(&td, d8, D, n_draw, (uint64_t)D, 128, DRAW_N))
      return cudaErrorInvalidValue;
  } else {
    td = tb;  // unused
  }
  ref8_kernel<<<M, REF_N * 32, 0, st>>>(h8, h_scale, w8, w_scale, inv_t, V, D, ref);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int grid = groups * p.cpg;
  if (n_draw > 0)
    e = (mt == 1) ? launch_heads<1, TILED_ROWS, true, true>(ta, tb, td, p, grid, st)
                  : launch_heads<2, TILED_ROWS, true, true>(ta, tb, td, p, grid, st);
  else
    e = (mt == 1) ? launch_heads<1, 256, false, true>(ta, tb, td, p, grid, st)
                  : launch_heads<2, 256, false, true>(ta, tb, td, p, grid, st);
  if (e != cudaSuccess) return e;
  const int row_blocks = (M + 7) / 8, draw_blocks = (n_draw + 7) / 8;
  heads_finalize_kernel<<<row_blocks + draw_blocks, 256, 0, st>>>(
      p.part, p.cpg, M, inv_t, out.lse, out.entropy, out.maxz, out.argmax, prob_scale, p.probs,
      p.ldp, p.n_tiles, bn, V, p.part_draw, n_draw, lse_draw, row_blocks, p.gl, p.status);
  return cudaGetLastError();
}

}  // namespace dgi
