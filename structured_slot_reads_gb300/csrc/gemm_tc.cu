// gemm_tc.cu -- tcgen05/TMEM GEMMs of the denoise step, fed by TMA.
//
// One persistent kernel template computes D[m, n] = sum_k A[m, k] B[n, k] for
// K-major bf16 operands (rows of A and B contiguous along k) with fp32
// accumulators in tensor memory, and consumes D in one of three epilogues:
//
//   EPI_STATS  lm-head pass (tau-home.com "Refusing JSON token generation";
//              24-ai.news "Token commit mechanism"): A = hidden rows, B = W.
//              Each epilogue thread owns one row and keeps an online
//              (max, sum 2^(v-max), sum v 2^(v-max), argmax) over the vocabulary
//              tiles it sees, and takes the logits of its row's allowed labels
//              as they pass (the label gather); the [M, V] logits never leave
//              the SM.  EPI_STATS8 / EPI_STATS4: the same on e4m3 operands, or
//              with B = NVFP4 weights widened to bf16 on chip.
//   EPI_PROBS  first half of self-conditioning (24-ai.news "Token commit
//              mechanism"): recompute the logits tile and write
//              p = exp(z - lse) in bf16, the A operand of the second GEMM.
//   EPI_ACCUM  second half: split-K over the vocabulary of P . E, fp32 tile
//              partials, summed by a reduction kernel in a fixed order.
//
// Warp roles (one CTA per SM): warps [0, 4*MT) are the epilogue (warp w reads
// TMEM lanes 32*(w%4)..+31 of M-tile w/4), warp 4*MT issues the TMA loads of a
// shared-memory ring whose stages hold MT 128x64 A tiles and one BNx64 B tile
// (128-byte swizzled), warp 4*MT+1 owns TMEM and issues tcgen05.mma from one
// thread.  B is K-major (W) or MN-major (E read as [V, d_model]).
//
// Up to 16 rows, the statistics pass takes skinny_stats_kernel instead: the
// operands swapped (A = the vocabulary tile, B = the rows, resident in shared
// memory), so only W streams and the MMAs are 16 columns wide.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
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
constexpr int EPI_STATS = 0;
constexpr int EPI_PROBS = 1;
constexpr int EPI_ACCUM = 2;
constexpr int EPI_ACCUM_MN = 3;  // as EPI_ACCUM with B given N-contiguous ([K, N] row-major)
constexpr int EPI_STATS8 = 4;    // as EPI_STATS with e4m3 operands and per-row scales
constexpr int EPI_ACCUM8 = 5;    // as EPI_ACCUM with e4m3 operands (both K-major) and scales
constexpr int EPI_STATS4 = 6;    // as EPI_STATS with B = NVFP4 weights widened to bf16 on chip
constexpr int EPI_STATS4X = 7;   // as EPI_STATS with A and B NVFP4 on the block-scaled kind
constexpr int RING_BUDGET = 232448 - 1024 - 512;  // operand rings (227 KB - alignment - barriers)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct GemmParams {
  int M, N, K;
  int cpg;           // CTAs per m-group (STATS/PROBS)
  int n_tiles;       // ceil(N / BN)
  int k_split;       // ACCUM: number of K ranges
  int kb_per_split;  // ACCUM: k-blocks per range
  const float* inv_t;
  const float* lse;
  const float* row_scale;  // STATS8 / ACCUM8: scale of each A row
  const float* col_scale;  // STATS8 / ACCUM8: scale of each B row (an output column)
  const uint8_t* codes4;   // STATS4: e2m1 codes [K/64][N][32 bytes]
  const uint8_t* scales4;  // STATS4: e4m3 block scales [K/64][N][4]
  const float* gscale;     // STATS4: the weights' tensor scale
  const uint8_t* sf4;      // skinny block-scaled: the weights' scale atoms [N/128][K/64][512]
  const uint8_t* sf_rows;  // skinny block-scaled: the rows' scale atoms [K/64][512]
  const float* gscale_rows;  // skinny block-scaled: the rows' tensor scale
  dgi::LabelGather gl;     // STATS kinds: label gather (gl.out null: none)
  float* part;            // STATS: 5 x [cpg][M]; ACCUM: [k_split][M][N]
  __nv_bfloat16* probs;   // PROBS: [M][ldp]
  long long ldp;
  int* status;
};

// PK > 0 (NVFP4 B): a second, deeper ring of PK-byte stages holds the packed
// codes and scales, so that their DRAM latency is hidden while the operand
// ring holds only the A rows and the widened B tile.  SF > 0 (block-scaled
// NVFP4 A and B): each stage also holds SF bytes of scale atoms, and one
// accumulator stage leaves tensor memory for the scales.
template <int MT, int BN, int PK = 0, int SF = 0>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;   // one 128-row A tile of a K block
  static constexpr int A_STAGE = MT * A_BYTES;
  static constexpr int B_STAGE = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_STAGE + B_STAGE + SF;
  static constexpr int PK_BYTES = PK;
  static constexpr int NS_FIT = PK == 0 ? RING_BUDGET / STAGE_BYTES
                                : (3 * STAGE_BYTES + 4 * PK <= RING_BUDGET ? 3 : 2);
  static constexpr int NSTAGE = NS_FIT > 8 ? 8 : NS_FIT;
  static constexpr int PK_FIT = PK == 0 ? 0 : (RING_BUDGET - NSTAGE * STAGE_BYTES) / PK;
  static constexpr int PK_STAGES = PK_FIT > 8 ? 8 : PK_FIT;
  static constexpr int ACC_COLS = MT * BN;
  // SF > 0: one set of scale columns per ring stage (MT A tiles + the B tile, four
  // steps of four columns), written by the scale warps while the stage is in flight
  static constexpr int SF_COLS = SF > 0 ? NSTAGE * 16 * (MT + BN / 128) : 0;
  static constexpr int ACC_STAGES = (2 * ACC_COLS + SF_COLS <= 512) ? 2 : 1;
  static constexpr int TMEM_NEED = ACC_STAGES * ACC_COLS + SF_COLS;
  static constexpr int TMEM_COLS = TMEM_NEED <= 32    ? 32
                                   : TMEM_NEED <= 64  ? 64
                                   : TMEM_NEED <= 128 ? 128
                                   : TMEM_NEED <= 256 ? 256
                                                      : 512;
  static constexpr int EPI_WARPS = 4 * MT;
  static constexpr int THREADS = (EPI_WARPS + 2) * 32;  // + producer, MMA issuer
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM_BYTES = 1024 + NSTAGE * STAGE_BYTES + PK_STAGES * PK + BAR_BYTES;
  static constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
  static constexpr uint32_t IDESC_BMN = idesc_bf16_f32_bmn(BM, BN);
  static_assert(TMEM_NEED <= 512, "accumulators exceed tensor memory");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(NSTAGE >= 2, "ring depth");
  static_assert(PK == 0 || (PK_STAGES >= 2 && PK % 1024 == 0), "packed ring");
  static_assert(SF % 1024 == 0 && (SF == 0 || BN % 128 == 0), "scale atoms");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// NVFP4 B staging of one K block: BN rows x (32 code bytes + 4 scale bytes)
constexpr int f4_pk_bytes(int bn) { return bn * 36; }
// Block-scaled NVFP4: the scale atoms of one 256-value K block (four 64-value
// steps, 512 bytes per 128 rows and step) for MT A tiles and BN B rows
constexpr int x4_sf_bytes(int mt, int bn) { return (mt + bn / 128) * 4 * 512; }
// Warps widening the packed B tile to bf16 (more where the block has fewer
// epilogue warps), plus the packed-ring producer.
constexpr int f4_conv_warps(int mt) { return mt == 1 ? 16 : 8; }
constexpr int f4_extra_warps(int mt) { return f4_conv_warps(mt) + 1; }

// Four bytes of e2m1 code pairs (the even element in the low nibble) as four
// f16x2 words, by the hardware conversion (exact: every e2m1 value is an f16).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t word, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(word));
}

template <int MT, int BN, int EPI>
__global__ void __launch_bounds__(Cfg<MT, BN>::THREADS + (EPI == EPI_STATS4    ? 32 * f4_extra_warps(MT)
                                                          : EPI == EPI_STATS4X ? 128
                                                                               : 0),
                                  1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, GemmParams p) {
  constexpr bool F4 = EPI == EPI_STATS4;
  constexpr bool X4 = EPI == EPI_STATS4X;
  using CF = Cfg<MT, BN, F4 ? f4_pk_bytes(BN) : 0, X4 ? x4_sf_bytes(MT, BN) : 0>;
  constexpr int NSTAGE = CF::NSTAGE;
  constexpr int PK_STAGES = CF::PK_STAGES;
  constexpr int PRODUCER_WARP = CF::EPI_WARPS;
  constexpr int MMA_WARP = CF::EPI_WARPS + 1;
  constexpr int CONV0 = CF::EPI_WARPS + 2;   // STATS4: first converter warp
  constexpr int CONV_WARPS = f4_conv_warps(MT);
  constexpr int PK_WARP = CONV0 + CONV_WARPS;   // STATS4: packed-ring producer
  constexpr bool B_MN = EPI == EPI_ACCUM_MN;
  constexpr bool ACCUM = EPI == EPI_ACCUM || B_MN || EPI == EPI_ACCUM8;
  constexpr bool F8 = EPI == EPI_STATS8 || EPI == EPI_ACCUM8;
  constexpr bool STATS = EPI == EPI_STATS || EPI == EPI_STATS8 || F4 || X4;
  // a stage holds 128-byte operand rows: 64 bf16, 128 e4m3 or 256 e2m1 values of K
  constexpr int KB = X4 ? 256 : F8 ? 128 : BK;
  constexpr uint32_t IDESC_F8 = idesc_e4m3_f32(BM, BN);
  constexpr uint32_t IDESC_X4 = idesc_nvf4_f32(BM, BN);
  // X4: tensor-memory columns of the scales, after the accumulator: two sets of
  // (MT A tiles + one 128-row B tile) x 4 steps x 4 columns
  constexpr int X4_SF_COL = CF::ACC_STAGES * CF::ACC_COLS;
  constexpr int X4_SF_SET = 16 * (MT + BN / 128);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  uint8_t* pk_ring = smem + NSTAGE * CF::STAGE_BYTES;   // STATS4: packed codes + scales
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(pk_ring + PK_STAGES * CF::PK_BYTES);
  uint64_t* empty_bar = full_bar + NSTAGE;
  uint64_t* tfull_bar = empty_bar + NSTAGE;
  uint64_t* tempty_bar = tfull_bar + CF::ACC_STAGES;
  uint64_t* drain_bar = tempty_bar + CF::ACC_STAGES;
  // STATS4: [NSTAGE] the widened B tile written; STATS4X: the stage's scales written
  uint64_t* bready_bar = drain_bar + 1;
  uint64_t* pkfull_bar = bready_bar + ((F4 || X4) ? NSTAGE : 0);  // STATS4: [PK_STAGES]
  uint64_t* pkempty_bar = pkfull_bar + PK_STAGES;                 // STATS4: [PK_STAGES]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pkempty_bar + PK_STAGES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
      if (F4) mbar_init(&bready_bar[i], CONV_WARPS);
      if (X4) mbar_init(&bready_bar[i], 4);
    }
    for (int i = 0; i < PK_STAGES; ++i) {
      mbar_init(&pkfull_bar[i], 1);
      mbar_init(&pkempty_bar[i], CONV_WARPS);
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
    if (!F4) prefetch_tmap(&tmB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // ---- work assignment --------------------------------------------------
  const int total_kb = (p.K + KB - 1) / KB;
  int gm, t_begin, t_end, kb_begin, kb_end;
  if (ACCUM) {
    const int per_group = p.n_tiles * p.k_split;
    gm = blockIdx.x / per_group;
    const int rem = blockIdx.x % per_group;
    t_begin = rem / p.k_split;
    t_end = t_begin + 1;
    const int split = rem % p.k_split;
    kb_begin = split * p.kb_per_split;
    kb_end = min(total_kb, kb_begin + p.kb_per_split);
  } else {
    gm = blockIdx.x / p.cpg;
    const int gn = blockIdx.x % p.cpg;
    t_begin = (int)((long long)gn * p.n_tiles / p.cpg);
    t_end = (int)((long long)(gn + 1) * p.n_tiles / p.cpg);
    kb_begin = 0;
    kb_end = total_kb;
  }
  const int m_base = gm * MT * BM;
  const bool has_work = (t_end > t_begin) && (kb_end > kb_begin);

  if (warp == PRODUCER_WARP) {
    // One ring: the A rows (re-read from L2) and the B tile (streamed from DRAM)
    // of a K block are requested together and fill one stage.  All CTAs walk K
    // in the same order, so CTAs sharing the A rows read the same lines close
    // together in time (P, larger than L2, is then fetched from DRAM once).
    if (lane == 0 && has_work) {
      const uint64_t pol_b = policy_evict_first();  // W or E: streamed once
      const uint64_t pol_a = policy_evict_last();   // hidden rows or P: re-read per tile
      int stage = 0;
      uint32_t phase = 0, issued_mask = 0, last_phase = 0;
      bool ok = true;
      for (int t = t_begin; t < t_end && ok; ++t) {
        for (int kb = kb_begin; kb < kb_end; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* s_a = stages + stage * CF::STAGE_BYTES;
          uint8_t* s_b = s_a + CF::A_STAGE;
          // STATS4: the A rows only; the converter warps write the B tile.  STATS4X:
          // the codes of A and B (128 bytes a row) and the scale atoms of this
          // K block's steps (the last block may have fewer than four)
          const int ns = X4 ? min(4, p.K / 64 - 4 * kb) : 0;
          // X4: the A tiles of this group that hold rows (their scale atoms exist)
          const int a_tiles = X4 ? min(MT, (p.M - m_base + BM - 1) / BM) : 0;
          mbar_arrive_expect_tx(&full_bar[stage],
                                F4   ? CF::A_STAGE
                                : X4 ? CF::A_STAGE + CF::B_STAGE + (a_tiles + BN / 128) * ns * 512
                                     : CF::STAGE_BYTES);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
            tma_load_2d_hint(s_a + mt * CF::A_BYTES, &tmA, &full_bar[stage],
                             X4 ? kb * 128 : kb * KB, m_base + mt * BM, pol_a);
          if (F4) {
          } else if (X4) {
            const int n_steps = p.K / 64;
            // the tiled codes: block (128-row tile t, K block kb) is one 16 KB run
            tma_load_4d_hint(s_b, &tmB, &full_bar[stage], 0, 0, kb, t, pol_b);
            uint8_t* s_sf = s_b + CF::B_STAGE;
            for (int mt = 0; mt < a_tiles; ++mt)
              bulk_load(s_sf + mt * 2048,
                        p.sf_rows + ((long long)(m_base / BM + mt) * n_steps + 4 * kb) * 512,
                        ns * 512, &full_bar[stage]);
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              bulk_load(s_sf + (MT + h) * 2048,
                        p.sf4 + ((long long)(t * (BN / 128) + h) * n_steps + 4 * kb) * 512,
                        ns * 512, &full_bar[stage]);
          } else if (B_MN) {
            // B [K, N] with N contiguous: BN/64 boxes of 64 N-columns x 64 K-rows
#pragma unroll
            for (int g = 0; g < BN / 64; ++g)
              tma_load_2d_hint(s_b + g * (BK * 128), &tmB, &full_bar[stage], t * BN + g * 64,
                               kb * BK, pol_b);
          } else {
            tma_load_2d_hint(s_b, &tmB, &full_bar[stage], kb * KB, t * BN, pol_b);
          }
          issued_mask |= 1u << stage;
          last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == NSTAGE) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {  // let every copy already issued land before the CTA exits
        for (int s = 0; s < NSTAGE; ++s)
          if (issued_mask & (1u << s)) mbar_wait_drain(&full_bar[s], (last_phase >> s) & 1u);
      }
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0 && has_work) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = t_begin; t < t_end && ok; ++t) {
        if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_base = tmem_base + acc * CF::ACC_COLS;
        for (int kb = kb_begin; kb < kb_end; ++kb) {
          // the A rows (and B, by TMA); STATS4: also the B tile the converters widened
          if (!mbar_wait(&full_bar[stage], phase, abort_flag, p.status) ||
              ((F4 || X4) && !mbar_wait(&bready_bar[stage], phase, abort_flag, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stages + stage * CF::STAGE_BYTES);
          const uint32_t b_addr = a_addr + CF::A_STAGE;
          if constexpr (X4) {
            // the scale warps have written this stage's scales into its column set
            const uint32_t sf_t = tmem_base + X4_SF_COL + stage * X4_SF_SET;
            const int ns = min(4, p.K / 64 - 4 * kb);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              if (ks < ns) {
                const uint64_t bdesc = sw128_kmajor_desc(b_addr + ks * 32);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
                  tc_mma_nvf4(d_base + mt * BN,
                              sw128_kmajor_desc(a_addr + mt * CF::A_BYTES + ks * 32), bdesc,
                              IDESC_X4, sf_t + mt * 16 + ks * 4, sf_t + MT * 16 + ks * 4,
                              (kb > kb_begin || ks > 0) ? 1u : 0u);
              }
            }
            tc_commit(&empty_bar[stage]);
            if (++stage == NSTAGE) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // K-major B: +32 bytes per 16 K inside the 128-byte row; MN-major B:
            // +2 KB (two 8-row K groups) per 16 K
            const uint64_t bdesc = B_MN ? sw128_mnmajor_desc(b_addr + kk * 2048, BK * 128, 1024)
                                        : sw128_kmajor_desc(b_addr + kk * 32);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              const uint64_t adesc = sw128_kmajor_desc(a_addr + mt * CF::A_BYTES + kk * 32);
              // 32 bytes of K per instruction: 16 bf16 (K = 16) or 32 e4m3 (K = 32)
              if (F8)
                tc_mma_f8(d_base + mt * BN, adesc, bdesc, IDESC_F8,
                          (kb > kb_begin || kk > 0) ? 1u : 0u);
              else
                tc_mma_f16(d_base + mt * BN, adesc, bdesc, B_MN ? CF::IDESC_BMN : CF::IDESC,
                           (kb > kb_begin || kk > 0) ? 1u : 0u);
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
      // every MMA issued by this thread has completed once drain_bar flips
      tc_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0);
    }
  } else if (X4 && warp >= CONV0 && warp < CONV0 + 4) {
    // ---- STATS4X scale warps, one per TMEM lane quarter: each stage's scale atoms
    // (32 rows of 16 bytes) into the stage's column set, every quarter the same
    // rows (the layout the block-scaled MMA reads), off the tensor pipe's queue ----
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = has_work;
    for (int t = t_begin; t < t_end && ok; ++t) {
      for (int kb = kb_begin; kb < kb_end; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(&full_bar[stage], phase, abort_flag, p.status));
        if (!ok) break;
        const uint8_t* sfs = stages + stage * CF::STAGE_BYTES + CF::A_STAGE + CF::B_STAGE;
        const uint32_t col = tmem_base + lane_base + X4_SF_COL + stage * X4_SF_SET;
        const int ns = min(4, p.K / 64 - 4 * kb);
#pragma unroll
        for (int u = 0; u < MT + BN / 128; ++u) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            if (ks < ns) {
              const uint4 v =
                  *reinterpret_cast<const uint4*>(sfs + u * 2048 + ks * 512 + lane * 16);
              tmem_st_32x32b_x4(col + u * 16 + ks * 4, v);
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bready_bar[stage]);
        if (++stage == NSTAGE) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (F4 && warp >= CONV0 && warp < PK_WARP) {
    // ---- STATS4 converter warps: each K block's packed B rows -> bf16 tile ----
    // (128-byte swizzled rows of 64 values, the layout TMA gives the other passes)
    const int ci = threadIdx.x - CONV0 * 32;
    int stage = 0, ps = 0;
    uint32_t phase = 0, pphase = 0;
    bool ok = has_work;
    for (int t = t_begin; t < t_end && ok; ++t) {
      const int rows = min(BN, p.N - t * BN);
      for (int kb = kb_begin; kb < kb_end; ++kb) {
        // the packed rows have landed and the MMAs are done with this B slot
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&pkfull_bar[ps], pphase, abort_flag, p.status) &&
                            mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.status));
        if (!ok) break;
        uint8_t* s_b = stages + stage * CF::STAGE_BYTES + CF::A_STAGE;
        const uint8_t* s_c = pk_ring + ps * CF::PK_BYTES;
        const uint8_t* s_s = s_c + BN * 32;
        // unit u = half hf of row r: elements [32 hf, 32 hf + 32), i.e. 16 code
        // bytes, 2 block scales and 16-byte chunks 4 hf .. 4 hf + 3 of the row
        for (int u = ci; u < 2 * BN; u += 32 * CONV_WARPS) {
          const int r = u >> 1, hf = u & 1;
          uint8_t* dst = s_b + r * 128;
          if (r >= rows) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4*>(dst + (((4 * hf + j) ^ (r & 7)) * 16)) =
                  make_uint4(0, 0, 0, 0);
            continue;
          }
          const uint4 cc = *reinterpret_cast<const uint4*>(s_c + r * 32 + hf * 16);
          const uint32_t sw = *reinterpret_cast<const uint16_t*>(s_s + r * 4 + hf * 2);
          const uint32_t cw[4] = {cc.x, cc.y, cc.z, cc.w};
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const __half_raw hr =
                __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)((sw >> (8 * q)) & 0xFF), __NV_E4M3);
            const __half2 s2 = __halves2half2(__half(hr), __half(hr));
            // 16 elements of one block scale: code words 2q, 2q+1.  e2m1 times an
            // e4m3 scale has at most 6 significant bits and lies in [2^-10, 2688]
            // (or is 0), so the f16 product and the bf16 result are exact.
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t f16[4], o[4];
              e2m1x8_to_f16x2(cw[2 * q + h], f16);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float2 f =
                    __half22float2(__hmul2(*reinterpret_cast<const __half2*>(&f16[k]), s2));
                const __nv_bfloat162 v = __floats2bfloat162_rn(f.x, f.y);
                o[k] = *reinterpret_cast<const uint32_t*>(&v);
              }
              const int c = 4 * hf + 2 * q + h;
              *reinterpret_cast<uint4*>(dst + ((c ^ (r & 7)) * 16)) =
                  make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
        }
        fence_proxy_async_smem();   // generic writes -> the MMA's operand reads
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bready_bar[stage]);
          mbar_arrive(&pkempty_bar[ps]);
        }
        if (++stage == NSTAGE) {
          stage = 0;
          phase ^= 1u;
        }
        if (++ps == PK_STAGES) {
          ps = 0;
          pphase ^= 1u;
        }
      }
    }
  } else if (F4 && warp == PK_WARP) {
    // ---- STATS4 packed-ring producer: codes and scales of each K block's B rows,
    // contiguous in the K-block-major layout, up to PK_STAGES blocks ahead ----
    if (lane == 0 && has_work) {
      int ps = 0;
      uint32_t pphase = 0, issued_mask = 0, last_phase = 0;
      bool ok = true;
      for (int t = t_begin; t < t_end && ok; ++t) {
        const int rows = min(BN, p.N - t * BN);
        for (int kb = kb_begin; kb < kb_end; ++kb) {
          if (!mbar_wait(&pkempty_bar[ps], pphase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* dst = pk_ring + ps * CF::PK_BYTES;
          mbar_arrive_expect_tx(&pkfull_bar[ps], rows * 36);
          const long long r0 = (long long)kb * p.N + (long long)t * BN;
          bulk_load(dst, p.codes4 + r0 * 32, rows * 32, &pkfull_bar[ps]);
          bulk_load(dst + BN * 32, p.scales4 + r0 * 4, rows * 4, &pkfull_bar[ps]);
          issued_mask |= 1u << ps;
          last_phase = (last_phase & ~(1u << ps)) | (pphase << ps);
          if (++ps == PK_STAGES) {
            ps = 0;
            pphase ^= 1u;
          }
        }
      }
      if (!ok) {  // let every copy already issued land before the CTA exits
        for (int q = 0; q < PK_STAGES; ++q)
          if (issued_mask & (1u << q)) mbar_wait_drain(&pkfull_bar[q], (last_phase >> q) & 1u);
      }
    }
  } else {
    // ---- epilogue warps ---------------------------------------------------
    const int mt = warp >> 2;
    const int quarter = warp & 3;
    const int row = m_base + mt * BM + quarter * 32 + lane;
    const bool row_ok = row < p.M;
    float scale = 0.f, lse2 = 0.f, rs = 1.f;
    if (!ACCUM && row_ok) scale = __ldg(p.inv_t + row) * LOG2E;
    if (F8 && row_ok) rs = __ldg(p.row_scale + row);
    const float gs = F4   ? __ldg(p.gscale)
                     : X4 ? __ldg(p.gscale) * __ldg(p.gscale_rows)
                          : 1.f;
    if (EPI == EPI_PROBS && row_ok) lse2 = __ldg(p.lse + row) * LOG2E;
    float m_run = -INFINITY, s_run = 0.f, t_run = 0.f, best = -INFINITY;
    int best_idx = 0x7fffffff;
    // Label gather: this row's slot, its label table, and the smallest of its
    // label ids at or past the current chunk (INT_MAX: none left in this CTA's
    // columns), so a chunk without one of the row's labels costs one compare.
    const int32_t* g_ids = nullptr;
    int g_n = 0, g_o = 0, g_next = 0x7fffffff;
    float g_it = 0.f;
    if (STATS && p.gl.out != nullptr && row_ok && has_work) {
      int gs = -1;
      if (p.gl.R > 0) {
        if (row < p.gl.S * p.gl.R) {
          gs = row / p.gl.R;
          g_o = row;
        }
      } else {
        gs = p.gl.row_slot[row];
        g_o = gs;
      }
      if (gs >= 0) {
        g_n = min(max(__ldg(p.gl.n_labels + gs), 0), p.gl.L);
        g_ids = p.gl.label_ids + (long long)gs * p.gl.L;
        g_it = __ldg(p.inv_t + row);
        const int lo = t_begin * BN;
        for (int k = 0; k < g_n; ++k) {
          const int id = __ldg(g_ids + k);
          if (id >= lo && id < g_next) g_next = id;
        }
      }
    }
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = t_begin; t < t_end && has_work; ++t) {
      if (!mbar_wait(&tfull_bar[acc], acc_phase, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * CF::ACC_COLS + mt * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld_32x32b_x32(taddr + c * 32, r);
        tmem_ld_wait();
        const int n0 = t * BN + c * 32;
        if (!row_ok) continue;
        if (F8) {
          // unscaled e4m3 products: times the row's and each column's scale
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            float4 cs = make_float4(0.f, 0.f, 0.f, 0.f);
            if (n0 + j + 4 <= p.N) {
              cs = __ldg(reinterpret_cast<const float4*>(p.col_scale + n0 + j));
            } else {
              if (n0 + j < p.N) cs.x = __ldg(p.col_scale + n0 + j);
              if (n0 + j + 1 < p.N) cs.y = __ldg(p.col_scale + n0 + j + 1);
              if (n0 + j + 2 < p.N) cs.z = __ldg(p.col_scale + n0 + j + 2);
            }
            r[j] = __float_as_uint(__uint_as_float(r[j]) * rs * cs.x);
            r[j + 1] = __float_as_uint(__uint_as_float(r[j + 1]) * rs * cs.y);
            r[j + 2] = __float_as_uint(__uint_as_float(r[j + 2]) * rs * cs.z);
            r[j + 3] = __float_as_uint(__uint_as_float(r[j + 3]) * rs * cs.w);
          }
        }
        if (F4 || X4) {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * gs);
        }
        if (STATS && g_next < n0 + 32) {
          // one or more of this row's labels fall in the chunk: take their
          // logits from the registers, and find the next label past the chunk
          int nn = 0x7fffffff;
          for (int k = 0; k < g_n; ++k) {
            const int id = __ldg(g_ids + k);
            const unsigned dj = (unsigned)(id - n0);
            if (dj < 32u) {
              float z = __uint_as_float(r[0]);
#pragma unroll
              for (int j = 1; j < 32; ++j) z = dj == (unsigned)j ? __uint_as_float(r[j]) : z;
              p.gl.out[(long long)g_o * p.gl.L + k] = z * g_it;
            } else if (id >= n0 + 32 && id < nn) {
              nn = id;
            }
          }
          g_next = nn;
        }
        if (STATS) {
          if (n0 + 32 <= p.N) {
            float cm = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float a = __uint_as_float(r[j]);
              if (a > best) {
                best = a;
                best_idx = n0 + j;
              }
              cm = fmaxf(cm, a * scale);
            }
            if (cm > m_run) {
              const float f = ex2(m_run - cm);
              s_run *= f;
              t_run *= f;
              m_run = cm;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float v = __uint_as_float(r[j]) * scale;
              const float e = ex2(v - m_run);
              s_run += e;
              t_run = fmaf(e, v, t_run);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (n0 + j >= p.N) continue;
              const float a = __uint_as_float(r[j]);
              if (a > best) {
                best = a;
                best_idx = n0 + j;
              }
              const float v = a * scale;
              if (v > m_run) {
                const float f = ex2(m_run - v);
                s_run *= f;
                t_run *= f;
                m_run = v;
              }
              const float e = ex2(v - m_run);
              s_run += e;
              t_run = fmaf(e, v, t_run);
            }
          }
        } else if (EPI == EPI_PROBS) {
          __nv_bfloat16* dst = p.probs + (long long)row * p.ldp + n0;
          if (n0 + 32 <= p.N) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint4 pk;
              __nv_bfloat162 b0 = __floats2bfloat162_rn(
                  ex2(fmaf(__uint_as_float(r[j + 0]), scale, -lse2)),
                  ex2(fmaf(__uint_as_float(r[j + 1]), scale, -lse2)));
              __nv_bfloat162 b1 = __floats2bfloat162_rn(
                  ex2(fmaf(__uint_as_float(r[j + 2]), scale, -lse2)),
                  ex2(fmaf(__uint_as_float(r[j + 3]), scale, -lse2)));
              __nv_bfloat162 b2 = __floats2bfloat162_rn(
                  ex2(fmaf(__uint_as_float(r[j + 4]), scale, -lse2)),
                  ex2(fmaf(__uint_as_float(r[j + 5]), scale, -lse2)));
              __nv_bfloat162 b3 = __floats2bfloat162_rn(
                  ex2(fmaf(__uint_as_float(r[j + 6]), scale, -lse2)),
                  ex2(fmaf(__uint_as_float(r[j + 7]), scale, -lse2)));
              pk.x = *reinterpret_cast<uint32_t*>(&b0);
              pk.y = *reinterpret_cast<uint32_t*>(&b1);
              pk.z = *reinterpret_cast<uint32_t*>(&b2);
              pk.w = *reinterpret_cast<uint32_t*>(&b3);
              *reinterpret_cast<uint4*>(dst + j) = pk;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n0 + j < p.N)
                dst[j] = __float2bfloat16_rn(ex2(fmaf(__uint_as_float(r[j]), scale, -lse2)));
          }
        } else {  // EPI_ACCUM
          const int split = (blockIdx.x % (p.n_tiles * p.k_split)) % p.k_split;
          float* dst = p.part + ((long long)split * p.M + row) * p.N + n0;
          if (n0 + 32 <= p.N) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(dst + j) =
                  make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                              __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n0 + j < p.N) dst[j] = __uint_as_float(r[j]);
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
    if (STATS && row_ok) {
      const int gn = blockIdx.x % p.cpg;
      const long long o = (long long)row * p.cpg + gn;
      const long long plane = (long long)p.cpg * p.M;
      p.part[o] = m_run;
      p.part[o + plane] = s_run;
      p.part[o + 2 * plane] = t_run;
      p.part[o + 3 * plane] = best;
      reinterpret_cast<int*>(p.part)[o + 4 * plane] = best_idx;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == MMA_WARP) tmem_dealloc(tmem_base, CF::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Skinny statistics pass (M <= 16 rows: the slot reads' draw rows) with the
// operands swapped: A = a 128-row slice of the vocabulary tile (streamed), B =
// the M rows, resident in shared memory for the whole pass (N = 16, rows past M
// zero).  Per K block only W (or its NVFP4 codes and scales) streams; the MMAs
// are 16 columns wide instead of 128 rows tall (most of them padding); the
// accumulator has the vocabulary on the TMEM lanes, so each epilogue thread
// owns one vocabulary row and keeps the online statistics of all 16 columns,
// merged over lanes and warps once, at the end.  The partial statistics leave
// in the planes of the STATS epilogue, so stats_finalize_kernel merges them.
//
// Three operand modes: bf16 W and rows (MODE 0); NVFP4 W widened on chip to f16
// against f16 rows (MODE 1); NVFP4 W and NVFP4 rows on the block-scaled tensor-core
// kind (MODE 2: kind::mxf4nvf4, scale_vec::4X).  MODE 2 streams the packed codes
// (K blocks of 256 values, 128 bytes a row, by TMA) and each K block's scale atoms
// (bulk copies); the MMA warp moves the scales into tensor memory with
// tcgen05.cp (.32x128b.warpx4, one 512-byte atom per 128 rows and 64-value
// K-step): the rows' scales once, after the rows arrive, and each K block's W
// scales before the MMAs that read them, alternating two sets of columns.
// ---------------------------------------------------------------------------
constexpr int SK_N = 16;                    // rows of B (the MMAs' N)
constexpr int SK_BN = 256;                  // vocabulary rows per tile: two M = 128 MMAs
constexpr int SK_W_BYTES = SK_BN * BK * 2;  // a W tile of one K block (32 KB)
constexpr int SK_B_BLOCK = SK_N * BK * 2;   // the rows' 64-column block (2 KB)
constexpr int SK_MAX_KB = 48;               // resident rows for d_model up to 3072
constexpr int SK_EPI_WARPS = 4;
constexpr int SK_CONV_WARPS = 10;    // 16 warps in all (128 registers a thread)
constexpr int SK_GBITS = 64;                // label-gather chunk bitmap words

constexpr int SK_X4_KB = 256;               // MODE 2: values of a K block (128 bytes a row)
constexpr int SK_X4_ROWS = SK_N * 128;      // MODE 2: the rows' codes of a K block (2 KB)
constexpr int SK_X4_CODES = 12 * SK_X4_ROWS;   // MODE 2: resident row codes, d_model <= 3072
constexpr int SK_X4_SFA = 2 * 4 * 512;      // MODE 2: W scale atoms of a K block (2 x 4 steps)
constexpr int SK_X4_SFW_COL = 64;           // MODE 2: tensor-memory columns of the W scales
constexpr int SK_X4_SFR_COL = 256;          // MODE 2: ... and of the rows' scales

template <int MODE>
struct SkCfg {
  static constexpr bool F4 = MODE == 1;
  static constexpr bool X4 = MODE == 2;
  // resident rows: bf16 K blocks; MODE 2: the codes, then the scale atoms
  static constexpr int B_BYTES = X4 ? 2 * SK_X4_CODES : SK_MAX_KB * SK_B_BLOCK;
  // one W ring stage: a 256-row tile of a K block (MODE 2: plus its scale atoms)
  static constexpr int W_STAGE = SK_W_BYTES + (X4 ? SK_X4_SFA : 0);
  // W tiles in flight; NVFP4: the widened tiles are made on chip, so two
  // suffice, and the room goes to the packed blocks, whose copies wait on DRAM
  static constexpr int NW = F4 ? 2 : 4;
  static constexpr int NP = F4 ? 7 : 0;
  static constexpr int PK = F4 ? f4_pk_bytes(SK_BN) : 0;
  // barriers (at most 19 x 8 bytes), the gather bitmap (256), the TMEM slot and
  // abort flag (8), the row scales and powers of two (2 x 64)
  static constexpr int BAR_BYTES = 1024;
  static constexpr int SMEM_BYTES = 1024 + B_BYTES + NW * W_STAGE + NP * PK + BAR_BYTES;
  static constexpr int PRODUCER = SK_EPI_WARPS;            // rows, then W (or the packed ring)
  static constexpr int MMA = SK_EPI_WARPS + 1;
  static constexpr int CONV0 = SK_EPI_WARPS + 2;           // F4: converter warps; X4: scale warps
  static constexpr int THREADS = (SK_EPI_WARPS + 2 + (F4 ? SK_CONV_WARPS : X4 ? 4 : 0)) * 32;
  static constexpr int NSF = X4 ? NW : 0;                  // X4: "scales written" barriers
  // 2 stages x 2 halves x 16 columns; MODE 2: then one set of 32 W scale columns
  // per W stage (2 halves x 4 steps x 4) and, from column 256, the rows' scales
  static constexpr int TMEM_COLS = X4 ? 512 : 64;
  // bf16 W: bf16 operands.  NVFP4 W: f16 operands (the widening is then two
  // instructions a code pair, and every e2m1 x e4m3 product is an f16)
  static constexpr uint32_t IDESC = X4   ? idesc_nvf4_f32(BM, SK_N)
                                    : F4 ? idesc_f16_f32(BM, SK_N)
                                         : idesc_bf16_f32(BM, SK_N);
  static_assert(W_STAGE % 1024 == 0, "W stages stay 1 KB aligned");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(SK_EPI_WARPS == 4, "one epilogue warp per TMEM lane quarter");
  static_assert((2 * NW + 2 * NP + NSF + 7) * 8 + SK_GBITS * 4 + 8 + 2 * SK_N * 4 <= BAR_BYTES,
                "barrier region");
};

__device__ __forceinline__ void sk_epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"r"(SK_EPI_WARPS * 32) : "memory");
}

template <int MODE>
__global__ void __launch_bounds__(SkCfg<MODE>::THREADS, 1)
    skinny_stats_kernel(const __grid_constant__ CUtensorMap tmH,
                        const __grid_constant__ CUtensorMap tmW, GemmParams p) {
  using CF = SkCfg<MODE>;
  constexpr bool F4 = CF::F4;
  constexpr bool X4 = CF::X4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* bres = smem;                              // [K blocks][16 rows x 128 B]
  uint8_t* wring = bres + CF::B_BYTES;               // [NW][SK_BN rows x 128 B]
  uint8_t* pring = wring + CF::NW * CF::W_STAGE;     // F4: [NP][codes, scales]
  uint64_t* wfull = reinterpret_cast<uint64_t*>(pring + CF::NP * CF::PK);
  uint64_t* wempty = wfull + CF::NW;
  uint64_t* pfull = wempty + CF::NW;
  uint64_t* pempty = pfull + CF::NP;
  uint64_t* sfready = pempty + CF::NP;   // X4: [NW] a stage's W scales written
  uint64_t* tfull = sfready + CF::NSF;
  uint64_t* tempty = tfull + 2;
  uint64_t* bres_bar = tempty + 2;
  uint64_t* drain_bar = bres_bar + 1;
  uint64_t* rows16_bar = drain_bar + 1;   // F4: the rows converted to f16
  uint32_t* gbits = reinterpret_cast<uint32_t*>(rows16_bar + 1);
  uint32_t* tmem_slot = gbits + SK_GBITS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* sscale = reinterpret_cast<float*>(tmem_slot + 2);   // [16] 1/T of each row, log2 units
  float* srow = sscale + SK_N;   // F4: [16] 2^k, the power of two row j was divided by

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < CF::NW; ++i) {
      mbar_init(&wfull[i], F4 ? SK_CONV_WARPS : 1);
      mbar_init(&wempty[i], 1);
    }
    for (int i = 0; i < CF::NP; ++i) {
      mbar_init(&pfull[i], 1);
      mbar_init(&pempty[i], SK_CONV_WARPS);
    }
    for (int i = 0; i < CF::NSF; ++i) mbar_init(&sfready[i], 4);
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], SK_EPI_WARPS);
    }
    mbar_init(bres_bar, 1);
    mbar_init(rows16_bar, SK_EPI_WARPS);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == CF::MMA) {
    tmem_alloc(tmem_slot, CF::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == CF::PRODUCER && lane == 0) {
    prefetch_tmap(&tmH);
    if (!F4) prefetch_tmap(&tmW);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total_kb = X4 ? (p.K + SK_X4_KB - 1) / SK_X4_KB : (p.K + BK - 1) / BK;
  const int n_steps = p.K / 64;   // MODE 2: 64-value K-steps (one scale atom each)
  const int gn = blockIdx.x;
  const int t_begin = (int)((long long)gn * p.n_tiles / p.cpg);
  const int t_end = (int)((long long)(gn + 1) * p.n_tiles / p.cpg);
  const bool has_work = t_end > t_begin;

  if (warp == CF::PRODUCER) {
    if (lane == 0 && has_work) {
      if (X4) {
        // the rows' codes (256-value K blocks of 16 rows), then their scale atoms
        mbar_arrive_expect_tx(bres_bar, total_kb * SK_X4_ROWS + n_steps * 512);
        for (int kb = 0; kb < total_kb; ++kb)
          tma_load_2d(bres + kb * SK_X4_ROWS, &tmH, bres_bar, kb * 128, 0);
        bulk_load(bres + SK_X4_CODES, p.sf_rows, n_steps * 512, bres_bar);
      } else {
        // the rows, once: every 64-column block of rows [0, 16) (rows >= M read as 0)
        mbar_arrive_expect_tx(bres_bar, total_kb * SK_B_BLOCK);
        for (int kb = 0; kb < total_kb; ++kb)
          tma_load_2d(bres + kb * SK_B_BLOCK, &tmH, bres_bar, kb * BK, 0);
      }
      const uint64_t pol = policy_evict_first();
      int st = 0;
      uint32_t ph = 0, issued = 0, last = 0;
      bool ok = true;
      constexpr int NR = F4 ? CF::NP : CF::NW;
      uint64_t* ring_full = F4 ? pfull : wfull;
      uint64_t* ring_empty = F4 ? pempty : wempty;
      for (int t = t_begin; t < t_end && ok; ++t) {
        const int rows = min(SK_BN, p.N - t * SK_BN);
        for (int kb = 0; kb < total_kb; ++kb) {
          if (!mbar_wait(&ring_empty[st], ph ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          if (F4) {
            uint8_t* dst = pring + st * CF::PK;
            mbar_arrive_expect_tx(&pfull[st], rows * 36);
            const long long r0 = (long long)kb * p.N + (long long)t * SK_BN;
            bulk_load(dst, p.codes4 + r0 * 32, rows * 32, &pfull[st]);
            bulk_load(dst + SK_BN * 32, p.scales4 + r0 * 4, rows * 4, &pfull[st]);
          } else if (X4) {
            // the codes of 256 vocabulary rows x 256 values (rows past N read as 0) and
            // the scale atoms of each existing 128-row half for this block's K-steps
            uint8_t* dst = wring + st * CF::W_STAGE;
            const int ns = min(4, n_steps - 4 * kb);
            const bool half1 = (2 * t + 1) * BM < p.N;
            mbar_arrive_expect_tx(&wfull[st], SK_W_BYTES + (half1 ? 2 : 1) * ns * 512);
            // the tiled codes: the 16 KB blocks of 128-row tiles 2t and 2t + 1
            tma_load_4d_hint(dst, &tmW, &wfull[st], 0, 0, kb, 2 * t, pol);
            for (int h = 0; h < (half1 ? 2 : 1); ++h)
              bulk_load(dst + SK_W_BYTES + h * 2048,
                        p.sf4 + ((long long)(2 * t + h) * n_steps + 4 * kb) * 512, ns * 512,
                        &wfull[st]);
          } else {
            mbar_arrive_expect_tx(&wfull[st], SK_W_BYTES);
            tma_load_2d_hint(wring + st * CF::W_STAGE, &tmW, &wfull[st], kb * BK, t * SK_BN, pol);
          }
          issued |= 1u << st;
          last = (last & ~(1u << st)) | (ph << st);
          if (++st == NR) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < NR; ++s)
          if (issued & (1u << s)) mbar_wait_drain(&ring_full[s], (last >> s) & 1u);
      }
      mbar_wait_drain(bres_bar, 0);
    }
  } else if (warp == CF::MMA) {
    if (lane == 0 && has_work) {
      int ws = 0, acc = 0;
      uint32_t wph = 0, aph = 0;
      bool ok = mbar_wait(F4 ? rows16_bar : bres_bar, 0, abort_flag, p.status);
      if (X4 && ok) {
        // the rows' scales, resident for the whole pass
        const uint32_t sfr = smem_u32(bres + SK_X4_CODES);
        for (int s = 0; s < n_steps; ++s)
          tc_cp_32x128b_warpx4(tmem_base + SK_X4_SFR_COL + 4 * s,
                               plain_kmajor_desc(sfr + s * 512, 128));
      }
      for (int t = t_begin; t < t_end && ok; ++t) {
        if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        for (int kb = 0; kb < total_kb; ++kb) {
          if (!mbar_wait(&wfull[ws], wph, abort_flag, p.status) ||
              (X4 && !mbar_wait(&sfready[ws], wph, abort_flag, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t w_addr = smem_u32(wring + ws * CF::W_STAGE);
          if constexpr (X4) {
            // the scale warps have written this stage's W scales into its column
            // set (half 0 steps, half 1 steps)
            const uint32_t b_addr = smem_u32(bres + kb * SK_X4_ROWS);
            const uint32_t sf_t = tmem_base + SK_X4_SFW_COL + ws * 32;
            const int ns = min(4, n_steps - 4 * kb);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              if (ks < ns) {
                const uint64_t bdesc = sw128_kmajor_desc(b_addr + ks * 32);
#pragma unroll
                for (int half = 0; half < 2; ++half)
                  tc_mma_nvf4(tmem_base + acc * 32 + half * SK_N,
                              sw128_kmajor_desc(w_addr + half * (BM * 128) + ks * 32), bdesc,
                              CF::IDESC, sf_t + half * 16 + ks * 4,
                              tmem_base + SK_X4_SFR_COL + 4 * (4 * kb + ks),
                              (kb > 0 || ks > 0) ? 1u : 0u);
              }
            }
          } else {
            const uint32_t b_addr = smem_u32(bres + kb * SK_B_BLOCK);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t bdesc = sw128_kmajor_desc(b_addr + kk * 32);
#pragma unroll
              for (int half = 0; half < 2; ++half)
                tc_mma_f16(tmem_base + acc * 32 + half * SK_N,
                           sw128_kmajor_desc(w_addr + half * (BM * 128) + kk * 32), bdesc,
                           CF::IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
            }
          }
          tc_commit(&wempty[ws]);
          if (++ws == CF::NW) {
            ws = 0;
            wph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          aph ^= 1u;
        }
      }
      tc_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0);
    }
  } else if (X4 && warp >= CF::CONV0) {
    // ---- MODE 2 scale warps, one per TMEM lane quarter: each W stage's scale
    // atoms into the stage's column set, every quarter the same 32 rows of 16
    // bytes (the layout the block-scaled MMA reads), off the tensor pipe's queue ----
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    int ws = 0;
    uint32_t wph = 0;
    bool ok = has_work;
    for (int t = t_begin; t < t_end && ok; ++t) {
      for (int kb = 0; kb < total_kb; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(&wfull[ws], wph, abort_flag, p.status));
        if (!ok) break;
        const uint8_t* sfw = wring + ws * CF::W_STAGE + SK_W_BYTES;
        const uint32_t col = tmem_base + lane_base + SK_X4_SFW_COL + ws * 32;
        const int ns = min(4, n_steps - 4 * kb);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            if (ks < ns) {
              const uint4 v =
                  *reinterpret_cast<const uint4*>(sfw + h * 2048 + ks * 512 + lane * 16);
              tmem_st_32x32b_x4(col + h * 16 + ks * 4, v);
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfready[ws]);
        if (++ws == CF::NW) {
          ws = 0;
          wph ^= 1u;
        }
      }
    }
  } else if (F4 && warp >= CF::CONV0) {
    // NVFP4: widen each K block's packed rows into the W ring (as in the GEMM)
    const int ci = threadIdx.x - CF::CONV0 * 32;
    int ws = 0, ps = 0;
    uint32_t wph = 0, pph = 0;
    bool ok = has_work;
    for (int t = t_begin; t < t_end && ok; ++t) {
      const int rows = min(SK_BN, p.N - t * SK_BN);
      for (int kb = 0; kb < total_kb; ++kb) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&pfull[ps], pph, abort_flag, p.status) &&
                            mbar_wait(&wempty[ws], wph ^ 1u, abort_flag, p.status));
        if (!ok) break;
        uint8_t* s_b = wring + ws * CF::W_STAGE;
        const uint8_t* s_c = pring + ps * CF::PK;
        const uint8_t* s_s = s_c + SK_BN * 32;
        for (int u = ci; u < 2 * SK_BN; u += 32 * SK_CONV_WARPS) {
          const int r = u >> 1, hf = u & 1;
          uint8_t* dst = s_b + r * 128;
          if (r >= rows) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4*>(dst + (((4 * hf + j) ^ (r & 7)) * 16)) =
                  make_uint4(0, 0, 0, 0);
            continue;
          }
          const uint4 cc = *reinterpret_cast<const uint4*>(s_c + r * 32 + hf * 16);
          const uint32_t sw = *reinterpret_cast<const uint16_t*>(s_s + r * 4 + hf * 2);
          const uint32_t cw[4] = {cc.x, cc.y, cc.z, cc.w};
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const __half_raw hr =
                __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)((sw >> (8 * q)) & 0xFF), __NV_E4M3);
            const __half2 s2 = __halves2half2(__half(hr), __half(hr));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              // f16 operands: the exact product stays in f16
              uint32_t f16[4], o[4];
              e2m1x8_to_f16x2(cw[2 * q + h], f16);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&f16[k]), s2);
                o[k] = *reinterpret_cast<const uint32_t*>(&v);
              }
              const int c = 4 * hf + 2 * q + h;
              *reinterpret_cast<uint4*>(dst + ((c ^ (r & 7)) * 16)) =
                  make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&wfull[ws]);
          mbar_arrive(&pempty[ps]);
        }
        if (++ws == CF::NW) {
          ws = 0;
          wph ^= 1u;
        }
        if (++ps == CF::NP) {
          ps = 0;
          pph ^= 1u;
        }
      }
    }
  } else if (warp < SK_EPI_WARPS) {
    // ---- epilogue: lane = vocabulary row of a 128-row half, 16 columns = rows ----
    const int q = warp;
    const int M = p.M;
    const float gs = F4   ? __ldg(p.gscale)
                     : X4 ? __ldg(p.gscale) * __ldg(p.gscale_rows)
                          : 1.f;
    float m[SK_N], s[SK_N], tt[SK_N], best[SK_N];
    int bidx[SK_N];
#pragma unroll
    for (int j = 0; j < SK_N; ++j) {
      m[j] = -INFINITY;
      s[j] = 0.f;
      tt[j] = 0.f;
      best[j] = -INFINITY;
      bidx[j] = 0x7fffffff;
    }
    if (threadIdx.x < SK_N) sscale[threadIdx.x] = threadIdx.x < M ? __ldg(p.inv_t + threadIdx.x) * LOG2E : 0.f;
    if (F4 && has_work) {
      // The resident rows to f16, in place (the same 16-bit slots): row j is
      // first divided by 2^k_j (exact), k_j >= 0 the least that keeps its
      // largest element below 2^15, so nothing overflows; the accumulators of
      // column j are multiplied back by 2^k_j.  An element is exact in f16 unless
      // it falls below 2^-14 there, where f16's subnormal spacing 2^-24 rounds it.
      // Thread i takes row i / 8 and the 16-byte chunks i % 8 of every K block.
      const bool rows_ok = mbar_wait(bres_bar, 0, abort_flag, p.status);
      const int j = threadIdx.x >> 3, c = threadIdx.x & 7;
      const int nkb = (p.K + BK - 1) / BK;
      float amax = 0.f;
      for (int kb = 0; kb < nkb && rows_ok; ++kb) {
        const uint4 u = *reinterpret_cast<const uint4*>(bres + kb * SK_B_BLOCK + j * 128 + c * 16);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
          amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
      }
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      // 2^k with k = max(0, e - 15), amax < 2^e (amax's exponent + 1)
      const int ex = amax > 0.f ? ((__float_as_int(amax) >> 23) & 0xFF) - 126 : 0;
      const int k = max(0, ex - 15);
      const float down = __int_as_float((127 - k) << 23);
      for (int kb = 0; kb < nkb && rows_ok; ++kb) {
        uint4* ptr = reinterpret_cast<uint4*>(bres + kb * SK_B_BLOCK + j * 128 + c * 16);
        uint4 u = *ptr;
        uint32_t* w4 = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
          const __half2 hv = __floats2half2_rn(f.x * down, f.y * down);
          w4[e] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        *ptr = u;
      }
      if (c == 0) srow[j] = __int_as_float((127 + k) << 23);
      fence_proxy_async_smem();   // generic writes -> the MMAs' operand reads
      __syncwarp();
      if (lane == 0) mbar_arrive(rows16_bar);
    }
    sk_epi_bar();
    // label gather: one bit per 32 vocabulary rows of this CTA's range holding a
    // label of one of the rows (aliased modulo SK_GBITS * 32 chunks)
    const bool gat = p.gl.out != nullptr && has_work;
    const int g_lo = t_begin * SK_BN;
    if (gat) {
      for (int i = threadIdx.x; i < SK_GBITS; i += SK_EPI_WARPS * 32) gbits[i] = 0;
      sk_epi_bar();
      const int hi = min(t_end * SK_BN, p.N);
      for (int i = threadIdx.x; i < M * p.gl.L; i += SK_EPI_WARPS * 32) {
        const int j = i / p.gl.L, k = i % p.gl.L;
        const int sl = p.gl.R > 0 ? (j < p.gl.S * p.gl.R ? j / p.gl.R : -1) : p.gl.row_slot[j];
        if (sl < 0 || k >= min(max(__ldg(p.gl.n_labels + sl), 0), p.gl.L)) continue;
        const int id = __ldg(p.gl.label_ids + (long long)sl * p.gl.L + k);
        if (id >= g_lo && id < hi) {
          const int c = ((id - g_lo) >> 5) & (SK_GBITS * 32 - 1);
          atomicOr(gbits + (c >> 5), 1u << (c & 31));
        }
      }
      sk_epi_bar();
    }
    int acc = 0;
    uint32_t aph = 0;
    for (int t = t_begin; t < t_end; ++t) {
      if (!mbar_wait(&tfull[acc], aph, abort_flag, p.status)) break;
      tc_fence_after();
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t r[SK_N];
        __syncwarp();
        tmem_ld_32x32b_x16(tmem_base + ((uint32_t)(q * 32) << 16) + acc * 32 + half * SK_N, r);
        tmem_ld_wait();
        const int v0 = t * SK_BN + half * BM + q * 32;   // this warp's first vocabulary row
        const int v = v0 + lane;
        if (v < p.N) {
#pragma unroll
          for (int j = 0; j < SK_N; ++j) {
            if (j >= M) break;
            const float a = __uint_as_float(r[j]) * (F4 ? gs * srow[j] : gs);
            if (a > best[j]) {   // rows ascend, so the first occurrence is the lowest id
              best[j] = a;
              bidx[j] = v;
            }
            const float x = a * sscale[j];
            const float mn = fmaxf(m[j], x);
            const float fo = ex2(m[j] - mn), fx = ex2(x - mn);
            s[j] = fmaf(s[j], fo, fx);
            tt[j] = fmaf(tt[j], fo, fx * x);
            m[j] = mn;
          }
        }
        if (gat) {
          const int c = ((v0 - g_lo) >> 5) & (SK_GBITS * 32 - 1);
          if ((gbits[c >> 5] >> (c & 31)) & 1u) {
            for (int j = 0; j < M && v < p.N; ++j) {
              int sl, o;
              if (p.gl.R > 0) {
                sl = j < p.gl.S * p.gl.R ? j / p.gl.R : -1;
                o = j;
              } else {
                sl = p.gl.row_slot[j];
                o = sl;
              }
              if (sl < 0) continue;
              const int n = min(max(__ldg(p.gl.n_labels + sl), 0), p.gl.L);
              for (int k = 0; k < n; ++k) {
                if (__ldg(p.gl.label_ids + (long long)sl * p.gl.L + k) != v) continue;
                float z = __uint_as_float(r[0]);
#pragma unroll
                for (int jj = 1; jj < SK_N; ++jj) z = j == jj ? __uint_as_float(r[jj]) : z;
                p.gl.out[(long long)o * p.gl.L + k] =
                    z * (F4 ? gs * srow[j] : gs) * __ldg(p.inv_t + j);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        aph ^= 1u;
      }
    }
    // merge over the lanes, then over the four warps (through the W ring, idle
    // now that every MMA has completed), and write this CTA's partials
#pragma unroll
    for (int j = 0; j < SK_N; ++j) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m[j], o);
        const float so = __shfl_xor_sync(0xffffffffu, s[j], o);
        const float to = __shfl_xor_sync(0xffffffffu, tt[j], o);
        const float bo = __shfl_xor_sync(0xffffffffu, best[j], o);
        const int io = __shfl_xor_sync(0xffffffffu, bidx[j], o);
        const float mn = fmaxf(m[j], mo);
        if (mn == -INFINITY) {
          s[j] = 0.f;
          tt[j] = 0.f;
        } else {
          const float f1 = ex2(m[j] - mn), f2 = ex2(mo - mn);
          s[j] = s[j] * f1 + so * f2;
          tt[j] = tt[j] * f1 + to * f2;
        }
        m[j] = mn;
        if (bo > best[j] || (bo == best[j] && io < bidx[j])) {
          best[j] = bo;
          bidx[j] = io;
        }
      }
    }
    float* red = reinterpret_cast<float*>(wring);   // [4 warps][16][5]
    if (lane == 0 && has_work) {
#pragma unroll
      for (int j = 0; j < SK_N; ++j) {
        float* e = red + (q * SK_N + j) * 5;
        e[0] = m[j];
        e[1] = s[j];
        e[2] = tt[j];
        e[3] = best[j];
        reinterpret_cast<int*>(e)[4] = bidx[j];
      }
    }
    sk_epi_bar();
    if (q == 0 && lane < M && has_work) {
      const int j = lane;
      float mm = -INFINITY, ss = 0.f, tv = 0.f, bb = -INFINITY;
      int ii = 0x7fffffff;
      for (int w = 0; w < SK_EPI_WARPS; ++w) {
        const float* e = red + (w * SK_N + j) * 5;
        const float mo = e[0];
        const float mn = fmaxf(mm, mo);
        if (mn != -INFINITY) {
          const float f1 = ex2(mm - mn), f2 = ex2(mo - mn);
          ss = ss * f1 + e[1] * f2;
          tv = tv * f1 + e[2] * f2;
        }
        mm = mn;
        const int io = reinterpret_cast<const int*>(e)[4];
        if (e[3] > bb || (e[3] == bb && io < ii)) {
          bb = e[3];
          ii = io;
        }
      }
      const long long o = (long long)j * p.cpg + gn;
      const long long plane = (long long)p.cpg * M;
      p.part[o] = mm;
      p.part[o + plane] = ss;
      p.part[o + 2 * plane] = tv;
      p.part[o + 3 * plane] = bb;
      reinterpret_cast<int*>(p.part)[o + 4 * plane] = ii;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == CF::MMA) tmem_dealloc(tmem_base, CF::TMEM_COLS);
}

// Merge the per-CTA online statistics of every row: one warp per row, lanes over
// the CTA partials (stored row-major, [M][cpg]), a fixed shuffle-tree order.
__global__ void stats_finalize_kernel(const float* part, int cpg, int M, const float* inv_t,
                                      float* lse, float* entropy, float* maxz, int32_t* argmax,
                                      dgi::LabelGather gl, int V, int* status) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const long long plane = (long long)cpg * M;
  const float* pm = part + (long long)row * cpg;
  float m = -INFINITY;
  for (int g = lane; g < cpg; g += 32) m = fmaxf(m, pm[g]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f, t = 0.f, best = -INFINITY;
  int idx = 0x7fffffff;
  for (int g = lane; g < cpg; g += 32) {
    const float mg = pm[g];
    if (mg != -INFINITY) {
      const float f = exp2f(mg - m);
      s += pm[g + plane] * f;
      t += pm[g + 2 * plane] * f;
    }
    const float bg = pm[g + 3 * plane];
    const int ig = reinterpret_cast<const int*>(pm)[g + 4 * plane];
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
  const float l = (m + log2f(s)) * LN2;
  if (lane == 0) {
    lse[row] = l;
    entropy[row] = l - (t / s) * LN2;
    maxz[row] = best * inv_t[row];
    argmax[row] = idx;
  }
  if (gl.out != nullptr) {
    // the gathered label logits of a slot row: ids checked, lse subtracted
    int gs = -1, go = 0;
    if (gl.R > 0) {
      if (row < gl.S * gl.R) {
        gs = row / gl.R;
        go = row;
      }
    } else {
      gs = gl.row_slot[row];
      go = gs;
    }
    if (gs >= 0) {
      const int n = min(max(gl.n_labels[gs], 0), gl.L);
      for (int k = lane; k < n; k += 32) {
        const int id = gl.label_ids[(long long)gs * gl.L + k];
        float* dst = gl.out + (long long)go * gl.L + k;
        if (id < 0 || id >= V) {
          atomicOr(status, 4 /* DG_DEV_BAD_LABEL */);
          *dst = -INFINITY;
        } else if (gl.sub_lse) {
          *dst -= l;
        }
      }
    }
  }
}

// Slot of every row for a label gather keyed by slot rows: row_slot was set to
// -1; a row outside [0, M) or claimed by two slots is flagged.
__global__ void row_slot_kernel(const int32_t* slot_row, int S, int M, int32_t* row_slot,
                                int* status) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= S) return;
  const int r = slot_row[s];
  if (r < 0 || r >= M || atomicCAS(row_slot + r, -1, s) != -1)
    atomicOr(status, 8 /* DG_DEV_BAD_INDEX */);
}

// Prepares a label gather (the row -> slot map when slots are given by row).
cudaError_t gather_prepare(const dgi::LabelGather* g, int M, cudaStream_t st) {
  if (!g || !g->out || g->R > 0 || g->S == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(g->row_slot, 0xFF, (size_t)M * sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  row_slot_kernel<<<(g->S + 255) / 256, 256, 0, st>>>(g->slot_row, g->S, M, g->row_slot,
                                                      dgi::status_ptr());
  return cudaGetLastError();
}

// out[m][n] = row_scale[m] * sum over splits of part[s][m][n], splits added in
// order (row_scale may be null: 1).
__global__ void split_reduce_kernel(const float4* part, int k_split, long long n4, int n_cols,
                                    const float* row_scale, float4* out) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    float4 a = part[i];
#pragma unroll 4
    for (int s = 1; s < k_split; ++s) {
      const float4 b = part[(long long)s * n4 + i];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    if (row_scale) {
      const float f = row_scale[(i * 4) / n_cols];
      a.x *= f;
      a.y *= f;
      a.z *= f;
      a.w *= f;
    }
    out[i] = a;
  }
}

template <int MT, int BN, int EPI>
cudaError_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                        int grid, cudaStream_t st) {
  using CF = Cfg<MT, BN, 0, EPI == EPI_STATS4X ? x4_sf_bytes(MT, BN) : 0>;
  static bool attr_done = false;  // per-process; the attribute is per function
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<MT, BN, EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         CF::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  // STATS4X: four scale warps besides the epilogue, producer and MMA warps
  const int threads = CF::THREADS + (EPI == EPI_STATS4X ? 128 : 0);
  gemm_tc_kernel<MT, BN, EPI><<<grid, threads, CF::SMEM_BYTES, st>>>(ta, tb, p);
  return cudaGetLastError();
}

// The skinny pass of M <= 16 rows (see skinny_stats_kernel).
bool skinny_ok(int M, int K) { return M <= SK_N && (K + BK - 1) / BK <= SK_MAX_KB; }

template <int MODE>
cudaError_t launch_skinny(const CUtensorMap& th, const CUtensorMap& tw, const GemmParams& p,
                          cudaStream_t st) {
  using CF = SkCfg<MODE>;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(skinny_stats_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         CF::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  skinny_stats_kernel<MODE><<<p.cpg, CF::THREADS, CF::SMEM_BYTES, st>>>(th, tw, p);
  return cudaGetLastError();
}

constexpr int STATS_BN = 256;

int stats_mt(int M) { return M <= BM ? 1 : 2; }

int stats_cpg(int M, int V) {
  const int mt = stats_mt(M);
  const int groups = (M + mt * BM - 1) / (mt * BM);
  const int n_tiles = (V + STATS_BN - 1) / STATS_BN;
  int cpg = std::max(1, dgi::num_sms() / groups);
  return std::min(cpg, n_tiles);
}

// Row statistics over the vocabulary: partials + finalize.
cudaError_t run_stats(const uint16_t* h, int M, const uint16_t* w, int V, int D,
                      const float* inv_t, dgi::RowStats out, float* part, cudaStream_t st,
                      const dgi::LabelGather* gather) {
  CUtensorMap ta, tb;
  if (!dgi::make_tmap_bf16_2d(&ta, h, D, M, (uint64_t)D * 2, BK, BM)) return cudaErrorInvalidValue;
  if (!dgi::make_tmap_bf16_2d(&tb, w, D, V, (uint64_t)D * 2, BK, STATS_BN)) return cudaErrorInvalidValue;
  const int mt = stats_mt(M);
  const int groups = (M + mt * BM - 1) / (mt * BM);
  if (cudaError_t e0 = gather_prepare(gather, M, st); e0 != cudaSuccess) return e0;
  GemmParams p{};
  p.M = M;
  p.N = V;
  p.K = D;
  p.cpg = stats_cpg(M, V);
  p.n_tiles = (V + STATS_BN - 1) / STATS_BN;
  p.inv_t = inv_t;
  p.part = part;
  p.status = dgi::status_ptr();
  if (gather) p.gl = *gather;
  cudaError_t e;
  if (skinny_ok(M, D)) {
    CUtensorMap th;   // the rows as 64 x 16 boxes (rows past M read as 0)
    if (!dgi::make_tmap_bf16_2d(&th, h, D, M, (uint64_t)D * 2, BK, SK_N))
      return cudaErrorInvalidValue;
    e = launch_skinny<0>(th, tb, p, st);
  } else {
    e = (mt == 1) ? launch_gemm<1, STATS_BN, EPI_STATS>(ta, tb, p, groups * p.cpg, st)
                  : launch_gemm<2, STATS_BN, EPI_STATS>(ta, tb, p, groups * p.cpg, st);
  }
  if (e != cudaSuccess) return e;
  stats_finalize_kernel<<<(M + 7) / 8, 256, 0, st>>>(part, p.cpg, M, inv_t, out.lse,
                                                     out.entropy, out.maxz, out.argmax, p.gl, V,
                                                     p.status);
  return cudaGetLastError();
}

// The statistics pass on e4m3 operands: K blocks of 128 values (128-byte rows).
cudaError_t run_stats_fp8(const uint8_t* h8, const float* h_scale, int M, const uint8_t* w8,
                          const float* w_scale, int V, int D, const float* inv_t,
                          dgi::RowStats out, float* part, cudaStream_t st,
                          const dgi::LabelGather* gather) {
  CUtensorMap ta, tb;
  if (!dgi::make_tmap_u8_2d(&ta, h8, D, M, (uint64_t)D, 128, BM)) return cudaErrorInvalidValue;
  if (!dgi::make_tmap_u8_2d(&tb, w8, D, V, (uint64_t)D, 128, STATS_BN))
    return cudaErrorInvalidValue;
  const int mt = stats_mt(M);
  const int groups = (M + mt * BM - 1) / (mt * BM);
  if (cudaError_t e0 = gather_prepare(gather, M, st); e0 != cudaSuccess) return e0;
  GemmParams p{};
  p.M = M;
  p.N = V;
  p.K = D;
  p.cpg = stats_cpg(M, V);
  p.n_tiles = (V + STATS_BN - 1) / STATS_BN;
  p.inv_t = inv_t;
  p.row_scale = h_scale;
  p.col_scale = w_scale;
  p.part = part;
  p.status = dgi::status_ptr();
  if (gather) p.gl = *gather;
  cudaError_t e =
      (mt == 1) ? launch_gemm<1, STATS_BN, EPI_STATS8>(ta, tb, p, groups * p.cpg, st)
                : launch_gemm<2, STATS_BN, EPI_STATS8>(ta, tb, p, groups * p.cpg, st);
  if (e != cudaSuccess) return e;
  stats_finalize_kernel<<<(M + 7) / 8, 256, 0, st>>>(part, p.cpg, M, inv_t, out.lse,
                                                     out.entropy, out.maxz, out.argmax, p.gl, V,
                                                     p.status);
  return cudaGetLastError();
}

// The statistics pass against NVFP4 weights: bf16 rows (TMA) times the codes
// and block scales (bulk copies) widened to bf16 on chip; the tensor scale is
// applied to the accumulators.
template <int MT>
cudaError_t launch_stats4(const CUtensorMap& ta, const GemmParams& p, int grid, cudaStream_t st) {
  using CF = Cfg<MT, STATS_BN, f4_pk_bytes(STATS_BN)>;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<MT, STATS_BN, EPI_STATS4>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         CF::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  gemm_tc_kernel<MT, STATS_BN, EPI_STATS4>
      <<<grid, CF::THREADS + 32 * f4_extra_warps(MT), CF::SMEM_BYTES, st>>>(ta, ta, p);
  return cudaGetLastError();
}

cudaError_t run_stats_nvfp4(const uint16_t* h, int M, const uint8_t* codes, const uint8_t* scales,
                            const float* g, int V, int D, const float* inv_t, dgi::RowStats out,
                            float* part, cudaStream_t st, const dgi::LabelGather* gather) {
  CUtensorMap ta;
  if (!dgi::make_tmap_bf16_2d(&ta, h, D, M, (uint64_t)D * 2, BK, BM)) return cudaErrorInvalidValue;
  const int mt = stats_mt(M);
  const int groups = (M + mt * BM - 1) / (mt * BM);
  if (cudaError_t e0 = gather_prepare(gather, M, st); e0 != cudaSuccess) return e0;
  GemmParams p{};
  p.M = M;
  p.N = V;
  p.K = D;
  p.cpg = stats_cpg(M, V);
  p.n_tiles = (V + STATS_BN - 1) / STATS_BN;
  p.inv_t = inv_t;
  p.codes4 = codes;
  p.scales4 = scales;
  p.gscale = g;
  p.part = part;
  p.status = dgi::status_ptr();
  if (gather) p.gl = *gather;
  cudaError_t e;
  if (skinny_ok(M, D)) {
    CUtensorMap th;
    if (!dgi::make_tmap_bf16_2d(&th, h, D, M, (uint64_t)D * 2, BK, SK_N))
      return cudaErrorInvalidValue;
    e = launch_skinny<1>(th, th, p, st);
  } else {
    e = (mt == 1) ? launch_stats4<1>(ta, p, groups * p.cpg, st)
                  : launch_stats4<2>(ta, p, groups * p.cpg, st);
  }
  if (e != cudaSuccess) return e;
  stats_finalize_kernel<<<(M + 7) / 8, 256, 0, st>>>(part, p.cpg, M, inv_t, out.lse,
                                                     out.entropy, out.maxz, out.argmax, p.gl, V,
                                                     p.status);
  return cudaGetLastError();
}

// Both operands NVFP4 on the block-scaled kind.  The rows are quantised into the
// workspace (codes, scale atoms, tensor scale; after the partials and the
// label-gather scratch); up to 16 rows take the skinny pass in MODE 2, more the
// GEMM form (EPI_STATS4X: rows on the TMEM lanes, 128-row vocabulary tiles).
constexpr int X4_BN = 128;

size_t x4_rows_offset(int M, int V) {
  return dgi::lmhead_ws_bytes(M, V) + dgi::align_up((size_t)M * 4, 256);
}

int x4_rows_padded(int M) { return M <= SK_N ? SK_N : M; }

cudaError_t run_stats_nvfp4_mma(const uint16_t* h, int M, const uint8_t* codes, const uint8_t* sf,
                                const float* g, int V, int D, const float* inv_t,
                                dgi::RowStats out, void* ws, cudaStream_t st,
                                const dgi::LabelGather* gather) {
  using dgi::align_up;
  const bool skinny = M <= SK_N;
  const int Mp = x4_rows_padded(M);
  uint8_t* rc = static_cast<uint8_t*>(ws) + x4_rows_offset(M, V);
  uint8_t* rsf = rc + align_up((size_t)Mp * (D / 2), 256);
  float* rg = reinterpret_cast<float*>(
      rsf + align_up((size_t)((Mp + 127) / 128) * (D / 64) * 512, 256));
  cudaError_t e =
      skinny ? dgi::quantize_rows_nvfp4_mma(h, M, D, rc, rsf, rg, st)
             : dgi::quantize_many_rows_nvfp4_mma(h, M, D, rc, rsf, rg,
                                                 reinterpret_cast<unsigned int*>(rg + 1), st);
  if (e != cudaSuccess) return e;
  CUtensorMap ta, tb;
  if (!dgi::make_tmap_u8_2d(&ta, rc, D / 2, Mp, D / 2, 128, skinny ? SK_N : BM))
    return cudaErrorInvalidValue;
  {
    // tiled codes [ceil(V/128)][ceil(D/256)][128 rows][128 bytes]; a box is one
    // 128-row block (the GEMM form) or two consecutive tiles' blocks (skinny)
    const int nkb = (D / 64 + 3) / 4;
    const uint64_t tiles = (uint64_t)(V + 127) / 128;
    const uint64_t dims[4] = {128, 128, (uint64_t)nkb, tiles};
    const uint64_t str[3] = {128, 128 * 128, (uint64_t)nkb * 128 * 128};
    const uint32_t box[4] = {128, 128, 1, skinny ? SK_BN / 128u : X4_BN / 128u};
    if (!dgi::make_tmap_u8_4d(&tb, codes, dims, str, box)) return cudaErrorInvalidValue;
  }
  if ((e = gather_prepare(gather, M, st)) != cudaSuccess) return e;
  GemmParams p{};
  p.M = M;
  p.N = V;
  p.K = D;
  p.cpg = stats_cpg(M, V);
  p.n_tiles = (V + (skinny ? SK_BN : X4_BN) - 1) / (skinny ? SK_BN : X4_BN);
  p.inv_t = inv_t;
  p.codes4 = codes;
  p.sf4 = sf;
  p.gscale = g;
  p.sf_rows = rsf;
  p.gscale_rows = rg;
  p.part = static_cast<float*>(ws);
  p.status = dgi::status_ptr();
  if (gather) p.gl = *gather;
  if (skinny) {
    e = launch_skinny<2>(ta, tb, p, st);
  } else {
    // two 128-row tiles a CTA when there are more than 128 rows (one accumulator
    // stage then, beside the scales): each W tile is copied and its scales moved
    // into tensor memory once for 256 rows.  One tile a CTA with two accumulator
    // stages, two groups sharing each W tile through L2, took 20% longer at 256
    // rows: twice the scale copies and barrier hand-offs per W byte.
    const int mt = stats_mt(M);
    const int groups = (M + mt * BM - 1) / (mt * BM);
    e = (mt == 1) ? launch_gemm<1, X4_BN, EPI_STATS4X>(ta, tb, p, groups * p.cpg, st)
                  : launch_gemm<2, X4_BN, EPI_STATS4X>(ta, tb, p, groups * p.cpg, st);
  }
  if (e != cudaSuccess) return e;
  stats_finalize_kernel<<<(M + 7) / 8, 256, 0, st>>>(p.part, p.cpg, M, inv_t, out.lse,
                                                     out.entropy, out.maxz, out.argmax, p.gl, V,
                                                     p.status);
  return cudaGetLastError();
}

constexpr int ACC_BN = 256;

// Split of the vocabulary (the K of P . E) over CTAs: every split non-empty.
// kb = K-block width (64 bf16 or 128 e4m3 values).
void accum_split(int M, int V, int D, int* k_split, int* kb_per_split, int kb = BK) {
  const int mt = stats_mt(M);
  const int groups = (M + mt * BM - 1) / (mt * BM);
  const int n_tiles = (D + ACC_BN - 1) / ACC_BN;
  const int total_kb = (V + kb - 1) / kb;
  const int tiles = groups * n_tiles, sms = dgi::num_sms();
  int ks;
  if (tiles <= sms * 7 / 16) {
    // Few output tiles: the GEMM is bound by the stream of E, which 7/8 of the
    // SMs keep saturated (256 x 262144 x 2816: 132 CTAs take 280 us against 279
    // for 143), so the split leaves the other eighth to work running beside it
    // on another stream.
    ks = std::max(1, (sms * 7 / 8) / tiles);
  } else {
    // Many output tiles: the CTAs are tensor-bound and come in waves; take the
    // split with the fewest rounds of whole-tile work, ceil(tiles ks / SMs) / ks
    // (2048 rows: 88 tiles on 88 SMs, or in 5 splits 440 CTAs in 3 waves of a
    // fifth of the work each), the smallest split on a tie.
    ks = 1;
    long long best_num = (tiles + sms - 1) / sms, best_den = 1;
    for (int c = 2; c <= 8; ++c) {
      const long long rounds = ((long long)tiles * c + sms - 1) / sms;
      if (rounds * best_den < best_num * c) {
        best_num = rounds;
        best_den = c;
        ks = c;
      }
    }
  }
  ks = std::min(ks, total_kb);
  const int kbps = (total_kb + ks - 1) / ks;
  *kb_per_split = kbps;
  *k_split = (total_kb + kbps - 1) / kbps;
}

}  // namespace

namespace dgi {

size_t lmhead_ws_bytes(int M, int V) {
  return align_up((size_t)5 * stats_cpg(M, V) * M * sizeof(float), 256);
}

cudaError_t lmhead_stats(const uint16_t* h, int M, const uint16_t* w, int V, int D,
                         const float* inv_t, RowStats out, void* ws, cudaStream_t st,
                         const LabelGather* gather) {
  return run_stats(h, M, w, V, D, inv_t, out, static_cast<float*>(ws), st, gather);
}

cudaError_t lmhead_stats_fp8(const uint8_t* h8, const float* h_scale, int M, const uint8_t* w8,
                             const float* w_scale, int V, int D, const float* inv_t, RowStats out,
                             void* ws, cudaStream_t st, const LabelGather* gather) {
  return run_stats_fp8(h8, h_scale, M, w8, w_scale, V, D, inv_t, out, static_cast<float*>(ws), st,
                       gather);
}

cudaError_t lmhead_stats_nvfp4(const uint16_t* h, int M, const uint8_t* codes,
                               const uint8_t* scales, const float* g, int V, int D,
                               const float* inv_t, RowStats out, void* ws, cudaStream_t st,
                               const LabelGather* gather) {
  return run_stats_nvfp4(h, M, codes, scales, g, V, D, inv_t, out, static_cast<float*>(ws), st,
                         gather);
}

size_t lmhead_nvfp4_mma_ws_bytes(int M, int V, int D) {
  const int Mp = x4_rows_padded(M);
  return x4_rows_offset(M, V) + align_up((size_t)Mp * (D / 2), 256) +
         align_up((size_t)((Mp + 127) / 128) * (D / 64) * 512, 256) + 256;
}

// (the last 256 bytes: g and, above 16 rows, the rows' largest magnitude)
bool lmhead_nvfp4_mma_ok(int M, int D) {
  return M >= 1 && D >= 64 && D % 64 == 0 && (M > SK_N || D <= 12 * SK_X4_KB);
}

cudaError_t lmhead_stats_nvfp4_mma(const uint16_t* h, int M, const uint8_t* codes,
                                   const uint8_t* sf, const float* g, int V, int D,
                                   const float* inv_t, RowStats out, void* ws, cudaStream_t st,
                                   const LabelGather* gather) {
  return run_stats_nvfp4_mma(h, M, codes, sf, g, V, D, inv_t, out, ws, st, gather);
}

size_t selfcond_ws_bytes(int M, int V, int D) {
  const size_t probs = align_up((size_t)M * align_up(V, 64) * 2, 256);
  int ks, kbps;
  accum_split(M, V, D, &ks, &kbps);
  const size_t part = align_up((size_t)ks * M * D * sizeof(float), 256);
  return probs + part;
}

cudaError_t selfcond(const uint16_t* h, int M, const uint16_t* w, const uint16_t* e, int V,
                     int D, const float* inv_t, const float* lse, float* out, void* ws,
                     cudaStream_t st) {
  const size_t ldp = align_up(V, 64);
  __nv_bfloat16* probs = static_cast<__nv_bfloat16*>(ws);
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                         align_up((size_t)M * ldp * 2, 256));
  const int mt = stats_mt(M);
  const int groups = (M + mt * BM - 1) / (mt * BM);
  // 1) probabilities p = exp(z - lse) in bf16
  {
    CUtensorMap ta, tb;
    if (!make_tmap_bf16_2d(&ta, h, D, M, (uint64_t)D * 2, BK, BM)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16_2d(&tb, w, D, V, (uint64_t)D * 2, BK, STATS_BN)) return cudaErrorInvalidValue;
    GemmParams p{};
    p.M = M;
    p.N = V;
    p.K = D;
    p.cpg = stats_cpg(M, V);
    p.n_tiles = (V + STATS_BN - 1) / STATS_BN;
    p.inv_t = inv_t;
    p.lse = lse;
    p.probs = probs;
    p.ldp = (long long)ldp;
    p.status = status_ptr();
    cudaError_t e = (mt == 1)
                        ? launch_gemm<1, STATS_BN, EPI_PROBS>(ta, tb, p, groups * p.cpg, st)
                        : launch_gemm<2, STATS_BN, EPI_PROBS>(ta, tb, p, groups * p.cpg, st);
    if (e != cudaSuccess) return e;
  }
  // 2) split-K partials of P . E over the vocabulary, 3) ordered reduction
  return probs_embed(reinterpret_cast<const uint16_t*>(probs), ldp, nullptr, M, e, V, D, out,
                     part, st);
}

size_t probs_embed_ws_bytes(int M, int V, int D) {
  int ks, kbps;
  accum_split(M, V, D, &ks, &kbps);
  return align_up((size_t)ks * M * D * sizeof(float), 256);
}

cudaError_t probs_embed(const uint16_t* probs, size_t ldp, const float* row_scale, int M,
                        const uint16_t* e, int V, int D, float* out, void* ws,
                        cudaStream_t st) {
  const int mt = stats_mt(M);
  const int groups = (M + mt * BM - 1) / (mt * BM);
  float* part = static_cast<float*>(ws);
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_2d(&ta, probs, V, M, (uint64_t)ldp * 2, BK, BM)) return cudaErrorInvalidValue;
  // E [V, D] row-major is the MN-major B operand: boxes of 64 d-columns x 64 vocabulary rows
  if (!make_tmap_bf16_2d(&tb, e, D, V, (uint64_t)D * 2, 64, BK)) return cudaErrorInvalidValue;
  GemmParams p{};
  p.M = M;
  p.N = D;
  p.K = V;
  p.n_tiles = (D + ACC_BN - 1) / ACC_BN;
  accum_split(M, V, D, &p.k_split, &p.kb_per_split);
  p.part = part;
  p.status = status_ptr();
  const int grid = groups * p.n_tiles * p.k_split;
  cudaError_t err = (mt == 1) ? launch_gemm<1, ACC_BN, EPI_ACCUM_MN>(ta, tb, p, grid, st)
                              : launch_gemm<2, ACC_BN, EPI_ACCUM_MN>(ta, tb, p, grid, st);
  if (err != cudaSuccess) return err;
  const long long n4 = (long long)M * D / 4;
  const int blocks = (int)std::min<long long>((n4 + 255) / 256, 4LL * num_sms());
  split_reduce_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(part), p.k_split,
                                              n4, D, row_scale, reinterpret_cast<float4*>(out));
  return cudaGetLastError();
}

size_t probs_embed8_ws_bytes(int M, int V, int D) {
  int ks, kbps;
  accum_split(M, V, D, &ks, &kbps, 128);
  return align_up((size_t)ks * M * D * sizeof(float), 256);
}

// P . E on e4m3 operands: p8 [M, V] (one scale per row), e8t = E transposed
// [D, V] (one scale per d_model column), both K-major with K = the vocabulary.
// out = row_scale * p_scale * e_scale * sum_v p8 e8t, split-K over the vocabulary.
cudaError_t probs_embed8(const uint8_t* p8, const float* p_scale, const float* row_scale, int M,
                         const uint8_t* e8t, const float* e_scale, int V, int D, float* out,
                         void* ws, cudaStream_t st) {
  const int mt = stats_mt(M);
  const int groups = (M + mt * BM - 1) / (mt * BM);
  float* part = static_cast<float*>(ws);
  CUtensorMap ta, tb;
  if (!make_tmap_u8_2d(&ta, p8, V, M, (uint64_t)V, 128, BM)) return cudaErrorInvalidValue;
  if (!make_tmap_u8_2d(&tb, e8t, V, D, (uint64_t)V, 128, ACC_BN)) return cudaErrorInvalidValue;
  GemmParams p{};
  p.M = M;
  p.N = D;
  p.K = V;
  p.n_tiles = (D + ACC_BN - 1) / ACC_BN;
  accum_split(M, V, D, &p.k_split, &p.kb_per_split, 128);
  p.row_scale = p_scale;
  p.col_scale = e_scale;
  p.part = part;
  p.status = status_ptr();
  const int grid = groups * p.n_tiles * p.k_split;
  cudaError_t err = (mt == 1) ? launch_gemm<1, ACC_BN, EPI_ACCUM8>(ta, tb, p, grid, st)
                              : launch_gemm<2, ACC_BN, EPI_ACCUM8>(ta, tb, p, grid, st);
  if (err != cudaSuccess) return err;
  const long long n4 = (long long)M * D / 4;
  const int blocks = (int)std::min<long long>((n4 + 255) / 256, 4LL * num_sms());
  split_reduce_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(part), p.k_split,
                                              n4, D, row_scale, reinterpret_cast<float4*>(out));
  return cudaGetLastError();
}

}  // namespace dgi
