// attn_tc.cu -- decoder-mode attention with 512-wide heads on the 5th-generation
// tensor cores (24-ai.news, "How does diffusion text generation differ?";
// thakicloud.com, "What is DiffusionGemma").
//
// Every canvas row attends to all prompt keys of its request (encoder KV,
// contiguous or in pages) and to the canvas keys within +-W of its position:
// one joint softmax, scale 1/sqrt(d).  A CTA owns 128 query rows = (128/G canvas
// positions) x (the G query heads of one KV head), so each key tile serves the
// whole GQA group.
//
// Tensor memory holds 512 fp32 columns per lane, exactly one 128 x 512 output
// accumulator, so the output columns are split over two CTAs: each keeps
// O[:, 256 h .. 256 h + 255] (256 columns) and recomputes the scores S = Q K^T
// (two 128-column buffers, so the softmax of one key tile overlaps the QK^T of
// the next).  Both CTAs of a pair compute bit-identical scores and therefore
// take identical softmax decisions.  Per 128-key tile:
//   MMA warp   S[j%2] = Q K_j^T                  (A, B from shared memory, TMA)
//   softmax    p = 2^(s*log2e/sqrt(d) - m), row sums; p (bf16) overwrites S in TMEM
//   MMA warp   O += P V_j                        (A = P from tensor memory, B = V)
// The reference m is raised only when a tile's maximum exceeds it by more than
// 2^8 (O is then rescaled in tensor memory), so p <= 256 and rescales are rare.
// The key range is split across CTAs (split-KV) and merged by the combine kernel.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace {

using namespace dgk;

constexpr int HD = 512;                 // head width
constexpr int DH = 256;                 // output columns per CTA
constexpr int BM = 128;                 // query rows per CTA
constexpr int BN = 128;                 // keys per tile
constexpr int BOX = BN * 128;           // one TMA box: 128 rows x 64 bf16 (16 KB)
constexpr int UNIT = 2 * BOX;           // one ring slot (32 KB)
constexpr int NSLOT = 3;
constexpr int Q_BYTES = BM * HD * 2;    // 128 KB, resident
constexpr int K_UNITS = HD / 128;       // 4 slots of K per tile (128 head columns each)
constexpr int V_UNITS = DH / 128;       // 2 slots of V per tile (this CTA's 256 columns)
constexpr int SOFT_WARPS = 8;           // two per TMEM lane quarter
constexpr int PRODUCER_WARP = SOFT_WARPS;
constexpr int MMA_WARP = SOFT_WARPS + 1;
constexpr int THREADS = (SOFT_WARPS + 2) * 32;
constexpr int TMEM_COLS = 512;
constexpr int O_COL = 0;                // O: columns [0, 256)
constexpr int S_COL = 256;              // S buffers: [256, 384) and [384, 512)
constexpr int BAR_BYTES = 256;
// per-tile row-maximum exchange of the two softmax warps of a lane quarter:
// [tile parity][warp half][128 rows] bf16
constexpr int XMAX_BYTES = 2 * 2 * BM * 2;
constexpr int SMEM_BYTES = 1024 + Q_BYTES + NSLOT * UNIT + BAR_BYTES + XMAX_BYTES;
constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN);
constexpr uint32_t IDESC_PV = idesc_bf16_f32_bmn(BM, 128);
constexpr uint32_t IDESC_QK_PAIR = idesc_bf16_f32(2 * BM, BN);
constexpr uint32_t IDESC_PV_PAIR = idesc_bf16_f32_bmn(2 * BM, DH);
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float LAZY = 8.f;             // log2 headroom before O is rescaled
constexpr int ORDER_MAX_B = 64;         // decoder batches up to this size go longest first
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct TcArgs {
  int B, C, Pmax, Hq, Hkv, W, G, npos, q_blocks, splits;
  int causal;              // encoder prefill: rows attend to keys j <= i of their own sequence
  const int32_t* seq_len;  // causal: valid rows (and keys) per request
  const int32_t* mode;     // mixed batch: per request 1 = causal, 0 = decoder (null: `causal`)
  const int32_t* rows_len; // mixed batch: valid rows per request (null: seq_len or C)
  const int32_t* page_table;
  int pages_per_req, n_pages, page_size;
  const int32_t* prompt_len;
  __nv_bfloat16* out;  // [B][C][Hq][512]
  float* lse;          // [B][Hq][C]
  float* ws_o;         // [splits][B][C][Hq][512]
  float* ws_ml;        // [splits][B][Hq][C][2]: reference (log2 units), sum
  int* status;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// bf16 bit pattern of the smallest bf16 value >= x (x finite or -inf): positive
// values round up, negative values truncate toward zero.
__device__ __forceinline__ uint16_t bf16_bits_up(float x) {
  uint32_t u = __float_as_uint(x);
  if (x > 0.f) u += 0xFFFFu;
  return (uint16_t)(u >> 16);
}
__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
  return __uint_as_float((uint32_t)h << 16);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Key-tile geometry of one CTA (shared by every role).
struct Tiles {
  int P, p0, npos, clo, chi, nbp, t_begin, t_end, len, causal;
  __device__ int key0(int t) const { return t < nbp ? t * BN : clo + (t - nbp) * BN; }
};

__device__ __forceinline__ Tiles tiles_of(const TcArgs& a, int b, int qb, int split) {
  Tiles T;
  T.p0 = qb * a.npos;
  T.npos = min(a.npos, a.C - T.p0);
  T.causal = a.mode ? (a.mode[b] != 0) : (a.causal != 0);
  const int32_t* lens = a.rows_len ? a.rows_len : (T.causal ? a.seq_len : nullptr);
  T.len = lens ? min(max(lens[b], 0), a.C) : a.C;
  if (T.causal) {
    // keys 0 .. (last row of the block), within the request's length
    T.P = 0;
    T.clo = 0;
    T.chi = T.p0 < T.len ? min(T.len, T.p0 + T.npos) : 0;  // no rows of this block: no keys
  } else if (T.p0 < T.len) {
    // prompt keys plus the rows of the request within +-W of the block
    T.P = min(max(a.prompt_len[b], 0), a.Pmax);
    T.clo = max(0, T.p0 - a.W);
    T.chi = min(T.len, T.p0 + T.npos - 1 + a.W + 1);
  } else {
    T.P = 0;
    T.clo = 0;
    T.chi = 0;
  }
  T.nbp = (T.P + BN - 1) / BN;
  const int nb = T.nbp + (T.chi - T.clo + BN - 1) / BN;
  T.t_begin = (int)((long long)split * nb / a.splits);
  T.t_end = (int)((long long)(split + 1) * nb / a.splits);
  return T;
}

// Page of prompt key k (k < P) of request b, or -1 when the table entry is invalid.
__device__ __forceinline__ int page_of(const TcArgs& a, int b, int k) {
  const int pg = a.page_table[(long long)b * a.pages_per_req + k / a.page_size];
  return (pg < 0 || pg >= a.n_pages) ? -1 : pg;
}

// Valid-key bit mask of one 32-key chunk for a row: keys [lo, hi) of the tile,
// minus the pages flagged in `bad` (bit i = tile keys [i ps, (i+1) ps)).
__device__ __forceinline__ uint32_t chunk_mask(int c, int lo, int hi, uint32_t bad, int ps) {
  const int a0 = max(lo - 32 * c, 0), a1 = min(hi - 32 * c, 32);
  if (a1 <= a0) return 0u;
  uint32_t m = (a1 == 32 ? 0xffffffffu : ((1u << a1) - 1u)) & ~((1u << a0) - 1u);
  if (bad) {
    for (int i = 0; i < BN / ps; ++i) {
      if (!((bad >> i) & 1u)) continue;
      const int k0 = i * ps - 32 * c, k1 = k0 + ps;
      const int b0 = max(k0, 0), b1 = min(k1, 32);
      if (b1 > b0) m &= ~((b1 == 32 ? 0xffffffffu : ((1u << b1) - 1u)) & ~((1u << b0) - 1u));
    }
  }
  return m;
}

// Softmax and output roles.  Warps w and w + 4 share query rows 32 (w % 4) .. +31
// (their TMEM lane quarter); warp half h = w / 4 takes keys [64 h, 64 h + 64) of
// every tile and output columns [128 h, 128 h + 128) of this CTA's 256.
// In the CTA-pair kernel the two CTAs hold consecutive row blocks of one pair
// tile (row_off = rank x 128/G positions) and the probabilities-ready barrier is
// the even CTA's (pready_c = its shared::cluster addresses).
template <bool PAIR>
__device__ __forceinline__ void softmax_and_store(const TcArgs& a, const Tiles& T, int n, int b,
                                                  int g, int dh, int split, int warp, int lane,
                                                  uint32_t tmem_base, uint64_t* sfull_bar,
                                                  uint64_t* pready_bar, uint64_t* pv_bar,
                                                  uint64_t* pair_bar, volatile int* abort_flag,
                                                  float* xch, int row_off, uint32_t pready_c0,
                                                  uint32_t pready_c1, uint16_t* xmax) {
  constexpr unsigned FULL = 0xffffffffu;
  const int quarter = warp & 3, half = warp >> 2;
  const int r = quarter * 32 + lane;
  const int lp = row_off + r / a.G;
  const int pos = T.p0 + lp;
  const bool row_ok = lp < T.npos && pos < T.len;
  const int head = g * a.G + r % a.G;
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  const float sl2 = LOG2E * rsqrtf((float)HD);
  float m_ref = -INFINITY, l = 0.f;
  bool ok = true;
  // page validity of a prompt tile: lane i checks the table entry of the tile's
  // page i, read one tile ahead so the table's latency overlaps the score wait
  const int npg = a.page_table ? BN / a.page_size : 0;
  auto page_bad = [&](int t) -> bool {
    if (!a.page_table || t >= T.nbp || lane >= npg) return false;
    const int k = t * BN + lane * a.page_size;
    return k < T.P && page_of(a, b, k) < 0;
  };
  bool bad_next = n > 0 && page_bad(T.t_begin);
  for (int j = 0; j < n; ++j) {
    const int t = T.t_begin + j;
    const bool bad_lane = bad_next;
    if (j + 1 < n) bad_next = page_bad(t + 1);
    ok = __all_sync(FULL, mbar_wait(&sfull_bar[j & 1], (j >> 1) & 1u, abort_flag, a.status));
    if (!ok) break;
    tc_fence_after();
    const uint32_t s_addr = tmem_base + lane_base + S_COL + (j & 1) * BN;
    const int key0 = T.key0(t);
    int lo, hi;
    uint32_t bad = 0;
    if (t < T.nbp) {
      lo = 0;
      hi = min(BN, T.P - key0);
      if (a.page_table) {
        bad = __ballot_sync(FULL, bad_lane);
        if (bad && r == 0 && half == 0) atomicOr(a.status, 2 /* DG_DEV_BAD_PAGE */);
      }
    } else if (T.causal) {
      lo = -key0;
      hi = min(T.chi, pos + 1) - key0;
    } else {
      lo = max(T.clo, pos - a.W) - key0;
      hi = min(T.chi, pos + a.W + 1) - key0;
    }
    // pass 1: this warp's 64 scores of the tile (keys [64 h, 64 h + 64)), read from
    // tensor memory once, and their masked maximum; the pair exchanges its partial
    // maxima in log2 units rounded up to bf16, so both warps take the same
    // reference and it is never below the row's true maximum (phase j of the
    // pair's barrier; slot parity j % 2 is rewritten two tiles later, after the
    // partner has passed phase j + 1 and so has read this value)
    uint32_t v0[32], v1[32];
    tmem_ld_32x32b_x32(s_addr + (2 * half) * 32, v0);
    tmem_ld_32x32b_x32(s_addr + (2 * half + 1) * 32, v1);
    const uint32_t vm0 = chunk_mask(2 * half, lo, hi, bad, a.page_size);
    const uint32_t vm1 = chunk_mask(2 * half + 1, lo, hi, bad, a.page_size);
    tmem_ld_wait();
    // every key of the warp's 64 valid for every row (the prompt tiles but the
    // last): the maximum and the exponentials without per-key masks
    const bool fast = __all_sync(FULL, (vm0 & vm1) == 0xffffffffu);
    float mh = -INFINITY;
    if (fast) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        mh = fmaxf(mh, fmaxf(__uint_as_float(v0[i]), __uint_as_float(v1[i])));
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if ((vm0 >> i) & 1u) mh = fmaxf(mh, __uint_as_float(v0[i]));
        if ((vm1 >> i) & 1u) mh = fmaxf(mh, __uint_as_float(v1[i]));
      }
    }
    const uint16_t own = bf16_bits_up(mh == -INFINITY ? -INFINITY : mh * sl2);
    uint16_t* xm = xmax + (j & 1) * 2 * BM;
    xm[half * BM + r] = own;
    __syncwarp();   // the warp's writes, ordered before its one arrival
    if (lane == 0) mbar_arrive(&pair_bar[quarter]);
    ok = __all_sync(FULL, mbar_wait(&pair_bar[quarter], j & 1u, abort_flag, a.status));
    if (!ok) break;
    const float mb = fmaxf(bf16_bits_to_float(own), bf16_bits_to_float(xm[(half ^ 1) * BM + r]));
    // lazy reference: raise it (and rescale O) only past LAZY log2 units
    const float m_new = fmaxf(m_ref, mb);
    const bool raise = m_new > m_ref + LAZY;
    const bool rescale = raise && m_ref != -INFINITY;
    const float f = rescale ? ex2(m_ref - m_new) : 1.f;
    if (__any_sync(FULL, rescale)) {
      // O holds tiles up to j-1: wait for the last P V, then scale this half's
      // columns in place.  The scores of tile j were committed after P V of tile
      // j-2, so the phase of tile j-2 is complete and this parity wait is unambiguous.
      ok = __all_sync(FULL, mbar_wait(pv_bar, (j - 1) & 1u, abort_flag, a.status));
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        const uint32_t o_addr = tmem_base + lane_base + O_COL + half * 128 + c * 32;
        tmem_ld_32x32b_x32(o_addr, o);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
        tmem_st_32x32b_x32(o_addr, o);
      }
      tmem_st_wait();
    }
    l *= f;
    if (raise) m_ref = m_new;
    const float mr = (m_ref == -INFINITY) ? 0.f : m_ref;
    // pass 2: p = 2^(s sl2 - m) from the registers, written as bf16 pairs over this
    // half's own score columns: keys [64 h, 64 h + 64) -> P columns [64 h, 64 h + 32)
    float psum = 0.f;
    auto probs = [&](const uint32_t (&v)[32], uint32_t vm, int cc) {
      uint32_t pk[16];
      if (fast) {
        // packed fp32 pairs: one FMA forms two exponents, one add keeps two partial sums
        const float2 sc = make_float2(sl2, sl2), off = make_float2(-mr, -mr);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 x = __ffma2_rn(
              make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), sc, off);
          const float2 pp = make_float2(ex2(x.x), ex2(x.y));
          acc = __fadd2_rn(acc, pp);
          pk[i] = pack_bf16(pp.x, pp.y);
        }
        psum += acc.x + acc.y;
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float x0 = fmaf(__uint_as_float(v[2 * i]), sl2, -mr);
          const float x1 = fmaf(__uint_as_float(v[2 * i + 1]), sl2, -mr);
          const float p0 = ((vm >> (2 * i)) & 1u) ? ex2(x0) : 0.f;
          const float p1 = ((vm >> (2 * i + 1)) & 1u) ? ex2(x1) : 0.f;
          psum += p0 + p1;
          pk[i] = pack_bf16(p0, p1);
        }
      }
      tmem_st_32x32b_x16(s_addr + half * 64 + cc * 16, pk);
    };
    probs(v0, vm0, 0);
    probs(v1, vm1, 1);
    l += psum;
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();   // one arrival per warp (a cluster-scope release in the pair)
    if (lane == 0) {
      if constexpr (PAIR)
        mbar_arrive_cluster((j & 1) ? pready_c1 : pready_c0);
      else
        mbar_arrive(&pready_bar[j & 1]);
    }
  }
  // the last two P V products: wait phase n-2 first, so that the parity wait for
  // phase n-1 cannot be satisfied by an older phase
  if (ok && n > 1) ok = __all_sync(FULL, mbar_wait(pv_bar, (n - 2) & 1u, abort_flag, a.status));
  if (ok && n > 0) ok = __all_sync(FULL, mbar_wait(pv_bar, (n - 1) & 1u, abort_flag, a.status));
  if (!ok) return;
  // row sum over both halves: phase n of the pair's barrier
  xch[half * 128 + r] = l;
  __syncwarp();
  if (lane == 0) mbar_arrive(&pair_bar[quarter]);
  if (!__all_sync(FULL, mbar_wait(&pair_bar[quarter], n & 1u, abort_flag, a.status))) return;
  l += xch[(half ^ 1) * 128 + r];
  tc_fence_after();
  const long long orow = (long long)(b * a.C + pos) * a.Hq + head;
  if (n == 0) {
    if (row_ok && dh == 0 && half == 0) {
      float* ml = a.ws_ml + (((long long)split * a.B + b) * a.Hq + head) * a.C * 2 + pos * 2;
      ml[0] = -INFINITY;
      ml[1] = 0.f;
    }
    return;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t o[32];
    tmem_ld_32x32b_x32(tmem_base + lane_base + O_COL + half * 128 + c * 32, o);
    tmem_ld_wait();
    if (!row_ok) continue;
    const int col = dh * DH + half * 128 + c * 32;
    if (a.splits == 1) {
      uint4* dst = reinterpret_cast<uint4*>(a.out + orow * HD + col);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 w;
        w.x = pack_bf16(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
        w.y = pack_bf16(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
        w.z = pack_bf16(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
        w.w = pack_bf16(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
        dst[q] = w;
      }
    } else {
      float4* dst = reinterpret_cast<float4*>(
          a.ws_o + (long long)split * a.B * a.C * a.Hq * HD + orow * HD + col);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[q] = make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                             __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3]));
    }
  }
  if (!row_ok || dh != 0 || half != 0) return;
  if (a.splits == 1) {
    a.lse[((long long)b * a.Hq + head) * a.C + pos] = (m_ref + log2f(l)) * LN2;
  } else {
    float* ml = a.ws_ml + (((long long)split * a.B + b) * a.Hq + head) * a.C * 2 + pos * 2;
    ml[0] = m_ref;
    ml[1] = l;
  }
}

// The kernel body.  PAIR: a cluster of two CTAs shares each MMA (cta_group::2,
// M = 256): CTA rank r holds query rows [128 r, 128 r + 128) of a 256-row pair
// tile, half of every key tile's K (keys [64 r, 64 r + 64), all 512 head
// columns: two ring units) and half of its V columns (this output half's
// columns [128 r, 128 r + 128): one unit), so one key tile (K and V) is three
// units, the whole ring: V(j) waits in one slot while K(j+1) fills the others.
template <bool PAIR>
__device__ __forceinline__ void attn_body(const CUtensorMap& tmQ, const CUtensorMap& tmKe,
                                          const CUtensorMap& tmVe, const CUtensorMap& tmKc,
                                          const CUtensorMap& tmVc, const TcArgs& a) {
  constexpr int KU = PAIR ? 2 : K_UNITS;  // ring units of K per tile
  constexpr int VU = PAIR ? 1 : V_UNITS;  // ring units of V per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* ring = smem + Q_BYTES;
  uint8_t* bar_base = ring + NSLOT * UNIT;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(bar_base);
  uint64_t* empty_bar = full_bar + NSLOT;
  uint64_t* q_bar = empty_bar + NSLOT;
  uint64_t* sfull_bar = q_bar + 1;       // [2] scores of tile j in buffer j % 2 ready
  uint64_t* pready_bar = sfull_bar + 2;  // [2] probabilities of tile j written over them
  uint64_t* pv_bar = pready_bar + 2;     // O += P V of a tile complete
  uint64_t* drain_bar = pv_bar + 1;
  uint64_t* pair_bar = drain_bar + 1;    // [4] the two softmax warps of a lane quarter
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pair_bar + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // row-sum exchange of the softmax warp pairs, after the last tile (the ring is idle then)
  float* xch = reinterpret_cast<float*>(ring);
  uint16_t* xmax = reinterpret_cast<uint16_t*>(bar_base + BAR_BYTES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  int bid = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int split = bid % a.splits;
  bid /= a.splits;
  const int dh = bid & 1;
  bid >>= 1;
  // causal prefill: the last query blocks see the most keys, so they go first
  const int qb = (a.causal || a.mode) ? a.q_blocks - 1 - bid % a.q_blocks : bid % a.q_blocks;
  bid /= a.q_blocks;
  const int g = bid % a.Hkv;
  const int rq = bid / a.Hkv;  // request slot in launch order
  // Decoder batches of ragged prompts: the blocks go out in launch order, so the
  // requests are taken longest prompt first (slot rq serves the request of rank
  // rq, ties to the lower index) and the last blocks to start are short ones.
  int* b_slot = reinterpret_cast<int*>(tmem_slot + 2);
  const bool by_len = !a.causal && !a.mode && a.prompt_len && a.B > 1 && a.B <= ORDER_MAX_B;
  if (by_len && (int)threadIdx.x < a.B) {
    const int i = threadIdx.x;
    const int li = a.prompt_len[i];
    int rank = 0;
    for (int j = 0; j < a.B; ++j) {
      const int lj = a.prompt_len[j];
      rank += (lj > li || (lj == li && j < i)) ? 1 : 0;
    }
    if (rank == rq) *b_slot = i;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    mbar_init(q_bar, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull_bar[i], 1);
      // the softmax threads of both CTAs arrive on the even CTA's barrier
      mbar_init(&pready_bar[i], (PAIR ? 2 : 1) * SOFT_WARPS);   // one arrival per softmax warp
    }
    mbar_init(pv_bar, 1);
    mbar_init(drain_bar, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&pair_bar[i], 2);   // the two warps of a lane quarter
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == MMA_WARP) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, TMEM_COLS);
      tmem_relinquish();
    }
  }
  if (warp == PRODUCER_WARP && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmKe);
    prefetch_tmap(&tmVe);
    prefetch_tmap(&tmKc);
    prefetch_tmap(&tmVc);
  }
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int b = by_len ? *b_slot : rq;
  const Tiles T = tiles_of(a, b, qb, split);
  const int n = T.t_end - T.t_begin;
  const int npos_cta = BM / a.G;                 // canvas positions of one CTA's rows
  const int row_off = (int)rank * npos_cta;     // this CTA's first position in the tile
  // barrier addresses the loads complete on: the even CTA's in a pair
  auto bar_of = [&](uint64_t* bar) -> uint32_t {
    return PAIR ? mapa_shared(smem_u32(bar), 0) : smem_u32(bar);
  };

  if (warp == PRODUCER_WARP) {
    // The whole warp produces: lane 0 waits on the ring and arms the barriers;
    // for paged prompts lane i loads page i of a box (up to 16 pages of a
    // 128-key box), so the page indices and the many small boxes go out in parallel.
    constexpr unsigned FULL = 0xffffffffu;
    int slot = 0;
    uint32_t phase = 0, issued = 0, last_phase = 0;
    bool ok = true;
    if (n > 0 && lane == 0) {
      if (!PAIR || rank == 0) mbar_arrive_expect_tx(q_bar, (PAIR ? 2 : 1) * Q_BYTES);
      const uint32_t qb_addr = bar_of(q_bar);
      for (int c = 0; c < HD / 64; ++c) {
        if constexpr (PAIR)
          tma_load_3d_pair(sQ + c * BOX, &tmQ, qb_addr, c * 64, g * a.G,
                           b * a.C + T.p0 + row_off);
        else
          tma_load_3d(sQ + c * BOX, &tmQ, q_bar, c * 64, g * a.G, b * a.C + T.p0);
      }
    }
    const int ps = a.page_table ? a.page_size : BN;
    // key rows of one box and this CTA's first key of a tile, per stream
    constexpr int K_ROWS = PAIR ? BN / 2 : BN;
    const int k_off = PAIR ? (int)rank * (BN / 2) : 0;
    // this lane's page of a prompt box of tile t (keys past the prompt read its
    // last page, a bad entry reads page 0: both are masked).  The page indices of a
    // tile are read from the table one tile ahead of its loads, so the table's
    // latency overlaps the waits on the ring instead of delaying the copies.
    auto page_idx = [&](int t, int koff, int rows) -> int {
      int v = 0;
      if (a.page_table && t < T.nbp && lane < rows / ps) {
        const int k = min(t * BN + koff + lane * ps, T.P - 1);
        v = a.page_table[(long long)b * a.pages_per_req + k / ps];
        if (v < 0 || v >= a.n_pages) v = 0;
      }
      return v;
    };
    // one ring slot of tile t: K unit u (PAIR: four boxes of 64 head columns x 64
    // keys; else two boxes of 64 head columns x 128 keys) or V unit u (two boxes
    // of 64 output columns x 128 keys); pg = this lane's page of the tile's box
    auto load_unit = [&](int t, bool is_v, int u, int pg) -> bool {
      int w_ok = 1;
      if (lane == 0) w_ok = mbar_wait(&empty_bar[slot], phase ^ 1u, abort_flag, a.status);
      if (!__shfl_sync(FULL, w_ok, 0)) return false;
      uint8_t* dst = ring + slot * UNIT;
      if (lane == 0 && (!PAIR || rank == 0))
        mbar_arrive_expect_tx(&full_bar[slot], (PAIR ? 2 : 1) * UNIT);
      __syncwarp();
      const uint32_t fb = bar_of(&full_bar[slot]);
      const int key0 = T.key0(t);
      const bool prompt = t < T.nbp;
      const bool paged = prompt && a.page_table;
      const CUtensorMap* m = prompt ? (is_v ? &tmVe : &tmKe) : (is_v ? &tmVc : &tmKc);
      const int rows = is_v ? BN : K_ROWS;       // key rows of one box
      const int koff = is_v ? 0 : k_off;         // this CTA's first key of the tile
      const int nbox = (PAIR && !is_v) ? 4 : 2;
      const int box_bytes = rows * 128;
      auto col_of = [&](int h) -> int {
        return PAIR ? (is_v ? dh * DH + (int)rank * 128 + h * 64 : u * 256 + h * 64)
                    : (is_v ? dh * DH : 0) + u * 128 + h * 64;
      };
      if (paged) {
        // one copy per (box, page), all from one instruction: lane l takes page
        // l % np of box l / np (np x nbox <= 32 for pages of 8 keys or more)
        const int np = rows / ps;
        const int pgl = __shfl_sync(FULL, pg, lane % np);
        if (lane < np * nbox) {
          const int h = lane / np;
          uint8_t* d = dst + h * box_bytes + (lane % np) * ps * 128;
          if constexpr (PAIR)
            tma_load_3d_pair(d, m, fb, col_of(h), g, pgl * ps);
          else
            tma_load_3d(d, m, &full_bar[slot], col_of(h), g, pgl * ps);
        }
      } else if (lane == 0) {
        const int row = (prompt ? b * a.Pmax : b * a.C) + key0 + koff;
        for (int h = 0; h < nbox; ++h) {
          if constexpr (PAIR)
            tma_load_3d_pair(dst + h * box_bytes, m, fb, col_of(h), g, row);
          else
            tma_load_3d(dst + h * box_bytes, m, &full_bar[slot], col_of(h), g, row);
        }
      }
      issued |= 1u << slot;
      last_phase = (last_phase & ~(1u << slot)) | (phase << slot);
      if (++slot == NSLOT) {
        slot = 0;
        phase ^= 1u;
      }
      return true;
    };
    // the MMA warp consumes K(t0), then K(t+1) before V(t) for every tile t;
    // pk1 / pv hold the pages of the next K and V loads, read one tile early
    int pk1 = 0, pv = 0;
    if (n > 0) {
      const int pk0 = page_idx(T.t_begin, k_off, K_ROWS);
      pv = page_idx(T.t_begin, 0, BN);
      if (n > 1) pk1 = page_idx(T.t_begin + 1, k_off, K_ROWS);
      for (int u = 0; u < KU && ok; ++u) ok = load_unit(T.t_begin, false, u, pk0);
    }
    for (int j = 0; j < n && ok; ++j) {
      const int t = T.t_begin + j;
      const int pk2 = j + 2 < n ? page_idx(t + 2, k_off, K_ROWS) : 0;
      const int pv1 = j + 1 < n ? page_idx(t + 1, 0, BN) : 0;
      if (j + 1 < n)
        for (int u = 0; u < KU && ok; ++u) ok = load_unit(t + 1, false, u, pk1);
      for (int u = 0; u < VU && ok; ++u) ok = load_unit(t, true, u, pv);
      pk1 = pk2;
      pv = pv1;
    }
    if (!ok && lane == 0 && (!PAIR || rank == 0)) {
      // the loads of both CTAs complete on the even CTA's barriers
      if (n > 0) mbar_wait_drain(q_bar, 0);
      for (int s = 0; s < NSLOT; ++s)
        if (issued & (1u << s)) mbar_wait_drain(&full_bar[s], (last_phase >> s) & 1u);
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0 && (!PAIR || rank == 0)) {
      int slot = 0;
      uint32_t phase = 0;
      bool ok = n > 0 && mbar_wait(q_bar, 0, abort_flag, a.status);
      tc_fence_after();
      const uint32_t q_addr = smem_u32(sQ);
      auto qk = [&](int j) -> bool {
        const uint32_t d_tmem = tmem_base + S_COL + (j & 1) * BN;
        for (int u = 0; u < KU; ++u) {
          if (!mbar_wait(&full_bar[slot], phase, abort_flag, a.status)) return false;
          tc_fence_after();
          const uint32_t base = smem_u32(ring + slot * UNIT);
          if constexpr (PAIR) {
            // 256 head columns per unit: four boxes of 64 keys x 64 columns
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
              const int h = kk >> 2, k16 = kk & 3;
              const uint64_t ad = sw128_kmajor_desc(q_addr + (4 * u + h) * BOX + k16 * 32);
              const uint64_t bd = sw128_kmajor_desc(base + h * (BOX / 2) + k16 * 32);
              tc_mma_f16_pair(d_tmem, ad, bd, IDESC_QK_PAIR, (u | kk) ? 1u : 0u);
            }
            tc_commit_pair(&empty_bar[slot], 0x3);
          } else {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const int h = kk >> 2, k16 = kk & 3;
              const uint64_t ad = sw128_kmajor_desc(q_addr + (2 * u + h) * BOX + k16 * 32);
              const uint64_t bd = sw128_kmajor_desc(base + h * BOX + k16 * 32);
              tc_mma_f16(d_tmem, ad, bd, IDESC_QK, (u | kk) ? 1u : 0u);
            }
            tc_commit(&empty_bar[slot]);
          }
          if (++slot == NSLOT) {
            slot = 0;
            phase ^= 1u;
          }
        }
        if constexpr (PAIR)
          tc_commit_pair(&sfull_bar[j & 1], 0x3);
        else
          tc_commit(&sfull_bar[j & 1]);
        return true;
      };
      auto pv = [&](int j) -> bool {
        if (!mbar_wait(&pready_bar[j & 1], (j >> 1) & 1u, abort_flag, a.status)) return false;
        tc_fence_after();
        const uint32_t p_tmem = tmem_base + S_COL + (j & 1) * BN;
        for (int u = 0; u < VU; ++u) {
          if (!mbar_wait(&full_bar[slot], phase, abort_flag, a.status)) return false;
          tc_fence_after();
          const uint32_t base = smem_u32(ring + slot * UNIT);
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks) {
            // V is MN-major: 64-column groups BOX bytes apart, 8-key atoms 1 KB apart
            const uint64_t bd = sw128_mnmajor_desc(base + ks * 2048, BOX, 1024);
            // P of keys [64 h, 64 h + 64) sits in columns [64 h, 64 h + 32)
            const uint32_t p_col = ks * 8 + (ks >= 4 ? 32 : 0);
            if constexpr (PAIR)
              tc_mma_f16_ts_pair(tmem_base + O_COL, p_tmem + p_col, bd, IDESC_PV_PAIR,
                                 (j | ks) ? 1u : 0u);
            else
              tc_mma_f16_ts(tmem_base + O_COL + u * 128, p_tmem + p_col, bd, IDESC_PV,
                            (j | ks) ? 1u : 0u);
          }
          if constexpr (PAIR)
            tc_commit_pair(&empty_bar[slot], 0x3);
          else
            tc_commit(&empty_bar[slot]);
          if (++slot == NSLOT) {
            slot = 0;
            phase ^= 1u;
          }
        }
        if constexpr (PAIR)
          tc_commit_pair(pv_bar, 0x3);
        else
          tc_commit(pv_bar);
        return true;
      };
      if (ok) ok = qk(0);
      for (int j = 0; j < n && ok; ++j) {
        if (j + 1 < n) ok = qk(j + 1);
        if (ok) ok = pv(j);
      }
      if constexpr (PAIR)
        tc_commit_pair(drain_bar, 0x1);
      else
        tc_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0);
    }
  } else {
    softmax_and_store<PAIR>(a, T, n, b, g, dh, split, warp, lane, tmem_base, sfull_bar,
                            pready_bar, pv_bar, pair_bar, abort_flag, xch, row_off,
                            bar_of(&pready_bar[0]), bar_of(&pready_bar[1]), xmax);
  }

  __syncwarp();
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
  if (warp == MMA_WARP) {
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

__global__ void __launch_bounds__(THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmKe,
                   const __grid_constant__ CUtensorMap tmVe,
                   const __grid_constant__ CUtensorMap tmKc,
                   const __grid_constant__ CUtensorMap tmVc, TcArgs a) {
  attn_body<false>(tmQ, tmKe, tmVe, tmKc, tmVc, a);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmKe,
                     const __grid_constant__ CUtensorMap tmVe,
                     const __grid_constant__ CUtensorMap tmKc,
                     const __grid_constant__ CUtensorMap tmVc, TcArgs a) {
  attn_body<true>(tmQ, tmKe, tmVe, tmKc, tmVc, a);
}

// Splits of the key range: enough CTAs to fill the SMs; for long key ranges a
// multiple of the SM count, as long as every split keeps at least 16 tiles.
// pair: CTA pairs over 256-row tiles (two CTAs per tile).  With a share of the
// SMs (sms < the device's), the splits fill the share while no CTA gets more
// than SHARE_MAX_TILES key tiles (about 100 us); beyond that the CTAs that do
// not fit beside the other work run after it, where shorter ones finish sooner,
// so the key range is split for the whole device instead.
constexpr int SHARE_MAX_TILES = 40;
int tc_splits(int B, int C, int Hq, int Hkv, int Pmax, int W, bool pair, int sms) {
  const int G = Hq / Hkv;
  const int npos = (pair ? 2 : 1) * (BM / G);      // canvas positions of one tile
  const int q_blocks = (C + npos - 1) / npos;
  const int base = B * Hkv * q_blocks * 2 * (pair ? 2 : 1);
  const int keys_c = std::min(C, npos + 2 * W);
  const int nb = std::max(1, (Pmax + BN - 1) / BN + (keys_c + BN - 1) / BN);
  const int all = dgi::num_sms();
  if (sms < all && (nb + std::max(1, sms / base) - 1) / std::max(1, sms / base) > SHARE_MAX_TILES)
    sms = all;
  int s = std::max(1, sms / base);
  for (int c = s + 1; c <= nb / 16; ++c)
    if ((long long)base * c % sms == 0) {
      s = c;
      break;
    }
  return std::min(s, nb);
}

}  // namespace

namespace dgi {

bool attn_tc_supported(const AttnArgs& x) {
  if (x.d != HD || x.Hkv < 1 || x.Hq % x.Hkv) return false;
  const int G = x.Hq / x.Hkv;
  if (BM % G) return false;
  if (x.page_table && (x.page_size < 8 || x.page_size > BN || BN % x.page_size ||
                       x.page_size % 8))
    return false;
  return true;
}

// The CTA-pair kernel loads half-tiles of 64 keys: pages must divide 64.
bool attn_pair_ok(const AttnArgs& x) {
  return attn_tc_supported(x) && (!x.page_table || (BN / 2) % x.page_size == 0);
}

size_t attn_tc_ws_bytes(int B, int C, int Pmax, int Hq, int Hkv, int W, int sms) {
  // sized for either kernel (the pair kernel is chosen per call from the page size)
  const int w = std::min(W, C);
  const int n = plan_sms(sms);
  const int s = std::max(tc_splits(B, C, Hq, Hkv, Pmax, w, false, n),
                         tc_splits(B, C, Hq, Hkv, Pmax, w, true, n));
  if (s == 1) return 256;
  return align_up((size_t)s * B * C * Hq * HD * 4 + (size_t)s * B * Hq * C * 8, 256);
}

cudaError_t attn_decode_tc(const AttnArgs& x, void* ws, cudaStream_t st) {
  TcArgs a{};
  a.B = x.B;
  a.C = x.C;
  a.Pmax = x.Pmax;
  a.Hq = x.Hq;
  a.Hkv = x.Hkv;
  a.W = std::min(x.W, x.C);
  a.G = x.Hq / x.Hkv;
  const bool pair = attn_pair_ok(x);
  a.npos = (pair ? 2 : 1) * (BM / a.G);   // canvas positions of one tile
  a.q_blocks = (x.C + a.npos - 1) / a.npos;
  a.splits = tc_splits(x.B, x.C, x.Hq, x.Hkv, x.Pmax, a.W, pair, plan_sms(x.sms));
  a.causal = x.causal;
  a.seq_len = x.seq_len;
  a.mode = x.mode;
  a.rows_len = x.rows_len;
  a.page_table = x.page_table;
  a.pages_per_req = x.pages_per_req;
  a.n_pages = x.n_pages;
  a.page_size = x.page_size;
  a.prompt_len = x.prompt_len;
  a.out = reinterpret_cast<__nv_bfloat16*>(x.out);
  a.lse = x.lse;
  a.ws_o = static_cast<float*>(ws);
  a.ws_ml = a.ws_o + (size_t)a.splits * x.B * x.C * x.Hq * HD;
  a.status = status_ptr();
  const uint64_t row = HD * 2;
  CUtensorMap tq, tke, tve, tkc, tvc;
  {
    const uint64_t dims[3] = {HD, (uint64_t)x.Hq, (uint64_t)x.B * x.C};
    const uint64_t str[2] = {row, row * x.Hq};
    // one CTA's rows: 128 / G positions x G heads
    const uint32_t box[3] = {64, (uint32_t)a.G, (uint32_t)(BM / a.G)};
    if (!make_tmap_bf16_3d(&tq, x.q, dims, str, box)) return cudaErrorInvalidValue;
  }
  // K boxes: a pair CTA loads half of a tile's keys
  const uint32_t k_rows = pair ? BN / 2 : BN;
  {
    const uint64_t dims[3] = {HD, (uint64_t)x.Hkv, (uint64_t)x.B * x.C};
    const uint64_t str[2] = {row, row * x.Hkv};
    const uint32_t kbox[3] = {64, 1, k_rows};
    const uint32_t vbox[3] = {64, 1, BN};
    if (!make_tmap_bf16_3d(&tkc, x.kc, dims, str, kbox)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16_3d(&tvc, x.vc, dims, str, vbox)) return cudaErrorInvalidValue;
  }
  if (x.Pmax > 0) {
    const bool paged = x.page_table != nullptr;
    const uint64_t rows = paged ? (uint64_t)x.n_pages * x.page_size : (uint64_t)x.B * x.Pmax;
    const uint64_t dims[3] = {HD, (uint64_t)x.Hkv, rows};
    const uint64_t str[2] = {row, row * x.Hkv};
    const uint32_t kbox[3] = {64, 1, paged ? (uint32_t)x.page_size : k_rows};
    const uint32_t vbox[3] = {64, 1, paged ? (uint32_t)x.page_size : (uint32_t)BN};
    if (!make_tmap_bf16_3d(&tke, x.kenc, dims, str, kbox)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16_3d(&tve, x.venc, dims, str, vbox)) return cudaErrorInvalidValue;
  } else {
    tke = tkc;  // no prompt tiles: never read
    tve = tvc;
  }
  static bool attr = false, attr_pair = false;
  bool& done = pair ? attr_pair : attr;
  if (!done) {
    cudaError_t e = pair ? cudaFuncSetAttribute(attn_pair_kernel,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                SMEM_BYTES)
                         : cudaFuncSetAttribute(attn_tc_kernel,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                SMEM_BYTES);
    if (e != cudaSuccess) return e;
    done = true;
  }
  const int grid = (pair ? 2 : 1) * a.splits * 2 * a.q_blocks * x.Hkv * x.B;
  if (pair)
    attn_pair_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(tq, tke, tve, tkc, tvc, a);
  else
    attn_tc_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(tq, tke, tve, tkc, tvc, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1) return e;
  return attn_combine(x.B, x.C, x.Hq, HD, a.splits, a.ws_o, a.ws_ml, x.out, x.lse, st,
                      x.rows_len ? x.rows_len : (x.causal ? x.seq_len : nullptr));
}

// Paged KV write of an encoder prefill: one warp per (request, key row, KV head)
// copies d bf16 values of K and of V with 16-byte loads and stores.
namespace {
__global__ void kv_page_write_kernel(const uint4* k, const uint4* v, int B, int P, int Hkv,
                                     int n16, const int32_t* seq_len, const int32_t* page_table,
                                     int pages_per_req, int n_pages, int page_size, uint4* pool_k,
                                     uint4* pool_v, int* status) {
  const long long item = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long n_items = (long long)B * P * Hkv;
  if (item >= n_items) return;
  const int h = (int)(item % Hkv);
  const int p = (int)((item / Hkv) % P);
  const int b = (int)(item / ((long long)Hkv * P));
  if (p >= min(max(seq_len[b], 0), P)) return;
  const int pg = page_table[(long long)b * pages_per_req + p / page_size];
  if (pg < 0 || pg >= n_pages) {
    if (lane == 0) atomicOr(status, 2 /* DG_DEV_BAD_PAGE */);
    return;
  }
  const long long src = item * n16;
  const long long dst = (((long long)pg * page_size + p % page_size) * Hkv + h) * n16;
  for (int i = lane; i < n16; i += 32) {
    pool_k[dst + i] = k[src + i];
    pool_v[dst + i] = v[src + i];
  }
}
}  // namespace

cudaError_t kv_page_write(const uint16_t* k, const uint16_t* v, int B, int P, int Hkv, int d,
                          const int32_t* seq_len, const int32_t* page_table, int pages_per_req,
                          int n_pages, int page_size, uint16_t* pool_k, uint16_t* pool_v,
                          cudaStream_t st) {
  const long long items = (long long)B * P * Hkv;
  if (items == 0) return cudaSuccess;
  const int grid = (int)((items + 7) / 8);
  kv_page_write_kernel<<<grid, 256, 0, st>>>(
      reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v), B, P, Hkv, d / 8,
      seq_len, page_table, pages_per_req, n_pages, page_size, reinterpret_cast<uint4*>(pool_k),
      reinterpret_cast<uint4*>(pool_v), status_ptr());
  return cudaGetLastError();
}

}  // namespace dgi
