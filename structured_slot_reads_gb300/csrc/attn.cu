// attn.cu -- decoder-mode attention of the canvas (24-ai.news, "How does
// diffusion text generation differ?"; thakicloud.com, "What is DiffusionGemma").
//
// Every canvas row attends to all prompt keys of its request (encoder KV,
// contiguous or in pages) and to the canvas keys within +-W of its position,
// one joint softmax, scale 1/sqrt(d).  The GQA group's query heads share the
// KV head, so a CTA packs 64 query rows = (64/G canvas positions) x (G heads)
// and streams the union of their keys once.  The key range is split across
// CTAs (split-KV) and the partial (max, sum, O) are merged by a combine kernel.
//
// This file serves the 64-wide heads of the tiny correctness shape: warp-level
// bf16 mma.sync m16n8k16 with fp32 accumulators, operands staged in
// XOR-swizzled shared memory by cp.async.  A 64 x 64 score tile and the whole
// 64 x 64 output fit one CTA's registers here, so this small case has none of
// the tensor-memory pressure that shapes the 512-wide kernel (attn_tc.cu),
// which every 512-wide call runs on.  The split-KV combine below serves both.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "internal.h"

namespace {

constexpr int BMQ = 64;  // query rows per CTA
constexpr int BNK = 64;  // keys per tile
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // src-size 0 writes zeros
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Offset (in bf16 elements) of chunk `c` (8 elements) of row `r` in a tile whose
// rows hold `cpr` chunks, 16-byte chunks XOR-swizzled within groups of 8.
__device__ __forceinline__ int swz(int r, int c, int cpr) {
  return r * cpr * 8 + ((c ^ (r & 7)) * 8);
}

struct Args {
  int B, C, Pmax, Hq, Hkv, W, G, npos, q_blocks, splits;
  const __nv_bfloat16 *q, *kc, *vc, *kenc, *venc;
  const int32_t* page_table;
  int pages_per_req, n_pages, page_size;
  const int32_t* prompt_len;
  __nv_bfloat16* out;
  float* lse;
  float* ws_o;   // [splits][B][C][Hq][d]
  float* ws_ml;  // [splits][B][Hq][C][2]
  int* status;
  const int32_t* seq_len;  // combine: rows at or past seq_len[b] are skipped (null: none)
};

template <int D>
struct AttnCfg {
  static constexpr int DSPLIT = (D >= 256) ? 2 : 1;
  static constexpr int WARPS = 4 * DSPLIT;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int CPR = D / 8;                 // 16-byte chunks per row
  static constexpr int KEYS_W = BNK / DSPLIT;       // score columns per warp
  static constexpr int NF_S = KEYS_W / 8;
  static constexpr int DW = D / DSPLIT;             // output columns per warp
  static constexpr int NF_O = DW / 8;
  static constexpr int TILE_ELEMS = BNK * D;
  static constexpr int SMEM = (BMQ * D + 2 * TILE_ELEMS + BMQ * BNK) * 2 + 4 * DSPLIT * BMQ * 4 +
                              BNK * 4 + 64;
};

template <int D>
__global__ void __launch_bounds__(AttnCfg<D>::THREADS, 1) attn_kernel(Args a) {
  using CF = AttnCfg<D>;
  extern __shared__ __align__(128) uint8_t sm[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(sm);
  __nv_bfloat16* sK = sQ + BMQ * D;
  __nv_bfloat16* sV = sK + CF::TILE_ELEMS;
  __nv_bfloat16* sP = sV + CF::TILE_ELEMS;
  float* red_max = reinterpret_cast<float*>(sP + BMQ * BNK);  // [DSPLIT][BMQ]
  float* red_sum = red_max + CF::DSPLIT * BMQ;                // [DSPLIT][BMQ]
  int* key_kind = reinterpret_cast<int*>(red_sum + CF::DSPLIT * BMQ);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int rg = warp & 3, sp = warp >> 2;
  const int g = lane >> 2, t4 = lane & 3;

  int bid = blockIdx.x;
  const int split = bid % a.splits;
  bid /= a.splits;
  const int qb = bid % a.q_blocks;
  bid /= a.q_blocks;
  const int kvh = bid % a.Hkv;
  const int b = bid / a.Hkv;

  const int p0 = qb * a.npos;
  const int npos = min(a.npos, a.C - p0);
  const int P = min(max(a.prompt_len[b], 0), a.Pmax);
  const int clo = max(0, p0 - a.W);
  const int chi = min(a.C, p0 + npos - 1 + a.W + 1);
  const int L = P + (chi - clo);
  const int ntiles = (L + BNK - 1) / BNK;
  const int t_begin = (int)((long long)split * ntiles / a.splits);
  const int t_end = (int)((long long)(split + 1) * ntiles / a.splits);
  const float sl2 = LOG2E * rsqrtf((float)D);

  // ---- load Q: row r = local position r / G, head r % G ------------------
  for (int i = tid; i < BMQ * CF::CPR; i += CF::THREADS) {
    const int r = i / CF::CPR, c = i % CF::CPR;
    const int pos = p0 + r / a.G;
    const bool ok = (r / a.G) < npos;
    const int h = kvh * a.G + r % a.G;
    const __nv_bfloat16* src = a.q + ((long long)(b * a.C + (ok ? pos : p0)) * a.Hq + h) * D + c * 8;
    cp_async16(sQ + swz(r, c, CF::CPR), src, ok);
  }

  // key source of virtual key k (prompt first, then canvas keys clo..chi-1)
  auto key_ptr = [&](const __nv_bfloat16* enc, const __nv_bfloat16* can, int k,
                     bool& ok) -> const __nv_bfloat16* {
    if (k >= L) {
      ok = false;
      return can;
    }
    if (k < P) {
      if (a.page_table) {
        const int pg = a.page_table[(long long)b * a.pages_per_req + k / a.page_size];
        if (pg < 0 || pg >= a.n_pages) {
          ok = false;
          return can;
        }
        ok = true;
        return enc + (((long long)pg * a.page_size + k % a.page_size) * a.Hkv + kvh) * D;
      }
      ok = true;
      return enc + (((long long)b * a.Pmax + k) * a.Hkv + kvh) * D;
    }
    ok = true;
    return can + (((long long)b * a.C + clo + (k - P)) * a.Hkv + kvh) * D;
  };
  auto load_tile = [&](__nv_bfloat16* dst, const __nv_bfloat16* enc, const __nv_bfloat16* can,
                       int tile) {
    for (int i = tid; i < BNK * CF::CPR; i += CF::THREADS) {
      const int r = i / CF::CPR, c = i % CF::CPR;
      bool ok;
      const __nv_bfloat16* src = key_ptr(enc, can, tile * BNK + r, ok);
      cp_async16(dst + swz(r, c, CF::CPR), ok ? src + c * 8 : can, ok);
    }
  };

  float o[CF::NF_O][4];
#pragma unroll
  for (int i = 0; i < CF::NF_O; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  const int row0 = rg * 16 + g;  // rows row0 and row0 + 8
  const int pos_r0 = p0 + row0 / a.G, pos_r1 = p0 + (row0 + 8) / a.G;

  if (t_begin < t_end) {
    load_tile(sK, a.kenc, a.kc, t_begin);
    cp_async_commit();  // Q + K0
    load_tile(sV, a.venc, a.vc, t_begin);
    cp_async_commit();  // V0
  } else {
    cp_async_commit();
  }

  for (int tile = t_begin; tile < t_end; ++tile) {
    // key kinds for masking: -1 invalid, -2 prompt, >=0 canvas position
    if (tid < BNK) {
      const int k = tile * BNK + tid;
      int kind = -1;
      if (k < L) {
        if (k < P) {
          kind = -2;
          if (a.page_table) {
            const int pg = a.page_table[(long long)b * a.pages_per_req + k / a.page_size];
            if (pg < 0 || pg >= a.n_pages) {
              kind = -1;
              atomicOr(a.status, 2 /* DG_DEV_BAD_PAGE */);
            }
          }
        } else {
          kind = clo + (k - P);
        }
      }
      key_kind[tid] = kind;
    }
    cp_async_wait<1>();
    __syncthreads();

    // ---- S = Q K^T for this warp's 16 rows x KEYS_W keys --------------
    float s[CF::NF_S][4];
#pragma unroll
    for (int i = 0; i < CF::NF_S; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll 4
    for (int kc = 0; kc < D / 16; ++kc) {
      uint32_t af[4];
      {
        const int r = rg * 16 + (lane & 15);
        const int c = kc * 2 + (lane >> 4);
        ldsm_x4(af, sQ + swz(r, c, CF::CPR));
      }
#pragma unroll
      for (int nf = 0; nf < CF::NF_S; nf += 2) {
        uint32_t bf[4];
        const int key = sp * CF::KEYS_W + nf * 8 + (lane & 7) + ((lane >> 4) << 3);
        const int c = kc * 2 + ((lane >> 3) & 1);
        ldsm_x4(bf, sK + swz(key, c, CF::CPR));
        mma_bf16(s[nf], af, bf[0], bf[1]);
        mma_bf16(s[nf + 1], af, bf[2], bf[3]);
      }
    }

    // ---- mask, scale (base 2), row max -------------------------------
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nf = 0; nf < CF::NF_S; ++nf) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = sp * CF::KEYS_W + nf * 8 + 2 * t4 + (e & 1);
        const int kind = key_kind[col];
        const int pr = (e < 2) ? pos_r0 : pos_r1;
        const bool ok = (kind == -2) || (kind >= 0 && abs(pr - kind) <= a.W);
        const float v = ok ? s[nf][e] * sl2 : -INFINITY;
        s[nf][e] = v;
        tmax[e >> 1] = fmaxf(tmax[e >> 1], v);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 1));
      tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 2));
    }
    if (CF::DSPLIT > 1) {
      if (t4 == 0) {
        red_max[sp * BMQ + row0] = tmax[0];
        red_max[sp * BMQ + row0 + 8] = tmax[1];
      }
      __syncthreads();
#pragma unroll
      for (int q = 0; q < CF::DSPLIT; ++q) {
        tmax[0] = fmaxf(tmax[0], red_max[q * BMQ + row0]);
        tmax[1] = fmaxf(tmax[1], red_max[q * BMQ + row0 + 8]);
      }
    }
    float alpha[2], mref[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float mn = fmaxf(m_run[h], tmax[h]);
      mref[h] = (mn == -INFINITY) ? 0.f : mn;
      alpha[h] = ex2(m_run[h] - mref[h]);
      m_run[h] = mn;
      l_run[h] *= alpha[h];
    }
    // ---- P = 2^(s - m) into shared memory (bf16) -----------------------
#pragma unroll
    for (int nf = 0; nf < CF::NF_S; ++nf) {
      const float p0v = ex2(s[nf][0] - mref[0]);
      const float p1v = ex2(s[nf][1] - mref[0]);
      const float p2v = ex2(s[nf][2] - mref[1]);
      const float p3v = ex2(s[nf][3] - mref[1]);
      l_run[0] += p0v + p1v;
      l_run[1] += p2v + p3v;
      const int col = sp * CF::KEYS_W + nf * 8 + 2 * t4;
      const int chunk = col >> 3, within = col & 7;
      *reinterpret_cast<__nv_bfloat162*>(sP + swz(row0, chunk, BNK / 8) + within) =
          __floats2bfloat162_rn(p0v, p1v);
      *reinterpret_cast<__nv_bfloat162*>(sP + swz(row0 + 8, chunk, BNK / 8) + within) =
          __floats2bfloat162_rn(p2v, p3v);
    }
#pragma unroll
    for (int i = 0; i < CF::NF_O; ++i) {
      o[i][0] *= alpha[0];
      o[i][1] *= alpha[0];
      o[i][2] *= alpha[1];
      o[i][3] *= alpha[1];
    }
    __syncthreads();  // P visible; every warp is done with K
    if (tile + 1 < t_end) load_tile(sK, a.kenc, a.kc, tile + 1);
    cp_async_commit();
    cp_async_wait<1>();  // V(tile)
    __syncthreads();

    // ---- O += P V over this warp's DW output columns ---------------------
#pragma unroll
    for (int kc = 0; kc < BNK / 16; ++kc) {
      uint32_t af[4];
      {
        const int r = rg * 16 + (lane & 15);
        const int c = kc * 2 + (lane >> 4);
        ldsm_x4(af, sP + swz(r, c, BNK / 8));
      }
#pragma unroll
      for (int nf = 0; nf < CF::NF_O; nf += 2) {
        uint32_t bf[4];
        const int key = kc * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int c = (sp * CF::DW + nf * 8) / 8 + (lane >> 4);
        ldsm_x4_t(bf, sV + swz(key, c, CF::CPR));
        mma_bf16(o[nf], af, bf[0], bf[1]);
        mma_bf16(o[nf + 1], af, bf[2], bf[3]);
      }
    }
    __syncthreads();  // done with V and P
    if (tile + 1 < t_end) load_tile(sV, a.venc, a.vc, tile + 1);
    cp_async_commit();
  }
  cp_async_wait<0>();

  // ---- row sums over the quad and the key-split warps -------------------
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
  if (CF::DSPLIT > 1) {
    __syncthreads();
    if (t4 == 0) {
      red_sum[sp * BMQ + row0] = l_run[0];
      red_sum[sp * BMQ + row0 + 8] = l_run[1];
    }
    __syncthreads();
    l_run[0] = l_run[1] = 0.f;
#pragma unroll
    for (int q = 0; q < CF::DSPLIT; ++q) {
      l_run[0] += red_sum[q * BMQ + row0];
      l_run[1] += red_sum[q * BMQ + row0 + 8];
    }
  }

  // ---- write: final (one split) or partial ------------------------------
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = row0 + h * 8;
    const int lp = r / a.G;
    if (lp >= npos) continue;
    const int pos = p0 + lp;
    const int head = kvh * a.G + r % a.G;
    const long long orow = ((long long)(b * a.C + pos) * a.Hq + head) * D;
    if (a.splits == 1) {
      const float inv = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f;
#pragma unroll
      for (int nf = 0; nf < CF::NF_O; ++nf) {
        const int col = sp * CF::DW + nf * 8 + 2 * t4;
        *reinterpret_cast<__nv_bfloat162*>(a.out + orow + col) =
            __floats2bfloat162_rn(o[nf][2 * h] * inv, o[nf][2 * h + 1] * inv);
      }
      if (sp == 0 && t4 == 0)
        a.lse[((long long)b * a.Hq + head) * a.C + pos] =
            (m_run[h] + log2f(l_run[h])) * LN2;
    } else {
      float* wo = a.ws_o + (long long)split * a.B * a.C * a.Hq * D + orow;
#pragma unroll
      for (int nf = 0; nf < CF::NF_O; ++nf) {
        const int col = sp * CF::DW + nf * 8 + 2 * t4;
        *reinterpret_cast<float2*>(wo + col) = make_float2(o[nf][2 * h], o[nf][2 * h + 1]);
      }
      if (sp == 0 && t4 == 0) {
        float* ml = a.ws_ml + (((long long)split * a.B + b) * a.Hq + head) * a.C * 2 + pos * 2;
        ml[0] = m_run[h];
        ml[1] = l_run[h];
      }
    }
  }
}

// Merge split partials: one thread per (b, pos, head) row and 4 output columns.
// Each thread first takes the row's reference over the splits (the (m, l) pairs
// are shared by the row's threads through L1), then sums the partial columns;
// a split that saw no key (m = -inf, partial never written) is dropped by a
// select.
template <int D>
__global__ void attn_combine_kernel(Args a) {
  constexpr int TPR = D / 4;  // threads per row
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = tid / TPR;
  const int c4 = (int)(tid % TPR);
  const long long nrows = (long long)a.B * a.C * a.Hq;
  if (row >= nrows) return;
  const int head = (int)(row % a.Hq);
  const int pos = (int)((row / a.Hq) % a.C);
  const int b = (int)(row / ((long long)a.Hq * a.C));
  if (a.seq_len && pos >= a.seq_len[b]) return;
  const long long split_o = (long long)a.B * a.C * a.Hq * D;
  const long long ml_split = (long long)a.B * a.Hq * a.C * 2;
  const float* ml0 = a.ws_ml + ((long long)b * a.Hq + head) * a.C * 2 + pos * 2;
  float mt = -INFINITY;
  for (int s = 0; s < a.splits; ++s) mt = fmaxf(mt, ml0[s * ml_split]);
  float lt = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* wo = reinterpret_cast<const float4*>(a.ws_o + row * D) + c4;
#pragma unroll 4
  for (int s = 0; s < a.splits; ++s) {
    const float m = ml0[s * ml_split], l = ml0[s * ml_split + 1];
    const bool live = m != -INFINITY;
    const float f = live ? exp2f(m - mt) : 0.f;
    lt += live ? l * f : 0.f;
    const float4 v = wo[s * (split_o / 4)];
    acc.x += live ? v.x * f : 0.f;
    acc.y += live ? v.y * f : 0.f;
    acc.z += live ? v.z * f : 0.f;
    acc.w += live ? v.w * f : 0.f;
  }
  const float inv = lt > 0.f ? 1.f / lt : 0.f;
  __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(a.out + row * D) + 2 * c4;
  o[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  o[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  if (c4 == 0) a.lse[((long long)b * a.Hq + head) * a.C + pos] = (mt + log2f(lt)) * LN2;
}

int pick_splits(int B, int C, int Hq, int Hkv, int Pmax, int W, int sms) {
  const int G = Hq / Hkv;
  const int npos = BMQ / G;
  const int q_blocks = (C + npos - 1) / npos;
  const int base = q_blocks * Hkv * B;
  const int keys = Pmax + std::min(C, npos + 2 * W);
  const int tiles = std::max(1, (keys + BNK - 1) / BNK);
  int s = std::max(1, sms / std::max(1, base));
  return std::min(s, tiles);
}

template <int D>
cudaError_t run(const dgi::AttnArgs& x, void* ws, cudaStream_t st) {
  using CF = AttnCfg<D>;
  Args a{};
  a.B = x.B;
  a.C = x.C;
  a.Pmax = x.Pmax;
  a.Hq = x.Hq;
  a.Hkv = x.Hkv;
  a.W = std::min(x.W, x.C);
  a.G = x.Hq / x.Hkv;
  a.npos = BMQ / a.G;
  a.q_blocks = (x.C + a.npos - 1) / a.npos;
  a.splits = pick_splits(x.B, x.C, x.Hq, x.Hkv, x.Pmax, a.W, dgi::plan_sms(x.sms));
  a.q = reinterpret_cast<const __nv_bfloat16*>(x.q);
  a.kc = reinterpret_cast<const __nv_bfloat16*>(x.kc);
  a.vc = reinterpret_cast<const __nv_bfloat16*>(x.vc);
  a.kenc = reinterpret_cast<const __nv_bfloat16*>(x.kenc);
  a.venc = reinterpret_cast<const __nv_bfloat16*>(x.venc);
  a.page_table = x.page_table;
  a.pages_per_req = x.pages_per_req;
  a.n_pages = x.n_pages;
  a.page_size = x.page_size;
  a.prompt_len = x.prompt_len;
  a.out = reinterpret_cast<__nv_bfloat16*>(x.out);
  a.lse = x.lse;
  a.ws_o = static_cast<float*>(ws);
  a.ws_ml = a.ws_o + (size_t)a.splits * x.B * x.C * x.Hq * D;
  a.status = dgi::status_ptr();
  static bool attr = false;
  if (!attr) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int grid = a.splits * a.q_blocks * x.Hkv * x.B;
  attn_kernel<D><<<grid, CF::THREADS, CF::SMEM, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1) return e;
  const long long threads = (long long)x.B * x.C * x.Hq * (D / 4);
  attn_combine_kernel<D><<<(int)((threads + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

namespace dgi {

size_t attn_ws_bytes(int B, int C, int Pmax, int Hq, int Hkv, int d, int W, int sms) {
  // d = 512 runs on the tensor-core kernel (attn_tc.cu)
  if (d == 512) return attn_tc_ws_bytes(B, C, Pmax, Hq, Hkv, W, sms);
  const int s = pick_splits(B, C, Hq, Hkv, Pmax, std::min(W, C), plan_sms(sms));
  if (s == 1) return 256;
  return align_up((size_t)s * B * C * Hq * d * 4 + (size_t)s * B * Hq * C * 8, 256);
}

cudaError_t attn_decode(const AttnArgs& a, void* ws, cudaStream_t st) {
  if (a.d == 64) return run<64>(a, ws, st);
  if (a.d == 512 && attn_tc_supported(a)) return attn_decode_tc(a, ws, st);
  return cudaErrorInvalidValue;
}

cudaError_t attn_combine(int B, int C, int Hq, int d, int splits, float* ws_o, float* ws_ml,
                         uint16_t* out, float* lse, cudaStream_t st, const int32_t* seq_len) {
  Args a{};
  a.seq_len = seq_len;
  a.B = B;
  a.C = C;
  a.Hq = Hq;
  a.splits = splits;
  a.ws_o = ws_o;
  a.ws_ml = ws_ml;
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  const long long rows = (long long)B * C * Hq;
  if (d == 64)
    attn_combine_kernel<64><<<(int)((rows * 16 + 255) / 256), 256, 0, st>>>(a);
  else if (d == 512)
    attn_combine_kernel<512><<<(int)((rows * 128 + 255) / 256), 256, 0, st>>>(a);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace dgi
