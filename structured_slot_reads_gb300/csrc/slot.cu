// slot.cu -- noise draws, the slot read, the entropy commit and the canvas update.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "internal.h"

namespace {

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC'11, section 3.2 and Table 2): per round the counter (x0..x3) becomes
// (hi(M1 x2) ^ x1 ^ k0, lo(M1 x2), hi(M0 x0) ^ x3 ^ k1, lo(M0 x0)); the key
// advances by (W0, W1) between rounds.
// ---------------------------------------------------------------------------
struct U4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ U4 philox10(U4 c, uint32_t k0, uint32_t k1) {
  constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
  constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint32_t hi0 = __umulhi(kM0, c.x), lo0 = kM0 * c.x;
    const uint32_t hi1 = __umulhi(kM1, c.z), lo1 = kM1 * c.z;
    c = U4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
  }
  return c;
}

__global__ void philox_fill_kernel(uint64_t seed, const uint4* ctr, int n, uint4* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint4 c = ctr[i];
  const U4 r = philox10(U4{c.x, c.y, c.z, c.w}, (uint32_t)seed, (uint32_t)(seed >> 32));
  out[i] = make_uint4(r.x, r.y, r.z, r.w);
}

// ---------------------------------------------------------------------------
// a0: one CTA per (slot, draw) row: token n from Philox, row = bf16(h + E[n]).
// ---------------------------------------------------------------------------
__global__ void slot_noise_kernel(const __nv_bfloat16* h, int M, const __nv_bfloat16* e, int V,
                                  int vbits, int D, const float* inv_t, const int32_t* slot_row,
                                  const int32_t* slot_req, int S, int R, uint64_t seed, int step,
                                  __nv_bfloat16* rows_out, float* inv_t_out, int32_t* tok_out,
                                  int* status) {
  const int s = blockIdx.x / R, r = blockIdx.x % R;
  const int row = slot_row[s];
  const bool row_ok = row >= 0 && row < M;
  const U4 c = philox10(U4{(uint32_t)slot_req[s], (uint32_t)step, (uint32_t)r, (uint32_t)s},
                        (uint32_t)seed, (uint32_t)(seed >> 32));
  const int tok = (int)(c.x >> (32 - vbits));
  if (threadIdx.x == 0) {
    if (tok_out) tok_out[s * R + r] = tok;
    inv_t_out[s * R + r] = row_ok ? inv_t[row] : 1.f;
    if (!row_ok) atomicOr(status, 8 /* DG_DEV_BAD_INDEX */);
  }
  // 16-byte chunks, each thread's loads issued before its adds (the E row is a
  // random row of a 1.5 GB table: one memory latency per row, not one per chunk)
  const uint4* hs = reinterpret_cast<const uint4*>(h + (long long)(row_ok ? row : 0) * D);
  const uint4* es = reinterpret_cast<const uint4*>(e + (long long)tok * D);
  uint4* dst = reinterpret_cast<uint4*>(rows_out + (long long)blockIdx.x * D);
  const int n16 = D / 8;
  constexpr int U = 4;
  for (int base = 0; base < n16; base += U * blockDim.x) {
    uint4 a[U], b[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * blockDim.x + threadIdx.x;
      a[u] = i < n16 ? hs[i] : make_uint4(0, 0, 0, 0);
      b[u] = i < n16 ? __ldg(es + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * blockDim.x + threadIdx.x;
      if (i >= n16) continue;
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[u]);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b[u]);
      uint4 o;
      __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 x = __bfloat1622float2(a2[q]);
        const float2 y = __bfloat1622float2(b2[q]);
        o2[q] = row_ok ? __floats2bfloat162_rn(x.x + y.x, x.y + y.y) : __floats2bfloat162_rn(0.f, 0.f);
      }
      dst[i] = o;
    }
  }
}

// ---------------------------------------------------------------------------
// a3: one CTA (256 threads) per slot.  Label logits of every draw are fp32 dot
// products (one warp per (draw, label)); then the renormalised distributions,
// the gate on draw 0's entropy, the average and the choice.
// ---------------------------------------------------------------------------
constexpr int MAXL = 26;

// Label logits of every (slot, draw, label): one warp per product, 8 labels per
// CTA, grid (S * R, ceil(L / 8)).  The fp32 logit z / T goes to lp_draws, which
// the epilogue below then turns into z - lse.
__global__ void slot_dots_kernel(const __nv_bfloat16* rows, const float* inv_t_rows,
                                 const __nv_bfloat16* w, int V, int D, const int32_t* label_ids,
                                 const int32_t* n_labels, int L, int R, float* lp_draws,
                                 int* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x / R, r = blockIdx.x % R;
  const int k = blockIdx.y * 8 + warp;
  const int n = n_labels[s];
  if (n < 0 || n > L || k >= n) return;  // a bad count is flagged by the epilogue
  int id = label_ids[(long long)s * L + k];
  if (id < 0 || id >= V) {
    if (lane == 0) atomicOr(status, 4 /* DG_DEV_BAD_LABEL */);
    id = 0;
  }
  const __nv_bfloat16* xr = rows + (long long)(s * R + r) * D;
  const __nv_bfloat16* yr = w + (long long)id * D;
  float acc = 0.f;
  if ((D % 8) == 0) {
    const uint4* x = reinterpret_cast<const uint4*>(xr);
    const uint4* y = reinterpret_cast<const uint4*>(yr);
    const int n16 = D / 8;
#pragma unroll 4
    for (int i = lane; i < n16; i += 32) {
      const uint4 xa = x[i];
      const uint4 ya = __ldg(y + i);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&xa);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&ya);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 a = __bfloat1622float2(a2[q]);
        const float2 b = __bfloat1622float2(b2[q]);
        acc = fmaf(a.x, b.x, acc);
        acc = fmaf(a.y, b.y, acc);
      }
    }
  } else {
    const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(xr);
    const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(yr);
    for (int i = lane; i < D / 2; i += 32) {
      const float2 a = __bfloat1622float2(x[i]);
      const float2 b = __bfloat1622float2(y[i]);
      acc = fmaf(a.x, b.x, acc);
      acc = fmaf(a.y, b.y, acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) lp_draws[((long long)s * R + r) * L + k] = acc * inv_t_rows[s * R + r];
}

// The slot read from the label logits: one warp per slot, lane holds labels
// lane + 32 i (i < LPL, label tables of stride L <= 32 LPL).
template <int LPL>
__global__ void slot_epilogue_kernel(const float* lse_rows, const int32_t* n_labels, int L, int R,
                                     int samples, float gate, float* q_avg, float* h_slot,
                                     int32_t* chosen, float* lp_draws, uint8_t* resampled,
                                     int32_t* n_reads, int* status) {
  const int s = blockIdx.x;
  const int lane = threadIdx.x & 31;
  int n = n_labels[s];
  // n == 0: a question whose ask_if condition did not fire -- not read
  if (n < 0 || n > L) {
    if (lane == 0) atomicOr(status, 4 /* DG_DEV_BAD_LABEL */);
    n = 0;
  }
  float qsum[LPL], q0[LPL];
#pragma unroll
  for (int i = 0; i < LPL; ++i) qsum[i] = q0[i] = 0.f;
  float h0 = 0.f;
  for (int r = 0; r < R; ++r) {
    float* lp = lp_draws + ((long long)s * R + r) * L;
    float zk[LPL];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < LPL; ++i) {
      const int k = lane + 32 * i;
      zk[i] = k < n ? lp[k] : -INFINITY;
      m = fmaxf(m, zk[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float ek[LPL], tot = 0.f;
#pragma unroll
    for (int i = 0; i < LPL; ++i) {
      ek[i] = (lane + 32 * i < n) ? expf(zk[i] - m) : 0.f;
      tot += ek[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    float hq = 0.f;
    const float lse_r = lse_rows[s * R + r];
#pragma unroll
    for (int i = 0; i < LPL; ++i) {
      const int k = lane + 32 * i;
      const float q = ek[i] / tot;
      if (k < n && q > 0.f) hq -= q * logf(q);
      if (k < L) lp[k] = k < n ? zk[i] - lse_r : 0.f;
      if (r < samples) qsum[i] += q;
      if (r == 0) q0[i] = q;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) hq += __shfl_xor_sync(0xffffffffu, hq, o);
    if (r == 0) h0 = hq;
  }
  const bool fire = samples > 1 && h0 > gate;
  float hs = 0.f, best = -1.f;
  int arg = 0x7fffffff;
#pragma unroll
  for (int i = 0; i < LPL; ++i) {
    const int k = lane + 32 * i;
    const bool kv = k < n;
    const float qk = kv ? (fire ? qsum[i] / (float)samples : q0[i]) : 0.f;
    if (kv && qk > 0.f) hs -= qk * logf(qk);
    if (kv && qk > best) {  // i ascends, so the lowest index wins within the lane
      best = qk;
      arg = k;
    }
    if (k < L) q_avg[(long long)s * L + k] = qk;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) hs += __shfl_xor_sync(0xffffffffu, hs, o);
  // argmax over lanes, lowest index on ties
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float bo = __shfl_xor_sync(0xffffffffu, best, o);
    const int ao = __shfl_xor_sync(0xffffffffu, arg, o);
    if (bo > best || (bo == best && ao < arg)) {
      best = bo;
      arg = ao;
    }
  }
  if (lane == 0) {
    chosen[s] = n > 0 ? arg : -1;
    h_slot[s] = hs;
    resampled[s] = (n > 0 && fire) ? 1 : 0;
    n_reads[s] = n == 0 ? 0 : (fire ? samples : 1);
  }
}

// ---------------------------------------------------------------------------
// a7: ask_if gating (sotaaz.com, "The server accepts at most 26 alternatives per
// question": a question carrying ask_if is read only when the earlier answer
// matches).  Thread per question: fired = chosen1[cond_slot] == cond_value.
// Warp per stage-2 slot: the first fired question that owns the slot copies
// its labels into the stage-2 table; with none, n_labels2 = 0 (not read).
// ---------------------------------------------------------------------------
__global__ void ask_if_kernel(const int32_t* chosen1, int S1, const int32_t* cond_slot,
                              const int32_t* cond_value, const int32_t* q_owner,
                              const int32_t* q_label_ids, const int32_t* q_n_labels, int Q,
                              int S2, int32_t* label_ids2, int32_t* n_labels2, uint8_t* fired,
                              int* status) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  auto fires = [&](int q) -> bool {
    const int cs = cond_slot[q];
    if (cs < 0 || cs >= S1) {
      atomicOr(status, 8 /* DG_DEV_BAD_INDEX */);
      return false;
    }
    return chosen1[cs] == cond_value[q];
  };
  // one thread per question: did it fire
  if (i < Q && fired) fired[i] = fires(i) ? 1 : 0;
  // one warp per stage-2 slot: the lowest-index fired question it owns (each
  // lane stops at its first, the warp takes the minimum), labels copied by lane
  const int slot = i >> 5, lane = threadIdx.x & 31;
  if (slot < S2) {
    int first = 0x7fffffff;
    for (int q = lane; q < Q; q += 32)
      if (q_owner[q] == slot && fires(q)) {
        first = q;
        break;
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
    const int pick = first == 0x7fffffff ? -1 : first;
    const int n = pick >= 0 ? q_n_labels[pick] : 0;
    if (lane == 0) {
      n_labels2[slot] = (n >= 0 && n <= MAXL) ? n : 0;
      if (n < 0 || n > MAXL) atomicOr(status, 4 /* DG_DEV_BAD_LABEL */);
    }
    if (lane < MAXL)
      label_ids2[slot * MAXL + lane] = (pick >= 0 && lane < n) ? q_label_ids[pick * MAXL + lane]
                                                              : -1;
  }
}

// ---------------------------------------------------------------------------
// a4: one CTA per request, one thread per canvas position (C <= 1024).  The
// candidates are put in confidence order by a stable block radix sort of
// (entropy, position): four passes over 8-bit digits of the entropy's
// order-preserving bit pattern, closed positions keyed last; within a pass a
// warp ranks equal digits with __match_any_sync and the per-warp digit counts
// are scanned digit-major, warp-minor, which keeps equal keys in position
// order.  A block scan of the sorted entropies then finds the cut.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_bits(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(1024) commit_kernel(int C, const float* entropy,
                                                     const int32_t* argmax, const uint8_t* cand,
                                                     const float* gamma,
                                                     uint8_t* committed_state,
                                                     int32_t* token_state, uint8_t* commit_out,
                                                     int32_t* tokens, int32_t* n_commit) {
  extern __shared__ uint32_t shu[];
  const int nw = blockDim.x >> 5;
  uint32_t* key_a = shu;                          // [C] keys in the current order
  uint16_t* pos_a = reinterpret_cast<uint16_t*>(key_a + C);      // [C] their positions
  uint32_t* hist = reinterpret_cast<uint32_t*>(pos_a + ((C + 1) & ~1));   // [256][nw]
  __shared__ uint32_t dig_tot[256];
  __shared__ int n_cand, cut;
  __shared__ float warp_tot[32];
  const int b = blockIdx.x, i = threadIdx.x;
  const int lane = i & 31, wid = i >> 5;
  const long long base = (long long)b * C;
  float hi = 0.f;
  int oi = 0;
  if (i < C) {
    hi = entropy[base + i];
    oi = cand[base + i] != 0 && !(committed_state && committed_state[base + i]);
  }
  if (i == 0) {
    n_cand = 0;
    cut = 0x7fffffff;
  }
  // this thread's element in the current order: initially position i
  // (+0.f turns a -0 entropy into +0, so that the two compare equal as floats do)
  uint32_t key = (i < C && oi) ? order_bits(hi + 0.f) : 0xffffffffu;
  int src = i;
  __syncthreads();
  if (i < C && oi) atomicAdd(&n_cand, 1);
#pragma unroll 1
  for (int shift = 0; shift < 32; shift += 8) {
    const bool live = i < C;
    const uint32_t d = (key >> shift) & 255u;
    for (int k = i; k < 256 * nw; k += blockDim.x) hist[k] = 0;
    __syncthreads();
    const unsigned act = __ballot_sync(0xffffffffu, live);
    unsigned peers = 0;
    if (live) {
      peers = __match_any_sync(act, d);
      // the lowest lane of each digit group records the warp's count
      if ((peers & ((1u << lane) - 1u)) == 0) hist[d * nw + wid] = __popc(peers);
    }
    __syncthreads();
    // digit totals, then the exclusive scan over (digit, warp); a block of fewer
    // than 256 threads takes several digits a thread
    for (int dg = i; dg < 256; dg += blockDim.x) {
      uint32_t t = 0;
      for (int w = 0; w < nw; ++w) t += hist[dg * nw + w];
      dig_tot[dg] = t;
    }
    __syncthreads();
    if (i < 32) {
      // one warp scans the 256 digit totals, 8 per lane
      uint32_t v[8], run = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        v[q] = dig_tot[i * 8 + q];
        run += v[q];
      }
      uint32_t inc = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (i >= o) inc += y;
      }
      uint32_t ex = inc - run;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t t = v[q];
        dig_tot[i * 8 + q] = ex;
        ex += t;
      }
    }
    __syncthreads();
    for (int dg = i; dg < 256; dg += blockDim.x) {
      uint32_t run = dig_tot[dg];
      for (int w = 0; w < nw; ++w) {
        const uint32_t c = hist[dg * nw + w];
        hist[dg * nw + w] = run;
        run += c;
      }
    }
    __syncthreads();
    if (live) {
      const int dst = (int)(hist[d * nw + wid] + __popc(peers & ((1u << lane) - 1u)));
      key_a[dst] = key;
      pos_a[dst] = (uint16_t)src;
    }
    __syncthreads();
    if (live) {
      key = key_a[i];
      src = pos_a[i];
    }
    __syncthreads();
  }
  // thread i holds the i-th element of the confidence order (position src);
  // prefix sums of the sorted entropies: the cut is the first k >= 1 whose prefix
  // passes gamma, else every candidate
  const int nc = n_cand;
  float run = (i < nc) ? entropy[base + src] : 0.f;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, run, o);
    if (lane >= o) run += y;
  }
  if (lane == 31) warp_tot[wid] = run;
  __syncthreads();
  for (int w2 = 0; w2 < wid; ++w2) run += warp_tot[w2];
  if (i == 0) cut = nc;
  __syncthreads();
  if (i >= 1 && i < nc && run > gamma[b]) atomicMin(&cut, i);
  __syncthreads();
  if (i == 0) n_commit[b] = cut;
  if (i < C) {
    // every position: accepted iff it is a candidate ranked before the cut
    const bool acc = i < cut && i < nc;
    const int p = src;
    const int tok = argmax[base + p];
    commit_out[base + p] = acc ? 1 : 0;
    tokens[base + p] = acc ? tok : -1;
    if (acc && committed_state) committed_state[base + p] = 1;
    if (acc && token_state) token_state[base + p] = tok;
  }
}

// ---------------------------------------------------------------------------
// a6: h_out = bf16(h0 + e_sc) for open rows, bf16(h0 + emb[tok]) for committed.
// ---------------------------------------------------------------------------
__global__ void canvas_update_kernel(const __nv_bfloat16* h0, const float* e_sc,
                                     const __nv_bfloat16* emb, int V, const int32_t* tokens,
                                     const uint8_t* committed, int D, __nv_bfloat16* h_out,
                                     int* status) {
  const int row = blockIdx.x;
  const bool cm = committed[row] != 0;
  int tok = cm ? tokens[row] : 0;
  if (cm && (tok < 0 || tok >= V)) {
    if (threadIdx.x == 0) atomicOr(status, 8);
    tok = 0;
  }
  const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(h0 + (long long)row * D);
  const float2* es = reinterpret_cast<const float2*>(e_sc + (long long)row * D);
  const __nv_bfloat162* et = reinterpret_cast<const __nv_bfloat162*>(emb + (long long)tok * D);
  __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(h_out + (long long)row * D);
  for (int i = threadIdx.x; i < D / 2; i += blockDim.x) {
    const float2 x = __bfloat1622float2(a[i]);
    const float2 y = cm ? __bfloat1622float2(et[i]) : es[i];
    dst[i] = __floats2bfloat162_rn(x.x + y.x, x.y + y.y);
  }
}


// The same with one thread per 8 consecutive values of a row (16-byte loads and
// stores, rows spread over many CTAs), for 16-byte aligned buffers and d_model a
// multiple of 8: the same fp32 adds and roundings, so the same bits.
__global__ void canvas_update_vec_kernel(const __nv_bfloat16* h0, const float* e_sc,
                                         const __nv_bfloat16* emb, int V, const int32_t* tokens,
                                         const uint8_t* committed, int M, int D,
                                         __nv_bfloat16* h_out, int* status) {
  const int n8 = D / 8;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)M * n8) return;
  const int row = (int)(i / n8), c = (int)(i % n8);
  const bool cm = committed[row] != 0;
  int tok = cm ? tokens[row] : 0;
  if (cm && (tok < 0 || tok >= V)) {
    if (c == 0) atomicOr(status, 8);
    tok = 0;
  }
  const uint4 a = reinterpret_cast<const uint4*>(h0 + (long long)row * D)[c];
  float y[8];
  if (cm) {
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(emb + (long long)tok * D) + c);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __bfloat1622float2(b2[q]);
      y[2 * q] = f.x;
      y[2 * q + 1] = f.y;
    }
  } else {
    const float4* es = reinterpret_cast<const float4*>(e_sc + (long long)row * D) + 2 * c;
    const float4 e0 = es[0], e1 = es[1];
    y[0] = e0.x; y[1] = e0.y; y[2] = e0.z; y[3] = e0.w;
    y[4] = e1.x; y[5] = e1.y; y[6] = e1.z; y[7] = e1.w;
  }
  const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
  uint4 o;
  __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 x = __bfloat1622float2(a2[q]);
    o2[q] = __floats2bfloat162_rn(x.x + y[2 * q], x.y + y[2 * q + 1]);
  }
  reinterpret_cast<uint4*>(h_out + (long long)row * D)[c] = o;
}

// Diagnostic: one warp waits on an mbarrier that nothing arrives on, with a
// limit of `limit_ns` of %globaltimer; when the limit passes it sets
// DG_DEV_TIMEOUT (bit 0) and returns, as every bounded wait of the library does.
__global__ void wait_timeout_kernel(uint64_t limit_ns, int* status, int* waited) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(&bar)))
                 : "memory");
  }
  __syncwarp();
  if (threadIdx.x != 0) return;
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  const uint32_t addr = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr)
        : "memory");
    if (ok) break;  // never: no thread arrives
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > limit_ns) {
      atomicOr(status, 1 /* DG_DEV_TIMEOUT */);
      break;
    }
  }
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  *waited = (int)((t - t0) / 1000);  // microseconds
}

}  // namespace

namespace dgi {

cudaError_t philox_fill(uint64_t seed, const uint32_t* ctr4, int n, uint32_t* out4,
                        cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  philox_fill_kernel<<<(n + 255) / 256, 256, 0, st>>>(seed, reinterpret_cast<const uint4*>(ctr4),
                                                       n, reinterpret_cast<uint4*>(out4));
  return cudaGetLastError();
}

cudaError_t slot_noise(const uint16_t* h, int M, const uint16_t* e, int V, int D,
                       const float* inv_t, const int32_t* slot_row, const int32_t* slot_req,
                       int S, int R, uint64_t seed, int step, uint16_t* rows_out,
                       float* inv_t_out, int32_t* tok_out, cudaStream_t st) {
  if (S * R == 0) return cudaSuccess;
  int vbits = 0;
  while ((1 << vbits) < V) ++vbits;
  slot_noise_kernel<<<S * R, 128, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(h), M, reinterpret_cast<const __nv_bfloat16*>(e), V,
      vbits, D, inv_t, slot_row, slot_req, S, R, seed, step,
      reinterpret_cast<__nv_bfloat16*>(rows_out), inv_t_out, tok_out, status_ptr());
  return cudaGetLastError();
}

// Label logits then the per-slot read (label tables of stride L <= 32 LPL).
// rows == null: lp_draws already holds the label logits z/T, gathered by the
// lm-head pass over the draw rows.
template <int LPL>
cudaError_t finish(const uint16_t* rows, const float* inv_t_rows, const float* lse_rows,
                   const uint16_t* w, int V, int D, const int32_t* label_ids,
                   const int32_t* n_labels, int L, int S, int R, int samples, float gate,
                   float* q_avg, float* h_slot, int32_t* chosen, float* lp_draws,
                   uint8_t* resampled, int32_t* n_reads, cudaStream_t st) {
  int* stp = status_ptr();
  if (rows != nullptr) {
    slot_dots_kernel<<<dim3(S * R, (L + 7) / 8), 256, 0, st>>>(
        reinterpret_cast<const __nv_bfloat16*>(rows), inv_t_rows,
        reinterpret_cast<const __nv_bfloat16*>(w), V, D, label_ids, n_labels, L, R, lp_draws,
        stp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  slot_epilogue_kernel<LPL><<<S, 32, 0, st>>>(lse_rows, n_labels, L, R, samples, gate, q_avg,
                                              h_slot, chosen, lp_draws, resampled, n_reads, stp);
  return cudaGetLastError();
}

cudaError_t slot_finish(const uint16_t* rows, const float* inv_t_rows, const float* lse_rows,
                        const uint16_t* w, int V, int D, const int32_t* label_ids,
                        const int32_t* n_labels, int S, int R, int samples, float gate,
                        float* q_avg, float* h_slot, int32_t* chosen, float* lp_draws,
                        uint8_t* resampled, int32_t* n_reads, cudaStream_t st) {
  if (S == 0) return cudaSuccess;
  return finish<1>(rows, inv_t_rows, lse_rows, w, V, D, label_ids, n_labels, MAXL, S, R, samples,
                   gate, q_avg, h_slot, chosen, lp_draws, resampled, n_reads, st);
}

cudaError_t slot_finish_wide(const uint16_t* rows, const float* inv_t_rows, const float* lse_rows,
                             const uint16_t* w, int V, int D, const int32_t* label_ids,
                             const int32_t* n_labels, int L, int S, int R, int samples,
                             float gate, float* q_avg, float* h_slot, int32_t* chosen,
                             float* lp_draws, uint8_t* resampled, int32_t* n_reads,
                             cudaStream_t st) {
  if (S == 0) return cudaSuccess;
  if (L < 1 || L > 256) return cudaErrorInvalidValue;
  if (L <= 64)
    return finish<2>(rows, inv_t_rows, lse_rows, w, V, D, label_ids, n_labels, L, S, R, samples,
                     gate, q_avg, h_slot, chosen, lp_draws, resampled, n_reads, st);
  if (L <= 128)
    return finish<4>(rows, inv_t_rows, lse_rows, w, V, D, label_ids, n_labels, L, S, R, samples,
                     gate, q_avg, h_slot, chosen, lp_draws, resampled, n_reads, st);
  return finish<8>(rows, inv_t_rows, lse_rows, w, V, D, label_ids, n_labels, L, S, R, samples,
                   gate, q_avg, h_slot, chosen, lp_draws, resampled, n_reads, st);
}

cudaError_t ask_if_select(const int32_t* chosen1, int S1, const int32_t* cond_slot,
                          const int32_t* cond_value, const int32_t* q_owner,
                          const int32_t* q_label_ids, const int32_t* q_n_labels, int Q, int S2,
                          int32_t* label_ids2, int32_t* n_labels2, uint8_t* fired,
                          cudaStream_t st) {
  const long long n = std::max<long long>(Q, 32LL * S2);
  if (n == 0) return cudaSuccess;
  ask_if_kernel<<<(int)((n + 127) / 128), 128, 0, st>>>(chosen1, S1, cond_slot, cond_value, q_owner,
                                                  q_label_ids, q_n_labels, Q, S2, label_ids2,
                                                  n_labels2, fired, status_ptr());
  return cudaGetLastError();
}

cudaError_t commit(int B, int C, const float* entropy, const int32_t* argmax,
                   const uint8_t* cand, const float* gamma, uint8_t* committed_state,
                   int32_t* token_state, uint8_t* commit_out, int32_t* tokens,
                   int32_t* n_commit, cudaStream_t st) {
  if (B == 0) return cudaSuccess;
  const int threads = ((C + 31) / 32) * 32;
  const size_t shm = (size_t)C * 4 + (size_t)((C + 1) & ~1) * 2 + (size_t)256 * (threads / 32) * 4;
  commit_kernel<<<B, threads, shm, st>>>(C, entropy, argmax, cand, gamma, committed_state,
                                         token_state, commit_out, tokens, n_commit);
  return cudaGetLastError();
}

cudaError_t check_wait_timeout(uint64_t limit_ns, int* waited_us, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(limit_ns, status_ptr(), waited_us);
  return cudaGetLastError();
}

cudaError_t canvas_update(const uint16_t* h0, const float* e_sc, const uint16_t* emb, int V,
                          const int32_t* tokens, const uint8_t* committed, int M, int D,
                          uint16_t* h_out, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
  if (D % 8 == 0 && a16(h0) && a16(e_sc) && a16(emb) && a16(h_out)) {
    const long long n = (long long)M * (D / 8);
    canvas_update_vec_kernel<<<(int)((n + 255) / 256), 256, 0, st>>>(
        reinterpret_cast<const __nv_bfloat16*>(h0), e_sc,
        reinterpret_cast<const __nv_bfloat16*>(emb), V, tokens, committed, M, D,
        reinterpret_cast<__nv_bfloat16*>(h_out), status_ptr());
  } else {
    canvas_update_kernel<<<M, 256, 0, st>>>(
        reinterpret_cast<const __nv_bfloat16*>(h0), e_sc,
        reinterpret_cast<const __nv_bfloat16*>(emb), V, tokens, committed, D,
        reinterpret_cast<__nv_bfloat16*>(h_out), status_ptr());
  }
  return cudaGetLastError();
}


}  // namespace dgi
