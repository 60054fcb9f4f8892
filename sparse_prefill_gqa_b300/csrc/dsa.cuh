// dsa.cuh -- token top-k sparse attention for decode: indexer scores, top-k selection, and the
// gather of the selected keys and values for the split-K decode.
//
// What it computes ("Attention in Code", section 5): a small scorer rates every cached token for
// the current query -- score[s] = sum_j w_j * relu(qi_j . ki[s]) over a few small query heads j,
// with one small key ki[s] per token -- and attention then reads only the k tokens with the
// highest scores.  The cache keeps every token; what shrinks is what attention reads.  Decode
// form: one query per sequence at position L_b - 1, which may see every cached token.
// Ties at the k-th score go to the lower token index.
#pragma once

#include "common.cuh"

namespace ga {

constexpr int kIdxWarps = 8;
constexpr int kIdxKeysPerWarp = 64;            // keys a warp scores per CTA

// grid: (ceil(L_max / (kIdxWarps * kIdxKeysPerWarp)), batch); block: 32 * kIdxWarps.
// DI = indexer key dim (64 or 128), HI = indexer heads (power of two, <= DI / 8).
// Lane l of a warp holds dims 8 (l % LD) .. + 7 of every head (LD = DI / 8 lanes per key) and
// scores keys l / LD, l / LD + 32 / LD, ...; scores past lens[b] are -inf.
template <int DI, int HI>
__global__ void __launch_bounds__(32 * kIdxWarps)
dsa_indexer_kernel(const __nv_bfloat16* __restrict__ qi, const float* __restrict__ wi,
                   const __nv_bfloat16* __restrict__ ki, const int32_t* __restrict__ lens,
                   int L_max, float* __restrict__ scores) {
  constexpr int LD = DI / 8, RP = 32 / LD;
  static_assert(HI >= 1 && HI <= LD && (HI & (HI - 1)) == 0, "indexer heads: power of two <= DI/8");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, b = blockIdx.y;
  const int L = seq_keys(lens, b, L_max);
  const int col = 8 * (lane % LD), r0 = lane / LD;
  float qreg[HI][8];
#pragma unroll
  for (int j = 0; j < HI; ++j) {
    float f[8];
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(qi + ((size_t)b * HI + j) * DI + col), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) qreg[j][e] = f[e];
  }
  // after the butterfly, lane l holds head idx = (bits of l below HI); its weight
  int idx = 0;
#pragma unroll
  for (int o = 1, w = 1; o < HI; o <<= 1, w <<= 1) idx += ((lane & o) ? 1 : 0) * (HI / (2 * w));
  const float wj = wi[(size_t)b * HI + idx];
  const int key_base = (blockIdx.x * kIdxWarps + warp) * kIdxKeysPerWarp;
  constexpr int BATCH = 8;                           // loads in flight per lane
  for (int rb = 0; rb < kIdxKeysPerWarp; rb += BATCH * RP) {
  uint4 xk[BATCH];
#pragma unroll
  for (int u = 0; u < BATCH; ++u) {
    const int s = key_base + rb + u * RP + r0;
    xk[u] = s < L ? __ldg(reinterpret_cast<const uint4*>(ki + ((size_t)b * L_max + s) * DI + col))
                  : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int u = 0; u < BATCH; ++u) {
    const int s = key_base + rb + u * RP + r0;
    float part[HI];
    if (s < L) {
      float f[8];
      bf16x8_to_f32(xk[u], f);
#pragma unroll
      for (int j = 0; j < HI; ++j) {
        float a = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) a = fmaf(qreg[j][e], f[e], a);
        part[j] = a;
      }
    } else {
#pragma unroll
      for (int j = 0; j < HI; ++j) part[j] = 0.0f;
    }
    // transposed butterfly over the low lane bits: each stage halves the heads a lane holds
    int cnt = HI;
#pragma unroll
    for (int o = 1; o < HI; o <<= 1) {
      const bool upper = (lane & o) != 0;
      cnt >>= 1;
#pragma unroll
      for (int j = 0; j < HI / 2; ++j) {
        if (j < cnt) {
          const float send = upper ? part[j] : part[j + cnt];
          const float keep = upper ? part[j + cnt] : part[j];
          part[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
    }
    float dot = part[0];                              // head idx, summed over HI lanes
#pragma unroll
    for (int o = HI; o < LD; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    float sc = wj * fmaxf(dot, 0.0f);
#pragma unroll
    for (int o = 1; o < HI; o <<= 1) sc += __shfl_xor_sync(0xffffffffu, sc, o);
    if (lane % LD == 0 && s < L_max) scores[(size_t)b * L_max + s] = s < L ? sc : -INFINITY;
  }
  }
}

// ---------------------------------------------------------------------------------------
// Top-k selection.  One CTA (kTopkThreads) per sequence: the k-th largest score by a radix
// select over order-preserving 32-bit keys (4 passes of 8 bits, most significant first), then an
// ordered compaction that keeps every score above it and, among scores equal to it, the lowest
// indices -- exactly k indices (all of them when L_b <= k), in increasing order.
constexpr int kTopkThreads = 1024;

__device__ __forceinline__ uint32_t order_key(float x) {     // larger float -> larger key
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix of `flag` over the CTA in thread order and the CTA total; wsum: 32 ints.
__device__ __forceinline__ int cta_prefix(bool flag, int* wsum, int& total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bal = __ballot_sync(0xffffffffu, flag);
  if (lane == 0) wsum[warp] = __popc(bal);
  __syncthreads();
  int before = 0;
  total = 0;
  for (int w = 0; w < kTopkThreads / 32; ++w) {
    if (w < warp) before += wsum[w];
    total += wsum[w];
  }
  __syncthreads();
  return before + __popc(bal & ((1u << lane) - 1u));
}

// grid: (batch); block: kTopkThreads.
__global__ void __launch_bounds__(kTopkThreads)
topk_select_kernel(const float* __restrict__ scores, const int32_t* __restrict__ lens, int L_max, int topk,
                   int32_t* __restrict__ idx, int32_t* __restrict__ n_sel) {
  __shared__ int hist[256];
  __shared__ int wsum[32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  const int b = blockIdx.x;
  const int L = seq_keys(lens, b, L_max);
  const float* row = scores + (size_t)b * L_max;
  int32_t* out = idx + (size_t)b * topk;
  const int k = min(topk, L);
  if (k == L) {                                  // every token: no selection
    for (int j = threadIdx.x; j < L; j += kTopkThreads) out[j] = j;
    for (int j = L + threadIdx.x; j < topk; j += kTopkThreads) out[j] = -1;
    if (threadIdx.x == 0) n_sel[b] = L;
    return;
  }
  // radix select of the k-th largest key
  if (threadIdx.x == 0) { s_prefix = 0u; s_need = k; }
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const uint32_t hi_mask = pass == 0 ? 0u : (0xFFFFFFFFu << (32 - 8 * pass));
    for (int i = threadIdx.x; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    for (int j = threadIdx.x; j < L; j += kTopkThreads) {
      const uint32_t key = order_key(row[j]);
      if ((key & hi_mask) == prefix) atomicAdd(&hist[(key >> shift) & 0xFFu], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {                      // walk the bins from the top
      int need = s_need, bin = 255;
      while (bin > 0 && hist[bin] < need) { need -= hist[bin]; --bin; }
      s_prefix = prefix | ((uint32_t)bin << shift);
      s_need = need;                             // how many of this bin's keys are in the top k
    }
    __syncthreads();
  }
  const uint32_t kth = s_prefix;                 // the k-th largest key
  const int quota = s_need;                      // keys equal to kth that are kept
  int eq_run = 0, out_run = 0;
  for (int base = 0; base < L; base += kTopkThreads) {
    const int j = base + (int)threadIdx.x;
    const uint32_t key = j < L ? order_key(row[j]) : 0u;
    const bool gt = j < L && key > kth, eq = j < L && key == kth;
    int eq_tot, sel_tot;
    const int eq_rank = eq_run + cta_prefix(eq, wsum, eq_tot);
    const bool sel = gt || (eq && eq_rank < quota);
    const int pos = out_run + cta_prefix(sel, wsum, sel_tot);
    if (sel) out[pos] = j;
    eq_run += eq_tot;
    out_run += sel_tot;
  }
  for (int j = k + threadIdx.x; j < topk; j += kTopkThreads) out[j] = -1;
  if (threadIdx.x == 0) n_sel[b] = k;
}

// ---------------------------------------------------------------------------------------
// Gather: rows idx[b, i] (i < n_sel[b]) of K and V of every kv head into a compact cache
// [batch, n_kv, topk, d], in the order of the index list.  grid: (ceil(topk / 8), n_kv, batch);
// block: 256 threads = 8 rows x 32 threads, 16 bytes a thread and step.
__global__ void __launch_bounds__(256)
dsa_gather_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                  const int32_t* __restrict__ idx, const int32_t* __restrict__ n_sel, int n_kv, int d,
                  int Tk_max, int topk, __nv_bfloat16* __restrict__ kc, __nv_bfloat16* __restrict__ vc) {
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (i >= min(n_sel[b], topk)) return;
  const int j = idx[(size_t)b * topk + i];
  if (j < 0 || j >= Tk_max) return;
  const size_t src = (((size_t)b * n_kv + kvh) * Tk_max + j) * d;
  const size_t dst = (((size_t)b * n_kv + kvh) * topk + i) * d;
  for (int c = 8 * (threadIdx.x & 31); c < d; c += 256) {
    *reinterpret_cast<uint4*>(kc + dst + c) = *reinterpret_cast<const uint4*>(k + src + c);
    *reinterpret_cast<uint4*>(vc + dst + c) = *reinterpret_cast<const uint4*>(v + src + c);
  }
}

}  // namespace ga
