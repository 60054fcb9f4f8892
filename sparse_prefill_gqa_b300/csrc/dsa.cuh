// dsa.cuh -- token top-k sparse attention for decode: indexer scores, top-k selection, and the
// gather of the selected keys and values for the split-K decode.
//
// What it computes ("Attention in Code", section 5): a small scorer rates every cached token for
// the current query -- score[s] = sum_j w_j * relu(qi_j . ki[s]) over a few small query heads j,
// with one small key ki[s] per token -- and attention then reads only the k tokens with the
// highest scores.  The cache keeps every token; what shrinks is what attention reads.  Decode
// form: one query per sequence at position L_b - 1, which may see every cached token.
// Ties at the k-th score go to the lower token index.  The decode over the selected tokens is the
// split-K decode kernel in its gathered form (decode.cuh), which loads the chosen cache rows itself.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace ga {

constexpr int kIdxWarps = 8;
constexpr int kIdxKeysPerWarp = 64;            // keys a warp scores per CTA
constexpr int kIdxGroups = 2;                  // 16-key groups whose loads a lane keeps in flight

// grid: (ceil(L_max / (kIdxWarps * kIdxKeysPerWarp)), batch); block: 32 * kIdxWarps.
// DI = indexer key dim (64 or 128), HI = indexer heads (power of two, <= DI / 8).
//
// The scores of 16 keys are mma.sync m16n8k16 contractions, one per 16 dims: the keys are the 16
// rows of A and the indexer heads the columns of B, eight per n-block (columns past HI hold zero
// queries and zero weights).  At 8 FLOP per byte the kernel is bound by HBM; the tensor cores
// only take the 1024 multiply-adds per key off the issue slots, so the loads stay in flight.
// A dot product does not depend on the order of its dims, so each lane takes whole 16-byte
// pieces of its key rows straight from global memory: lane (g, c) = (lane / 4, lane % 4) loads
// pieces c, c + 4, ... of keys g and g + 8, and its query fragment (head g) the same pieces.
// In the k16 step that covers dims 0..3 (or 4..7) of piece u, the lane's four dims of a row sit
// at the k indices 2c, 2c + 1, 2c + 8, 2c + 9 that the fragment layout assigns to it, on the A
// and the B side alike.  The result is C[key][head]; lane (g, c) holds heads 2c, 2c + 1 (of
// each n-block) of keys g and g + 8, so the weighted relu sum over the heads takes two shuffles
// within each group of four lanes.  Scores past lens[b] are -inf.
template <int DI, int HI>
__global__ void __launch_bounds__(32 * kIdxWarps)
dsa_indexer_kernel(const __nv_bfloat16* __restrict__ qi, const float* __restrict__ wi,
                   const __nv_bfloat16* __restrict__ ki, const int32_t* __restrict__ lens,
                   int L_max, float* __restrict__ scores) {
  constexpr int NU = DI / 32;                  // 16-byte pieces per lane and key row
  constexpr int NB = (HI + 7) / 8;             // n8 blocks of indexer heads
  static_assert(HI >= 1 && HI <= DI / 8 && (HI & (HI - 1)) == 0, "indexer heads: power of two <= DI/8");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, b = blockIdx.y;
  const int g = lane >> 2, c = lane & 3;
  griddep_launch_dependents();                 // the top-k select may start its launch
  const int L = seq_keys(lens, b, L_max);
  uint4 qf[NB][NU];
  float w[NB][2];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int head = 8 * nb + g;
#pragma unroll
    for (int u = 0; u < NU; ++u)
      qf[nb][u] = head < HI
          ? __ldg(reinterpret_cast<const uint4*>(qi + ((size_t)b * HI + head) * DI + 8 * (c + 4 * u)))
          : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int hw = 8 * nb + 2 * c + e;
      w[nb][e] = hw < HI ? wi[(size_t)b * HI + hw] : 0.0f;
    }
  }
  const int key_base = (blockIdx.x * kIdxWarps + warp) * kIdxKeysPerWarp;
  const __nv_bfloat16* kb = ki + (size_t)b * L_max * DI;
  float* sb = scores + (size_t)b * L_max;
  for (int rb = 0; rb < kIdxKeysPerWarp; rb += 16 * kIdxGroups) {
    uint4 ka[kIdxGroups][2][NU];               // [group][key g or g + 8][piece]
#pragma unroll
    for (int gi = 0; gi < kIdxGroups; ++gi)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int s = key_base + rb + 16 * gi + 8 * r + g;
#pragma unroll
        for (int u = 0; u < NU; ++u)
          ka[gi][r][u] = s < L ? __ldg(reinterpret_cast<const uint4*>(kb + (size_t)s * DI + 8 * (c + 4 * u)))
                               : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
    for (int gi = 0; gi < kIdxGroups; ++gi) {
      float acc[NB][4];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.0f;
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        // A registers: (key g, k 2c..), (key g + 8, k 2c..), (key g, k 2c + 8..), (key g + 8, k 2c + 8..)
        const uint32_t a_lo[4] = {ka[gi][0][u].x, ka[gi][1][u].x, ka[gi][0][u].y, ka[gi][1][u].y};
        const uint32_t a_hi[4] = {ka[gi][0][u].z, ka[gi][1][u].z, ka[gi][0][u].w, ka[gi][1][u].w};
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          mma_bf16_16816(acc[nb], a_lo, qf[nb][u].x, qf[nb][u].y);
          mma_bf16_16816(acc[nb], a_hi, qf[nb][u].z, qf[nb][u].w);
        }
      }
      float s0 = 0.0f, s1 = 0.0f;              // keys g and g + 8 over this lane's heads
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        s0 = fmaf(w[nb][0], fmaxf(acc[nb][0], 0.0f), s0);
        s0 = fmaf(w[nb][1], fmaxf(acc[nb][1], 0.0f), s0);
        s1 = fmaf(w[nb][0], fmaxf(acc[nb][2], 0.0f), s1);
        s1 = fmaf(w[nb][1], fmaxf(acc[nb][3], 0.0f), s1);
      }
      s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
      s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
      const int s = key_base + rb + 16 * gi + g + 8 * c;      // lane c = 0: key g, c = 1: key g + 8
      if (c < 2 && s < L_max) sb[s] = s < L ? (c ? s1 : s0) : -INFINITY;
    }
  }
}

// ---------------------------------------------------------------------------------------
// Top-k selection.  One CTA (kTopkThreads) per sequence: the k-th largest score by a radix
// select over order-preserving 32-bit keys (4 passes of 8 bits, most significant first), then an
// ordered compaction that keeps every score above it and, among scores equal to it, the lowest
// indices -- exactly k indices (all of them when L_b <= k), in increasing order.
constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkCandMax = 8192;            // keys of the chosen bins kept for the later passes
constexpr int kTopkFixedSmem = (kTopkWarps * 256 + kTopkCandMax) * 4;   // dynamic, before the row
constexpr int kTopkStageMax = 40960;          // longest row whose keys are staged in shared memory

__device__ __forceinline__ uint32_t order_key(float x) {     // larger float -> larger key
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// grid: (batch); block: kTopkThreads (32 warps); dynamic shared memory kTopkFixedSmem (+ 4 L_max
// bytes when STAGED).
//   radix select: per 8-bit digit, a histogram of the keys that match the digits chosen so far,
//     one private histogram per warp (indexer scores are non-negative and concentrated, so the
//     top digits fall into one or a few bins: a shared histogram would serialise every warp on
//     them), counted by plain shared-memory atomics and summed per bin; warp 0 finds the bin that holds the k-th largest key by a suffix
//     scan, each lane covering 8 bins from the top.  Once the chosen bin holds at most
//     kTopkCandMax keys they are copied to a candidate list, and the remaining digits histogram
//     only those;
//   compaction: warp w owns a contiguous segment of the scores; a first sweep counts its keys
//     above and equal to the k-th, a second writes its selected indices at its offset, which
//     keeps the indices in increasing order with one barrier in all.
// STAGED: the row's keys are read from global memory once, into shared memory (L_max <=
// kTopkStageMax), and every pass and sweep reads them there; otherwise each reads the row again.
template <bool STAGED>
__global__ void __launch_bounds__(kTopkThreads)
topk_select_kernel(const float* __restrict__ scores, const int32_t* __restrict__ lens, int L_max, int topk,
                   int32_t* __restrict__ idx, int32_t* __restrict__ n_sel) {
  constexpr int NW = kTopkWarps;
  extern __shared__ uint32_t dyn[];
  int* whist = reinterpret_cast<int*>(dyn);      // NW x 256 per-warp histograms
  uint32_t* cand = dyn + NW * 256;               // candidate keys
  uint32_t* skeys = cand + kTopkCandMax;         // STAGED: the row's order-preserving keys
  __shared__ int hist[256];
  __shared__ int w_gt[NW], w_eq[NW];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need, s_ncand;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t lt_mask = (1u << lane) - 1u;
  const int b = blockIdx.x;
  // Launched as a programmatic dependent of the indexer: nothing is read before it has completed.
  griddep_wait();
  griddep_launch_dependents();                   // the gathered decode may start its launch
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
  if (STAGED) {
    // 16-byte loads when the row is 16-byte aligned (all of them in flight: at most 10 a thread)
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    const int n4 = vec ? L / 4 : 0;
#pragma unroll 4
    for (int i = threadIdx.x; i < n4; i += kTopkThreads) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(row) + i);
      *reinterpret_cast<uint4*>(skeys + 4 * i) = make_uint4(order_key(x.x), order_key(x.y), order_key(x.z), order_key(x.w));
    }
    for (int j = 4 * n4 + threadIdx.x; j < L; j += kTopkThreads) skeys[j] = order_key(row[j]);
  }
  auto key_at = [&](int j) -> uint32_t { return STAGED ? skeys[j] : order_key(row[j]); };
  // ---- radix select of the k-th largest key ------------------------------------------------
  if (threadIdx.x == 0) { s_prefix = 0u; s_need = k; s_ncand = -1; }
  int* my_hist = whist + warp * 256;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const uint32_t hi_mask = pass == 0 ? 0u : (0xFFFFFFFFu << (32 - 8 * pass));
    for (int i = threadIdx.x; i < NW * 256; i += kTopkThreads) whist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    const int n_cand = s_ncand;                  // -1: no candidate list yet
    auto count = [&](uint32_t key, bool in) {
      if (in) atomicAdd(&my_hist[(key >> shift) & 0xFF], 1);
    };
    if (n_cand >= 0) {
      for (int base = 0; base < n_cand; base += kTopkThreads) {
        const int j = base + (int)threadIdx.x;
        const uint32_t key = j < n_cand ? cand[j] : 0u;
        count(key, j < n_cand && (key & hi_mask) == prefix);
      }
    } else {
      for (int base = 0; base < L; base += kTopkThreads) {       // uniform trip count per warp
        const int j = base + (int)threadIdx.x;
        const uint32_t key = j < L ? key_at(j) : 0u;
        count(key, j < L && (key & hi_mask) == prefix);
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 256; i += kTopkThreads) {
      int t = 0;
#pragma unroll 8
      for (int w = 0; w < NW; ++w) t += whist[w * 256 + i];
      hist[i] = t;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l covers bins 255 - 8l down to 248 - 8l; the chosen bin is the highest b >= 1 whose
      // suffix count (keys in bins >= b) reaches `need`, else 0
      const int need = s_need;
      int cnt = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) cnt += hist[255 - 8 * lane - e];
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const uint32_t reach = __ballot_sync(0xffffffffu, incl >= need);
      const int ls = reach ? __ffs(reach) - 1 : 31;
      if (lane == ls) {
        int running = incl - cnt;                // keys in the bins above this lane's
        int bin = 255 - 8 * lane;
        while (bin > 0 && running + hist[bin] < need) { running += hist[bin]; --bin; }
        s_prefix = prefix | ((uint32_t)bin << shift);
        s_need = need - running;                 // how many of this bin's keys are in the top k
        hist[0] = hist[bin];                     // keys that share the chosen digits (read below)
      }
    }
    __syncthreads();
    // the first time the chosen bin is small enough, its keys become the candidate list
    if (pass < 3 && n_cand < 0 && hist[0] <= kTopkCandMax) {
      const uint32_t pre = s_prefix, m = 0xFFFFFFFFu << (24 - 8 * pass);
      if (threadIdx.x == 0) s_ncand = 0;
      __syncthreads();
      for (int base = 0; base < L; base += kTopkThreads) {
        const int j = base + (int)threadIdx.x;
        const uint32_t key = j < L ? key_at(j) : 0u;
        const bool in = j < L && (key & m) == pre;
        const uint32_t bal = __ballot_sync(0xffffffffu, in);
        int at = 0;
        if (lane == 0 && bal) at = atomicAdd(&s_ncand, __popc(bal));
        at = __shfl_sync(0xffffffffu, at, 0);
        if (in) cand[at + __popc(bal & lt_mask)] = key;
      }
      __syncthreads();
    }
  }
  const uint32_t kth = s_prefix;                 // the k-th largest key
  const int quota = s_need;                      // keys equal to kth that are kept
  // ---- ordered compaction over per-warp segments ------------------------------------------
  const int seg = (L + kTopkThreads - 1) / kTopkThreads * 32;   // a multiple of 32 keys
  const int j0 = warp * seg, j1 = min(L, j0 + seg);
  int n_gt = 0, n_eq = 0;
  for (int base = j0; base < j1; base += 32) {
    const int j = base + lane;
    const uint32_t key = j < j1 ? key_at(j) : 0u;
    n_gt += __popc(__ballot_sync(0xffffffffu, j < j1 && key > kth));
    n_eq += __popc(__ballot_sync(0xffffffffu, j < j1 && key == kth));
  }
  if (lane == 0) { w_gt[warp] = n_gt; w_eq[warp] = n_eq; }
  __syncthreads();
  int gt_before = lane < warp ? w_gt[lane] : 0;
  int eq_run = lane < warp ? w_eq[lane] : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    gt_before += __shfl_xor_sync(0xffffffffu, gt_before, o);
    eq_run += __shfl_xor_sync(0xffffffffu, eq_run, o);
  }
  int out_run = gt_before + min(eq_run, quota);
  for (int base = j0; base < j1; base += 32) {
    const int j = base + lane;
    const uint32_t key = j < j1 ? key_at(j) : 0u;
    const bool gt = j < j1 && key > kth, eq = j < j1 && key == kth;
    const uint32_t eq_bal = __ballot_sync(0xffffffffu, eq);
    const bool sel = gt || (eq && eq_run + __popc(eq_bal & lt_mask) < quota);
    const uint32_t sel_bal = __ballot_sync(0xffffffffu, sel);
    if (sel && GA_BOUNDS(out_run + __popc(sel_bal & lt_mask) < topk, 6, out_run + __popc(sel_bal & lt_mask)))
      out[out_run + __popc(sel_bal & lt_mask)] = j;
    eq_run += __popc(eq_bal);
    out_run += __popc(sel_bal);
  }
  for (int j = k + threadIdx.x; j < topk; j += kTopkThreads) out[j] = -1;
  if (threadIdx.x == 0) n_sel[b] = k;
}

}  // namespace ga
