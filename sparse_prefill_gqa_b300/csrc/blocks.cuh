// blocks.cuh -- block statistics (centroid and maximum radius per key block) for radius-bounded sparse prefill.
//
// "RBS-Attention review" (patty.io): keys are grouped into blocks represented by their
// centroid; a block's maximum radius is the distance from the centroid to its farthest
// key.  Memory-bound reductions on the CUDA cores; the selection that uses the statistics is
// in select.cuh.
#pragma once

#include "attend_simt.cuh"
#include "common.cuh"

namespace ga {

// ---------------------------------------------------------------------------------------
// Block statistics: one CTA per (key block, kv head, sequence).  Pass 1 sums the block's
// keys per dimension (thread = dimension, rows read coalesced); pass 2 re-reads the block
// (now in L1) and takes the largest squared distance to the centroid, one warp per key.
// HBM traffic: the keys once, plus d + 1 floats per block written.
// ---------------------------------------------------------------------------------------
constexpr int kStatsThreads = 128;

template <typename T>
__global__ void __launch_bounds__(kStatsThreads)
block_stats_kernel(const T* __restrict__ k, const int32_t* __restrict__ k_lens, int n_kv, int d,
                   int Tk_max, int k_block, int nKb, float* __restrict__ centroid,
                   float* __restrict__ radius) {
  __shared__ float c_s[kSimtMaxD];
  __shared__ float r2_s[kStatsThreads / 32];
  const int beta = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int Tk = seq_keys(k_lens, b, Tk_max);
  const long long j0 = (long long)beta * k_block;
  const int n = (int)max(0LL, min((long long)k_block, (long long)Tk - j0));
  const size_t blk = ((size_t)b * n_kv + kvh) * nKb + beta;
  float* c_out = centroid + blk * d;
  if (n == 0) {
    for (int c = threadIdx.x; c < d; c += kStatsThreads) c_out[c] = 0.0f;
    if (threadIdx.x == 0) radius[blk] = 0.0f;
    return;
  }
  const T* kb = k + (((size_t)b * n_kv + kvh) * Tk_max + j0) * d;
  for (int c = threadIdx.x; c < d; c += kStatsThreads) {
    float s = 0.0f;
    for (int j = 0; j < n; ++j) s += to_f32(kb[(size_t)j * d + c]);
    const float mean = s / (float)n;
    c_s[c] = mean;
    c_out[c] = mean;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float best = 0.0f;
  for (int j = warp; j < n; j += kStatsThreads / 32) {
    float acc = 0.0f;
    for (int c = lane; c < d; c += 32) {
      const float diff = to_f32(kb[(size_t)j * d + c]) - c_s[c];
      acc = fmaf(diff, diff, acc);
    }
    best = fmaxf(best, warp_sum(acc));
  }
  if (lane == 0) r2_s[warp] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r2 = r2_s[0];
    for (int w = 1; w < kStatsThreads / 32; ++w) r2 = fmaxf(r2, r2_s[w]);
    radius[blk] = sqrtf(r2);
  }
}

// ---------------------------------------------------------------------------------------
// Block statistics, bf16 keys with d = 8 * L (L = 1, 2, 4, 8, 16 or 32): one warp per key
// block.  Lane l reads 16 bytes (8 dimensions, 8 * (l % L) ..) of rows l / L, l / L + 32 / L,
// ...; the per-dimension sums meet by shuffles across the lanes of equal l % L.  Pass 2
// re-reads the block (L1 hits) and keeps the largest squared distance to the centroid.
// Each key byte crosses HBM once, in 16-byte loads.
// ---------------------------------------------------------------------------------------
constexpr int kStatsVecWarps = 4;


template <int L>
__global__ void __launch_bounds__(32 * kStatsVecWarps)
block_stats_vec_kernel(const __nv_bfloat16* __restrict__ k, const int32_t* __restrict__ k_lens,
                       int batch, int n_kv, int Tk_max, int k_block, int nKb,
                       float* __restrict__ centroid, float* __restrict__ radius) {
  constexpr int D = 8 * L, RP = 32 / L;          // head dim, rows per warp-wide load
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long blk = (long long)blockIdx.x * kStatsVecWarps + warp;   // (b, kvh, beta)
  if (blk >= (long long)batch * n_kv * nKb) return;
  const int beta = (int)(blk % nKb);
  const int bk = (int)(blk / nKb);               // b * n_kv + kvh
  const int b = bk / n_kv;
  const int Tk = seq_keys(k_lens, b, Tk_max);
  const long long j0 = (long long)beta * k_block;
  const int n = (int)max(0LL, min((long long)k_block, (long long)Tk - j0));
  float* c_out = centroid + blk * D;
  const int col = 8 * (lane % L), r0 = lane / L;
  if (n == 0) {
    if (r0 == 0) {
      *reinterpret_cast<float4*>(c_out + col) = make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(c_out + col + 4) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (lane == 0) radius[blk] = 0.0f;
    return;
  }
  const __nv_bfloat16* kb = k + ((size_t)bk * Tk_max + j0) * D + col;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int r = r0; r < n; r += RP) {
    float f[8];
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(kb + (size_t)r * D)), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += f[i];
  }
#pragma unroll
  for (int o = L; o < 32; o <<= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
  const float inv_n = 1.0f / (float)n;
  float c[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) c[i] = acc[i] * inv_n;
  if (r0 == 0) {
    *reinterpret_cast<float4*>(c_out + col) = make_float4(c[0], c[1], c[2], c[3]);
    *reinterpret_cast<float4*>(c_out + col + 4) = make_float4(c[4], c[5], c[6], c[7]);
  }
  float best = 0.0f;
#pragma unroll 4
  for (int rb = 0; rb < n; rb += RP) {           // every lane runs the same trip count
    const int r = rb + r0;
    float part = 0.0f;
    if (r < n) {
      float f[8];
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(kb + (size_t)r * D)), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float e = f[i] - c[i];
        part = fmaf(e, e, part);
      }
    }
#pragma unroll
    for (int o = 1; o < L; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    best = fmaxf(best, part);
  }
#pragma unroll
  for (int o = L; o < 32; o <<= 1) best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, o));
  if (lane == 0) radius[blk] = sqrtf(best);
}

// Register-resident form (bf16, d = 8 L with L in {4, 8, 16}, key blocks of at most 64 keys):
// one warp per key block reads the block once -- each lane keeps its R = 2 L rows (16 bytes
// each) in registers -- sums them for the centroid, then takes the distances from the same
// registers, so HBM sees every key byte exactly once.  Same arithmetic as the two-pass form:
// fp32 sums in row order per lane, a shuffle tree over the lanes of a column, squared
// distances summed over each lane's 8 dimensions then over the L lanes of a row.
template <int L>
__global__ void __launch_bounds__(32 * kStatsVecWarps)
block_stats_reg_kernel(const __nv_bfloat16* __restrict__ k, const int32_t* __restrict__ k_lens,
                       int batch, int n_kv, int Tk_max, int k_block, int nKb,
                       float* __restrict__ centroid, float* __restrict__ radius) {
  constexpr int D = 8 * L, RP = 32 / L, R = 64 / RP;   // rows per warp-wide load; rows per lane
  static_assert(L == 4 || L == 8 || L == 16, "head dim 32, 64 or 128");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long blk = (long long)blockIdx.x * kStatsVecWarps + warp;   // (b, kvh, beta)
  if (blk >= (long long)batch * n_kv * nKb) return;
  const int beta = (int)(blk % nKb);
  const int bk = (int)(blk / nKb);               // b * n_kv + kvh
  const int b = bk / n_kv;
  const int Tk = seq_keys(k_lens, b, Tk_max);
  const long long j0 = (long long)beta * k_block;
  const int n = (int)max(0LL, min((long long)k_block, (long long)Tk - j0));   // n <= 64
  float* c_out = centroid + blk * D;
  const int col = 8 * (lane % L), r0 = lane / L;
  if (n == 0) {
    if (r0 == 0) {
      *reinterpret_cast<float4*>(c_out + col) = make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(c_out + col + 4) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (lane == 0) radius[blk] = 0.0f;
    return;
  }
  const __nv_bfloat16* kb = k + ((size_t)bk * Tk_max + j0) * D + col;
  uint4 x[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int r = r0 + RP * i;
    x[i] = r < n ? __ldg(reinterpret_cast<const uint4*>(kb + (size_t)r * D)) : make_uint4(0u, 0u, 0u, 0u);
  }
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < R; ++i) {                  // rows past n hold zeros: they add nothing
    float f[8];
    bf16x8_to_f32(x[i], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += f[e];
  }
#pragma unroll
  for (int o = L; o < 32; o <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
  const float inv_n = 1.0f / (float)n;
  float c[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) c[e] = acc[e] * inv_n;
  if (r0 == 0) {
    *reinterpret_cast<float4*>(c_out + col) = make_float4(c[0], c[1], c[2], c[3]);
    *reinterpret_cast<float4*>(c_out + col + 4) = make_float4(c[4], c[5], c[6], c[7]);
  }
  // The packed rows stay in registers; hide them from common-subexpression elimination so the
  // compiler converts them again here instead of keeping all R x 8 floats of the first pass.
#pragma unroll
  for (int i = 0; i < R; ++i) asm volatile("" : "+r"(x[i].x), "+r"(x[i].y), "+r"(x[i].z), "+r"(x[i].w));
  // squared distance of each of the lane's rows over its 8 dimensions
  float part[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    float f[8];
    bf16x8_to_f32(x[i], f);
    float a = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float d2 = f[e] - c[e];
      a = fmaf(d2, d2, a);
    }
    part[i] = a;
  }
  // Sum each row over its L lanes by a transposed butterfly: at the stage of lane bit o the
  // lane keeps the half of its rows selected by that bit and adds its partner's copy of them,
  // so after log2(L) stages each lane holds the full sums of R / L rows.  Stages run over lane
  // bits 1, 2, 4, ..., the order of a per-row shuffle tree, so every sum is the same.
  int cnt = R;
#pragma unroll
  for (int o = 1; o < L; o <<= 1) {
    const bool upper = (lane & o) != 0;
    cnt >>= 1;
#pragma unroll
    for (int i = 0; i < R / 2; ++i) {
      if (i < cnt) {
        const float send = upper ? part[i] : part[i + cnt];
        const float keep = upper ? part[i + cnt] : part[i];
        part[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
  }
  // the lane now holds rows idx + t, t < R / L: stage k (lane bit 2^k) chose the upper half of
  // a set of R / 2^k rows
  int idx = 0;
#pragma unroll
  for (int o = 1, w = 1; o < L; o <<= 1, w <<= 1) idx += ((lane & o) ? 1 : 0) * (R / (2 * w));
  float best = 0.0f;
#pragma unroll
  for (int t = 0; t < R / L; ++t)
    if (r0 + RP * (idx + t) < n) best = fmaxf(best, part[t]);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, o));
  if (lane == 0) radius[blk] = sqrtf(best);
}

}  // namespace ga
