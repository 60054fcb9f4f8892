// blocks.cuh -- block statistics and block selection for radius-bounded sparse prefill.
//
// "RBS-Attention review" (patty.io): keys are grouped into blocks represented by their
// centroid; a block's maximum radius is the distance from the centroid to its farthest
// key; a query block scores a key block by its inner product with the centroid (mean
// branch); blocks whose radius is unusually large against the radius distribution of that
// prompt and head are rescued (radius branch); the two thresholded masks are joined by a
// union.  Both kernels are memory-bound reductions on the CUDA cores.
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

// ---------------------------------------------------------------------------------------
// Block selection.  One CTA per (kSelQT query blocks, query head, sequence), 8 warps.
//   1. radius mean and population std over the kv head's key blocks, in fp64 (fixed tree,
//      so every CTA of the kv head gets identical values), and the rescue flags;
//   2. the mean query row of each query block (q read once, 16-byte loads), stored
//      dimension-major: qmt[c][a];
//   3. per query block, the visible key-block range [vlo, vhi) and the diagonal range;
//   4. pass A: the scores q_mean . c / sqrt(d) of tiles of kSelBT key blocks (centroids
//      staged dimension-major, ctt[c][beta]); warp w owns query blocks 4w .. 4w+3 and lane
//      l key blocks 4l .. 4l+3 of the tile, so each step is one broadcast 16-byte load of
//      four query means and one 16-byte load of four centroids for 16 FMAs; the row
//      maximum over visible blocks needs no atomics (one warp owns the row);
//   5. pass B: the same scores recomputed bit for bit (same operations, same order),
//      thresholded, OR-ed with the rescue and diagonal flags, written as the mask row.
// Scores are not stored, so any number of key blocks fits in a fixed amount of shared
// memory; the recomputation doubles a cost that is small next to the attention itself.
// ---------------------------------------------------------------------------------------
constexpr int kSelThreads = 256;
constexpr int kSelQT = 32;        // query blocks per CTA (4 per warp)
constexpr int kSelBT = 128;       // key blocks per centroid tile (4 per lane)
constexpr int kSelQS = kSelQT + 4;   // row stride (floats) of qmt
constexpr int kSelCS = kSelBT + 4;   // row stride (floats) of ctt

struct SelectShape {
  int batch, n_heads, n_kv, d, Tq, Tk, nKb_out, q_block, k_block, causal, window;
  int nQb, nKb;                   // query blocks, key blocks holding keys (ceil(Tk/k_block))
  float tau_mean, lambda_radius;
  int radius_rule;                // 0: z-score (mean, population std); 1: median and MAD
  int sort_len;                   // rule 1: power of two >= nKb (the sort buffer); else 0
  float tau_bound;                // bound branch threshold; -inf: no bound branch
  int group_shared;               // 1: one selection per kv head (grid over kv heads), from the
                                  // query rows of its g heads pooled; every head gets the mask
};

// shared memory: qmt [d][kSelQS] | ctt [d][kSelCS] | red [8] double | sortbuf [sort_len] double
// | rowmax [QT] | qnrm [QT] | nsel [QT] | ranges [QT][4] | rescue [nKb]
__host__ __device__ inline size_t select_smem_bytes(int d, int nKb, int sort_len) {
  return (size_t)d * (kSelQS + kSelCS) * 4 + (kSelThreads / 32) * 8 + (size_t)sort_len * 8 +
         kSelQT * 4 * 7 + (size_t)nKb + 16;
}

// Ascending bitonic sort of buf[0, n) (n a power of two) by the CTA's kSelThreads threads.
__device__ inline void select_sort(double* buf, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += kSelThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const double a = buf[i], b = buf[ixj];
          if ((a > b) == ((i & k) == 0)) { buf[i] = b; buf[ixj] = a; }
        }
      }
      __syncthreads();
    }
  }
}

// Median of a sorted buf[0, n): the middle value, or the mean of the two middle values.
__device__ inline double sorted_median(const double* buf, int n) {
  return (n & 1) ? buf[n / 2] : (buf[n / 2 - 1] + buf[n / 2]) * 0.5;
}

template <typename T>
__global__ void __launch_bounds__(kSelThreads)
select_blocks_kernel(const T* __restrict__ q, const float* __restrict__ centroid,
                     const float* __restrict__ radius, uint8_t* __restrict__ block_mask,
                     int32_t* __restrict__ n_selected, SelectShape s) {
  extern __shared__ __align__(16) unsigned char sel_smem_raw[];
  const int d = s.d;
  float* qmt = reinterpret_cast<float*>(sel_smem_raw);                 // [d][kSelQS]
  float* ctt = qmt + (size_t)d * kSelQS;                               // [d][kSelCS]
  double* red = reinterpret_cast<double*>(ctt + (size_t)d * kSelCS);   // [8]
  double* sortbuf = red + kSelThreads / 32;                            // [sort_len]
  float* rowmax = reinterpret_cast<float*>(sortbuf + s.sort_len);      // [QT]
  float* qnrm = rowmax + kSelQT;                                       // [QT]
  int* nsel = reinterpret_cast<int*>(qnrm + kSelQT);                   // [QT]
  int* rng = nsel + kSelQT;                                            // [QT][4]
  uint8_t* rescue = reinterpret_cast<uint8_t*>(rng + 4 * kSelQT);      // [nKb]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int a0 = blockIdx.x * kSelQT, b = blockIdx.z;
  const int g = s.n_heads / s.n_kv;
  // group-shared: blockIdx.y is the kv head and the pooled heads are its g query heads
  const int h = s.group_shared ? blockIdx.y * g : blockIdx.y;        // first head of the CTA
  const int n_pool = s.group_shared ? g : 1;                         // heads pooled and written
  const int kvh = h / g;
  const float* rrow = radius + ((size_t)b * s.n_kv + kvh) * s.nKb_out;
  const float* cbase = centroid + ((size_t)b * s.n_kv + kvh) * (size_t)s.nKb_out * d;

  // ---- 1. radius distribution of (b, kvh): mean, population std, rescue flags ----------
  auto block_sum = [&](double x) -> double {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    __syncthreads();
    if (lane == 0) red[warp] = x;
    __syncthreads();
    double tot = 0.0;
    for (int w = 0; w < kSelThreads / 32; ++w) tot += red[w];
    return tot;
  };
  if (s.radius_rule == 0) {
    double part = 0.0;
    for (int x = tid; x < s.nKb; x += kSelThreads) part += (double)rrow[x];
    const double mu = block_sum(part) / s.nKb;
    part = 0.0;
    for (int x = tid; x < s.nKb; x += kSelThreads) {
      const double e = (double)rrow[x] - mu;
      part += e * e;
    }
    const double sigma = sqrt(block_sum(part) / s.nKb);
    for (int x = tid; x < s.nKb; x += kSelThreads)
      rescue[x] = (sigma > 0.0 && ((double)rrow[x] - mu) / sigma >= (double)s.lambda_radius) ? 1 : 0;
  } else {
    // robust form: (r - median) / (1.4826 MAD), median and MAD by sorting (fp64, exact)
    for (int x = tid; x < s.sort_len; x += kSelThreads) sortbuf[x] = x < s.nKb ? (double)rrow[x] : INFINITY;
    __syncthreads();
    select_sort(sortbuf, s.sort_len);
    const double med = sorted_median(sortbuf, s.nKb);
    __syncthreads();
    for (int x = tid; x < s.sort_len; x += kSelThreads)
      sortbuf[x] = x < s.nKb ? fabs((double)rrow[x] - med) : INFINITY;
    __syncthreads();
    select_sort(sortbuf, s.sort_len);
    const double mad = sorted_median(sortbuf, s.nKb);
    const double scale_r = 1.4826 * mad;   // consistency factor of the MAD for normal data
    for (int x = tid; x < s.nKb; x += kSelThreads)
      rescue[x] = (mad > 0.0 && ((double)rrow[x] - med) / scale_r >= (double)s.lambda_radius) ? 1 : 0;
  }

  // ---- 2. mean query row of each query block of this CTA -> qmt[c][a] --------------------
  // Warp w pools query blocks 4w .. 4w+3 on its own (no CTA-wide barrier between blocks).
  const int vec_l = d / 8;
  for (int i = 0; i < 4; ++i) {
    const int a = 4 * warp + i, alpha = a0 + a;
    if (alpha >= s.nQb) {                                             // padding rows: zeros
      for (int c = lane; c < d; c += 32) qmt[c * kSelQS + a] = 0.0f;
      continue;
    }
    const int t0 = alpha * s.q_block, t1 = min(s.Tq, t0 + s.q_block);
    const float inv_n = 1.0f / (float)((t1 - t0) * n_pool);
    const T* qb = q + (((size_t)b * s.n_heads + h) * s.Tq) * d;
    if (sizeof(T) == 2 && d % 8 == 0 && 32 % vec_l == 0) {
      // 16-byte loads: lane l reads dims 8*(l % L) .. of rows l / L, l / L + 32/L, ...
      const int rpw = 32 / vec_l, col = 8 * (lane % vec_l), r0 = lane / vec_l;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int hp = 0; hp < n_pool; ++hp) {                         // the pooled heads' rows
        const T* qh = qb + (size_t)hp * s.Tq * d;
#pragma unroll 8
        for (int t = t0 + r0; t < t1; t += rpw) {
          float f[8];
          bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(qh + (size_t)t * d + col)), f);
#pragma unroll
          for (int k = 0; k < 8; ++k) acc[k] += f[k];
        }
      }
      for (int o = vec_l; o < 32; o <<= 1)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
      if (r0 == 0)
#pragma unroll
        for (int k = 0; k < 8; ++k) qmt[(col + k) * kSelQS + a] = acc[k] * inv_n;
    } else {
      for (int c = lane; c < d; c += 32) {
        float acc = 0.0f;
        for (int hp = 0; hp < n_pool; ++hp)
          for (int t = t0; t < t1; ++t) acc += to_f32(qb[((size_t)hp * s.Tq + t) * d + c]);
        qmt[c * kSelQS + a] = acc * inv_n;
      }
    }
  }
  __syncthreads();

  // ---- 3. visible and diagonal key-block ranges of each query block ----------------------
  if (tid < kSelQT) {
    const int alpha = a0 + tid;
    int vlo = 0, vhi = 0, dlo = 1, dhi = 0;                            // empty by default
    if (alpha < s.nQb) {
      const long long t0 = (long long)alpha * s.q_block;
      const long long t1 = min((long long)s.Tq, t0 + s.q_block);
      const long long i_first = (long long)s.Tk - s.Tq + t0, i_last = (long long)s.Tk - s.Tq + t1 - 1;
      vhi = s.causal ? (int)min((long long)s.nKb, i_last / s.k_block + 1) : s.nKb;
      if (s.causal && s.window > 0) {
        const long long x = i_first - s.window + 1;                    // first key a row may see
        vlo = x <= 0 ? 0 : (int)(x / s.k_block);
      }
      dlo = (int)(i_first / s.k_block);
      dhi = (int)min((long long)s.nKb - 1, i_last / s.k_block);
    }
    rng[4 * tid + 0] = vlo; rng[4 * tid + 1] = vhi; rng[4 * tid + 2] = dlo; rng[4 * tid + 3] = dhi;
    rowmax[tid] = -INFINITY;
    nsel[tid] = 0;
    float n2 = 0.0f;                                                   // |q_mean| of the block
    for (int c = 0; c < d; ++c) n2 = fmaf(qmt[c * kSelQS + tid], qmt[c * kSelQS + tid], n2);
    qnrm[tid] = sqrtf(n2);
  }
  __syncthreads();
  int beta_lo = s.nKb, beta_hi = 0;                                   // union over the CTA
  for (int a = 0; a < kSelQT; ++a) {
    if (rng[4 * a + 1] > rng[4 * a]) {
      beta_lo = min(beta_lo, rng[4 * a]);
      beta_hi = max(beta_hi, rng[4 * a + 1]);
    }
  }
  if (beta_hi <= beta_lo) beta_lo = beta_hi = 0;
  int my_vlo[4], my_vhi[4], my_dlo[4], my_dhi[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int a = 4 * warp + i;
    my_vlo[i] = rng[4 * a]; my_vhi[i] = rng[4 * a + 1]; my_dlo[i] = rng[4 * a + 2]; my_dhi[i] = rng[4 * a + 3];
  }
  const float scale = 1.0f / sqrtf((float)d);
  const bool vec_mask = (s.nKb_out % 4) == 0 && (reinterpret_cast<uintptr_t>(block_mask) & 3) == 0;

  for (int pass = 0; pass < 2; ++pass) {
    for (int bt = beta_lo; bt < beta_hi; bt += kSelBT) {
      // stage centroids of key blocks bt .. bt+127 dimension-major (zeros past beta_hi)
      __syncthreads();
      if (d % 4 == 0) {                                               // rows are 16-byte aligned
        for (int e = tid; e < kSelBT * (d / 4); e += kSelThreads) {
          const int r = e % kSelBT, c4 = e / kSelBT;
          const int beta = bt + r;
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (beta < beta_hi) v = *reinterpret_cast<const float4*>(cbase + (size_t)beta * d + 4 * c4);
          ctt[(4 * c4 + 0) * kSelCS + r] = v.x;
          ctt[(4 * c4 + 1) * kSelCS + r] = v.y;
          ctt[(4 * c4 + 2) * kSelCS + r] = v.z;
          ctt[(4 * c4 + 3) * kSelCS + r] = v.w;
        }
      } else {
        for (int e = tid; e < kSelBT * d; e += kSelThreads) {
          const int r = e % kSelBT, c = e / kSelBT;
          const int beta = bt + r;
          ctt[c * kSelCS + r] = beta < beta_hi ? cbase[(size_t)beta * d + c] : 0.0f;
        }
      }
      __syncthreads();
      float acc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc[i][jj] = 0.0f;
      const float* qp = qmt + 4 * warp;
      const float* cp = ctt + 4 * lane;
#pragma unroll 4
      for (int c = 0; c < d; ++c) {       // fused multiply-adds in dimension order, two per op
        const float4 x = *reinterpret_cast<const float4*>(qp + c * kSelQS);
        const float4 y = *reinterpret_cast<const float4*>(cp + c * kSelCS);
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ffma2(acc[i][0], acc[i][1], y.x, y.y, xs[i], xs[i], acc[i][0], acc[i][1]);
          ffma2(acc[i][2], acc[i][3], y.z, y.w, xs[i], xs[i], acc[i][2], acc[i][3]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int a = 4 * warp + i, alpha = a0 + a;
        if (alpha >= s.nQb) continue;                                  // warp-uniform
        if (pass == 0) {
          float m = -INFINITY;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int beta = bt + 4 * lane + jj;
            if (beta >= my_vlo[i] && beta < my_vhi[i]) m = fmaxf(m, __fmul_rn(acc[i][jj], scale));
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (lane == 0) rowmax[a] = fmaxf(rowmax[a], m);
        } else {
          const float thr = rowmax[a] - s.tau_mean;
          // bound branch: (q_mean . c + |q_mean| r) / sqrt(d) >= best mean score - tau_bound
          const bool bound = s.tau_bound != -INFINITY;
          const float thr_b = rowmax[a] - s.tau_bound, qn = qnrm[a];
          uint32_t bytes = 0u;
          int kept = 0;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int beta = bt + 4 * lane + jj;
            const bool vis = beta >= my_vlo[i] && beta < my_vhi[i];
            const float sc = __fmul_rn(acc[i][jj], scale);
            bool keep = vis && (sc >= thr || rescue[beta] != 0 || (beta >= my_dlo[i] && beta <= my_dhi[i]));
            if (bound && vis && !keep) keep = __fmaf_rn(qn, __fmul_rn(rrow[beta], scale), sc) >= thr_b;
            bytes |= (keep ? 1u : 0u) << (8 * jj);
            kept += keep ? 1 : 0;
          }
          const int beta0 = bt + 4 * lane;
          for (int hp = 0; hp < n_pool; ++hp) {                       // every head of the CTA
            uint8_t* mrow = block_mask + (((size_t)b * s.n_heads + h + hp) * s.nQb + alpha) * s.nKb_out;
            if (vec_mask && beta0 + 3 < s.nKb_out) {
              *reinterpret_cast<uint32_t*>(mrow + beta0) = bytes;
            } else {
#pragma unroll
              for (int jj = 0; jj < 4; ++jj)
                if (beta0 + jj < s.nKb_out) mrow[beta0 + jj] = (uint8_t)((bytes >> (8 * jj)) & 1u);
            }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) kept += __shfl_xor_sync(0xffffffffu, kept, o);
          if (lane == 0) nsel[a] += kept;
        }
      }
    }
    __syncthreads();
  }
  // zero the rest of each mask row (key blocks outside the CTA's tiles)
  const int tiles_end = beta_lo + ((beta_hi - beta_lo + kSelBT - 1) / kSelBT) * kSelBT;
  for (int a = 0; a < kSelQT; ++a) {
    const int alpha = a0 + a;
    if (alpha >= s.nQb) break;
    for (int hp = 0; hp < n_pool; ++hp) {
      uint8_t* mrow = block_mask + (((size_t)b * s.n_heads + h + hp) * s.nQb + alpha) * s.nKb_out;
      for (int beta = tid; beta < s.nKb_out; beta += kSelThreads)
        if (beta < beta_lo || beta >= tiles_end) mrow[beta] = 0;
      if (tid == 0 && n_selected) n_selected[((size_t)b * s.n_heads + h + hp) * s.nQb + alpha] = nsel[a];
    }
  }
}

}  // namespace ga
