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

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

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

// ---------------------------------------------------------------------------------------
// Block selection.  One CTA per (group of kSelQT query blocks, query head, sequence).
//   1. radius mean and population std over the kv head's key blocks, in fp64 (fixed tree,
//      so every CTA of the kv head gets identical values), and the rescue flags;
//   2. the mean query row of each query block (q read once, coalesced);
//   3. pass A: every visible (query block, key block) score q_mean . c / sqrt(d) in fp32,
//      reduced to the row maximum;
//   4. pass B: the same scores recomputed bit for bit, thresholded, OR-ed with the rescue
//      and diagonal flags, and written as the mask row (0 beyond the visible range).
// Scores are not stored, so the kernel takes any number of key blocks in little shared
// memory; the recomputation doubles a cost that is small next to the attention itself.
// ---------------------------------------------------------------------------------------
constexpr int kSelThreads = 256;
constexpr int kSelQT = 16;        // query blocks per CTA (2 per thread row group)
constexpr int kSelBT = 64;        // key blocks per centroid tile (2 per thread)

struct SelectShape {
  int batch, n_heads, n_kv, d, Tq, Tk, nKb_out, q_block, k_block, causal, window;
  int nQb, nKb;                   // query blocks, key blocks holding keys (ceil(Tk/k_block))
  float tau_mean, lambda_radius;
};

__device__ __forceinline__ bool block_visible(const SelectShape& s, int alpha, int beta) {
  if (!s.causal) return beta < s.nKb;
  const long long t0 = (long long)alpha * s.q_block;
  const long long t1 = min((long long)s.Tq, t0 + s.q_block);
  const long long i_first = (long long)s.Tk - s.Tq + t0, i_last = (long long)s.Tk - s.Tq + t1 - 1;
  const long long j_lo = (long long)beta * s.k_block;
  const long long j_hi = min(j_lo + s.k_block, (long long)s.Tk) - 1;
  if (beta >= s.nKb || j_lo > i_last) return false;
  if (s.window > 0 && j_hi <= i_first - s.window) return false;
  return true;
}

__device__ __forceinline__ bool block_diagonal(const SelectShape& s, int alpha, int beta) {
  const long long t0 = (long long)alpha * s.q_block;
  const long long t1 = min((long long)s.Tq, t0 + s.q_block);
  const long long i_first = (long long)s.Tk - s.Tq + t0, i_last = (long long)s.Tk - s.Tq + t1 - 1;
  const long long j_lo = (long long)beta * s.k_block;
  const long long j_hi = min(j_lo + s.k_block, (long long)s.Tk) - 1;
  return j_lo <= i_last && j_hi >= i_first;
}

template <int D4>   // padded row stride (floats) of the shared q_mean / centroid tiles
struct SelectSmem {
  float qm[kSelQT][D4];
  float ct[kSelBT][D4];
  double red[kSelThreads / 32];
  float rowmax[kSelQT];
  int nsel[kSelQT];
};

template <typename T>
__global__ void __launch_bounds__(kSelThreads)
select_blocks_kernel(const T* __restrict__ q, const float* __restrict__ centroid,
                     const float* __restrict__ radius, uint8_t* __restrict__ block_mask,
                     int32_t* __restrict__ n_selected, SelectShape s) {
  extern __shared__ __align__(16) unsigned char sel_smem_raw[];
  const int D4 = (s.d + 3) / 4 * 4 + 4;
  float* qm = reinterpret_cast<float*>(sel_smem_raw);                 // [kSelQT][D4]
  float* ct = qm + kSelQT * D4;                                       // [kSelBT][D4]
  double* red = reinterpret_cast<double*>(ct + kSelBT * D4);          // [kSelThreads/32]
  float* rowmax = reinterpret_cast<float*>(red + kSelThreads / 32);   // [kSelQT]
  int* nsel = reinterpret_cast<int*>(rowmax + kSelQT);                // [kSelQT]
  uint8_t* rescue = reinterpret_cast<uint8_t*>(nsel + kSelQT);        // [nKb]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int a0 = blockIdx.x * kSelQT, h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / (s.n_heads / s.n_kv);
  const int d = s.d;
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
  double part = 0.0;
  for (int x = tid; x < s.nKb; x += kSelThreads) part += (double)rrow[x];
  const double mu = block_sum(part) / s.nKb;
  part = 0.0;
  for (int x = tid; x < s.nKb; x += kSelThreads) {
    const double e = (double)rrow[x] - mu;
    part += e * e;
  }
  const double sigma = sqrt(block_sum(part) / s.nKb);
  for (int x = tid; x < s.nKb; x += kSelThreads) {
    rescue[x] = (sigma > 0.0 && ((double)rrow[x] - mu) / sigma >= (double)s.lambda_radius) ? 1 : 0;
  }

  // ---- 2. mean query row of each query block of this CTA --------------------------------
  const int vec_l = d / 8;                       // lanes per row for 16-byte bf16 loads
  if (sizeof(T) == 2 && d % 8 == 0 && 32 % vec_l == 0) {
    // 16-byte loads: lane l reads dims 8*(l % L) .. of rows l / L, l / L + 32/L, ... of the
    // warp's share; sums meet by shuffles, then across the 8 warps in shared memory
    const int rpw = 32 / vec_l;                  // rows per warp-wide load
    const int col = 8 * (lane % vec_l), r0 = lane / vec_l;
    for (int a = 0; a < kSelQT; ++a) {
      const int alpha = a0 + a;
      if (alpha >= s.nQb) break;
      const int t0 = alpha * s.q_block, t1 = min(s.Tq, t0 + s.q_block);
      const T* qb = q + (((size_t)b * s.n_heads + h) * s.Tq) * d + col;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int t = t0 + warp * rpw + r0; t < t1; t += (kSelThreads / 32) * rpw) {
        float f[8];
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(qb + (size_t)t * d)), f);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += f[i];
      }
      for (int o = vec_l; o < 32; o <<= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
      if (r0 == 0)
#pragma unroll
        for (int i = 0; i < 8; ++i) ct[warp * D4 + col + i] = acc[i];   // ct used as scratch here
      __syncthreads();
      for (int c = tid; c < d; c += kSelThreads) {
        float sum = 0.0f;
        for (int w = 0; w < kSelThreads / 32; ++w) sum += ct[w * D4 + c];
        qm[a * D4 + c] = sum / (float)(t1 - t0);
      }
      __syncthreads();
    }
  } else {
    const int groups = min(kSelBT, max(1, kSelThreads / d));
    const int gidx = tid / d, dim = tid % d;
    for (int a = 0; a < kSelQT; ++a) {
      const int alpha = a0 + a;
      if (alpha >= s.nQb) break;
      const int t0 = alpha * s.q_block, t1 = min(s.Tq, t0 + s.q_block);
      const T* qb = q + (((size_t)b * s.n_heads + h) * s.Tq) * d;
      for (int c = dim; c < d; c += (d > kSelThreads ? kSelThreads : d)) {
        float acc = 0.0f;
        if (gidx < groups)
          for (int t = t0 + gidx; t < t1; t += groups) acc += to_f32(qb[(size_t)t * d + c]);
        if (gidx < groups) ct[gidx * D4 + c] = acc;   // ct used as scratch here
      }
      __syncthreads();
      for (int c = tid; c < d; c += kSelThreads) {
        float acc = 0.0f;
        for (int g = 0; g < groups; ++g) acc += ct[g * D4 + c];
        qm[a * D4 + c] = acc / (float)(t1 - t0);
      }
      __syncthreads();
    }
  }
  // rowmax holds an order-preserving integer image of the float maximum during pass A
  for (int c = tid; c < kSelQT; c += kSelThreads) {
    reinterpret_cast<int*>(rowmax)[c] = INT_MIN;
    nsel[c] = 0;
  }
  if (tid < kSelQT) {
    for (int c = d; c < D4; ++c) qm[tid * D4 + c] = 0.0f;
  }

  // key-block range seen by any query block of the CTA
  const int a_last = min(s.nQb, a0 + kSelQT) - 1;
  int beta_hi = s.nKb;
  if (s.causal) {
    const long long t1 = min((long long)s.Tq, (long long)(a_last + 1) * s.q_block);
    const long long i_last = (long long)s.Tk - s.Tq + t1 - 1;
    beta_hi = (int)min((long long)s.nKb, i_last / s.k_block + 1);
  }
  int beta_lo = 0;
  if (s.causal && s.window > 0) {
    const long long i_first = (long long)s.Tk - s.Tq + (long long)a0 * s.q_block;
    beta_lo = (int)max(0LL, (i_first - s.window + 1) / s.k_block);
  }
  const float scale = 1.0f / sqrtf((float)d);
  // thread -> 2 query blocks x 2 key blocks of the tile
  const int ta = 2 * (tid / (kSelBT / 2));
  const int tb = 2 * (tid % (kSelBT / 2));

  for (int pass = 0; pass < 2; ++pass) {
    __syncthreads();
    for (int bt = beta_lo; bt < beta_hi; bt += kSelBT) {
      // stage centroid tile [kSelBT][d] (zero-padded) into shared memory
      for (int e = tid; e < kSelBT * D4; e += kSelThreads) {
        const int r = e / D4, c = e % D4;
        const int beta = bt + r;
        ct[e] = (beta < beta_hi && c < d) ? cbase[(size_t)beta * d + c] : 0.0f;
      }
      __syncthreads();
      float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      const float* q0 = qm + ta * D4;
      const float* q1 = qm + (ta + 1) * D4;
      const float* c0 = ct + tb * D4;
      const float* c1 = ct + (tb + 1) * D4;
      for (int c = 0; c < D4; c += 4) {
        const float4 x0 = *reinterpret_cast<const float4*>(q0 + c);
        const float4 x1 = *reinterpret_cast<const float4*>(q1 + c);
        const float4 y0 = *reinterpret_cast<const float4*>(c0 + c);
        const float4 y1 = *reinterpret_cast<const float4*>(c1 + c);
        acc[0][0] = __fmaf_rn(x0.x, y0.x, acc[0][0]); acc[0][0] = __fmaf_rn(x0.y, y0.y, acc[0][0]);
        acc[0][0] = __fmaf_rn(x0.z, y0.z, acc[0][0]); acc[0][0] = __fmaf_rn(x0.w, y0.w, acc[0][0]);
        acc[0][1] = __fmaf_rn(x0.x, y1.x, acc[0][1]); acc[0][1] = __fmaf_rn(x0.y, y1.y, acc[0][1]);
        acc[0][1] = __fmaf_rn(x0.z, y1.z, acc[0][1]); acc[0][1] = __fmaf_rn(x0.w, y1.w, acc[0][1]);
        acc[1][0] = __fmaf_rn(x1.x, y0.x, acc[1][0]); acc[1][0] = __fmaf_rn(x1.y, y0.y, acc[1][0]);
        acc[1][0] = __fmaf_rn(x1.z, y0.z, acc[1][0]); acc[1][0] = __fmaf_rn(x1.w, y0.w, acc[1][0]);
        acc[1][1] = __fmaf_rn(x1.x, y1.x, acc[1][1]); acc[1][1] = __fmaf_rn(x1.y, y1.y, acc[1][1]);
        acc[1][1] = __fmaf_rn(x1.z, y1.z, acc[1][1]); acc[1][1] = __fmaf_rn(x1.w, y1.w, acc[1][1]);
      }
#pragma unroll
      for (int ia = 0; ia < 2; ++ia) {
        const int alpha = a0 + ta + ia;
        if (alpha >= s.nQb) continue;
#pragma unroll
        for (int ib = 0; ib < 2; ++ib) {
          const int beta = bt + tb + ib;
          if (beta >= beta_hi || !block_visible(s, alpha, beta)) continue;
          const float score = __fmul_rn(acc[ia][ib], scale);
          if (pass == 0) {
            // scores are finite; order-preserving integer max on the float bits
            atomicMax(reinterpret_cast<int*>(&rowmax[ta + ia]),
                      __float_as_int(score) >= 0 ? __float_as_int(score) : (int)(0x80000000u ^ ~__float_as_uint(score)));
          } else {
            const bool keep = score >= rowmax[ta + ia] - s.tau_mean || rescue[beta] ||
                              block_diagonal(s, alpha, beta);
            block_mask[(((size_t)b * s.n_heads + h) * s.nQb + alpha) * s.nKb_out + beta] = keep;
            if (keep) atomicAdd(&nsel[ta + ia], 1);
          }
        }
      }
      __syncthreads();
    }
    if (pass == 0) {
      __syncthreads();
      if (tid < kSelQT) {   // decode the order-preserving integer back to the float
        const int x = reinterpret_cast<int*>(rowmax)[tid];
        rowmax[tid] = x >= 0 ? __int_as_float(x) : __uint_as_float(~((unsigned)x ^ 0x80000000u));
      }
    }
  }
  __syncthreads();
  // zero the rest of each mask row (invisible key blocks and blocks without keys)
  for (int a = 0; a < kSelQT; ++a) {
    const int alpha = a0 + a;
    if (alpha >= s.nQb) break;
    uint8_t* mrow = block_mask + (((size_t)b * s.n_heads + h) * s.nQb + alpha) * s.nKb_out;
    for (int beta = tid; beta < s.nKb_out; beta += kSelThreads) {
      if (beta < beta_lo || beta >= beta_hi || !block_visible(s, alpha, beta)) mrow[beta] = 0;
    }
    if (tid == 0 && n_selected) n_selected[((size_t)b * s.n_heads + h) * s.nQb + alpha] = nsel[a];
  }
}

}  // namespace ga
