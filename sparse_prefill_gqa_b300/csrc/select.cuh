// select.cuh -- block selection for radius-bounded sparse prefill, in four launches.
//
// "RBS-Attention review" (patty.io): a query block scores each key block by the inner product
// of its (pooled) query with the key block's centroid -- the mean branch, kept when the score
// is close enough to the row's best; a key block whose maximum radius is unusually large
// against the radius distribution of its prompt and head is rescued -- the radius branch; the
// two thresholded masks are joined by a union.  Readings fixed here (the pages print no
// formula): the mean branch keeps s >= max_visible s - tau_mean, the radius branch is a z-score
// (or its median/MAD form) over the kv head's key blocks, the query block's own diagonal key
// blocks are always kept, and an optional bound branch keeps a block whose Cauchy-Schwarz bound
// (q_mean . c + |q_mean| r) / sqrt(d) reaches max_visible s - tau_bound.
//
//   1. select_pool_kernel     the mean query row of every query block (and its norm), q read
//                             once at the copy rate; each row maximum starts at -inf
//   2. select_rescue_kernel   per (sequence, kv head): the radius statistics in fp64 and the
//                             rescue flag of every key block, once
//   3. select_score_kernel    scores of 128 query blocks x 128 key blocks per CTA, fp32 fused
//                             multiply-adds in dimension order, stored once; the row maxima by
//                             atomicMax
//   4. select_decide_kernel   per row: the stored scores thresholded, OR-ed with rescue, diagonal
//                             and bound, written as the mask rows, and the per-row counts
// The pooled queries, row maxima, rescue flags and scores live in the caller's workspace.
#pragma once

#include "attend_simt.cuh"
#include "common.cuh"

namespace ga {

struct SelectShape {
  int batch, n_heads, n_kv, d, Tq, Tk, nKb_out, q_block, k_block, causal, window;
  int nQb, nKb;                   // query blocks, key blocks holding keys (ceil(Tk/k_block))
  float tau_mean, lambda_radius;
  int radius_rule;                // 0: z-score (mean, population std); 1: median and MAD
  int sort_len;                   // rule 1: power of two >= nKb (the sort buffer); else 0
  float tau_bound;                // bound branch threshold; -inf: no bound branch
  int group_shared;               // 1: one selection per kv head from the rows of its g heads
  int n_hp;                       // pooled rows: n_heads, or n_kv when group-shared
  float* qmean;                   // workspace [batch, n_hp, nQb, d]: mean query rows
  float* qnorm;                   // workspace [batch, n_hp, nQb]: their Euclidean norms
  int* rowmax;                    // workspace [batch, n_hp, nQb]: row maxima, order-preserving ints
  uint8_t* rescue;                // workspace [batch, n_kv, nKb]: radius-branch flags
  float* scores;                  // workspace [batch, n_hp, nQb, stride]: the mean-branch scores
};

// Bytes of each workspace part, 256-byte aligned.
__host__ __device__ inline size_t sel_up256(size_t x) { return (x + 255) / 256 * 256; }

// Float <-> int with the same order (NaN-free values), so that atomicMax on ints is a max on
// floats: non-negative floats keep their bits, negative ones have their 31 low bits flipped.
__device__ __forceinline__ int f2ord(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float ord2f(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7fffffff); }

// Key blocks query block alpha may see, [vlo, vhi): rows at absolute positions i_first .. i_last
// = Tk - Tq + those rows; with the causal rule the last visible block holds key i_last, with a
// window the first holds key i_first - W + 1.
__device__ __forceinline__ void sel_visible(const SelectShape& s, int alpha, int& vlo, int& vhi) {
  const long long t0 = (long long)alpha * s.q_block;
  const long long t1 = min((long long)s.Tq, t0 + s.q_block);
  const long long i_first = (long long)s.Tk - s.Tq + t0, i_last = (long long)s.Tk - s.Tq + t1 - 1;
  vhi = s.causal ? (int)min((long long)s.nKb, i_last / s.k_block + 1) : s.nKb;
  vlo = 0;
  if (s.causal && s.window > 0) {
    const long long x = i_first - s.window + 1;
    vlo = x <= 0 ? 0 : (int)(x / s.k_block);
  }
}

// Key blocks overlapping the query block's own positions [i_first, i_last]: [dlo, dhi].
__device__ __forceinline__ void sel_diagonal(const SelectShape& s, int alpha, int& dlo, int& dhi) {
  const long long t0 = (long long)alpha * s.q_block;
  const long long t1 = min((long long)s.Tq, t0 + s.q_block);
  const long long i_first = (long long)s.Tk - s.Tq + t0, i_last = (long long)s.Tk - s.Tq + t1 - 1;
  dlo = (int)(i_first / s.k_block);
  dhi = (int)min((long long)s.nKb - 1, i_last / s.k_block);
}

// ---------------------------------------------------------------------------------------
// 1. Pooling: one CTA per (query block, pooled head, sequence).  bf16 rows with d = 8 L
// (L = 1 .. 32): lane l reads 16 bytes (8 dims, 8 (l % L) ..) of rows l / L + k 32 / L, the
// four warps interleaved, every load in flight before the sums; the lanes of a column meet by
// shuffles, the warps in shared memory.  Other dtypes and head dims: one thread per dimension.
// ---------------------------------------------------------------------------------------
constexpr int kPoolThreads = 128;

__device__ void rescue_zscore(const float* __restrict__ radius, SelectShape s, int kvh, int b);

template <typename T>
__global__ void __launch_bounds__(kPoolThreads)
select_pool_kernel(const T* __restrict__ q, const float* __restrict__ radius, SelectShape s) {
  __shared__ float part[kPoolThreads / 32][kSimtMaxD];
  __shared__ float mean_s[kSimtMaxD];
  const int alpha = blockIdx.x, hp = blockIdx.y, b = blockIdx.z;
  if (alpha == s.nQb) {         // the extra column: the z-score radius branch, beside the pooling
    if (s.radius_rule == 0 && hp < s.n_kv) rescue_zscore(radius, s, hp, b);
    return;
  }
  const int d = s.d, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = s.n_heads / s.n_kv;
  const int h0 = s.group_shared ? hp * g : hp, n_pool = s.group_shared ? g : 1;
  const int t0 = alpha * s.q_block, t1 = min(s.Tq, t0 + s.q_block);
  const float inv_n = 1.0f / (float)((t1 - t0) * n_pool);
  const size_t row = ((size_t)b * s.n_hp + hp) * s.nQb + alpha;
  float* dst = s.qmean + row * d;
  if (sizeof(T) == 2 && d % 8 == 0 && 32 % (d / 8) == 0) {
    const int L = d / 8, RP = 32 / L;               // lanes per row, rows per warp step
    const int col = 8 * (lane % L), r0 = lane / L;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int p = 0; p < n_pool; ++p) {
      const T* qh = q + (((size_t)b * s.n_heads + h0 + p) * s.Tq) * d + col;
#pragma unroll 8
      for (int t = t0 + warp * RP + r0; t < t1; t += 4 * RP) {
        float f[8];
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(qh + (size_t)t * d)), f);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] += f[k];
      }
    }
    for (int o = L; o < 32; o <<= 1)
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
    if (r0 == 0)
#pragma unroll
      for (int k = 0; k < 8; ++k) part[warp][col + k] = acc[k];
    __syncthreads();
    for (int c = threadIdx.x; c < d; c += kPoolThreads)
      mean_s[c] = ((part[0][c] + part[1][c]) + (part[2][c] + part[3][c])) * inv_n;
  } else {
    for (int c = threadIdx.x; c < d; c += kPoolThreads) {
      float acc = 0.0f;
      for (int p = 0; p < n_pool; ++p) {
        const T* qh = q + (((size_t)b * s.n_heads + h0 + p) * s.Tq) * d + c;
        for (int t = t0; t < t1; ++t) acc += to_f32(qh[(size_t)t * d]);
      }
      mean_s[c] = acc * inv_n;
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < d; c += kPoolThreads) dst[c] = mean_s[c];
  if (threadIdx.x == 0) {
    float n2 = 0.0f;                                  // |q_mean| (bound branch)
    for (int c = 0; c < d; ++c) n2 = fmaf(mean_s[c], mean_s[c], n2);
    s.qnorm[row] = sqrtf(n2);
    s.rowmax[row] = f2ord(-INFINITY);
  }
}

// ---------------------------------------------------------------------------------------
// 2. Radius branch: one CTA per (kv head, sequence) -- extra CTAs of the pooling launch for the z
// rule (mean and population std of the kv head's radii in fp64, a fixed reduction tree), a launch
// of its own for the MAD rule (median and median absolute deviation by an exact fp64 bitonic sort
// in shared memory).  rescue = z >= lambda (nothing when the scale is zero).
// ---------------------------------------------------------------------------------------
constexpr int kRescueThreads = 512;

__device__ inline void rescue_sort(double* buf, int n) {     // ascending, n a power of two
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += kRescueThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const double a = buf[i], c = buf[ixj];
          if ((a > c) == ((i & k) == 0)) { buf[i] = c; buf[ixj] = a; }
        }
      }
      __syncthreads();
    }
  }
}

__device__ inline double sorted_median(const double* buf, int n) {
  return (n & 1) ? buf[n / 2] : (buf[n / 2 - 1] + buf[n / 2]) * 0.5;
}

// z rule by the CTA's threads (any multiple of 32 up to 1024): mean and population std of the kv
// head's radii in fp64 over a fixed reduction tree (strided per-thread sums, then the warps in
// order), and z >= lambda tested as r - mu >= lambda sigma (no fp64 division, which is slow here).
__device__ void rescue_zscore(const float* __restrict__ radius, SelectShape s, int kvh, int b) {
  __shared__ double zred[32];
  const int tid = threadIdx.x, nt = blockDim.x, warp = tid >> 5, lane = tid & 31, nw = nt >> 5;
  const float* rrow = radius + ((size_t)b * s.n_kv + kvh) * s.nKb_out;
  uint8_t* out = s.rescue + ((size_t)b * s.n_kv + kvh) * s.nKb;
  auto block_sum = [&](double x) -> double {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    __syncthreads();
    if (lane == 0) zred[warp] = x;
    __syncthreads();
    double tot = 0.0;
    for (int w = 0; w < nw; ++w) tot += zred[w];
    return tot;
  };
  double acc = 0.0;
  for (int x = tid; x < s.nKb; x += nt) acc += (double)rrow[x];
  const double mu = block_sum(acc) / s.nKb;
  acc = 0.0;
  for (int x = tid; x < s.nKb; x += nt) {
    const double e = (double)rrow[x] - mu;
    acc += e * e;
  }
  const double sigma = sqrt(block_sum(acc) / s.nKb);
  const double bar = (double)s.lambda_radius * sigma;
  for (int x = tid; x < s.nKb; x += nt) out[x] = (sigma > 0.0 && (double)rrow[x] - mu >= bar) ? 1 : 0;
}

// The MAD rule (the z rule runs inside the pooling launch).
__global__ void __launch_bounds__(kRescueThreads)
select_rescue_kernel(const float* __restrict__ radius, SelectShape s) {
  extern __shared__ double sortbuf[];                // rule 1: sort_len doubles
  __shared__ double red[kRescueThreads / 32];
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float* rrow = radius + ((size_t)b * s.n_kv + kvh) * s.nKb_out;
  uint8_t* out = s.rescue + ((size_t)b * s.n_kv + kvh) * s.nKb;
  auto block_sum = [&](double x) -> double {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    __syncthreads();
    if (lane == 0) red[warp] = x;
    __syncthreads();
    double tot = 0.0;
    for (int w = 0; w < kRescueThreads / 32; ++w) tot += red[w];
    return tot;
  };
  if (s.radius_rule == 0) {
    rescue_zscore(radius, s, kvh, b);
  } else {
    for (int x = tid; x < s.sort_len; x += kRescueThreads) sortbuf[x] = x < s.nKb ? (double)rrow[x] : INFINITY;
    __syncthreads();
    rescue_sort(sortbuf, s.sort_len);
    const double med = sorted_median(sortbuf, s.nKb);
    __syncthreads();
    for (int x = tid; x < s.sort_len; x += kRescueThreads)
      sortbuf[x] = x < s.nKb ? fabs((double)rrow[x] - med) : INFINITY;
    __syncthreads();
    rescue_sort(sortbuf, s.sort_len);
    const double mad = sorted_median(sortbuf, s.nKb);
    const double scale_r = 1.4826 * mad;   // consistency factor of the MAD for normal data
    const double bar = (double)s.lambda_radius * scale_r;
    for (int x = tid; x < s.nKb; x += kRescueThreads)
      out[x] = (mad > 0.0 && (double)rrow[x] - med >= bar) ? 1 : 0;
  }
}

// ---------------------------------------------------------------------------------------
// 3. Scores.  One CTA per (128 key blocks, 128 query blocks, pooled head x sequence), 8 warps,
// two CTAs per SM.  Lane l owns query blocks l, l + 32, l + 64, l + 96 of the tile, warp w key
// blocks 16 w .. 16 w + 15, so each dimension step is four conflict-free loads of query means
// (one per query block, consecutive across the lanes), four broadcast 16-byte loads of centroids,
// and 64 fused multiply-adds (32 packed instructions); the query means and centroids are staged
// 64 dimensions at a time, dimension-major.  Every score s = acc / sqrt(d) (fp32) is stored in the
// workspace through shared memory (whole 512-byte row segments) and the row maxima over the
// visible key blocks go to the workspace by atomicMax.  Tiles no query block of which sees a key
// block of the CTA's range store nothing.
// ---------------------------------------------------------------------------------------
constexpr int kScThreads = 256;
constexpr int kScA = 128;            // query blocks per CTA
constexpr int kScB = 128;            // key blocks per CTA
constexpr int kScDC = 64;            // dimensions staged at a time
constexpr int kScQS = kScA + 4;      // row stride (floats) of the staged query means [c][a]
constexpr int kScCS = kScB + 4;      // row stride (floats) of the staged centroids [c][beta]
constexpr int kScSS = kScB + 4;      // row stride (floats) of the staged scores [a][beta]
// shared memory: query means | centroids (the scores reuse both) | per-row ranges | warp maxima
constexpr int kScSmem = kScDC * (kScQS + kScCS) * 4 + kScA * 4 * 4 + (kScThreads / 32) * kScA * 4;
static_assert(kScA * kScSS <= kScDC * (kScQS + kScCS), "scores fit in the staging area");

// Row stride of the stored scores: the key blocks rounded up to whole CTA ranges.
__host__ __device__ inline int sel_score_stride(int nKb) { return (nKb + kScB - 1) / kScB * kScB; }

__global__ void __launch_bounds__(kScThreads, 2)
select_score_kernel(const float* __restrict__ centroid, SelectShape s) {
  extern __shared__ __align__(16) unsigned char sc_smem[];
  float* sq = reinterpret_cast<float*>(sc_smem);                       // [DC][QS]
  float* sc = sq + kScDC * kScQS;                                      // [DC][CS]
  float* ss = sq;                                                      // [A][SS] (after the dot products)
  int* rng = reinterpret_cast<int*>(sc + kScDC * kScCS);               // [A][2]: visible [vlo, vhi)
  int* wpart = rng + kScA * 4;                                         // [8][A]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int beta0 = blockIdx.x * kScB, a0 = blockIdx.y * kScA;
  const int b = blockIdx.z / s.n_hp, hp = blockIdx.z % s.n_hp;
  const int g = s.n_heads / s.n_kv;
  const int kvh = s.group_shared ? hp : hp / g;
  const int d = s.d;
  const size_t row0 = ((size_t)b * s.n_hp + hp) * s.nQb;             // first pooled row of (b, hp)

  for (int i = tid; i < kScA; i += kScThreads) {
    const int alpha = a0 + i;
    int vlo = 0, vhi = 0;
    if (alpha < s.nQb) sel_visible(s, alpha, vlo, vhi);
    rng[4 * i + 0] = vlo;
    rng[4 * i + 1] = vhi;
  }
  __syncthreads();
  // does any query block of the tile see a key block of this CTA's range?
  bool mine = false;
  for (int i = lane; i < kScA; i += 32) mine |= max(rng[4 * i], beta0) < min(rng[4 * i + 1], beta0 + kScB);
  if (__syncthreads_or(mine ? 1 : 0) == 0) return;

  float acc[4][16];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[i][j] = 0.0f;
  const float* cbase = centroid + ((size_t)b * s.n_kv + kvh) * (size_t)s.nKb_out * d;
  const float* qbase = s.qmean + row0 * d;
  for (int c0 = 0; c0 < d; c0 += kScDC) {
    const int dc = min(kScDC, d - c0);
    __syncthreads();
    // stage query means and centroids of dims c0 .. c0 + dc, dimension-major (zeros outside):
    // 16-byte loads along a row, the block index fastest across threads, so that the
    // transposed stores of a warp fall in consecutive banks
    if (d % 4 == 0) {
      for (int e = tid; e < kScA * (kScDC / 4); e += kScThreads) {
        const int a = e % kScA, c = 4 * (e / kScA);
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < dc && a0 + a < s.nQb) v = *reinterpret_cast<const float4*>(qbase + (size_t)(a0 + a) * d + c0 + c);
        sq[(c + 0) * kScQS + a] = v.x;
        sq[(c + 1) * kScQS + a] = v.y;
        sq[(c + 2) * kScQS + a] = v.z;
        sq[(c + 3) * kScQS + a] = v.w;
      }
      for (int e = tid; e < kScB * (kScDC / 4); e += kScThreads) {
        const int j = e % kScB, c = 4 * (e / kScB);
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < dc && beta0 + j < s.nKb) v = *reinterpret_cast<const float4*>(cbase + (size_t)(beta0 + j) * d + c0 + c);
        sc[(c + 0) * kScCS + j] = v.x;
        sc[(c + 1) * kScCS + j] = v.y;
        sc[(c + 2) * kScCS + j] = v.z;
        sc[(c + 3) * kScCS + j] = v.w;
      }
    } else {
      for (int e = tid; e < kScA * kScDC; e += kScThreads) {
        const int a = e % kScA, c = e / kScA;
        sq[c * kScQS + a] = (c < dc && a0 + a < s.nQb) ? qbase[(size_t)(a0 + a) * d + c0 + c] : 0.0f;
      }
      for (int e = tid; e < kScB * kScDC; e += kScThreads) {
        const int j = e % kScB, c = e / kScB;
        sc[c * kScCS + j] = (c < dc && beta0 + j < s.nKb) ? cbase[(size_t)(beta0 + j) * d + c0 + c] : 0.0f;
      }
    }
    __syncthreads();
    const float* qp = sq + lane;
    const float* cp = sc + 16 * warp;
#pragma unroll 2
    for (int c = 0; c < dc; ++c) {       // fused multiply-adds in dimension order, two per op
      float x[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = qp[c * kScQS + 32 * i];
      const float4 y0 = *reinterpret_cast<const float4*>(cp + c * kScCS);
      const float4 y1 = *reinterpret_cast<const float4*>(cp + c * kScCS + 4);
      const float4 y2 = *reinterpret_cast<const float4*>(cp + c * kScCS + 8);
      const float4 y3 = *reinterpret_cast<const float4*>(cp + c * kScCS + 12);
      const float ys[16] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w,
                            y2.x, y2.y, y2.z, y2.w, y3.x, y3.y, y3.z, y3.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 16; j += 2)
          ffma2(acc[i][j], acc[i][j + 1], ys[j], ys[j + 1], x[i], x[i], acc[i][j], acc[i][j + 1]);
    }
  }
  const float scale = 1.0f / sqrtf((float)d);
  __syncthreads();                                   // the staging area now holds the scores
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int a = lane + 32 * i;
    const int vlo = rng[4 * a], vhi = rng[4 * a + 1];
    float sv[16];
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      sv[j] = __fmul_rn(acc[i][j], scale);
      const int beta = beta0 + 16 * warp + j;
      if (beta >= vlo && beta < vhi) m = fmaxf(m, sv[j]);
    }
#pragma unroll
    for (int j = 0; j < 16; j += 4)
      *reinterpret_cast<float4*>(ss + a * kScSS + 16 * warp + j) = make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]);
    wpart[warp * kScA + a] = f2ord(m);
  }
  __syncthreads();
  const int n_rows = min(kScA, s.nQb - a0);
  const int stride = sel_score_stride(s.nKb);
  for (int a = tid; a < n_rows; a += kScThreads) {
    int m = wpart[a];
    for (int w = 1; w < kScThreads / 32; ++w) m = max(m, wpart[w * kScA + a]);
    if (m > f2ord(-INFINITY)) atomicMax(&s.rowmax[row0 + a0 + a], m);
  }
  float* dst = s.scores + (row0 + a0) * stride + beta0;
  for (int e = tid; e < n_rows * (kScB / 4); e += kScThreads) {
    const int a = e / (kScB / 4), q4 = e % (kScB / 4);
    *reinterpret_cast<float4*>(dst + (size_t)a * stride + 4 * q4) = *reinterpret_cast<const float4*>(ss + a * kScSS + 4 * q4);
  }
}

// ---------------------------------------------------------------------------------------
// 4. Decisions.  One warp per (query block, pooled head, sequence) row: keep = visible && (s >=
// max - tau_mean || rescue || diagonal || bound), read from the stored scores and written as
// the mask row of every head of the row (all g heads of the group when group-shared), with the
// row's count.  Lane l takes key blocks 4 l + 128 t .. + 3: 16-byte score loads, 4-byte mask
// stores where the row length allows.
// ---------------------------------------------------------------------------------------
constexpr int kDecWarps = 8;

__global__ void __launch_bounds__(32 * kDecWarps)
select_decide_kernel(const float* __restrict__ radius, uint8_t* __restrict__ block_mask,
                     int32_t* __restrict__ n_selected, SelectShape s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kDecWarps + warp;    // (b, hp, alpha)
  if (row >= (long long)s.batch * s.n_hp * s.nQb) return;
  const int alpha = (int)(row % s.nQb);
  const int bh = (int)(row / s.nQb), b = bh / s.n_hp, hp = bh % s.n_hp;
  const int g = s.n_heads / s.n_kv;
  const int kvh = s.group_shared ? hp : hp / g;
  const int h_out0 = s.group_shared ? hp * g : hp, n_out = s.group_shared ? g : 1;
  int vlo, vhi, dlo, dhi;
  sel_visible(s, alpha, vlo, vhi);
  sel_diagonal(s, alpha, dlo, dhi);
  const float rmax = ord2f(s.rowmax[row]);
  const float thr = rmax - s.tau_mean, thr_b = rmax - s.tau_bound, qn = s.qnorm[row];
  const bool bound = s.tau_bound != -INFINITY;
  const float scale = 1.0f / sqrtf((float)s.d);
  const float* srow = s.scores + (size_t)row * sel_score_stride(s.nKb);
  const float* rrow = radius + ((size_t)b * s.n_kv + kvh) * s.nKb_out;
  const uint8_t* resc = s.rescue + ((size_t)b * s.n_kv + kvh) * s.nKb;
  const bool vec4 = (s.nKb_out % 4) == 0 && (reinterpret_cast<uintptr_t>(block_mask) & 3) == 0;
  int kept = 0;
  for (int base = 4 * lane; base < s.nKb_out; base += 4 * 128) {
    float4 sv[4];                                   // four steps' scores in flight
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int beta0 = base + 128 * u;
      sv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (beta0 < s.nKb_out && beta0 + 3 >= vlo && beta0 < vhi)    // stored for every visible block
        sv[u] = *reinterpret_cast<const float4*>(srow + beta0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
    const int beta0 = base + 128 * u;
    if (beta0 >= s.nKb_out) break;
    uint32_t bytes = 0u;
    const float sa[4] = {sv[u].x, sv[u].y, sv[u].z, sv[u].w};
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int beta = beta0 + jj;
      const bool vis = beta >= vlo && beta < vhi;
      bool keep = vis && (sa[jj] >= thr || resc[beta] != 0 || (beta >= dlo && beta <= dhi));
      if (bound && vis && !keep) keep = __fmaf_rn(qn, __fmul_rn(rrow[beta], scale), sa[jj]) >= thr_b;
      bytes |= (keep ? 1u : 0u) << (8 * jj);
      kept += keep ? 1 : 0;
    }
    for (int o = 0; o < n_out; ++o) {
      uint8_t* mrow = block_mask + (((size_t)b * s.n_heads + h_out0 + o) * s.nQb + alpha) * s.nKb_out;
      if (vec4) {
        *reinterpret_cast<uint32_t*>(mrow + beta0) = bytes;
      } else {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
          if (beta0 + jj < s.nKb_out) mrow[beta0 + jj] = (uint8_t)((bytes >> (8 * jj)) & 1u);
      }
    }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kept += __shfl_xor_sync(0xffffffffu, kept, o);
  if (lane == 0 && n_selected)
    for (int o = 0; o < n_out; ++o) n_selected[((size_t)b * s.n_heads + h_out0 + o) * s.nQb + alpha] = kept;
}

}  // namespace ga
