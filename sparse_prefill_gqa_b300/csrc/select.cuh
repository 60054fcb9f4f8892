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
//   3. select_score_kernel    scores of 128 query blocks x 128 key blocks per CTA on the tensor
//                             cores (three TF32 products of split operands, fp32 accumulation),
//                             stored once; the row maxima by atomicMax
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
  int dp;                         // d rounded up to 32 (the operand rows' length, zero padded)
  float* q_hi;                    // workspace [batch, n_hp, nQb, dp]: mean query rows, high part
  float* q_lo;                    //   and the rest (q_hi + q_lo = the fp32 mean exactly)
  float* c_hi;                    // workspace [batch, n_kv, nKb, dp]: centroids, split the same way
  float* c_lo;
  uint64_t timeout_ns;            // limit of the score kernel's pipeline waits
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

// x = hi + lo exactly: hi keeps the sign, exponent and top 10 mantissa bits (a TF32 value), lo
// the remaining 13 bits (a TF32 value up to its last bit, which the split leaves below 2^-21 x).
__device__ __forceinline__ void tf32_split(float x, float& hi, float& lo) {
  hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
  lo = x - hi;
}

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
select_pool_kernel(const T* __restrict__ q, const float* __restrict__ radius,
                   const float* __restrict__ centroid, SelectShape s) {
  __shared__ float part[kPoolThreads / 32][kSimtMaxD];
  __shared__ float mean_s[kSimtMaxD];
  const int alpha = blockIdx.x, hp = blockIdx.y, b = blockIdx.z;
  griddep_launch_dependents();  // the next launch of the selection may start its set-up
  if (alpha == s.nQb) {         // the extra column: the z-score radius branch, beside the pooling
    if (s.radius_rule == 0 && hp < s.n_kv) rescue_zscore(radius, s, hp, b);
    return;
  }
  if (alpha > s.nQb) {          // further columns: 128 centroids of kv head hp, split for the scores
    if (hp >= s.n_kv) return;
    const int beta0 = (alpha - s.nQb - 1) * 128, nb = min(128, s.nKb - beta0);
    const float* src = centroid + (((size_t)b * s.n_kv + hp) * s.nKb_out + beta0) * s.d;
    const size_t o = (((size_t)b * s.n_kv + hp) * s.nKb + beta0) * s.dp;
    for (int e = threadIdx.x; e < nb * s.dp; e += kPoolThreads) {
      const int r = e / s.dp, c = e % s.dp;
      float hi, lo;
      tf32_split(c < s.d ? src[(size_t)r * s.d + c] : 0.0f, hi, lo);
      s.c_hi[o + e] = hi;
      s.c_lo[o + e] = lo;
    }
    return;
  }
  const int d = s.d, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = s.n_heads / s.n_kv;
  const int h0 = s.group_shared ? hp * g : hp, n_pool = s.group_shared ? g : 1;
  const int t0 = alpha * s.q_block, t1 = min(s.Tq, t0 + s.q_block);
  const float inv_n = 1.0f / (float)((t1 - t0) * n_pool);
  const size_t row = ((size_t)b * s.n_hp + hp) * s.nQb + alpha;
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
  for (int c = threadIdx.x; c < s.dp; c += kPoolThreads) {
    float hi, lo;
    tf32_split(c < d ? mean_s[c] : 0.0f, hi, lo);
    s.q_hi[row * s.dp + c] = hi;
    s.q_lo[row * s.dp + c] = lo;
  }
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
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x;
  griddep_wait();               // launched as a programmatic dependent of the pooling
  griddep_launch_dependents();
  const float* rrow = radius + ((size_t)b * s.n_kv + kvh) * s.nKb_out;
  uint8_t* out = s.rescue + ((size_t)b * s.n_kv + kvh) * s.nKb;
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
// 3. Scores.  128 x 128 tiles (128 query blocks x 128 key blocks of one pooled head and
// sequence) S = Q C^T on the tensor cores, a persistent CTA per SM walking every tile with a
// visible pair (tiles t = blockIdx.x, + gridDim.x, ... in (head, query tile, key tile) order).
// fp32 operands are split as x = hi + lo (tf32_split) and every product takes three TF32 MMAs,
// hi.hi + hi.lo + lo.hi, accumulated in fp32: the dropped lo.lo term and the TF32 reading of lo
// are below 2^-20 of each product, far inside the decision band, at five times the fp32 fused
// multiply-add rate.  The operands stream through a ring of two stages of 32 dimensions (four
// 16 KB TMA boxes: Q hi, Q lo, C hi, C lo; 128-byte swizzle); tile j of the CTA accumulates in
// tensor-memory buffer j % 2, so the loads and MMAs of the next tile overlap the epilogue of
// this one.
//   warp 0   TMA producer;
//   warp 1   MMA issuer (the whole warp, one elected lane issuing);
//   warps 2-5  epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31, i.e. its query
//            blocks' rows of S, scales them by 1/sqrt(d), takes each row's maximum over the
//            visible key blocks (atomicMax into the workspace), stages the rows in shared
//            memory and stores them as whole 512-byte row segments.
// ---------------------------------------------------------------------------------------
constexpr int kScThreads = 192;
constexpr int kScA = 128;            // query blocks per tile (MMA M)
constexpr int kScB = 128;            // key blocks per tile (MMA N)
constexpr int kScKC = 32;            // dimensions per stage: one 128-byte fp32 row
constexpr int kScBox = 128 * 128;    // bytes of one 128-row x 32-dim box
constexpr int kScStageBytes = 4 * kScBox;
constexpr int kScSS = kScB + 4;      // row stride (floats) of the staged scores [a][beta]
constexpr int kScOffSS = 2 * kScStageBytes;
constexpr int kScOffBar = kScOffSS + kScA * kScSS * 4;
constexpr int kScSmem = kScOffBar + 128 + 1024;

struct ScoreBars {
  uint64_t full[2], empty[2], acc_full[2], acc_empty[2], drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(ScoreBars) <= 128, "score barriers");

// Row stride of the stored scores: the key blocks rounded up to whole tiles.
__host__ __device__ inline int sel_score_stride(int nKb) { return (nKb + kScB - 1) / kScB * kScB; }

// Tiles of a launch (every pooled head and sequence) and whether tile t holds a visible pair:
// the rows' visible ranges are intervals moving right with the row, and consecutive rows'
// intervals touch, so their union is [vlo(first row), vhi(last row)).
__host__ __device__ inline long long sel_score_tiles(int batch, int n_hp, int nQb, int nKb) {
  return (long long)batch * n_hp * ((nQb + kScA - 1) / kScA) * ((nKb + kScB - 1) / kScB);
}
__device__ __forceinline__ bool sel_tile(const SelectShape& s, long long t, int& x, int& y, int& bh) {
  const int nx = (s.nKb + kScB - 1) / kScB, ny = (s.nQb + kScA - 1) / kScA;
  x = (int)(t % nx);
  y = (int)((t / nx) % ny);
  bh = (int)(t / ((long long)nx * ny));
  int vlo0, vhi0, vlo1, vhi1;
  sel_visible(s, y * kScA, vlo0, vhi0);
  sel_visible(s, min(s.nQb, (y + 1) * kScA) - 1, vlo1, vhi1);
  return vlo0 < (x + 1) * kScB && vhi1 > x * kScB;
}

// tm_qh, tm_ql: [1, batch * n_hp * nQb, dp] fp32; tm_ch, tm_cl: [1, batch * n_kv * nKb, dp] fp32;
// boxes of 32 x 128 with the 128-byte swizzle.  Rows past a head's last block belong to the next
// head (or read as zero past the end): their scores are never visible, stored past the row's
// blocks or kept.
__global__ void __launch_bounds__(kScThreads, 1)
select_score_kernel(const __grid_constant__ CUtensorMap tm_qh, const __grid_constant__ CUtensorMap tm_ql,
                    const __grid_constant__ CUtensorMap tm_ch, const __grid_constant__ CUtensorMap tm_cl,
                    SelectShape s) {
  extern __shared__ unsigned char sc_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(sc_raw) + 1023) & ~uintptr_t(1023));
  float* ss = reinterpret_cast<float*>(smem + kScOffSS);              // [A][SS]
  ScoreBars* bars = reinterpret_cast<ScoreBars*>(smem + kScOffBar);
  volatile int* abort_flag = &bars->abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = s.n_heads / s.n_kv;
  const uint64_t tmo = s.timeout_ns;
  const long long n_tiles = sel_score_tiles(s.batch, s.n_hp, s.nQb, s.nKb);
  const int n_ch = s.dp / kScKC;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
      mbar_init(&bars->acc_full[i], 1);
      mbar_init(&bars->acc_empty[i], 4);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&bars->tmem_base, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // Launched as a programmatic dependent of the pooling (or the MAD rescue): the set-up above ran
  // while it finished; its pooled rows, centroids and row maxima are read only from here on.
  griddep_wait();
  griddep_launch_dependents();  // the decisions may start their launch

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_qh);
      tma_prefetch_desc(&tm_ql);
      tma_prefetch_desc(&tm_ch);
      tma_prefetch_desc(&tm_cl);
      int q = 0;                                       // chunks issued over the CTA's tiles
      bool ok = true;
      for (long long t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        int x, y, bh;
        if (!sel_tile(s, t, x, y, bh)) continue;
        const int b = bh / s.n_hp, hp = bh % s.n_hp, kvh = s.group_shared ? hp : hp / g;
        const int qrow = bh * s.nQb + y * kScA, crow = (b * s.n_kv + kvh) * s.nKb + x * kScB;
        for (int k = 0; k < n_ch; ++k, ++q) {
          const int st = q & 1;
          if (q >= 2 && !(ok = mbar_wait(&bars->empty[st], ((q >> 1) - 1) & 1, tmo, abort_flag))) break;
          unsigned char* dst = smem + st * kScStageBytes;
          mbar_arrive_expect_tx(&bars->full[st], kScStageBytes);
          tma_load_3d(dst + 0 * kScBox, &tm_qh, &bars->full[st], kScKC * k, qrow, 0);
          tma_load_3d(dst + 1 * kScBox, &tm_ql, &bars->full[st], kScKC * k, qrow, 0);
          tma_load_3d(dst + 2 * kScBox, &tm_ch, &bars->full[st], kScKC * k, crow, 0);
          tma_load_3d(dst + 3 * kScBox, &tm_cl, &bars->full[st], kScKC * k, crow, 0);
        }
      }
      // every load issued has landed before the CTA may exit
      for (int k = max(0, q - 2); k < q; ++k) mbar_wait(&bars->full[k & 1], (k >> 1) & 1, tmo, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_tf32_f32(kScA, kScB);
    bool ok = true;
    int q = 0, j = 0;                                  // chunks consumed, tiles done
    for (long long t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
      int x, y, bh;
      if (!sel_tile(s, t, x, y, bh)) continue;
      const int acc = j & 1;
      // the epilogue has read this buffer's previous tile
      if (j >= 2 && !(ok = warp_wait(&bars->acc_empty[acc], ((j >> 1) - 1) & 1, tmo, abort_flag))) break;
      tc_fence_after();
      const uint32_t d = tmem + 128 * acc;
      for (int k = 0; k < n_ch; ++k, ++q) {
        const int st = q & 1;
        if (!(ok = warp_wait(&bars->full[st], (q >> 1) & 1, tmo, abort_flag))) break;
        tc_fence_after();
        const uint32_t base = smem_u32(smem + st * kScStageBytes);
        const uint64_t dqh = sdesc_sw128(base + 0 * kScBox, 16, 1024), dql = sdesc_sw128(base + 1 * kScBox, 16, 1024);
        const uint64_t dch = sdesc_sw128(base + 2 * kScBox, 16, 1024), dcl = sdesc_sw128(base + 3 * kScBox, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kScKC / 8; ++kk) {       // 4 steps of 8 dimensions (32 bytes)
          const uint64_t o = (uint64_t)((kk * 32) >> 4);
          umma_tf32_ss_elect(d, dqh + o, dch + o, idesc, (k > 0 || kk > 0) ? 1u : 0u);
          umma_tf32_ss_elect(d, dqh + o, dcl + o, idesc, 1u);
          umma_tf32_ss_elect(d, dql + o, dch + o, idesc, 1u);
        }
        umma_commit_elect(&bars->empty[st]);
      }
      if (!ok) break;
      umma_commit_elect(&bars->acc_full[acc]);
      ++j;
    }
    // every MMA issued has completed before tensor memory is released
    umma_commit_elect(&bars->drain);
    warp_wait(&bars->drain, 0, tmo, nullptr);
  } else {
    // ------------------------------------------------------------------ epilogue
    const int a = 32 * (warp & 3) + lane;                // query block of the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const float scale = 1.0f / sqrtf((float)s.d);
    const int stride = sel_score_stride(s.nKb);
    const int et = tid - 64;                              // 0 .. 127 over the epilogue warps
    int j = 0;
    for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x) {
      int x, y, bh;
      if (!sel_tile(s, t, x, y, bh)) continue;
      const int acc = j & 1;
      const bool ok = warp_wait(&bars->acc_full[acc], (j >> 1) & 1, tmo, abort_flag);
      // every epilogue warp takes the same branch
      uint32_t all;
      asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                   "bar.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                   : "=r"(all) : "r"(ok && *abort_flag == 0 ? 1u : 0u) : "memory");
      if (!all) break;
      tc_fence_after();
      const int a0 = y * kScA, beta0 = x * kScB;
      const int alpha = a0 + a;
      int vlo = 0, vhi = 0;
      if (alpha < s.nQb) sel_visible(s, alpha, vlo, vhi);
      float m = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < kScB; c += 32) {
        float v[32];
        tmem_ld32(tmem + 128 * acc + lane_off + c, v);
        tmem_wait_ld();
        if (c == kScB - 32) {                            // the accumulator is read: release it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->acc_empty[acc]);
        }
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          v[jj] = __fmul_rn(v[jj], scale);
          const int beta = beta0 + c + jj;
          if (beta >= vlo && beta < vhi) m = fmaxf(m, v[jj]);
        }
#pragma unroll
        for (int jj = 0; jj < 32; jj += 4)
          *reinterpret_cast<float4*>(ss + a * kScSS + c + jj) = make_float4(v[jj], v[jj + 1], v[jj + 2], v[jj + 3]);
      }
      const int n_rows = min(kScA, s.nQb - a0);
      const size_t row0 = (size_t)bh * s.nQb;
      if (a < n_rows && m > -INFINITY) atomicMax(&s.rowmax[row0 + a0 + a], f2ord(m));
      asm volatile("bar.sync 1, 128;" ::: "memory");       // the tile's rows are staged
      float* dst = s.scores + (row0 + a0) * stride + beta0;
      for (int e = et; e < n_rows * (kScB / 4); e += 128) {
        const int r = e / (kScB / 4), q4 = e % (kScB / 4);
        [[maybe_unused]] const size_t off = (row0 + a0 + r) * stride + beta0 + 4 * q4;
        if (GA_BOUNDS(off + 4 <= (size_t)s.batch * s.n_hp * s.nQb * stride, 7, off))
          *reinterpret_cast<float4*>(dst + (size_t)r * stride + 4 * q4) = *reinterpret_cast<const float4*>(ss + r * kScSS + 4 * q4);
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");       // staged rows read: the next tile may write
      ++j;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
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

__global__ void __launch_bounds__(32 * kDecWarps, 3)
select_decide_kernel(const float* __restrict__ radius, uint8_t* __restrict__ block_mask,
                     int32_t* __restrict__ n_selected, SelectShape s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();               // launched as a programmatic dependent of the score kernel
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
  // the rescue flags (and radii, for the bound branch) of a lane's four key blocks come with
  // its scores, as whole words, when the rows are word (16-byte) aligned
  const bool rvec = (s.nKb % 4) == 0 && (reinterpret_cast<uintptr_t>(resc) & 3) == 0;
  const bool bvec = bound && (s.nKb_out % 4) == 0 && (reinterpret_cast<uintptr_t>(rrow) & 15) == 0;
  uint8_t* mrow0 = block_mask + (((size_t)b * s.n_heads + h_out0) * s.nQb + alpha) * s.nKb_out;
  const size_t mhead = (size_t)s.nQb * s.nKb_out;       // next head's row
  // The row's invisible ends (before vlo, from vhi on: about half of a causal row) keep nothing:
  // when the rows are 16-byte aligned they are written as 16-byte words of zeros, and only the
  // 16-block-aligned span [gbeg, gend) around the visible blocks goes through the tests below.
  int gbeg = 0, gend = s.nKb_out;
  if ((s.nKb_out % 16) == 0 && (reinterpret_cast<uintptr_t>(mrow0) & 15) == 0) {
    gbeg = vlo / 16 * 16;
    gend = min(s.nKb_out, (vhi + 15) / 16 * 16);
    for (int o = 0; o < n_out; ++o) {
      uint8_t* mrow = mrow0 + o * mhead;
      for (int z = 16 * lane; z < s.nKb_out; z += 16 * 32) {
        if (z >= gbeg && z < gend) continue;
        [[maybe_unused]] const size_t zoff = (size_t)(mrow - block_mask) + z;
        if (GA_BOUNDS(zoff + 16 <= (size_t)s.batch * s.n_heads * s.nQb * s.nKb_out, 8, zoff))
          *reinterpret_cast<uint4*>(mrow + z) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  int kept = 0;
  for (int base = gbeg + 4 * lane; base < gend; base += 4 * 128) {
    float4 sv[4], rv[4];                            // four steps' scores (radii) in flight
    uint32_t fl[4];                                 // and rescue flags
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int beta0 = base + 128 * u;
      sv[u] = rv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      fl[u] = 0u;
      if (beta0 < gend && beta0 + 3 >= vlo && beta0 < vhi) {        // stored for every visible block
        sv[u] = *reinterpret_cast<const float4*>(srow + beta0);
        if (rvec) fl[u] = __ldg(reinterpret_cast<const uint32_t*>(resc + beta0));
        if (bvec) rv[u] = __ldg(reinterpret_cast<const float4*>(rrow + beta0));
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int beta0 = base + 128 * u;
      if (beta0 >= gend) break;
      // keep bytes (0 or 1 each) of key blocks beta0 .. beta0 + 3; groups wholly outside the
      // visible range keep nothing, wholly inside it and off the diagonal need no per-block
      // range tests, and the rescue flags are already bytes of 0 and 1
      uint32_t bytes = 0u;
      if (beta0 + 3 >= vlo && beta0 < vhi) {
        const float sa[4] = {sv[u].x, sv[u].y, sv[u].z, sv[u].w};
        uint32_t mean = 0u;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) mean |= (sa[jj] >= thr ? 1u : 0u) << (8 * jj);
        uint32_t resc4 = fl[u];
        if (!rvec) {
          resc4 = 0u;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
            if (beta0 + jj < s.nKb) resc4 |= (resc[beta0 + jj] != 0 ? 1u : 0u) << (8 * jj);
        }
        bytes = mean | resc4;
        const bool interior = beta0 >= vlo && beta0 + 3 < vhi && (beta0 + 3 < dlo || beta0 > dhi);
        if (!interior) {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int beta = beta0 + jj;
            const uint32_t bit = 1u << (8 * jj);
            if (beta >= dlo && beta <= dhi) bytes |= bit;
            if (beta < vlo || beta >= vhi) bytes &= ~bit;
          }
        }
        if (bound) {
          const float ra[4] = {rv[u].x, rv[u].y, rv[u].z, rv[u].w};
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int beta = beta0 + jj;
            const uint32_t bit = 1u << (8 * jj);
            if (!(bytes & bit) && beta >= vlo && beta < vhi &&
                __fmaf_rn(qn, __fmul_rn(bvec ? ra[jj] : rrow[beta], scale), sa[jj]) >= thr_b)
              bytes |= bit;
          }
        }
      }
      kept += __popc(bytes);
      for (int o = 0; o < n_out; ++o) {
        uint8_t* mrow = mrow0 + o * mhead;
        [[maybe_unused]] const size_t moff = (size_t)(mrow - block_mask) + beta0;
        if (!GA_BOUNDS(moff < (size_t)s.batch * s.n_heads * s.nQb * s.nKb_out, 8, moff)) continue;
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
