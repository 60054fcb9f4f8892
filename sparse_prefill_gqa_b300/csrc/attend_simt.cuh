// attend_simt.cuh -- attention on the CUDA cores, fp32 arithmetic throughout.
//
// Serves the fp32 storage mode (where tensor-core TF32 would miss an fp32 tolerance) and
// every shape the tensor-core kernels do not take (odd head dims, odd block sizes, tiny
// problems).  One warp per query row; keys are scored 32 at a time (one per lane), folded
// into a running max / running sum, and the lanes then accumulate the value rows over
// their share of the head dimension.
//
// What it computes ("Attention in Code", "one function all designs use"; section 1 for the
// head grouping; section 3 for the sink): for query row t of head h at absolute position
// i = Tk_b - Tq + t, the softmax over the allowed keys of q.k_j / sqrt(d), with a sink logit
// joining the normaliser, applied to the value rows of kv head h / (n_heads / n_kv).
#pragma once

#include "common.cuh"

namespace ga {

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

constexpr int kSimtWarps = 4;      // query rows per CTA
constexpr int kSimtMaxD = 256;

// grid: (ceil(Tq / kSimtWarps), n_heads, batch); block: 32 * kSimtWarps threads.
template <typename T>
__global__ void __launch_bounds__(32 * kSimtWarps)
attend_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   T* __restrict__ out, float* __restrict__ lse, AttnShape sh) {
  __shared__ float q_s[kSimtWarps][kSimtMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kSimtWarps + warp;
  const int h = blockIdx.y, b = blockIdx.z;
  if (t >= sh.Tq) return;
  const int d = sh.d;
  const int kvh = h / (sh.n_heads / sh.n_kv);
  const int Tk = seq_keys(sh.k_lens, b, sh.Tk_max);
  const long long i = (long long)Tk - sh.Tq + t;           // absolute position of row t
  const long long hi = sh.causal ? min((long long)Tk, i + 1) : (long long)Tk;  // exclusive
  const long long lo = sh.window > 0 ? max(0LL, i - sh.window + 1) : 0LL;

  const size_t row = ((size_t)b * sh.n_heads + h) * sh.Tq + t;
  const T* qr = q + row * d;
  const T* kb = k + ((size_t)b * sh.n_kv + kvh) * (size_t)sh.Tk_max * d;
  const T* vb = v + ((size_t)b * sh.n_kv + kvh) * (size_t)sh.Tk_max * d;
  const uint8_t* mrow = nullptr;
  if (sh.block_mask) {
    mrow = sh.block_mask + (((size_t)b * sh.n_heads + h) * sh.nQb + t / sh.q_block) * sh.nKb;
  }
  for (int c = lane; c < d; c += 32) q_s[warp][c] = to_f32(qr[c]);
  __syncwarp();

  const float scale = 1.0f / sqrtf((float)d);
  float m = -INFINITY, l = 0.0f;
  if (sh.sink) { m = sh.sink[h]; l = 1.0f; }
  float acc[kSimtMaxD / 32];
#pragma unroll
  for (int c = 0; c < kSimtMaxD / 32; ++c) acc[c] = 0.0f;

  for (long long j0 = lo; j0 < hi; j0 += 32) {
    const long long j = j0 + lane;
    bool ok = j < hi && (mrow == nullptr || mrow[j / sh.k_block] != 0);
    float s = -INFINITY;
    if (ok) {
      const T* kr = kb + (size_t)j * d;
      float dot = 0.0f;
      for (int c = 0; c < d; ++c) dot = fmaf(q_s[warp][c], to_f32(kr[c]), dot);
      s = dot * scale;
    }
    const float m_new = fmaxf(m, warp_max(s));
    if (m_new == -INFINITY) continue;                     // nothing allowed so far
    const float alpha = expf(m - m_new);                  // 0 when m was -inf
    const float p = ok ? expf(s - m_new) : 0.0f;
    l = l * alpha + warp_sum(p);
#pragma unroll
    for (int c = 0; c < kSimtMaxD / 32; ++c) acc[c] *= alpha;
    const int n = (int)min(32LL, hi - j0);
    for (int jj = 0; jj < n; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      if (pj == 0.0f) continue;                           // masked key: value never read
      const T* vr = vb + (size_t)(j0 + jj) * d;
#pragma unroll
      for (int c = 0; c < kSimtMaxD / 32; ++c) {
        const int dim = lane + 32 * c;
        if (dim < d) acc[c] = fmaf(pj, to_f32(vr[dim]), acc[c]);
      }
    }
    m = m_new;
  }

  const float inv = l > 0.0f ? 1.0f / l : 0.0f;
  T* orow = out + row * d;
#pragma unroll
  for (int c = 0; c < kSimtMaxD / 32; ++c) {
    const int dim = lane + 32 * c;
    if (dim < d) orow[dim] = from_f32<T>(acc[c] * inv);
  }
  if (lse && lane == 0) lse[row] = l > 0.0f ? m + logf(l) : -INFINITY;
}

}  // namespace ga
