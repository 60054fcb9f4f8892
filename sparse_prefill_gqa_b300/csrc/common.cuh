// common.cuh -- shapes passed to every attention kernel, and shared constants.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace ga {

// Everything an attention kernel needs to know about one ga_attend call.
// n / d for 0 <= n < 2^31 and 1 <= d < 2^31 by a multiply and a shift (the round-up method of
// Granlund and Montgomery, "Division by invariant integers using multiplication", 1994): with
// s = ceil(log2 d) and m = floor(2^32 (2^s - d) / d) + 1, n / d = (mulhi(n, m) + n) >> s, the
// sum staying below 2^32 because n < 2^31.
struct FastDiv {
  uint32_t m = 1;
  int s = 0;
  void init(uint32_t d) {
    s = 0;
    while ((1ull << s) < d) ++s;
    m = (uint32_t)((((1ull << 32) * ((1ull << s) - d)) / d) + 1);
  }
  __device__ __forceinline__ int div(int n) const { return (int)((__umulhi((uint32_t)n, m) + (uint32_t)n) >> s); }
};

struct AttnShape {
  int batch, n_heads, n_kv, d, Tq, Tk_max;
  const int32_t* k_lens;        // device [batch] or null
  int causal, window;
  const float* sink;            // device [n_heads] or null
  const uint8_t* block_mask;    // device [batch, n_heads, nQb, nKb] or null
  int q_block, k_block, nQb, nKb;
  uint64_t timeout_ns;          // limit for every device-side wait
  int item_qt_block;            // query tiles per block of the prefill item order (>= 1)
  // divisors of the prefill item decode: heads x batch, heads, query heads per kv head, kv
  // heads, items per block of query tiles, items per kv head in a full and in the last block
  FastDiv fd_hb, fd_h, fd_g, fd_nkv, fd_pb, fd_cg, fd_cgl;
};

constexpr float kLog2e = 1.4426950408889634f;

// Keys present in sequence b: k_lens[b] clamped to [0, Tk_max] (Tk_max when k_lens is null),
// so a bad length can shrink or empty a row but never move a read past the cache.
__device__ __forceinline__ int seq_keys(const int32_t* k_lens, int b, int Tk_max) {
  return k_lens ? min(max(k_lens[b], 0), Tk_max) : Tk_max;
}

// Widens 8 packed bf16 values (one 16-byte load) to fp32, exactly.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

}  // namespace ga
