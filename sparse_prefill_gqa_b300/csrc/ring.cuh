// ring.cuh -- append one token per sequence to a sliding-window ring cache.
//
// What it computes ("Attention in Code", section 2): a layer that only looks at the last W
// tokens keeps W slots per kv head; token number n (from 0) is written to slot n mod W, so
// once the cache is full the new token replaces the oldest one.  Attention over the ring
// (ga_attend_ring) then runs the split-K decode over the min(n, W) filled slots.
#pragma once

#include "common.cuh"

namespace ga {

constexpr int kRingThreads = 256;

// grid: (batch); block: kRingThreads.  One CTA per sequence reads the counter once, copies the
// new key and value of every kv head into the slot (16 bytes a thread and step), then bumps
// the counter after all copies of the CTA are issued.
__global__ void __launch_bounds__(kRingThreads)
ring_append_kernel(__nv_bfloat16* __restrict__ k_ring, __nv_bfloat16* __restrict__ v_ring,
                   const __nv_bfloat16* __restrict__ k_new, const __nv_bfloat16* __restrict__ v_new,
                   int32_t* __restrict__ n_seen, int n_kv, int d, int W) {
  const int b = blockIdx.x;
  const int n = n_seen[b];
  __syncthreads();                                  // every thread has read the counter
  if (n >= 0) {
    const int slot = n % W;
    const int per_head = d / 8;                     // 16-byte pieces of one row
    for (int e = threadIdx.x; e < n_kv * per_head; e += kRingThreads) {
      const int kvh = e / per_head, c = 8 * (e % per_head);
      const size_t src = ((size_t)b * n_kv + kvh) * d + c;
      const size_t dst = (((size_t)b * n_kv + kvh) * W + slot) * d + c;
      *reinterpret_cast<uint4*>(k_ring + dst) = *reinterpret_cast<const uint4*>(k_new + src);
      *reinterpret_cast<uint4*>(v_ring + dst) = *reinterpret_cast<const uint4*>(v_new + src);
    }
    __syncthreads();                                // the counter moves after every read of it
    if (threadIdx.x == 0) n_seen[b] = n + 1;
  }
}

}  // namespace ga
