// mla.cuh -- multi-head latent attention, absorbed form, for decode.
//
// What it computes ("Attention in Code", section 4): each cached token stores a latent c_kv (512
// numbers) and one rope key k_rope (64) shared by all heads; head h's key is c_kv w_uk[h] plus
// k_rope and its value c_kv w_uv[h].  The absorbed form never builds per-head keys or values:
//   q_lat = q_nope w_uk[h]^T                          (the query moved into latent space)
//   s_j   = (q_lat . c_kv_j + q_rope . k_rope_j) / sqrt(dn + dr)
//   o_lat = softmax(s) c_kv,   out = o_lat w_uv[h]   (expanded once per head)
// so every head reads the same 576 numbers per cached token.  Decode: one new token per
// sequence at position lens[b] - 1, which sees every cached token.
//
// Kernels: mla_absorb_kernel (q_lat, then q = [q_lat | q_rope] in bf16), mla_decode_kernel
// (split over token chunks; the heads are the 16 rows of mma.sync m16n8k16), mla_combine_kernel
// (log-sum-exp re-association of the chunks), mla_expand_kernel (o_lat w_uv).
#pragma once

#include "common.cuh"

namespace ga {

struct MlaCfg {
  static constexpr int R = 512, DR = 64, DN = 128, DV = 128;
  static constexpr int DK = R + DR;                     // 576 numbers per cached token
  static constexpr int SLABS = DK / 64;                 // 9 SW128 boxes of 64 columns
  static constexpr int TILE = 64;                       // tokens per stage
  static constexpr int STAGES = 2;
  static constexpr int STAGE_BYTES = TILE * DK * 2;     // 73728
  static constexpr int QROW = DK * 2 + 16;              // padded row of the query tile (bytes)
  static constexpr int PROW = TILE * 2 + 16;            // padded row of the P tile (bytes)
  static constexpr int OFF_Q = STAGES * STAGE_BYTES;
  static constexpr int OFF_P = OFF_Q + 16 * QROW;
  static constexpr int OFF_X = OFF_P + 16 * PROW;       // [4][16] float exchange
  static constexpr int OFF_BAR = OFF_X + 4 * 16 * 4;
  static constexpr int SMEM_BYTES = OFF_BAR + 64 + 1024;
  static constexpr int THREADS = 160;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

struct MlaShape {
  int batch, n_heads, L_max, chunk_len, n_chunks;
  const int32_t* lens;
  uint64_t timeout_ns;
};

// grid: (n_heads, batch); block: 256.  q[b, h] = [q_nope w_uk[h]^T (fp32 sums, rounded to bf16) |
// q_rope].  Warp w computes latent dims w, w + 8, ...: lanes split the 128 nope dims (4 each).
// One (sequence, head) per CTA: the grid's many warps hide the latency of the weight rows,
// which L2 serves to every sequence.
__global__ void __launch_bounds__(256)
mla_absorb_kernel(const __nv_bfloat16* __restrict__ q_nope, const __nv_bfloat16* __restrict__ q_rope,
                  const __nv_bfloat16* __restrict__ w_uk, __nv_bfloat16* __restrict__ q_abs, int n_heads) {
  using C = MlaCfg;
  const int h = blockIdx.x, b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row = (size_t)b * n_heads + h;
  float qn[4];
  {
    const __nv_bfloat16* src = q_nope + row * C::DN + 4 * lane;
#pragma unroll
    for (int e = 0; e < 4; ++e) qn[e] = __bfloat162float(src[e]);
  }
  __nv_bfloat16* dst = q_abs + row * C::DK;
  for (int c = warp; c < C::R; c += 8) {
    const __nv_bfloat16* w = w_uk + ((size_t)h * C::R + c) * C::DN + 4 * lane;
    float a = 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) a = fmaf(__bfloat162float(w[e]), qn[e], a);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (lane == 0) dst[c] = __float2bfloat16_rn(a);
  }
  for (int e = threadIdx.x; e < C::DR; e += 256) dst[C::R + e] = q_rope[row * C::DR + e];
}

struct MlaBars {
  uint64_t full[2], empty[2];
  int abort_flag;
};

// AND of `ok` over the 128 consumer threads (named barrier 1): every consumer warp takes the
// same branch, so a wait that gave up in one warp can never leave another at a barrier.
__device__ __forceinline__ bool consumers_all(bool ok) {
  uint32_t res;
  asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
               "bar.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
               : "=r"(res) : "r"(ok ? 1u : 0u) : "memory");
  return res != 0;
}

// grid: (n_chunks, batch); block: 160 -- warps 0-3 compute, warp 4 loads 64-token tiles of the
// latent cache [batch, L_max, 576] by TMA (9 boxes of 64 columns, 128-byte swizzle).
// Per tile: warp w scores its 16 tokens for the 16 query rows (the heads; rows >= n_heads are
// zero), the warps agree on each row's tile maximum through shared memory, write their
// probabilities into a shared 16 x 64 P tile, and each accumulates latent dims 128 w .. 128 w +
// 127 of P c_kv over all 64 tokens.
__global__ void __launch_bounds__(MlaCfg::THREADS, 1)
mla_decode_kernel(const __grid_constant__ CUtensorMap tm_lat, const __nv_bfloat16* __restrict__ q_abs,
                  float* __restrict__ ws_o, float* __restrict__ ws_ml, float* __restrict__ o_lat, MlaShape s) {
  using C = MlaCfg;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  MlaBars* bars = reinterpret_cast<MlaBars*>(smem + C::OFF_BAR);
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, b = blockIdx.y, H = s.n_heads;
  const int L = seq_keys(s.lens, b, s.L_max);
  const int kbeg = c * s.chunk_len, kend = min((c + 1) * s.chunk_len, L);
  if (kbeg >= kend) return;                          // chunk holds no token (uniform)
  const int n_tiles = (kend - kbeg + C::TILE - 1) / C::TILE;
  const uint64_t tmo = s.timeout_ns;

  if (threadIdx.x == 0) {
    for (int st = 0; st < C::STAGES; ++st) {
      mbar_init(&bars->full[st], 1);
      mbar_init(&bars->empty[st], 4);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp < 4) {                                    // query tile, zero rows past the heads
    for (int e = threadIdx.x; e < 16 * (C::DK / 8); e += 128) {
      const int r = e / (C::DK / 8), ch = e % (C::DK / 8);
      const uint4 v = r < H ? *reinterpret_cast<const uint4*>(q_abs + ((size_t)b * H + r) * C::DK + 8 * ch)
                            : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(smem + C::OFF_Q + r * C::QROW + ch * 16) = v;
    }
  }
  __syncthreads();

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_lat);
      int issued = 0;
      for (int it = 0; it < n_tiles; ++it) {
        const int st = it % C::STAGES, use = it / C::STAGES;
        if (it >= C::STAGES && !mbar_wait(&bars->empty[st], (use + 1) & 1, tmo, abort_flag)) break;
        unsigned char* dst = smem + st * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&bars->full[st], C::STAGE_BYTES);
        ++issued;
        const int key0 = kbeg + it * C::TILE;
        for (int sl = 0; sl < C::SLABS; ++sl)
          tma_load_3d(dst + sl * C::TILE * 128, &tm_lat, &bars->full[st], 64 * sl, key0, b);
      }
      for (int k = max(0, issued - C::STAGES); k < issued; ++k)
        mbar_wait(&bars->full[k % C::STAGES], (k / C::STAGES) & 1, tmo, nullptr);
    }
    __syncthreads();                                 // matches the consumers' one block barrier
    return;
  }

  // ---------------------------------------------------------------------- consumer warps
  const int r_lo = lane >> 2, r_hi = r_lo + 8;
  const float scale_log2 = kLog2e / sqrtf((float)(C::DN + C::DR));
  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.0f, 0.0f};
  const uint32_t sbase = smem_u32(smem);
  const uint32_t qs = sbase + C::OFF_Q, ps = sbase + C::OFF_P;
  float* xs = reinterpret_cast<float*>(smem + C::OFF_X);             // [4][16]
  const int mi = lane >> 3, rr = lane & 7;

  for (int it = 0; it < n_tiles; ++it) {
    const int st = it % C::STAGES;
    const bool got = warp_wait(&bars->full[st], (it / C::STAGES) & 1, tmo, abort_flag);
    if (!consumers_all(got)) break;
    const uint32_t kb = sbase + st * C::STAGE_BYTES;
    const int t0 = kbeg + it * C::TILE;                // first token of the tile
    // ---- scores of this warp's 16 tokens ------------------------------------------------
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int keyr = 16 * warp + ((mi >> 1) << 3) + rr;
#pragma unroll 4
      for (int kk = 0; kk < C::DK / 16; ++kk) {
        uint32_t a[4];
        ldmatrix_x4(qs + (lane & 15) * C::QROW + (kk * 16 + (lane >> 4) * 8) * 2, a[0], a[1], a[2], a[3]);
        const int dchunk = 2 * kk + (mi & 1);
        const uint32_t addr = kb + (dchunk >> 3) * (C::TILE * 128) + keyr * 128 + (((dchunk & 7) ^ (keyr & 7)) << 4);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(addr, b0, b1, b2, b3);
        mma_bf16_16816(sc[0], a, b0, b1);
        mma_bf16_16816(sc[1], a, b2, b3);
      }
    }
    float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = t0 + 16 * warp + 8 * n + 2 * (lane & 3) + (e & 1);
        sc[n][e] = j < kend ? sc[n][e] * scale_log2 : -INFINITY;
        mt[e >> 1] = fmaxf(mt[e >> 1], sc[n][e]);
      }
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      mt[row] = fmaxf(mt[row], __shfl_xor_sync(0xffffffffu, mt[row], 1));
      mt[row] = fmaxf(mt[row], __shfl_xor_sync(0xffffffffu, mt[row], 2));
    }
    if ((lane & 3) == 0) {
      xs[warp * 16 + r_lo] = mt[0];
      xs[warp * 16 + r_hi] = mt[1];
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    float alpha[2], m_use[2];
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      const int r = row ? r_hi : r_lo;
      const float tmax = fmaxf(fmaxf(xs[r], xs[16 + r]), fmaxf(xs[32 + r], xs[48 + r]));
      const float m_new = fmaxf(m_run[row], tmax);
      alpha[row] = m_new == -INFINITY ? 1.0f : ex2(m_run[row] - m_new);
      m_run[row] = m_new;
      m_use[row] = m_new == -INFINITY ? 0.0f : m_new;
      l_part[row] *= alpha[row];
    }
    unsigned char* pb = smem + C::OFF_P;
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        p[e] = ex2(sc[n][e] - m_use[e >> 1]);
        l_part[e >> 1] += p[e];
      }
      const int col = 16 * warp + 8 * n + 2 * (lane & 3);
      *reinterpret_cast<uint32_t*>(pb + r_lo * C::PROW + col * 2) = pack_bf16x2(p[0], p[1]);
      *reinterpret_cast<uint32_t*>(pb + r_hi * C::PROW + col * 2) = pack_bf16x2(p[2], p[3]);
    }
    if (alpha[0] != 1.0f || alpha[1] != 1.0f) {
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        o[n][0] *= alpha[0]; o[n][1] *= alpha[0];
        o[n][2] *= alpha[1]; o[n][3] *= alpha[1];
      }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");   // the P tile is complete
    // ---- o += P c_kv over the tile's 64 tokens, latent dims 128 warp .. -------------------
    const int lim = kend - t0;                        // first tile row past the end
    const bool tail = lim < C::TILE;
#pragma unroll
    for (int kk = 0; kk < C::TILE / 16; ++kk) {
      uint32_t pa[4];
      ldmatrix_x4(ps + (lane & 15) * C::PROW + (kk * 16 + (lane >> 4) * 8) * 2, pa[0], pa[1], pa[2], pa[3]);
      const int key = 16 * kk + ((mi & 1) << 3) + rr;
      const int kb0 = 16 * kk + 2 * (lane & 3);
#pragma unroll
      for (int n = 0; n < 16; n += 2) {
        const int dchunk = 16 * warp + n + (mi >> 1);
        const uint32_t addr = kb + (dchunk >> 3) * (C::TILE * 128) + key * 128 + (((dchunk & 7) ^ (key & 7)) << 4);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(addr, b0, b1, b2, b3);
        if (tail) {                                   // latent rows past the end may hold anything
          auto clip = [&](uint32_t x, int r0) -> uint32_t {
            const uint32_t lo16 = (r0 < lim) ? (x & 0xFFFFu) : 0u;
            const uint32_t hi16 = (r0 + 1 < lim) ? (x & 0xFFFF0000u) : 0u;
            return lo16 | hi16;
          };
          b0 = clip(b0, kb0); b1 = clip(b1, kb0 + 8);
          b2 = clip(b2, kb0); b3 = clip(b3, kb0 + 8);
        }
        mma_bf16_16816(o[n], pa, b0, b1);
        mma_bf16_16816(o[n + 1], pa, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->empty[st]);
  }
  // ---- row sums over the 4 warps' tokens, then this chunk's result ----------------------
#pragma unroll
  for (int row = 0; row < 2; ++row) {
    l_part[row] += __shfl_xor_sync(0xffffffffu, l_part[row], 1);
    l_part[row] += __shfl_xor_sync(0xffffffffu, l_part[row], 2);
  }
  if ((lane & 3) == 0) {
    xs[warp * 16 + r_lo] = l_part[0];
    xs[warp * 16 + r_hi] = l_part[1];
  }
  __syncthreads();
  if (*abort_flag != 0) return;
  float lsum[2];
#pragma unroll
  for (int row = 0; row < 2; ++row) {
    const int r = row ? r_hi : r_lo;
    lsum[row] = (xs[r] + xs[16 + r]) + (xs[32 + r] + xs[48 + r]);
  }
  const bool final_out = s.n_chunks == 1;
#pragma unroll
  for (int row = 0; row < 2; ++row) {
    const int h = row ? r_hi : r_lo;
    if (h >= H) continue;
    const size_t qrow = (size_t)b * H + h;
    const float inv = lsum[row] > 0.0f ? 1.0f / lsum[row] : 0.0f;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      const int dim = 128 * warp + 8 * n + 2 * (lane & 3);
      const float v0 = o[n][2 * row], v1 = o[n][2 * row + 1];
      if (final_out) {
        o_lat[qrow * C::R + dim] = v0 * inv;
        o_lat[qrow * C::R + dim + 1] = v1 * inv;
      } else {
        float* dst = ws_o + (qrow * s.n_chunks + c) * C::R + dim;
        dst[0] = v0;
        dst[1] = v1;
      }
    }
    if (!final_out && warp == 0 && (lane & 3) == 0) {
      ws_ml[(qrow * s.n_chunks + c) * 2 + 0] = m_run[row];
      ws_ml[(qrow * s.n_chunks + c) * 2 + 1] = lsum[row];
    }
  }
}

// grid: (n_heads, batch); block: 512 (one latent dim each).  o_lat = sum_c 2^(m_c - M) o_c /
// sum_c 2^(m_c - M) l_c over the chunks that hold tokens.
__global__ void __launch_bounds__(MlaCfg::R)
mla_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_ml, float* __restrict__ o_lat,
                   MlaShape s) {
  using C = MlaCfg;
  const int h = blockIdx.x, b = blockIdx.y, dim = threadIdx.x;
  const int L = seq_keys(s.lens, b, s.L_max);
  const size_t qrow = (size_t)b * s.n_heads + h;
  const int n_used = min(s.n_chunks, (L + s.chunk_len - 1) / s.chunk_len);
  float M = -INFINITY;
  for (int c = 0; c < n_used; ++c) M = fmaxf(M, ws_ml[(qrow * s.n_chunks + c) * 2]);
  float Lsum = 0.0f, O = 0.0f;
  if (M != -INFINITY) {
    for (int c = 0; c < n_used; ++c) {
      const float mc = ws_ml[(qrow * s.n_chunks + c) * 2];
      if (mc == -INFINITY) continue;
      const float f = ex2(mc - M);
      Lsum += f * ws_ml[(qrow * s.n_chunks + c) * 2 + 1];
      O += f * ws_o[(qrow * s.n_chunks + c) * C::R + dim];
    }
  }
  o_lat[qrow * C::R + dim] = Lsum > 0.0f ? O / Lsum : 0.0f;
}

// grid: (n_heads, batch); block: 128 (one output dim each).  out = o_lat w_uv[h] (fp32 sums).
__global__ void __launch_bounds__(MlaCfg::DV)
mla_expand_kernel(const float* __restrict__ o_lat, const __nv_bfloat16* __restrict__ w_uv,
                  __nv_bfloat16* __restrict__ out, int n_heads) {
  using C = MlaCfg;
  __shared__ float lat[C::R];
  const int h = blockIdx.x, b = blockIdx.y, e = threadIdx.x;
  const size_t qrow = (size_t)b * n_heads + h;
  for (int c = e; c < C::R; c += C::DV) lat[c] = o_lat[qrow * C::R + c];
  __syncthreads();
  const __nv_bfloat16* w = w_uv + (size_t)h * C::R * C::DV + e;
  float a = 0.0f;
  for (int c = 0; c < C::R; ++c) a = fmaf(lat[c], __bfloat162float(w[(size_t)c * C::DV]), a);
  out[qrow * C::DV + e] = __float2bfloat16_rn(a);
}

}  // namespace ga
