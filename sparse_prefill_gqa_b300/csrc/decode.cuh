// decode.cuh -- split-K decode attention over a KV cache (bf16), and the log-sum-exp combine.
//
// What it computes: the same attention as the prefill kernels ("Attention in Code", "one
// function all designs use" and section 1), for a few query rows per kv head -- the
// token-by-token decode of the cached GQA layer, one new row at absolute position Tk_b - 1
// (or a few rows at Tk_b - Tq .. Tk_b - 1).  The sum over keys is split into chunks; each
// chunk yields a partial output with its own running max m_c and sum l_c, and the combine
// applies o = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c, an exact re-association.
//
// The work is bound by reading K and V once from HBM (every byte of a kv head serves all
// its g query heads).  One CTA per (key chunk, kv head, sequence):
//   warp 4   TMA producer: 64-key K and V tiles (128-byte swizzled) into a ring of stages (in the
//            gathered form, which reads the keys an index list names, the consumer warps load
//            their own rows instead);
//   warps 0-3  each takes 16 keys of every tile.  The rows of the MMA are the g * Tq query
//            rows of the kv head (padded to 16); scores and the value sum run on the tensor
//            cores through mma.sync m16n8k16 (a contraction of 16 x d x 16 per warp and tile,
//            so the instruction count stays far below the memory time), with the online
//            softmax on the accumulator fragments.  The 4 warps' partial states are merged
//            through shared memory at the end of the chunk.
#pragma once

#include "common.cuh"

namespace ga {

// 16-byte asynchronous copy global -> shared through L2 only, and its group bookkeeping.
__device__ __forceinline__ void cp_async_16(uint32_t smem_dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <int D>
struct DecodeCfg {
  static constexpr int TILE = 64;                       // keys per stage
  static constexpr int SLABS = D / 64;
  static constexpr int TILE_BYTES = TILE * D * 2;       // one K or V tile
  static constexpr int STAGES = D >= 256 ? 3 : (D >= 128 ? 4 : 8);
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int OFF_BAR = STAGES * STAGE_BYTES;
  static constexpr int MERGE_BYTES = 4 * 16 * D * 4 + 4 * 16 * 2 * 4;  // per-warp O, m, l
  static constexpr int BODY = OFF_BAR > MERGE_BYTES ? OFF_BAR : MERGE_BYTES;
  static constexpr int SMEM_BYTES = BODY + 256 + 1024;
  static constexpr int THREADS = 160;
  // gathered form: each warp keeps GSTAGES - 1 of its tiles in flight; then the barriers, then
  // the chunk's cache rows (at most kGatherMaxKeys).  Up to d = 128 two CTAs fit on an SM, so one
  // streams while the other starts or finishes.
  static constexpr int GSTAGES = D >= 128 ? 3 : 6;
  static constexpr int GBODY = GSTAGES * STAGE_BYTES > MERGE_BYTES ? GSTAGES * STAGE_BYTES : MERGE_BYTES;
  static constexpr int GATHER_SMEM_BYTES = GBODY + 256 + 4 * 1024 + 1024;
};

constexpr int kGatherMaxKeys = 1024;              // longest key chunk of the gathered form

struct DecodeBars {
  uint64_t full[8], empty[8];
  int abort_flag;
};

struct DecodeShape {
  AttnShape a;
  int chunk_len;        // keys per chunk (multiple of 64)
  int n_chunks;
  int rows;             // query rows per kv head: g * Tq (<= 16)
  int g;
  // Gathered form only: key j of sequence b is cache row gidx[b * gidx_stride + j] of its kv
  // head in gk / gv [batch, n_kv, cache_T, D] (the tensor maps are not used).
  const int32_t* gidx;
  int gidx_stride;
  int cache_T;
  const __nv_bfloat16* gk;
  const __nv_bfloat16* gv;
};

// Key range [lo, hi) that any row of sequence b may use, and the chunk's share of it.
__device__ __forceinline__ void decode_chunk_range(const DecodeShape& s, int Tk, int c, int& kbeg,
                                                   int& kend) {
  const int lo = s.a.window > 0 ? max(0, Tk - s.a.Tq - s.a.window + 1) : 0;
  kbeg = max(c * s.chunk_len, lo / 64 * 64);
  kend = min((c + 1) * s.chunk_len, Tk);
}

// grid: (n_chunks, n_kv, batch); block: 160 threads.
// GATHER = false: keys kbeg.. of the chunk are consecutive cache rows, loaded by the TMA producer
// warp (3-D maps, one box per slab).
// GATHER = true: the keys are the cache rows that s.gidx names.  Each consumer warp reads only its
// own 16 rows of every tile, so each loads them itself with 16-byte cp.async copies into the same
// swizzled layout, GSTAGES - 1 tiles ahead, and needs nothing but __syncwarp; the producer warp
// idles.  (Indexed TMA copies, tile::gather4, four 128-byte rows per copy issued by the producer
// warp, were measured at about 6 bytes per clock per SM on this workload, half the rate of these
// copies.)
template <int D, bool GATHER = false>
__global__ void __launch_bounds__(160, D >= 256 ? 1 : 2)
decode_splitk_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ out,
                     float* __restrict__ lse, float* __restrict__ ws_o, float* __restrict__ ws_ml,
                     DecodeShape s) {
  using C = DecodeCfg<D>;
  constexpr int NST = GATHER ? C::GSTAGES : C::STAGES;       // stages of the ring
  constexpr int BODY = GATHER ? C::GBODY : C::BODY;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DecodeBars* bars = reinterpret_cast<DecodeBars*>(smem + BODY);
  int* rows = reinterpret_cast<int*>(smem + BODY + 256);     // gathered form: the chunk's cache rows
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  // The gathered form is launched as a programmatic dependent of the top-k select (its index
  // lists): nothing is read before that kernel has completed.  Otherwise a no-op.
  griddep_wait();
  griddep_launch_dependents();                    // the combine may start its launch
  const int Tk = seq_keys(s.a.k_lens, b, s.a.Tk_max);
  int kbeg, kend;
  decode_chunk_range(s, Tk, c, kbeg, kend);
  if (kbeg >= kend) {                             // chunk holds no usable key (uniform)
    // Only an empty sequence (Tk = 0) leaves every chunk without keys.  With several chunks
    // the combine writes its rows; as the only chunk, this CTA does: no allowed key, so
    // out = 0 and lse = the sink's logit (or -inf).
    if (s.n_chunks == 1) {
      for (int e = threadIdx.x; e < s.rows * D; e += C::THREADS) {
        const int m = e / D, dim = e % D;
        const int hh = kvh * s.g + m % s.g;
        const size_t qrow = ((size_t)b * s.a.n_heads + hh) * s.a.Tq + m / s.g;
        if (GA_BOUNDS(qrow < (size_t)s.a.batch * s.a.n_heads * s.a.Tq && dim < D, 5, qrow)) out[qrow * D + dim] = __float2bfloat16_rn(0.0f);
        if (lse && dim == 0 && GA_BOUNDS(qrow < (size_t)s.a.batch * s.a.n_heads * s.a.Tq, 5, qrow)) lse[qrow] = s.a.sink ? s.a.sink[hh] : -INFINITY;
      }
    }
    return;
  }
  const int n_tiles = (kend - kbeg + C::TILE - 1) / C::TILE;
  const uint64_t tmo = s.a.timeout_ns;

  if constexpr (GATHER) {
    // The chunk's cache rows, once per CTA: rows past the chunk's end repeat its last key (the
    // consumers mask them), and an index outside the cache is clamped into it.  The host keeps
    // the chunk within kGatherMaxKeys keys.
    const long long row0 = (long long)(b * s.a.n_kv + kvh) * s.cache_T;
    const int32_t* gi = s.gidx + (size_t)b * s.gidx_stride + kbeg;
    const int n_keys = kend - kbeg;
    for (int j = threadIdx.x; j < n_tiles * C::TILE; j += C::THREADS) {
      const int t = __ldg(gi + min(j, n_keys - 1));
      rows[j] = (int)(row0 + min(max(t, 0), s.cache_T - 1));
    }
  }
  if (threadIdx.x == 0) {
    for (int st = 0; st < C::STAGES; ++st) {
      mbar_init(&bars->full[st], 1);
      mbar_init(&bars->empty[st], 4);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  __syncthreads();

  if (warp == 4 && GATHER) {                      // the consumers load their own rows
    __syncthreads();
    return;
  }
  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int kz = b * s.a.n_kv + kvh;
      int issued = 0;
      for (int it = 0; it < n_tiles; ++it) {
        const int st = it % C::STAGES, use = it / C::STAGES;
        if (it >= C::STAGES && !mbar_wait(&bars->empty[st], (use + 1) & 1, tmo, abort_flag)) break;
        unsigned char* dk = smem + st * C::STAGE_BYTES;
        unsigned char* dv = dk + C::TILE_BYTES;
        mbar_arrive_expect_tx(&bars->full[st], C::STAGE_BYTES);
        ++issued;
        const int key0 = kbeg + it * C::TILE;
        for (int sl = 0; sl < C::SLABS; ++sl) {
          tma_load_3d(dk + sl * C::TILE * 128, &tm_k, &bars->full[st], 64 * sl, key0, kz);
          tma_load_3d(dv + sl * C::TILE * 128, &tm_v, &bars->full[st], 64 * sl, key0, kz);
        }
      }
      for (int k = max(0, issued - C::STAGES); k < issued; ++k)
        mbar_wait(&bars->full[k % C::STAGES], (k / C::STAGES) & 1, tmo, nullptr);
    }
    __syncthreads();
    return;
  }

  // ---------------------------------------------------------------------- consumer warps
  // MMA row m (0..15) <-> (query row tq = m / g, query head kvh * g + m % g); rows >= s.rows pad.
  const int g = s.g;
  const int r_lo = lane >> 2, r_hi = r_lo + 8;
  const float scale_log2 = kLog2e / sqrtf((float)D);
  const long long pos0 = (long long)Tk - s.a.Tq;  // absolute position of query row 0
  auto row_q = [&](int m) -> const __nv_bfloat16* {
    const int tq = m / g, hh = kvh * g + m % g;
    return q + (((size_t)b * s.a.n_heads + hh) * s.a.Tq + tq) * D;
  };
  // A fragments of Q (rows r_lo / r_hi, dims 2*(lane%4) + {0,1} (+8)) for every 16-dim step
  uint32_t qa[D / 16][4];
  {
    const bool v_lo = r_lo < s.rows, v_hi = r_hi < s.rows;
    const __nv_bfloat16* q_lo = v_lo ? row_q(r_lo) : nullptr;
    const __nv_bfloat16* q_hi = v_hi ? row_q(r_hi) : nullptr;
    const int cc = 2 * (lane & 3);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][0] = v_lo ? *reinterpret_cast<const uint32_t*>(q_lo + 16 * kk + cc) : 0u;
      qa[kk][1] = v_hi ? *reinterpret_cast<const uint32_t*>(q_hi + 16 * kk + cc) : 0u;
      qa[kk][2] = v_lo ? *reinterpret_cast<const uint32_t*>(q_lo + 16 * kk + cc + 8) : 0u;
      qa[kk][3] = v_hi ? *reinterpret_cast<const uint32_t*>(q_hi + 16 * kk + cc + 8) : 0u;
    }
  }
  // causal / window limits per row (absolute key index must be in [lo, hi))
  int lo_r[2], hi_r[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int m = e ? r_hi : r_lo;
    if (m < s.rows) {
      const long long i = pos0 + m / g;
      hi_r[e] = s.a.causal ? (int)min((long long)Tk, i + 1) : Tk;
      lo_r[e] = s.a.window > 0 ? (int)max(0LL, i - s.a.window + 1) : 0;
    } else {
      hi_r[e] = 0; lo_r[e] = 0;                   // padding row: nothing allowed
    }
  }

  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_part[2] = {0.0f, 0.0f};                 // this lane's share of the row sums

  const uint32_t sbase = smem_u32(smem);
  // gathered form: copy this warp's 16 rows of tile t (K and V) into stage t % NST, as one group
  auto gather_rows = [&](int t) {
    if (t < n_tiles) {
      constexpr int CH = D / 8, LPR = CH < 32 ? CH : 32, RPP = 32 / LPR;   // 16-byte pieces per row
      const int pc = lane % LPR;
      const uint32_t kst = sbase + (t % NST) * C::STAGE_BYTES;
#pragma unroll
      for (int p = 0; p < 16 / RPP; ++p) {
        const int kt = 16 * warp + p * RPP + lane / LPR;                    // row of the tile
        const size_t src = (size_t)rows[t * C::TILE + kt] * D + 8 * pc;
        const uint32_t off = (pc >> 3) * (C::TILE * 128) + kt * 128 + (((pc & 7) ^ (kt & 7)) << 4);
        cp_async_16(kst + off, s.gk + src);
        cp_async_16(kst + C::TILE_BYTES + off, s.gv + src);
      }
    }
    cp_async_commit();                            // empty groups past the end keep the count
  };
  if constexpr (GATHER) {
#pragma unroll 1
    for (int t = 0; t < NST - 1; ++t) gather_rows(t);
  }
  for (int it = 0; it < n_tiles; ++it) {
    const int st = it % NST;
    if constexpr (GATHER) {
      gather_rows(it + NST - 1);                  // into the stage this warp finished last
      cp_async_wait<NST - 1>();                   // tile it has landed
      __syncwarp();
    } else {
      if (!warp_wait(&bars->full[st], (it / C::STAGES) & 1, tmo, abort_flag)) break;
    }
    const uint32_t kb = sbase + st * C::STAGE_BYTES;
    const uint32_t vb = kb + C::TILE_BYTES;
    const int key0 = kbeg + it * C::TILE + 16 * warp;   // this warp's 16 keys

    // ---- S = Q K^T for 16 keys (two n-tiles of 8) --------------------------------------
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int key = 16 * warp + ((mi >> 1) << 3) + rr;      // row of the K tile
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int dchunk = 2 * kk + (mi & 1);
        const uint32_t addr = kb + (dchunk >> 3) * (C::TILE * 128) + key * 128 +
                              (((dchunk & 7) ^ (key & 7)) << 4);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(addr, b0, b1, b2, b3);
        mma_bf16_16816(sc[0], qa[kk], b0, b1);
        mma_bf16_16816(sc[1], qa[kk], b2, b3);
      }
    }
    // ---- mask, online softmax (log2 domain) ----------------------------------------------
    float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = e >> 1;
        const int j = key0 + 8 * n + 2 * (lane & 3) + (e & 1);
        const bool ok = j >= lo_r[row] && j < hi_r[row] && j < kend;
        sc[n][e] = ok ? sc[n][e] * scale_log2 : -INFINITY;
        mt[row] = fmaxf(mt[row], sc[n][e]);
      }
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      mt[row] = fmaxf(mt[row], __shfl_xor_sync(0xffffffffu, mt[row], 1));
      mt[row] = fmaxf(mt[row], __shfl_xor_sync(0xffffffffu, mt[row], 2));
    }
    float alpha[2], m_use[2];
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      const float m_new = fmaxf(m_run[row], mt[row]);
      alpha[row] = m_new == -INFINITY ? 1.0f : ex2(m_run[row] - m_new);
      m_run[row] = m_new;
      m_use[row] = m_new == -INFINITY ? 0.0f : m_new;
      l_part[row] *= alpha[row];
    }
    uint32_t pa[4];
    {
      float p[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          p[n][e] = ex2(sc[n][e] - m_use[e >> 1]);
          l_part[e >> 1] += p[n][e];
        }
      pa[0] = pack_bf16x2(p[0][0], p[0][1]);
      pa[1] = pack_bf16x2(p[0][2], p[0][3]);
      pa[2] = pack_bf16x2(p[1][0], p[1][1]);
      pa[3] = pack_bf16x2(p[1][2], p[1][3]);
    }
    if (alpha[0] != 1.0f || alpha[1] != 1.0f) {
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= alpha[0]; o[n][1] *= alpha[0];
        o[n][2] *= alpha[1]; o[n][3] *= alpha[1];
      }
    }
    // ---- O += P V for the warp's 16 keys --------------------------------------------------
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int key = 16 * warp + ((mi & 1) << 3) + rr;       // row of the V tile
      // value rows at or past the sequence end may hold anything: zero their B elements
      const bool tail = key0 + 16 > kend;
      const int kb0 = 16 * warp + 2 * (lane & 3);             // tile rows of this lane's B pairs
      const int lim = kend - (kbeg + it * C::TILE);           // first tile row past the end
#pragma unroll
      for (int n = 0; n < D / 8; n += 2) {
        const int dchunk = n + (mi >> 1);
        const uint32_t addr = vb + (dchunk >> 3) * (C::TILE * 128) + key * 128 +
                              (((dchunk & 7) ^ (key & 7)) << 4);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(addr, b0, b1, b2, b3);
        if (tail) {
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
    if (!GATHER && lane == 0) mbar_arrive(&bars->empty[st]);
  }
  if constexpr (GATHER) cp_async_wait_all();
  // row sums of this warp
#pragma unroll
  for (int row = 0; row < 2; ++row) {
    l_part[row] += __shfl_xor_sync(0xffffffffu, l_part[row], 1);
    l_part[row] += __shfl_xor_sync(0xffffffffu, l_part[row], 2);
  }

  // ---- merge the 4 warps' partial states (stage buffers are free after the barrier) -------
  __syncthreads();
  const bool aborted = *abort_flag != 0;
  float* mo = reinterpret_cast<float*>(smem);               // [4][16][D]
  float* mml = mo + 4 * 16 * D;                             // [4][16][2]
  {
    const int cc = 2 * (lane & 3);
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      float* r0 = mo + ((warp * 16 + r_lo) * D) + 8 * n + cc;
      float* r1 = mo + ((warp * 16 + r_hi) * D) + 8 * n + cc;
      r0[0] = o[n][0]; r0[1] = o[n][1];
      r1[0] = o[n][2]; r1[1] = o[n][3];
    }
    if ((lane & 3) == 0) {
      mml[(warp * 16 + r_lo) * 2 + 0] = m_run[0];
      mml[(warp * 16 + r_lo) * 2 + 1] = l_part[0];
      mml[(warp * 16 + r_hi) * 2 + 0] = m_run[1];
      mml[(warp * 16 + r_hi) * 2 + 1] = l_part[1];
    }
  }
  asm volatile("bar.sync 1, 128;" ::: "memory");             // consumer warps only
  const bool final_out = s.n_chunks == 1;
  for (int e = threadIdx.x; e < s.rows * D; e += 128) {
    const int m = e / D, dim = e % D;
    if (aborted) {
      // A wait ran out (the status word says so): publish an empty chunk -- zero output, or a
      // partial with max -inf and sum 0 that the combine skips -- never what an earlier call
      // left in the workspace.
      const size_t qrow = ((size_t)b * s.a.n_heads + kvh * g + m % g) * s.a.Tq + m / g;
      if (final_out) {
        if (GA_BOUNDS(qrow < (size_t)s.a.batch * s.a.n_heads * s.a.Tq && dim < D, 5, qrow)) out[qrow * D + dim] = __float2bfloat16_rn(0.0f);
        if (lse && dim == 0 && GA_BOUNDS(qrow < (size_t)s.a.batch * s.a.n_heads * s.a.Tq, 5, qrow)) lse[qrow] = -INFINITY;
      } else {
        const size_t slot = qrow * s.n_chunks + c;
        if (GA_BOUNDS(slot < (size_t)s.a.batch * s.a.n_heads * s.a.Tq * s.n_chunks && dim < D, 4, slot)) ws_o[slot * D + dim] = 0.0f;
        if (dim == 0 && GA_BOUNDS(slot < (size_t)s.a.batch * s.a.n_heads * s.a.Tq * s.n_chunks, 4, slot)) {
          ws_ml[slot * 2 + 0] = -INFINITY;
          ws_ml[slot * 2 + 1] = 0.0f;
        }
      }
      continue;
    }
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, mml[(w * 16 + m) * 2]);
    float L = 0.0f, O = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float mw = mml[(w * 16 + m) * 2];
      const float f = mw == -INFINITY ? 0.0f : ex2(mw - M);
      L += f * mml[(w * 16 + m) * 2 + 1];
      O += f * mo[(w * 16 + m) * D + dim];
    }
    const int tq = m / g, hh = kvh * g + m % g;
    const size_t qrow = ((size_t)b * s.a.n_heads + hh) * s.a.Tq + tq;
    if (final_out) {
      float Mf = M, Lf = L;
      if (s.a.sink) {
        const float sk = s.a.sink[hh] * kLog2e;
        const float Mn = fmaxf(M, sk);
        Lf = (M == -INFINITY ? 0.0f : L * ex2(M - Mn)) + ex2(sk - Mn);
        O = M == -INFINITY ? 0.0f : O * ex2(M - Mn);
        Mf = Mn;
      }
      if (GA_BOUNDS(qrow < (size_t)s.a.batch * s.a.n_heads * s.a.Tq && dim < D, 5, qrow)) out[qrow * D + dim] = __float2bfloat16_rn(Lf > 0.0f ? O / Lf : 0.0f);
      if (lse && dim == 0 && GA_BOUNDS(qrow < (size_t)s.a.batch * s.a.n_heads * s.a.Tq, 5, qrow)) lse[qrow] = Lf > 0.0f ? (Mf + log2f(Lf)) * 0.6931471805599453f : -INFINITY;
    } else {
      const size_t slot = qrow * s.n_chunks + c;
      if (GA_BOUNDS(slot < (size_t)s.a.batch * s.a.n_heads * s.a.Tq * s.n_chunks && dim < D, 4, slot)) ws_o[slot * D + dim] = O;
      if (dim == 0 && GA_BOUNDS(slot < (size_t)s.a.batch * s.a.n_heads * s.a.Tq * s.n_chunks, 4, slot)) {
        ws_ml[slot * 2 + 0] = M;
        ws_ml[slot * 2 + 1] = L;
      }
    }
  }
}

// Combine the chunk partials of one (b, h, query row).  grid: (Tq, n_heads, batch), D threads.
// Launched as a programmatic dependent of the decode kernel: its CTAs may become resident while
// the decode's last CTAs run, and read nothing before the decode grid has completed.
template <int D>
__global__ void __launch_bounds__(D)
decode_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_ml,
                      __nv_bfloat16* __restrict__ out, float* __restrict__ lse, DecodeShape s) {
  const int tq = blockIdx.x, hh = blockIdx.y, b = blockIdx.z;
  const int dim = threadIdx.x;
  griddep_wait();                                 // the partials of the decode kernel
  const int Tk = seq_keys(s.a.k_lens, b, s.a.Tk_max);
  const size_t qrow = ((size_t)b * s.a.n_heads + hh) * s.a.Tq + tq;
  float M = -INFINITY;
  for (int c = 0; c < s.n_chunks; ++c) {
    int kbeg, kend;
    decode_chunk_range(s, Tk, c, kbeg, kend);
    if (kbeg >= kend) continue;
    M = fmaxf(M, ws_ml[(qrow * s.n_chunks + c) * 2]);
  }
  float Mf = M;
  if (s.a.sink) Mf = fmaxf(M, s.a.sink[hh] * kLog2e);
  float L = 0.0f, O = 0.0f;
  if (Mf != -INFINITY) {
    for (int c = 0; c < s.n_chunks; ++c) {
      int kbeg, kend;
      decode_chunk_range(s, Tk, c, kbeg, kend);
      if (kbeg >= kend) continue;
      const size_t slot = qrow * s.n_chunks + c;
      const float mc = ws_ml[slot * 2];
      if (mc == -INFINITY) continue;
      const float f = ex2(mc - Mf);
      L += f * ws_ml[slot * 2 + 1];
      O += f * ws_o[slot * D + dim];
    }
    if (s.a.sink) L += ex2(s.a.sink[hh] * kLog2e - Mf);
  }
  if (GA_BOUNDS(qrow < (size_t)s.a.batch * s.a.n_heads * s.a.Tq && dim < D, 5, qrow)) out[qrow * D + dim] = __float2bfloat16_rn(L > 0.0f ? O / L : 0.0f);
  if (lse && dim == 0 && GA_BOUNDS(qrow < (size_t)s.a.batch * s.a.n_heads * s.a.Tq, 5, qrow)) lse[qrow] = L > 0.0f ? (Mf + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

}  // namespace ga
