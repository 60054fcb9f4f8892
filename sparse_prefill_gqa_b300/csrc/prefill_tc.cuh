// prefill_tc.cuh -- bf16 attention prefill on the 5th-generation tensor cores (tcgen05).
//
// What it computes: "Attention in Code", "one function all designs use" (scores q.k/sqrt(d),
// masked positions removed, optional sink logit in the normaliser, weighted sum of values),
// with the grouped-query mapping of section 1 and the absolute-position causal rule; and,
// with a block mask, the block-sparse execution of the "RBS-Attention review" section on
// regular block sparsity: key blocks outside the mask are never loaded nor multiplied.
//
// One CTA per (128-row query tile, query head, sequence).  Warp roles:
//   warp 4  TMA producer: Q once, then K and V tiles (64-key halves) into a 2-stage ring;
//   warp 5  MMA issuer (lane 0): S = Q K^T into one of two TMEM score buffers, and
//           O += P V into the TMEM output accumulator; completions signalled by
//           tcgen05.commit on mbarriers;
//   warps 0-3  softmax: thread r owns query row r = TMEM lane r, so the row max and the row
//           sum need no shuffles.  Each tile: tcgen05.ld the S row, mask from indices,
//           online softmax in the log2 domain, P (bf16) written to shared memory in the
//           128-byte-swizzled K-major layout the MMA reads.  The running output is rescaled
//           in TMEM only when the running max grows by more than 2^8 (exponents stay <= 8,
//           so P <= 256 never overflows), which is rare after the first tiles.
// Key tiles that the causal rule, the window, the sequence length or the block mask leave
// empty are skipped before any load; within a tile, an unselected 64-key half is neither
// loaded nor multiplied.
//
// Shared memory (bytes, D=128/BN=128 | D=256/BN=64): Q 32K|64K, K 2x32K|2x32K,
// V 2x32K|2x32K, P 32K|16K.  TMEM: O in columns [0, D), S buffers at D and D + BN.
#pragma once

#include "common.cuh"

namespace ga {

template <int D_, int BN_>
struct PrefillCfg {
  static constexpr int D = D_;
  static constexpr int BN = BN_;
  static constexpr int BM = 128;
  static constexpr int SLABS = D / 64;            // 64-column slabs of 128-byte rows
  static constexpr int HALVES = BN / 64;
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int P_BYTES = BM * BN * 2;
  static constexpr int STAGES = 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_P = OFF_V + STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;   // + alignment slack
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 192;
  static_assert(D + 2 * BN <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct PrefillBars {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], s_free[2], p_full;
  uint64_t o_done, mma_drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Per-CTA view of the key range and tile mask of one (b, h, query tile).
struct TileRange {
  int key_lo, key_hi;          // union over valid rows of the allowed key range [lo, hi)
  int kt_lo, kt_hi;            // tile index range (tiles of BN keys)
  int t0, rows;                // first query row of the tile, number of valid rows
  long long i_first, i_last;   // absolute positions of the first and last valid rows
  int Tk;                      // keys present in this sequence
  const uint8_t* mrow;         // block-mask row for this query tile, or null
};

template <int BN>
__device__ __forceinline__ uint32_t tile_half_mask(const TileRange& r, const AttnShape& sh, int j) {
  uint32_t hm = 0;
#pragma unroll
  for (int hf = 0; hf < BN / 64; ++hf) {
    const int k0 = j * BN + 64 * hf;
    if (k0 >= r.key_hi || k0 + 64 <= r.key_lo) continue;
    if (r.mrow && r.mrow[k0 / sh.k_block] == 0) continue;
    hm |= 1u << hf;
  }
  return hm;
}

template <int BN>
__device__ __forceinline__ int next_tile(const TileRange& r, const AttnShape& sh, int j) {
  for (++j; j < r.kt_hi; ++j)
    if (tile_half_mask<BN>(r, sh, j)) return j;
  return r.kt_hi;
}

template <int D, int BN>
__global__ void __launch_bounds__(192, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ out,
                  float* __restrict__ lse, AttnShape sh) {
  using C = PrefillCfg<D, BN>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sQ = smem + C::OFF_Q;
  unsigned char* sK = smem + C::OFF_K;
  unsigned char* sV = smem + C::OFF_V;
  unsigned char* sP = smem + C::OFF_P;
  PrefillBars* bars = reinterpret_cast<PrefillBars*>(smem + C::OFF_BAR);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = (sh.Tq + C::BM - 1) / C::BM;
  const int qt = n_qt - 1 - (int)blockIdx.x;            // heaviest causal tiles first
  const int h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / (sh.n_heads / sh.n_kv);
  const uint64_t tmo = sh.timeout_ns;

  TileRange r;
  r.Tk = seq_keys(sh.k_lens, b, sh.Tk_max);
  r.t0 = qt * C::BM;
  r.rows = min(C::BM, sh.Tq - r.t0);
  r.i_first = (long long)r.Tk - sh.Tq + r.t0;
  r.i_last = r.i_first + r.rows - 1;
  r.key_lo = sh.window > 0 ? (int)max(0LL, r.i_first - sh.window + 1) : 0;
  r.key_hi = sh.causal ? (int)min((long long)r.Tk, r.i_last + 1) : r.Tk;
  r.kt_lo = r.key_lo / BN;
  r.kt_hi = r.key_hi > r.key_lo ? (r.key_hi + BN - 1) / BN : r.kt_lo;
  r.mrow = sh.block_mask
               ? sh.block_mask + (((size_t)b * sh.n_heads + h) * sh.nQb + r.t0 / sh.q_block) * sh.nKb
               : nullptr;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_free[s], 4);
    }
    mbar_init(&bars->p_full, 4);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->mma_drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 5) tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tmem_O = tmem;                       // columns [0, D)
  const uint32_t tmem_S = tmem + D;                   // buffer s at D + s*BN

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int qz = b * sh.n_heads + h, kz = b * sh.n_kv + kvh;
      mbar_arrive_expect_tx(&bars->q_full, C::Q_BYTES);
      for (int s = 0; s < C::SLABS; ++s)
        tma_load_3d(sQ + s * C::BM * 128, &tm_q, &bars->q_full, 64 * s, r.t0, qz);
      int it = 0, k_issued = 0, v_issued = 0;
      for (int j = next_tile<BN>(r, sh, r.kt_lo - 1); j < r.kt_hi; j = next_tile<BN>(r, sh, j), ++it) {
        const uint32_t hm = tile_half_mask<BN>(r, sh, j);
        const int st = it & 1;
        const uint32_t bytes = (uint32_t)__popc(hm) * 64u * D * 2u;
        if (it >= 2 && !mbar_wait(&bars->k_empty[st], ((it >> 1) + 1) & 1, tmo, abort_flag)) break;
        mbar_arrive_expect_tx(&bars->k_full[st], bytes);
        ++k_issued;
        for (int hf = 0; hf < C::HALVES; ++hf) {
          if (!((hm >> hf) & 1)) continue;
          for (int s = 0; s < C::SLABS; ++s)
            tma_load_3d(sK + st * C::KV_BYTES + s * BN * 128 + hf * 64 * 128, &tm_k, &bars->k_full[st],
                        64 * s, j * BN + 64 * hf, kz);
        }
        if (it >= 2 && !mbar_wait(&bars->v_empty[st], ((it >> 1) + 1) & 1, tmo, abort_flag)) break;
        mbar_arrive_expect_tx(&bars->v_full[st], bytes);
        ++v_issued;
        for (int hf = 0; hf < C::HALVES; ++hf) {
          if (!((hm >> hf) & 1)) continue;
          for (int s = 0; s < C::SLABS; ++s)
            tma_load_3d(sV + st * C::KV_BYTES + s * BN * 128 + hf * 64 * 128, &tm_v, &bars->v_full[st],
                        64 * s, j * BN + 64 * hf, kz);
        }
      }
      // Drain: the most recent load of every stage has landed before the CTA can exit.
      mbar_wait(&bars->q_full, 0, tmo, nullptr);
      for (int k = max(0, k_issued - 2); k < k_issued; ++k)
        mbar_wait(&bars->k_full[k & 1], (k >> 1) & 1, tmo, nullptr);
      for (int k = max(0, v_issued - 2); k < v_issued; ++k)
        mbar_wait(&bars->v_full[k & 1], (k >> 1) & 1, tmo, nullptr);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_s_full = idesc_bf16_f32(128, BN, false);
    constexpr uint32_t idesc_s_half = idesc_bf16_f32(128, 64, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
    const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV),
                   p_addr = smem_u32(sP);
    bool ok = warp_wait(&bars->q_full, 0, tmo, abort_flag);
    uint32_t pv_started = 0;

    auto issue_s = [&](int it, int j) -> bool {
      const int st = it & 1;
      if (!warp_wait(&bars->k_full[st], (it >> 1) & 1, tmo, abort_flag)) return false;
      if (it >= 2 && !warp_wait(&bars->s_free[st], ((it >> 1) + 1) & 1, tmo, abort_flag)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t hm = tile_half_mask<BN>(r, sh, j);
        const uint32_t kb = k_addr + st * C::KV_BYTES;
        const uint32_t d_s = tmem_S + st * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * C::BM * 128 + (kk & 3) * 32;
          const uint64_t a = sdesc_sw128(q_addr + koff, 16, 1024);
          const uint32_t boff = (kk >> 2) * BN * 128 + (kk & 3) * 32;
          if (hm == (1u << C::HALVES) - 1) {
            umma_bf16_ss(d_s, a, sdesc_sw128(kb + boff, 16, 1024), idesc_s_full, kk > 0);
          } else {
#pragma unroll
            for (int hf = 0; hf < C::HALVES; ++hf)
              if ((hm >> hf) & 1)
                umma_bf16_ss(d_s + 64 * hf, a, sdesc_sw128(kb + boff + hf * 64 * 128, 16, 1024),
                             idesc_s_half, kk > 0);
          }
        }
        umma_commit(&bars->s_full[st]);
        umma_commit(&bars->k_empty[st]);
      }
      __syncwarp();
      return true;
    };

    auto issue_pv = [&](int it, int j) -> bool {
      const int st = it & 1;
      if (!warp_wait(&bars->p_full, it & 1, tmo, abort_flag)) return false;
      if (!warp_wait(&bars->v_full[st], (it >> 1) & 1, tmo, abort_flag)) return false;
      tc_fence_after();
      const uint32_t hm = tile_half_mask<BN>(r, sh, j);
      const int key0 = j * BN;
      if (key0 + BN > r.Tk) {
        // Value rows at or beyond the sequence length may hold anything (even NaN); P is 0
        // there, but 0 * NaN is NaN, so the rows are cleared before the MMA reads them.
        unsigned char* vs = sV + st * C::KV_BYTES;
        const int first = max(0, r.Tk - key0);
        for (int e = lane; e < (BN - first) * C::SLABS * 8; e += 32) {
          const int row = first + e / (C::SLABS * 8);
          const int rest = e % (C::SLABS * 8);
          const int s = rest / 8, chunk = rest % 8;
          if (!((hm >> (row / 64)) & 1)) continue;
          *reinterpret_cast<uint4*>(vs + s * BN * 128 + row * 128 + chunk * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        const uint32_t vb = v_addr + st * C::KV_BYTES;
        const uint32_t pb = p_addr;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          if (!((hm >> (kk >> 2)) & 1)) continue;
          const uint64_t a = sdesc_sw128(pb + (kk >> 2) * C::BM * 128 + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(vb + kk * 2048, BN * 128, 1024);
          umma_bf16_ss(tmem_O, a, bd, idesc_pv, pv_started);
          pv_started = 1;
        }
        umma_commit(&bars->o_done);
        umma_commit(&bars->v_empty[st]);
      }
      __syncwarp();
      return true;
    };

    if (ok) {
      int j = next_tile<BN>(r, sh, r.kt_lo - 1);
      if (j < r.kt_hi) ok = issue_s(0, j);
      for (int it = 0; ok && j < r.kt_hi; ++it) {
        const int jn = next_tile<BN>(r, sh, j);
        if (jn < r.kt_hi) ok = issue_s(it + 1, jn);
        if (ok) ok = issue_pv(it, j);
        j = jn;
      }
    }
    // Drain: every MMA this thread issued has completed before TMEM can be released.
    if (lane == 0) umma_commit(&bars->mma_drain);
    __syncwarp();
    warp_wait(&bars->mma_drain, 0, tmo, nullptr);
  } else {
    // ------------------------------------------------------------------ softmax warps 0-3
    const int row = threadIdx.x;                      // query row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const long long i = r.i_first + row;              // absolute position of this row
    const int lo = sh.window > 0 ? (int)max(0LL, i - sh.window + 1) : 0;
    const int hi = sh.causal ? (int)min((long long)r.Tk, i + 1) : r.Tk;
    // the tile is interior when every valid row may use every key of it
    const int lo_all = sh.window > 0 ? (int)max(0LL, r.i_last - sh.window + 1) : 0;
    const int hi_all = sh.causal ? (int)min((long long)r.Tk, r.i_first + 1) : r.Tk;
    const float scale_log2 = kLog2e / sqrtf((float)D);
    float m_run = -INFINITY, l_run = 0.0f;
    if (sh.sink) { m_run = sh.sink[h] * kLog2e; l_run = 1.0f; }

    int it = 0;
    for (int j = next_tile<BN>(r, sh, r.kt_lo - 1); j < r.kt_hi; j = next_tile<BN>(r, sh, j), ++it) {
      const int st = it & 1;
      if (!warp_wait(&bars->s_full[st], (it >> 1) & 1, tmo, abort_flag)) break;
      tc_fence_after();
      float sv[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
        tmem_ld32(tmem_S + st * BN + 32 * c + lane_off, *reinterpret_cast<float(*)[32]>(&sv[32 * c]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free[st]);

      const uint32_t hm = tile_half_mask<BN>(r, sh, j);
      const int key0 = j * BN;
      const bool interior = hm == (1u << C::HALVES) - 1 && key0 >= lo_all && key0 + BN <= hi_all;
      if (!interior) {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const int jj = key0 + c;
          const bool okc = jj >= lo && jj < hi && ((hm >> (c >> 6)) & 1);
          sv[c] = okc ? sv[c] : -INFINITY;
        }
      }
      float mx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx[u] = sv[u];
#pragma unroll
      for (int c = 8; c < BN; ++c) mx[c & 7] = fmaxf(mx[c & 7], sv[c]);
      const float m_tile =
          fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) *
          scale_log2;

      // lazy rescale: move the reference max only when the new one exceeds it by > 8
      const bool need = m_tile > m_run + 8.0f;
      const float m_new = need ? m_tile : m_run;
      const float alpha = need ? ex2(m_run - m_new) : 1.0f;   // ex2(-inf) = 0
      const float m_use = m_new == -INFINITY ? 0.0f : m_new;
      uint32_t pk[BN / 2];
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < BN; c += 2) {
        const float p0 = ex2(fmaf(sv[c], scale_log2, -m_use));
        const float p1 = ex2(fmaf(sv[c + 1], scale_log2, -m_use));
        ls[(c >> 1) & 3] += p0 + p1;
        pk[c >> 1] = pack_bf16x2(p0, p1);
      }
      l_run = l_run * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      m_run = m_new;

      // PV of the previous tile must be complete before O is rescaled or the P buffer is
      // overwritten.  Waiting at every tile keeps this warp within one phase of o_done.
      if (it > 0) {
        if (!warp_wait(&bars->o_done, (it - 1) & 1, tmo, abort_flag)) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            float o[32];
            tmem_ld32(tmem_O + c + lane_off, o);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) o[u] *= alpha;
            tmem_st32(tmem_O + c + lane_off, o);
          }
          tmem_wait_st();
        }
      }
      unsigned char* prow = sP + row * 128;
#pragma unroll
      for (int c8 = 0; c8 < BN / 8; ++c8) {
        const uint4 v4 = make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
        const int slab = c8 >> 3, chunk = c8 & 7;
        *reinterpret_cast<uint4*>(prow + slab * C::BM * 128 + ((chunk ^ (row & 7)) << 4)) = v4;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full);
    }

    // ---- epilogue: O / l from TMEM to global ------------------------------------------
    const int n_tiles = it;
    bool ok = __all_sync(0xffffffffu, *abort_flag == 0);
    if (ok && n_tiles > 0) ok = warp_wait(&bars->o_done, (n_tiles - 1) & 1, tmo, abort_flag);
    tc_fence_after();
    const int t = r.t0 + row;
    const float inv_l = l_run > 0.0f ? 1.0f / l_run : 0.0f;
    __nv_bfloat16* orow = out + (((size_t)b * sh.n_heads + h) * sh.Tq + t) * D;
    if (ok) {
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        float o[32];
        if (n_tiles > 0) {
          tmem_ld32(tmem_O + c + lane_off, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = 0.0f;
        }
        if (row < r.rows) {
#pragma unroll
          for (int u = 0; u < 32; u += 8) {
            uint4 pk;
            pk.x = pack_bf16x2(o[u + 0] * inv_l, o[u + 1] * inv_l);
            pk.y = pack_bf16x2(o[u + 2] * inv_l, o[u + 3] * inv_l);
            pk.z = pack_bf16x2(o[u + 4] * inv_l, o[u + 5] * inv_l);
            pk.w = pack_bf16x2(o[u + 6] * inv_l, o[u + 7] * inv_l);
            *reinterpret_cast<uint4*>(orow + c + u) = pk;
          }
        }
      }
      if (lse && row < r.rows)
        lse[((size_t)b * sh.n_heads + h) * sh.Tq + t] =
            l_run > 0.0f ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace ga
