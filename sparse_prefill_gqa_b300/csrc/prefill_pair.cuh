// prefill_pair.cuh -- bf16 attention prefill, head dim 128, two query tiles per CTA.
//
// What it computes: the same attention as prefill_tc.cuh ("Attention in Code", "one function
// all designs use": scores q.k/sqrt(d), masked positions removed, optional sink logit in the
// normaliser, weighted sum of values; section 1 head grouping; the absolute-position causal
// rule; the "RBS-Attention review" block-sparse execution, where key blocks outside the mask
// are neither loaded nor multiplied).
//
// The CTA owns 256 query rows of one (sequence, query head) as two 128-row tiles X = 0, 1.
// The tensor core alternates between them, so the softmax of one tile overlaps the MMAs of
// the other:   ... PV0(j)  S0(j+1)  PV1(j)  S1(j+1)  PV0(j+1) ...
//   warps 0-3  softmax of tile 0 (thread r = query row r = TMEM lane r);
//   warps 4-7  softmax of tile 1;
//   warp 8     TMA producer: Q0, Q1 once; K and V tiles of 128 keys into 2-stage rings;
//   warp 9     MMA issuer (one lane);
//   warps 10-11  idle (they complete the third warpgroup, whose registers move to the
//              softmax warpgroups: 168 per thread at launch; 200 for warps 0-7 and 96 for
//              warps 8-11 after setmaxnreg, 256 x 200 + 128 x 96 = 63488 <= 384 x 168).
// Tensor memory (512 columns): O0 [0,128), O1 [128,256), S0 [256,384), S1 [384,512).  The
// softmax writes P (bf16, two per 32-bit column) over the first 64 columns of its own S
// buffer and the PV MMA reads it from there (A operand in TMEM).  tcgen05 operations of one
// issuing thread complete in order, so:
//   - S_X(j+1) is issued after PV_X(j) and overwrites P_X(j) only after PV_X(j) read it;
//   - when the softmax sees S_X(j+1) complete, PV_X(j) is complete too, so it may rescale
//     O_X in TMEM without any other wait.
// The running output is rescaled only when the running max grows by more than 2^8 (P <= 256
// in bf16 never overflows), which is rare after the first tiles of a row.
// Key tiles left empty by the causal rule, the window, the sequence length or the block mask
// are skipped before any load, per query tile; an unselected 64-key half is neither loaded
// nor multiplied.  CTAs are numbered heaviest first (the last 256 rows of every head first).
//
// Shared memory: Q 2 x 32 KB, K 2 x 32 KB, V 2 x 32 KB (128-byte swizzle), barriers.
#pragma once

#include "common.cuh"
#include "prefill_tc.cuh"

namespace ga {

struct PairCfg {
  static constexpr int D = 128;
  static constexpr int BM = 128;                 // rows per query tile
  static constexpr int BN = 128;                 // keys per key tile
  static constexpr int SLABS = D / 64;
  static constexpr int HALVES = BN / 64;
  static constexpr int QT_BYTES = BM * D * 2;    // one query tile
  static constexpr int KV_BYTES = BN * D * 2;    // one K or V tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * QT_BYTES;
  static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + 2 * KV_BYTES;
  static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
  static constexpr int THREADS = 384;
  static constexpr int LAUNCH_REGS = 168;        // ptxas register count at launch (384 threads)
  static constexpr int SOFTMAX_REGS = 200, OTHER_REGS = 96;
  static_assert(256 * SOFTMAX_REGS + 128 * OTHER_REGS <= THREADS * LAUNCH_REGS, "register split");
  static constexpr uint32_t COL_O = 0, COL_S = 2 * D;  // O_X at X*D, S_X at 2D + X*BN
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct PairBars {
  uint64_t q_full[2];
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2], o_final[2];
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Key range, rows and mask row of query tile X of the CTA (rows <= 0: the tile is empty).
__device__ __forceinline__ TileRange pair_range(const AttnShape& sh, int b, int h, int t0, int Tk) {
  TileRange r;
  r.Tk = Tk;
  r.t0 = t0;
  r.rows = min(PairCfg::BM, sh.Tq - t0);
  if (r.rows <= 0) {
    r.rows = 0; r.key_lo = 0; r.key_hi = 0; r.kt_lo = 0; r.kt_hi = 0;
    r.i_first = r.i_last = 0; r.mrow = nullptr;
    return r;
  }
  r.i_first = (long long)Tk - sh.Tq + t0;
  r.i_last = r.i_first + r.rows - 1;
  r.key_lo = sh.window > 0 ? (int)max(0LL, r.i_first - sh.window + 1) : 0;
  r.key_hi = sh.causal ? (int)min((long long)Tk, r.i_last + 1) : Tk;
  if (r.key_hi < r.key_lo) r.key_hi = r.key_lo;
  r.kt_lo = r.key_lo / PairCfg::BN;
  r.kt_hi = r.key_hi > r.key_lo ? (r.key_hi + PairCfg::BN - 1) / PairCfg::BN : r.kt_lo;
  r.mrow = sh.block_mask
               ? sh.block_mask + (((size_t)b * sh.n_heads + h) * sh.nQb + t0 / sh.q_block) * sh.nKb
               : nullptr;
  return r;
}

__device__ __forceinline__ uint32_t pair_half_mask(const TileRange& r, const AttnShape& sh, int j) {
  if (r.rows == 0 || j < r.kt_lo || j >= r.kt_hi) return 0u;
  // without a block mask every tile strictly inside the range uses both halves
  if (r.mrow == nullptr && j > r.kt_lo && j + 1 < r.kt_hi) return 3u;
  return tile_half_mask<PairCfg::BN>(r, sh, j);
}

// Next key tile after j that either query tile uses (kt_end when none).
__device__ __forceinline__ int pair_next(const TileRange& r0, const TileRange& r1, const AttnShape& sh,
                                         int j, int kt_end) {
  ++j;
  // without a block mask, the next tile inside either contiguous range is used
  if (r0.mrow == nullptr && r1.mrow == nullptr && j < kt_end &&
      ((j >= r0.kt_lo && j < r0.kt_hi) || (j >= r1.kt_lo && j < r1.kt_hi)))
    return j;
  for (; j < kt_end; ++j)
    if (pair_half_mask(r0, sh, j) | pair_half_mask(r1, sh, j)) return j;
  return kt_end;
}

// grid: (n_pairs * n_heads * batch); block: 384 threads; 1 CTA per SM.
__global__ void __launch_bounds__(384, 1)
prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ out,
                    float* __restrict__ lse, AttnShape sh) {
  using C = PairCfg;
  constexpr int D = C::D, BN = C::BN;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sQ = smem + C::OFF_Q;
  unsigned char* sK = smem + C::OFF_K;
  unsigned char* sV = smem + C::OFF_V;
  PairBars* bars = reinterpret_cast<PairBars*>(smem + C::OFF_BAR);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heaviest first: CTA index -> (pair from the end, head, sequence)
  const int n_pairs = (sh.Tq + 2 * C::BM - 1) / (2 * C::BM);
  const int hb = sh.n_heads * sh.batch;
  const int pr = (int)(blockIdx.x / hb), rem = (int)(blockIdx.x % hb);
  const int h = rem % sh.n_heads, b = rem / sh.n_heads;
  const int pair = n_pairs - 1 - pr;
  const int kvh = h / (sh.n_heads / sh.n_kv);
  const uint64_t tmo = sh.timeout_ns;
  const int Tk = seq_keys(sh.k_lens, b, sh.Tk_max);
  const TileRange r0 = pair_range(sh, b, h, pair * 2 * C::BM, Tk);
  const TileRange r1 = pair_range(sh, b, h, pair * 2 * C::BM + C::BM, Tk);
  const int kt_begin = r1.rows ? min(r0.kt_lo, r1.kt_lo) : r0.kt_lo;
  const int kt_end = r1.rows ? max(r0.kt_hi, r1.kt_hi) : r0.kt_hi;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 4);
      mbar_init(&bars->o_final[s], 1);
    }
    mbar_init(&bars->mma_drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 9) tmem_alloc(&bars->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp >= 8) {
  // warps 8-11: one warpgroup gives registers back, then takes the producer / MMA roles
  regs_dec<C::OTHER_REGS>();
  if (warp == 8) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int qz = b * sh.n_heads + h, kz = b * sh.n_kv + kvh;
      bool q_loaded[2] = {false, false};
      for (int x = 0; x < 2; ++x) {
        const TileRange& r = x ? r1 : r0;
        if (r.rows == 0) continue;
        mbar_arrive_expect_tx(&bars->q_full[x], C::QT_BYTES);
        for (int s = 0; s < C::SLABS; ++s)
          tma_load_3d(sQ + x * C::QT_BYTES + s * C::BM * 128, &tm_q, &bars->q_full[x], 64 * s, r.t0, qz);
        q_loaded[x] = true;
      }
      int u = 0, k_issued = 0, v_issued = 0;
      for (int j = pair_next(r0, r1, sh, kt_begin - 1, kt_end); j < kt_end;
           j = pair_next(r0, r1, sh, j, kt_end), ++u) {
        const uint32_t hm = pair_half_mask(r0, sh, j) | pair_half_mask(r1, sh, j);
        const int st = u & 1;
        const uint32_t bytes = (uint32_t)__popc(hm) * 64u * D * 2u;
        if (u >= 2 && !mbar_wait(&bars->k_empty[st], ((u >> 1) + 1) & 1, tmo, abort_flag)) break;
        mbar_arrive_expect_tx(&bars->k_full[st], bytes);
        ++k_issued;
        for (int hf = 0; hf < C::HALVES; ++hf) {
          if (!((hm >> hf) & 1)) continue;
          for (int s = 0; s < C::SLABS; ++s)
            tma_load_3d(sK + st * C::KV_BYTES + s * BN * 128 + hf * 64 * 128, &tm_k, &bars->k_full[st],
                        64 * s, j * BN + 64 * hf, kz);
        }
        if (u >= 2 && !mbar_wait(&bars->v_empty[st], ((u >> 1) + 1) & 1, tmo, abort_flag)) break;
        mbar_arrive_expect_tx(&bars->v_full[st], bytes);
        ++v_issued;
        for (int hf = 0; hf < C::HALVES; ++hf) {
          if (!((hm >> hf) & 1)) continue;
          for (int s = 0; s < C::SLABS; ++s)
            tma_load_3d(sV + st * C::KV_BYTES + s * BN * 128 + hf * 64 * 128, &tm_v, &bars->v_full[st],
                        64 * s, j * BN + 64 * hf, kz);
        }
      }
      // Drain: every load this thread issued has landed before the CTA may exit.
      for (int x = 0; x < 2; ++x)
        if (q_loaded[x]) mbar_wait(&bars->q_full[x], 0, tmo, nullptr);
      for (int k = max(0, k_issued - 2); k < k_issued; ++k)
        mbar_wait(&bars->k_full[k & 1], (k >> 1) & 1, tmo, nullptr);
      for (int k = max(0, v_issued - 2); k < v_issued; ++k)
        mbar_wait(&bars->v_full[k & 1], (k >> 1) & 1, tmo, nullptr);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------------ MMA issuer
    // One thread runs the whole issue loop: a tcgen05.mma costs the issuing thread about
    // as long as a 128x128x16 MMA takes to execute, so this thread does nothing else
    // (descriptors are built once and advanced by constant offsets; waits are one thread's).
    if (lane == 0) {
      constexpr uint32_t idesc_s_full = idesc_bf16_f32(128, BN, false);
      constexpr uint32_t idesc_s_half = idesc_bf16_f32(128, 64, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
      const uint64_t dq0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dk0 = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(smem_u32(sV), BN * 128, 1024);
      bool ok = true;
      if (r0.rows) ok = mbar_wait(&bars->q_full[0], 0, tmo, abort_flag);
      if (ok && r1.rows) ok = mbar_wait(&bars->q_full[1], 0, tmo, abort_flag);
      int pv_total0 = 0, pv_total1 = 0;   // key tiles each query tile uses
      for (int j = pair_next(r0, r1, sh, kt_begin - 1, kt_end); j < kt_end; j = pair_next(r0, r1, sh, j, kt_end)) {
        pv_total0 += pair_half_mask(r0, sh, j) ? 1 : 0;
        pv_total1 += pair_half_mask(r1, sh, j) ? 1 : 0;
      }
      int n_pv0 = 0, n_pv1 = 0;
      uint32_t o_acc0 = 0u, o_acc1 = 0u;  // O_X already holds an accumulated value

      // S_X = Q_X K^T for the key tile in stage st (N=128, or N=64 per used half)
      auto issue_s = [&](int x, int st, uint32_t hm) {
        const uint64_t aq = dq0 + (uint64_t)((x * C::QT_BYTES) >> 4);
        const uint64_t bk = dk0 + (uint64_t)((st * C::KV_BYTES) >> 4);
        const uint32_t d_s = tmem + C::COL_S + x * BN;
        if (hm == 3u) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * C::BM * 128 + (kk & 3) * 32) >> 4);
            const uint64_t offb = (uint64_t)(((kk >> 2) * BN * 128 + (kk & 3) * 32) >> 4);
            umma_bf16_ss(d_s, aq + off, bk + offb, idesc_s_full, kk > 0);
          }
        } else {                               // one used 64-key half: N = 64
          const int hf = hm == 2u ? 1 : 0;
          const uint64_t bh = bk + (uint64_t)((hf * 64 * 128) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * C::BM * 128 + (kk & 3) * 32) >> 4);
            const uint64_t offb = (uint64_t)(((kk >> 2) * BN * 128 + (kk & 3) * 32) >> 4);
            umma_bf16_ss(d_s + 64 * hf, aq + off, bh + offb, idesc_s_half, kk > 0);
          }
        }
        umma_commit(&bars->s_full[x]);
      };
      // O_X += P_X V for the key tile in stage st (P_X in TMEM over S_X's first 64 columns)
      // (one branch per group: the MMAs of a group are issued straight-line)
      auto issue_pv = [&](int x, int st, uint32_t hm, uint32_t& o_acc) {
        const uint64_t bv = dv0 + (uint64_t)((st * C::KV_BYTES) >> 4);
        const uint32_t p_col = tmem + C::COL_S + x * BN;
        const uint32_t d_o = tmem + C::COL_O + x * D;
        if (hm == 3u) {
          umma_bf16_ts(d_o, p_col, bv, idesc_pv, o_acc);
#pragma unroll
          for (int kk = 1; kk < BN / 16; ++kk)
            umma_bf16_ts(d_o, p_col + kk * 8, bv + (uint64_t)((kk * 2048) >> 4), idesc_pv, 1u);
        } else {
          const int k0 = hm == 2u ? 4 : 0;     // the one used 64-key half
          const uint64_t bh = bv + (uint64_t)((k0 * 2048) >> 4);
          const uint32_t ph = p_col + k0 * 8;
          umma_bf16_ts(d_o, ph, bh, idesc_pv, o_acc);
#pragma unroll
          for (int kk = 1; kk < 4; ++kk)
            umma_bf16_ts(d_o, ph + kk * 8, bh + (uint64_t)((kk * 2048) >> 4), idesc_pv, 1u);
        }
        o_acc = 1u;
      };
      // zero value rows at or past the sequence end in the used halves (P is 0 there, but
      // 0 * NaN = NaN for an uninitialised cache); only a sequence's last tile needs it
      auto clear_v_tail = [&](int j, int st, uint32_t hm) {
        const int key0 = j * BN;
        if (key0 + BN <= Tk) return;
        unsigned char* vs = sV + st * C::KV_BYTES;
        for (int row = max(0, Tk - key0); row < BN; ++row) {
          if (!((hm >> (row / 64)) & 1)) continue;
          for (int sl = 0; sl < C::SLABS; ++sl)
            for (int chunk = 0; chunk < 8; ++chunk)
              *reinterpret_cast<uint4*>(vs + sl * BN * 128 + row * 128 + chunk * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      };

      int j = pair_next(r0, r1, sh, kt_begin - 1, kt_end);
      if (ok && j < kt_end) {
        ok = mbar_wait(&bars->k_full[0], 0, tmo, abort_flag);
        if (ok) {
          tc_fence_after();
          const uint32_t h0 = pair_half_mask(r0, sh, j), h1 = pair_half_mask(r1, sh, j);
          if (h0) issue_s(0, 0, h0);
          if (h1) issue_s(1, 0, h1);
          umma_commit(&bars->k_empty[0]);
        }
      }
      uint32_t h0 = ok && j < kt_end ? pair_half_mask(r0, sh, j) : 0u;
      uint32_t h1 = ok && j < kt_end ? pair_half_mask(r1, sh, j) : 0u;
      for (int u = 0; ok && j < kt_end; ++u) {
        const int st = u & 1, stn = st ^ 1;
        const int jn = pair_next(r0, r1, sh, j, kt_end);
        const uint32_t n0 = jn < kt_end ? pair_half_mask(r0, sh, jn) : 0u;
        const uint32_t n1 = jn < kt_end ? pair_half_mask(r1, sh, jn) : 0u;
        // both TMA waits first (the loads were released two tiles ago), so that each PV
        // and the following S go to the tensor core back to back
        if (!(ok = mbar_wait(&bars->v_full[st], (u >> 1) & 1, tmo, abort_flag))) break;
        if (jn < kt_end && !(ok = mbar_wait(&bars->k_full[stn], ((u + 1) >> 1) & 1, tmo, abort_flag))) break;
        tc_fence_after();
        clear_v_tail(j, st, h0 | h1);
        if (h0) {
          if (!(ok = mbar_wait(&bars->p_full[0], n_pv0 & 1, tmo, abort_flag))) break;
          tc_fence_after();
          issue_pv(0, st, h0, o_acc0);
          if (++n_pv0 == pv_total0) umma_commit(&bars->o_final[0]);
        }
        if (n0) issue_s(0, stn, n0);
        if (h1) {
          if (!(ok = mbar_wait(&bars->p_full[1], n_pv1 & 1, tmo, abort_flag))) break;
          tc_fence_after();
          issue_pv(1, st, h1, o_acc1);
          if (++n_pv1 == pv_total1) umma_commit(&bars->o_final[1]);
        }
        umma_commit(&bars->v_empty[st]);
        if (jn < kt_end) {
          if (n1) issue_s(1, stn, n1);
          umma_commit(&bars->k_empty[stn]);
        }
        j = jn; h0 = n0; h1 = n1;
      }
      // Drain: every MMA this thread issued has completed before TMEM can be released.
      umma_commit(&bars->mma_drain);
      mbar_wait(&bars->mma_drain, 0, tmo, nullptr);
    }
    __syncwarp();
  }
  } else {
    // ------------------------------------------------------------------ softmax warps 0-7
    regs_inc<C::SOFTMAX_REGS>();
    const int x = warp >> 2;                          // query tile of this warpgroup
    const TileRange& r = x ? r1 : r0;
    const int row = threadIdx.x & 127;                // row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + C::COL_S + x * BN + lane_off;
    const uint32_t t_o = tmem + C::COL_O + x * D + lane_off;
    const long long i = r.i_first + row;              // absolute position of this row
    const int lo = sh.window > 0 ? (int)max(0LL, i - sh.window + 1) : 0;
    const int hi = sh.causal ? (int)min((long long)Tk, i + 1) : Tk;
    const int lo_all = sh.window > 0 ? (int)max(0LL, r.i_last - sh.window + 1) : 0;
    const int hi_all = sh.causal ? (int)min((long long)Tk, r.i_first + 1) : Tk;
    const float scale_log2 = kLog2e / sqrtf((float)D);
    float m_run = -INFINITY, l_run = 0.0f;
    if (sh.sink) { m_run = sh.sink[h] * kLog2e; l_run = 1.0f; }

    int n = 0;
    if (r.rows > 0) {
      for (int j = pair_next(r, r, sh, r.kt_lo - 1, r.kt_hi); j < r.kt_hi; j = pair_next(r, r, sh, j, r.kt_hi), ++n) {
        if (!warp_wait(&bars->s_full[x], n & 1, tmo, abort_flag)) break;
        tc_fence_after();
        float sv[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
          tmem_ld32(t_s + 32 * c, *reinterpret_cast<float(*)[32]>(&sv[32 * c]));
        tmem_wait_ld();

        const uint32_t hm = pair_half_mask(r, sh, j);
        const int key0 = j * BN;
        const bool interior = hm == 3u && key0 >= lo_all && key0 + BN <= hi_all;
        if (!interior) {
#pragma unroll
          for (int c = 0; c < BN; ++c) {
            const int jj = key0 + c;
            const bool okc = jj >= lo && jj < hi && ((hm >> (c >> 6)) & 1);
            sv[c] = okc ? sv[c] : -INFINITY;
          }
        }
        // row max: 3-input max over 128 values in 4 independent chains
        static_assert(BN % 8 == 0, "max chains take 8 columns per step");
        float mx[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) mx[u] = fmaxf(sv[u], sv[u + 4]);
#pragma unroll
        for (int c = 8; c < BN; c += 8)
#pragma unroll
          for (int u = 0; u < 4; ++u) mx[u] = fmax3(mx[u], sv[c + u], sv[c + u + 4]);
        const float m_tile = fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]) * scale_log2;
        const bool need = m_tile > m_run + 8.0f;
        const float m_new = need ? m_tile : m_run;
        const float alpha = need ? ex2(m_run - m_new) : 1.0f;   // ex2(-inf) = 0
        const float m_use = m_new == -INFINITY ? 0.0f : m_new;
        // p = 2^(s * scale_log2 - m): the scale-and-shift two columns per instruction
        float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // four independent pairs
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            float t0, t1, t2, t3;
            ffma2(t0, t1, sv[c0 + c], sv[c0 + c + 1], scale_log2, scale_log2, -m_use, -m_use);
            ffma2(t2, t3, sv[c0 + c + 2], sv[c0 + c + 3], scale_log2, scale_log2, -m_use, -m_use);
            const float p0 = ex2(t0), p1 = ex2(t1), p2 = ex2(t2), p3 = ex2(t3);
            const int q = (c >> 1) & 2;
            fadd2(ls[q], ls[q + 1], ls[q], ls[q + 1], p0, p1);
            fadd2(ls[q + 4], ls[q + 5], ls[q + 4], ls[q + 5], p2, p3);
            pk[c >> 1] = pack_bf16x2(p0, p1);
            pk[(c >> 1) + 1] = pack_bf16x2(p2, p3);
          }
          tmem_st16(t_s + c0 / 2, pk);
        }
        l_run = l_run * alpha + (((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7])));
        m_run = m_new;
        // S_X complete => PV_X of the previous tile complete: O_X may be rescaled now (after
        // P is out of registers, so the score row and the O chunk are never live together)
        if (n > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            float o[32];
            tmem_ld32(t_o + c, o);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) o[u] *= alpha;
            tmem_st32(t_o + c, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[x]);
      }
    }

    // ---- epilogue: O / l from TMEM to global ------------------------------------------
    if (r.rows > 0) {
      bool ok = __all_sync(0xffffffffu, *abort_flag == 0);
      if (ok && n > 0) ok = warp_wait(&bars->o_final[x], 0, tmo, abort_flag);
      tc_fence_after();
      const int t = r.t0 + row;
      const float inv_l = l_run > 0.0f ? 1.0f / l_run : 0.0f;
      __nv_bfloat16* orow = out + (((size_t)b * sh.n_heads + h) * sh.Tq + t) * D;
      if (ok) {
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float o[32];
          if (n > 0) {
            tmem_ld32(t_o + c, o);
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
  }

  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace ga
