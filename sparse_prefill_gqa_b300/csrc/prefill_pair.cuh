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
// are skipped before any load; an unselected 64-key unit is neither loaded nor multiplied.
// With a block mask, the selected 64-key units are compacted at the start of the CTA into a
// list of full 128-key tiles (units both query tiles use, then those only tile 0 uses, then
// those only tile 1 uses, paired within each group), so sparse work runs on full-width MMAs
// and costs in proportion to the selected units.  CTAs are numbered heaviest first (the
// last 256 rows of every head first).
//
// Shared memory: Q 2 x 32 KB, K 2 x 32 KB, V 2 x 32 KB (128-byte swizzle), barriers, and the
// tile list (2 x 2048 unit indices).
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
  static constexpr int BAR_BYTES = 512;
  static constexpr int LIST_MAX = 2048;          // tiles in the shared-memory list
  static constexpr int OFF_LIST = OFF_BAR + BAR_BYTES;
  static constexpr int SMEM_BYTES = OFF_LIST + 2 * LIST_MAX * 4 + 1024;
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
  int lcnt[3];                  // tile-list build: units per group
  int lwarp[3][12];             // tile-list build: units per group and warp in a chunk
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

// The CTA's key-tile schedule.  A tile is two 64-key units ua, ub (keys 64*ua .. 64*ua+63
// and 64*ub ..) and, per query tile X, the halves it uses (bit 0: ua, bit 1: ub).
//   dense: tile j is units 2j, 2j+1 over the contiguous key ranges of the two query tiles
//          (no block mask, or a block mask whose list would not fit);
//   list:  tiles [0, c0) are used by both query tiles, [c0, c1) by tile 0 only, [c1, n) by
//          tile 1 only; lb = kNoUnit marks a tile holding one unit.
constexpr uint32_t kNoUnit = 0xFFFFFFFFu;

struct PairSched {
  int list;
  int kt_begin, kt_end;
  int n, c0, c1;
  const uint32_t* la;
  const uint32_t* lb;
};

struct PairTile {
  int ua, ub;
  uint32_t h0, h1;
};

__device__ __forceinline__ PairTile sched_tile(const PairSched& s, const TileRange& r0, const TileRange& r1,
                                               const AttnShape& sh, int pos) {
  PairTile t;
  if (!s.list) {
    t.ua = 2 * pos;
    t.ub = 2 * pos + 1;
    t.h0 = pair_half_mask(r0, sh, pos);
    t.h1 = pair_half_mask(r1, sh, pos);
  } else {
    const uint32_t b = s.lb[pos];
    const uint32_t present = b == kNoUnit ? 1u : 3u;
    t.ua = (int)s.la[pos];
    t.ub = b == kNoUnit ? t.ua : (int)b;
    t.h0 = pos < s.c1 ? present : 0u;
    t.h1 = (pos < s.c0 || pos >= s.c1) ? present : 0u;
  }
  return t;
}

// x < 0: the tiles either query tile uses; x = 0 / 1: the tiles query tile x uses.
__device__ __forceinline__ int sched_end(const PairSched& s, const TileRange& r0, const TileRange& r1, int x) {
  if (!s.list) return x < 0 ? s.kt_end : (x == 0 ? r0.kt_hi : r1.kt_hi);
  return x == 0 ? s.c1 : s.n;
}

// The position after pos (pos = -1: the first), or sched_end when none is left.
__device__ __forceinline__ int sched_next(const PairSched& s, const TileRange& r0, const TileRange& r1,
                                          const AttnShape& sh, int pos, int x) {
  if (!s.list) {
    if (x < 0) return pair_next(r0, r1, sh, pos < 0 ? s.kt_begin - 1 : pos, s.kt_end);
    const TileRange& r = x == 0 ? r0 : r1;
    return pair_next(r, r, sh, pos < 0 ? r.kt_lo - 1 : pos, r.kt_hi);
  }
  int p = pos + 1;
  if (x == 1 && p == s.c0) p = s.c1;
  return p;
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

  // ---- schedule: with a block mask, compact the selected units into a tile list ---------
  PairSched sched;
  sched.list = 0;
  sched.kt_begin = kt_begin;
  sched.kt_end = kt_end;
  sched.n = sched.c0 = sched.c1 = 0;
  uint32_t* list_a = reinterpret_cast<uint32_t*>(smem + C::OFF_LIST);
  uint32_t* list_b = list_a + C::LIST_MAX;
  sched.la = list_a;
  sched.lb = list_b;
  if (sh.block_mask) {
    const int u_lo = (r1.rows ? min(r0.key_lo, r1.key_lo) : r0.key_lo) / 64;
    const int u_hi = ((r1.rows ? max(r0.key_hi, r1.key_hi) : r0.key_hi) + 63) / 64;
    // group of unit u: 0 both query tiles use it, 1 only tile 0, 2 only tile 1, -1 neither
    auto unit_group = [&](int u) -> int {
      if (u >= u_hi) return -1;
      const int k0 = 64 * u;
      const bool s0 = r0.rows && k0 < r0.key_hi && k0 + 64 > r0.key_lo && r0.mrow[k0 / sh.k_block] != 0;
      const bool s1 = r1.rows && k0 < r1.key_hi && k0 + 64 > r1.key_lo && r1.mrow[k0 / sh.k_block] != 0;
      return s0 && s1 ? 0 : (s0 ? 1 : (s1 ? 2 : -1));
    };
    if (threadIdx.x < 3) bars->lcnt[threadIdx.x] = 0;
    __syncthreads();
    for (int u = u_lo + (int)threadIdx.x; u < u_hi; u += C::THREADS) {
      const int g = unit_group(u);
      if (g >= 0) atomicAdd(&bars->lcnt[g], 1);
    }
    __syncthreads();
    const int cnt0 = bars->lcnt[0], cnt1 = bars->lcnt[1], cnt2 = bars->lcnt[2];
    const int tiles0 = (cnt0 + 1) / 2, tiles1 = (cnt1 + 1) / 2, tiles2 = (cnt2 + 1) / 2;
    if (tiles0 + tiles1 + tiles2 <= C::LIST_MAX) {
      sched.list = 1;
      sched.c0 = tiles0;
      sched.c1 = tiles0 + tiles1;
      sched.n = sched.c1 + tiles2;
      int run0 = 0, run1 = 0, run2 = 0;             // units placed per group (same in all threads)
      const uint32_t lt = (1u << lane) - 1u;
      for (int base = u_lo; base < u_hi; base += C::THREADS) {   // ordered compaction
        const int u = base + (int)threadIdx.x;
        const int g = unit_group(u);
        const uint32_t bal0 = __ballot_sync(0xffffffffu, g == 0);
        const uint32_t bal1 = __ballot_sync(0xffffffffu, g == 1);
        const uint32_t bal2 = __ballot_sync(0xffffffffu, g == 2);
        if (lane == 0) {
          bars->lwarp[0][warp] = __popc(bal0);
          bars->lwarp[1][warp] = __popc(bal1);
          bars->lwarp[2][warp] = __popc(bal2);
        }
        __syncthreads();
        if (g >= 0) {
          const uint32_t bal = g == 0 ? bal0 : (g == 1 ? bal1 : bal2);
          int rank = (g == 0 ? run0 : (g == 1 ? run1 : run2)) + __popc(bal & lt);
          for (int w = 0; w < warp; ++w) rank += bars->lwarp[g][w];
          const int tb = g == 0 ? 0 : (g == 1 ? sched.c0 : sched.c1);
          (rank & 1 ? list_b : list_a)[tb + (rank >> 1)] = (uint32_t)u;
        }
        for (int w = 0; w < C::THREADS / 32; ++w) {
          run0 += bars->lwarp[0][w];
          run1 += bars->lwarp[1][w];
          run2 += bars->lwarp[2][w];
        }
        __syncthreads();
      }
      // a group's odd last unit stands alone in its tile
      if (threadIdx.x == 0) {
        if (cnt0 & 1) list_b[cnt0 / 2] = kNoUnit;
        if (cnt1 & 1) list_b[sched.c0 + cnt1 / 2] = kNoUnit;
        if (cnt2 & 1) list_b[sched.c1 + cnt2 / 2] = kNoUnit;
      }
      __syncthreads();
    }
  }

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
      const int pend = sched_end(sched, r0, r1, -1);
      for (int pos = sched_next(sched, r0, r1, sh, -1, -1); pos < pend;
           pos = sched_next(sched, r0, r1, sh, pos, -1), ++u) {
        const PairTile ti = sched_tile(sched, r0, r1, sh, pos);
        const uint32_t hm = ti.h0 | ti.h1;
        const int st = u & 1;
        const uint32_t bytes = (uint32_t)__popc(hm) * 64u * D * 2u;
        if (u >= 2 && !mbar_wait(&bars->k_empty[st], ((u >> 1) + 1) & 1, tmo, abort_flag)) break;
        mbar_arrive_expect_tx(&bars->k_full[st], bytes);
        ++k_issued;
        for (int hf = 0; hf < C::HALVES; ++hf) {
          if (!((hm >> hf) & 1)) continue;
          for (int s = 0; s < C::SLABS; ++s)
            tma_load_3d(sK + st * C::KV_BYTES + s * BN * 128 + hf * 64 * 128, &tm_k, &bars->k_full[st],
                        64 * s, 64 * (hf ? ti.ub : ti.ua), kz);
        }
        if (u >= 2 && !mbar_wait(&bars->v_empty[st], ((u >> 1) + 1) & 1, tmo, abort_flag)) break;
        mbar_arrive_expect_tx(&bars->v_full[st], bytes);
        ++v_issued;
        for (int hf = 0; hf < C::HALVES; ++hf) {
          if (!((hm >> hf) & 1)) continue;
          for (int s = 0; s < C::SLABS; ++s)
            tma_load_3d(sV + st * C::KV_BYTES + s * BN * 128 + hf * 64 * 128, &tm_v, &bars->v_full[st],
                        64 * s, 64 * (hf ? ti.ub : ti.ua), kz);
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
      const int pend = sched_end(sched, r0, r1, -1);
      int pv_total0 = 0, pv_total1 = 0;   // key tiles each query tile uses
      if (sched.list) {
        pv_total0 = sched.c1;
        pv_total1 = sched.c0 + (sched.n - sched.c1);
      } else {
        for (int j = sched_next(sched, r0, r1, sh, -1, -1); j < pend; j = sched_next(sched, r0, r1, sh, j, -1)) {
          pv_total0 += pair_half_mask(r0, sh, j) ? 1 : 0;
          pv_total1 += pair_half_mask(r1, sh, j) ? 1 : 0;
        }
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
      auto clear_v_tail = [&](const PairTile& ti, int st, uint32_t hm) {
        bool any = false;
        unsigned char* vs = sV + st * C::KV_BYTES;
        for (int hf = 0; hf < C::HALVES; ++hf) {
          const int key0 = 64 * (hf ? ti.ub : ti.ua);
          if (!((hm >> hf) & 1) || key0 + 64 <= Tk) continue;
          any = true;
          for (int row = max(0, Tk - key0); row < 64; ++row)
            for (int sl = 0; sl < C::SLABS; ++sl)
              for (int chunk = 0; chunk < 8; ++chunk)
                *reinterpret_cast<uint4*>(vs + sl * BN * 128 + (hf * 64 + row) * 128 + chunk * 16) =
                    make_uint4(0, 0, 0, 0);
        }
        if (any) fence_proxy_async_smem();
      };

      int j = sched_next(sched, r0, r1, sh, -1, -1);
      PairTile ti = j < pend ? sched_tile(sched, r0, r1, sh, j) : PairTile{0, 0, 0u, 0u};
      if (ok && j < pend) {
        ok = mbar_wait(&bars->k_full[0], 0, tmo, abort_flag);
        if (ok) {
          tc_fence_after();
          if (ti.h0) issue_s(0, 0, ti.h0);
          if (ti.h1) issue_s(1, 0, ti.h1);
          umma_commit(&bars->k_empty[0]);
        }
      }
      for (int u = 0; ok && j < pend; ++u) {
        const int st = u & 1, stn = st ^ 1;
        const uint32_t h0 = ti.h0, h1 = ti.h1;
        const int jn = sched_next(sched, r0, r1, sh, j, -1);
        const PairTile tn = jn < pend ? sched_tile(sched, r0, r1, sh, jn) : PairTile{0, 0, 0u, 0u};
        const uint32_t n0 = tn.h0, n1 = tn.h1;
        // both TMA waits first (the loads were released two tiles ago), so that each PV
        // and the following S go to the tensor core back to back
        if (!(ok = mbar_wait(&bars->v_full[st], (u >> 1) & 1, tmo, abort_flag))) break;
        if (jn < pend && !(ok = mbar_wait(&bars->k_full[stn], ((u + 1) >> 1) & 1, tmo, abort_flag))) break;
        tc_fence_after();
        clear_v_tail(ti, st, h0 | h1);
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
        if (jn < pend) {
          if (n1) issue_s(1, stn, n1);
          umma_commit(&bars->k_empty[stn]);
        }
        j = jn;
        ti = tn;
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
      const int pend = sched_end(sched, r0, r1, x);
      for (int pos = sched_next(sched, r0, r1, sh, -1, x); pos < pend; pos = sched_next(sched, r0, r1, sh, pos, x), ++n) {
        if (!warp_wait(&bars->s_full[x], n & 1, tmo, abort_flag)) break;
        tc_fence_after();
        float sv[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
          tmem_ld32(t_s + 32 * c, *reinterpret_cast<float(*)[32]>(&sv[32 * c]));
        tmem_wait_ld();

        const PairTile ti = sched_tile(sched, r0, r1, sh, pos);
        const uint32_t hm = x ? ti.h1 : ti.h0;
        const int kb0 = 64 * ti.ua, kb1 = 64 * ti.ub;   // first key of each 64-key half
        const bool interior = hm == 3u && kb0 >= lo_all && kb0 + 64 <= hi_all && kb1 >= lo_all &&
                              kb1 + 64 <= hi_all;
        if (!interior) {
#pragma unroll
          for (int c = 0; c < BN; ++c) {
            const int jj = (c < 64 ? kb0 : kb1) + (c & 63);
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
