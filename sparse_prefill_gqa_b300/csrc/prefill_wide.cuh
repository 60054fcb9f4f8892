// prefill_wide.cuh -- bf16 attention prefill, one 128-row query tile per CTA, head dim 128 or
// 256: causal, window, sink, and block-sparse (a block mask over 64-key units).
//
// What it computes ("Attention in Code", "one function all designs use": scores q.k/sqrt(d),
// masked positions removed, optional sink logit in the normaliser, weighted sum of values;
// section 1 head grouping; the absolute-position causal rule; the sliding window of section 2),
// restricted to the selected key blocks when a block mask is given ("RBS-Attention review":
// attention is computed only over the blocks the selection keeps).
//
// Block masks: the CTA first lists the selected 64-key units of its query tile, in key order,
// and pairs them into 128-key tiles; each half of a tile is loaded as its own 64-key box and
// masked from its own key base, so the work is proportional to the selected units and the MMAs
// stay full width.  Launches without a block mask use the instantiation UNITS = false, which
// has no list and loads contiguous 128-key tiles.
//
// One CTA per (128-row query tile, query head, sequence), heaviest causal tiles first.
//
// d = 128 (12 warps): two softmax warpgroups split the key tiles of the query tile between them,
// warpgroup 0 the even tiles and warpgroup 1 the odd ones, each with its own running max and sum
// and its own output accumulator in tensor memory; the epilogue merges the two partial results
// by the log-sum-exp rule (the same re-association as split-K decode).  The two softmaxes run
// concurrently, so each scheduler holds two softmax warps and the tensor core sees tile j+1
// ready while tile j is still being exponentiated.
//   warps 0-3, 4-7  softmax of even / odd tiles: thread r of a warpgroup = query row r = TMEM lane r;
//   warp 8          TMA producer (one lane): Q once, then K and V through a ring of 32 KB chunks
//                   (4 slots), K one tile ahead of V;
//   warp 9          S issuer (one lane): S(j) = Q K(j)^T into S buffer j & 1;
//   warp 10         PV issuer (one lane): O_(j&1) += P(j) V(j);
//   warp 11         idle (completes the warpgroup whose registers move to the softmax).
// Two issuers, because the tensor core's queue is short: a thread that issues an MMA waits while
// earlier MMAs execute, so one thread that also waited for P would leave the pipe idle.
// Tensor memory: O_0 [0,128), O_1 [128,256), S buffers [256,384) and [384,512).
// P(j) (bf16) is written over the first 64 columns of S buffer j&1 and read from there by the PV
// MMA, in two halves of 64 keys: the PV issuer starts on the first half while the softmax still
// exponentiates the second.  S(j+2) overwrites P(j), so the S issuer waits for PV(j) to complete
// before it issues S(j+2); by the time a warpgroup sees S(j+2), its previous PV into the same
// accumulator is therefore complete, and a rescale of that accumulator (done right after the row
// maximum, before P is produced) needs no further wait.
//
// d = 256 (6 warps): one softmax warpgroup (warps 0-3) takes every tile, warp 4 is the producer,
// warp 5 alone issues S(j+1) before PV(j) (a tile keeps the tensor core busy twice as long, and
// in-order completion makes S overwrite P only after PV read it).  Tensor memory: O [0,256),
// S buffers [256,384) and [384,512).  A rescale waits for PV(j-1) on a per-PV barrier.
//
// Value rows past a sequence's end are zeroed by the producer before the chunk is published
// (P is 0 there, but 0 * NaN = NaN for an uninitialised cache).
#pragma once

#include "common.cuh"

namespace ga {

template <int D_>
struct WideCfg {
  static constexpr int D = D_;
  static constexpr int BM = 128, BN = 128;
  static constexpr int Q_BYTES = BM * D * 2;            // D/64 slabs of 128 rows x 128 B
  static constexpr int CHUNK = 32768;                   // ring chunk
  static constexpr int KCH = D / 128;                   // K chunks per key tile (128 dims each)
  static constexpr int VCH = D / 128;                   // V chunks per key tile
  static constexpr int VK = 16384 / D;                  // keys per V chunk
  static constexpr int RING = 4;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = OFF_Q + Q_BYTES;
  static constexpr int OFF_BAR = OFF_RING + RING * CHUNK;
  static constexpr int OFF_XCH = OFF_BAR + 256;         // epilogue (m, l) exchange (d = 128)
  static constexpr int LIST_MAX = 2048;                 // block-mask tile list: tiles (2 units each)
  static constexpr int OFF_LIST = OFF_XCH + 2 * BM * 8;
  static constexpr int SMEM_BYTES = OFF_LIST + 2 * LIST_MAX * 4 + 1024;
  // d = 128: two softmax warpgroups on alternate key tiles, separate S and PV issuers.
  // d = 256 (O alone fills half of tensor memory): one softmax warpgroup, one issuer.
  static constexpr bool DUAL = D == 128;
  static constexpr int NWG = DUAL ? 2 : 1;              // softmax warpgroups
  static constexpr int W_PROD = 4 * NWG;                // producer warp
  static constexpr int W_S = W_PROD + 1;                // S issuer (the only issuer for d = 256)
  static constexpr int W_PV = W_PROD + 2;               // PV issuer (d = 128)
  static constexpr int THREADS = DUAL ? 384 : 192;
  static constexpr uint32_t COL_O = 0, COL_S = 256;     // O_b at 128 b (d = 128); S_b at 256 + 128 b
  // register split (d = 128): launched at 168 a thread (384 threads, one CTA per SM)
  static constexpr int LAUNCH_REGS = 168, SOFTMAX_REGS = 200, OTHER_REGS = 96;
  static_assert(!DUAL || 256 * SOFTMAX_REGS + 128 * OTHER_REGS <= THREADS * LAUNCH_REGS, "register split");
  static_assert(D == 128 || D == 256, "head dim");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(NWG * D + 2 * BN <= 512 && COL_S == NWG * D, "tensor memory budget");
};

struct WideBars {
  uint64_t q_full;
  uint64_t full[6], empty[6];
  uint64_t s_full[2], p_full[2][2], o_done, o_final, v_tail, mma_drain[2];
  uint64_t p_free[2];           // PV of the tile in S buffer b has completed (d = 128)
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(WideBars) <= 256, "barrier area");

// What the epilogue writes.  Differential attention ("Attention Variants": (A1 - lambda A2) V)
// runs the kernel twice: the first pass keeps its normalised output in fp32 (mode 1), the
// second subtracts lambda times its own from it before the single rounding to bf16 (mode 2),
// so the cancellation between the two maps happens in fp32.
struct WideEpi {
  int mode;             // 0: out (bf16); 1: out32 (fp32); 2: out = sub - lam * result (bf16)
  float* out32;         // mode 1: [batch, n_heads, Tq, D]
  const float* sub;     // mode 2: [batch, n_heads, Tq, D]
  float lam;
};

// A list entry naming no unit: the tile holds one unit, in its first half.
constexpr uint32_t kUnitNone = 0xFFFFFFFFu;

// grid: (n_qt * n_heads * batch); block: 384 threads (d = 128) or 192 (d = 256); 1 CTA per SM.
// Tensor maps (64-column SW128 boxes): tm_q 128 rows; tm_k 128 keys; tm_v 16384/d keys;
// tm_k64 and tm_v64 64 keys (the 64-key units of a block-masked tile).
// UNITS: the launch has a block mask (tiles are lists of 64-key units); without one the
// kernel compiles to contiguous 128-key tiles only.
// EPI: the epilogue's mode (WideEpi::mode), fixed at compile time so that plain launches carry
// none of the other modes' code.
template <int D_, bool UNITS, int EPI = 0>
__global__ void __launch_bounds__(WideCfg<D_>::THREADS, 1)
prefill_wide_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_k64,
                    const __grid_constant__ CUtensorMap tm_v64, __nv_bfloat16* __restrict__ out,
                    float* __restrict__ lse, AttnShape sh, WideEpi epi) {
  using C = WideCfg<D_>;
  constexpr int D = C::D, BN = C::BN;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sQ = smem + C::OFF_Q;
  unsigned char* sR = smem + C::OFF_RING;
  WideBars* bars = reinterpret_cast<WideBars*>(smem + C::OFF_BAR);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = (sh.Tq + C::BM - 1) / C::BM;
  const int hb = sh.n_heads * sh.batch;
  const int qr = (int)(blockIdx.x / hb), rem = (int)(blockIdx.x % hb);
  const int h = rem % sh.n_heads, b = rem / sh.n_heads;
  const int qt = n_qt - 1 - qr;                          // heaviest causal tiles first
  const int kvh = h / (sh.n_heads / sh.n_kv);
  const uint64_t tmo = sh.timeout_ns;
  const int Tk = seq_keys(sh.k_lens, b, sh.Tk_max);

  // key range of the tile's rows and its 128-key tiles
  const int t0 = qt * C::BM;
  const int rows = min(C::BM, sh.Tq - t0);
  const long long i_first = (long long)Tk - sh.Tq + t0, i_last = i_first + rows - 1;
  const int key_lo = sh.window > 0 ? (int)max(0LL, i_first - sh.window + 1) : 0;
  int key_hi = sh.causal ? (int)min((long long)Tk, i_last + 1) : Tk;
  if (key_hi < key_lo) key_hi = key_lo;
  const int kt_lo = key_lo / BN;
  int n_tiles = key_hi > key_lo ? (key_hi + BN - 1) / BN - kt_lo : 0;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::RING; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->s_full[0], 1);
    mbar_init(&bars->s_full[1], 1);
    for (int b2 = 0; b2 < 4; ++b2) mbar_init(&bars->p_full[b2 >> 1][b2 & 1], 4);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->o_final, 1);
    mbar_init(&bars->v_tail, 1);
    mbar_init(&bars->mma_drain[0], 1);
    mbar_init(&bars->mma_drain[1], 1);
    mbar_init(&bars->p_free[0], 1);
    mbar_init(&bars->p_free[1], 1);
    bars->abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == C::W_S) tmem_alloc(&bars->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  // ---- block mask: the selected 64-key units of this query tile, in key order, paired into
  // 128-key tiles (unit list_a[t] in the first half of tile t, list_b[t] in the second).  Keys
  // of a tile need not be adjacent -- the softmax masks each half from its own base -- and the
  // order of tiles does not change the result, so the work is proportional to the selected
  // units.  A list that would not fit leaves the contiguous tiles, masked per half.
  const uint8_t* mrow = UNITS && sh.block_mask
      ? sh.block_mask + (((size_t)b * sh.n_heads + h) * sh.nQb + t0 / sh.q_block) * sh.nKb
      : nullptr;
  uint32_t* list_a = reinterpret_cast<uint32_t*>(smem + C::OFF_LIST);
  uint32_t* list_b = list_a + C::LIST_MAX;
  bool list = false;
  if (UNITS && mrow != nullptr && n_tiles > 0) {
    int* cnt = reinterpret_cast<int*>(smem + C::OFF_XCH);   // [0] total, [1 + w] per warp
    const int u_lo = key_lo / 64, u_hi = (key_hi + 63) / 64;
    auto selected = [&](int u) -> bool { return u < u_hi && mrow[(64 * u) / sh.k_block] != 0; };
    if (threadIdx.x == 0) cnt[0] = 0;
    __syncthreads();
    int mine = 0;
    for (int u = u_lo + (int)threadIdx.x; u < u_hi; u += C::THREADS) mine += selected(u) ? 1 : 0;
    mine = __reduce_add_sync(0xffffffffu, mine);
    if (lane == 0 && mine) atomicAdd(&cnt[0], mine);
    __syncthreads();
    const int total = cnt[0];
    if (total <= 2 * C::LIST_MAX) {
      list = true;
      int run = 0;                                   // units placed so far (same in all threads)
      const uint32_t lt = (1u << lane) - 1u;
      for (int base = u_lo; base < u_hi; base += C::THREADS) {
        const int u = base + (int)threadIdx.x;
        const bool sel = selected(u);
        const uint32_t bal = __ballot_sync(0xffffffffu, sel);
        if (lane == 0) cnt[1 + warp] = __popc(bal);
        __syncthreads();
        if (sel) {
          int rank = run + __popc(bal & lt);
          for (int w = 0; w < warp; ++w) rank += cnt[1 + w];
          (rank & 1 ? list_b : list_a)[rank >> 1] = (uint32_t)u;
        }
        for (int w = 0; w < C::THREADS / 32; ++w) run += cnt[1 + w];
        __syncthreads();
      }
      if (threadIdx.x == 0 && (total & 1)) list_b[total >> 1] = kUnitNone;
      __syncthreads();
      n_tiles = (total + 1) / 2;
    }
  }
  // Tile t: the 64-key units of its two halves and which halves hold keys of this query tile
  // (bit 0: first half, bit 1: second).  A lone unit is loaded into both halves, the second
  // masked, so that no half ever holds unloaded data.
  auto tile_units = [&](int t, int& ua, int& ub, uint32_t& present) {
    if (UNITS && list) {
      const uint32_t lb = list_b[t];
      ua = (int)list_a[t];
      ub = lb == kUnitNone ? ua : (int)lb;
      present = lb == kUnitNone ? 1u : 3u;
    } else {
      ua = 2 * (kt_lo + t);
      ub = ua + 1;
      present = 3u;
      if (UNITS && mrow != nullptr)
        present = (mrow[(64 * ua) / sh.k_block] ? 1u : 0u) |
                  ((64 * ub < sh.Tk_max && mrow[(64 * ub) / sh.k_block]) ? 2u : 0u);
    }
  };

  if (warp >= C::W_PROD) {
    if constexpr (C::DUAL) regs_dec<C::OTHER_REGS>();
    if (warp == C::W_PROD) {
      // ------------------------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        const int qz = b * sh.n_heads + h, kz = b * sh.n_kv + kvh;
        mbar_arrive_expect_tx(&bars->q_full, C::Q_BYTES);
        for (int s = 0; s < D / 64; ++s)
          tma_load_3d(sQ + s * C::BM * 128, &tm_q, &bars->q_full, 64 * s, t0, qz);
        int cnt = 0, n_tail = 0;                           // chunks issued, tail chunks
        bool ok = true;
        // acquire ring slot for chunk number cnt
        auto slot_acquire = [&](int& slot) -> bool {
          slot = cnt % C::RING;
          if (cnt >= C::RING && !mbar_wait(&bars->empty[slot], ((cnt / C::RING) + 1) & 1, tmo, abort_flag))
            return false;
          return true;
        };
        // With a block mask every half of a tile is a 64-key unit of its own (64-row boxes);
        // otherwise tile j is the contiguous keys 128 (kt_lo + j) ... (128-row boxes).
        constexpr bool units = UNITS;
        auto load_k = [&](int j) -> bool {                 // K(j): chunks of 128 dims
          int ua, ub;
          uint32_t pr;
          tile_units(j, ua, ub, pr);
          for (int c = 0; c < C::KCH; ++c) {
            int slot;
            if (!slot_acquire(slot)) return false;
            unsigned char* dst = sR + slot * C::CHUNK;
            mbar_arrive_expect_tx(&bars->full[slot], C::CHUNK);
            for (int s = 0; s < 2; ++s) {
              if (!units) {
                tma_load_3d(dst + s * BN * 128, &tm_k, &bars->full[slot], 128 * c + 64 * s, (kt_lo + j) * BN, kz);
              } else {
                tma_load_3d(dst + s * BN * 128, &tm_k64, &bars->full[slot], 128 * c + 64 * s, 64 * ua, kz);
                tma_load_3d(dst + s * BN * 128 + 64 * 128, &tm_k64, &bars->full[slot], 128 * c + 64 * s, 64 * ub, kz);
              }
            }
            ++cnt;
          }
          return true;
        };
        auto load_v = [&](int j) -> bool {                 // V(j): chunks of VK keys x D dims
          int ua, ub;
          uint32_t pr;
          tile_units(j, ua, ub, pr);
          constexpr int PARTS = C::VK / 64;                // 64-key units per chunk
          for (int c = 0; c < C::VCH; ++c) {
            int slot;
            if (!slot_acquire(slot)) return false;
            unsigned char* dst = sR + slot * C::CHUNK;
            // unit of part p: half PARTS * c + p of the tile
            auto part_unit = [&](int p) { return (PARTS * c + p) == 0 ? ua : ub; };
            bool tail = false;
            for (int p = 0; p < PARTS; ++p) tail |= 64 * part_unit(p) + 64 > Tk;
            uint64_t* bar = tail ? &bars->v_tail : &bars->full[slot];
            mbar_arrive_expect_tx(bar, C::CHUNK);
            for (int s = 0; s < D / 64; ++s) {
              if (!units) {
                tma_load_3d(dst + s * C::VK * 128, &tm_v, bar, 64 * s, (kt_lo + j) * BN + C::VK * c, kz);
              } else {
                for (int p = 0; p < PARTS; ++p)
                  tma_load_3d(dst + s * C::VK * 128 + p * 64 * 128, &tm_v64, bar, 64 * s, 64 * part_unit(p), kz);
              }
            }
            if (tail) {
              if (!mbar_wait(&bars->v_tail, n_tail & 1, tmo, abort_flag)) return false;
              ++n_tail;
              for (int p = 0; p < PARTS; ++p)
                for (int row = max(0, Tk - 64 * part_unit(p)); row < 64; ++row)
                  for (int s = 0; s < D / 64; ++s)
                    for (int q16 = 0; q16 < 8; ++q16)
                      *reinterpret_cast<uint4*>(dst + s * C::VK * 128 + (p * 64 + row) * 128 + q16 * 16) =
                          make_uint4(0, 0, 0, 0);
              fence_proxy_async_smem();
              mbar_arrive(&bars->full[slot]);
            }
            ++cnt;
          }
          return true;
        };
        if (n_tiles > 0) ok = load_k(0);
        for (int j = 0; ok && j < n_tiles; ++j) {
          if (j + 1 < n_tiles) ok = load_k(j + 1);
          if (ok) ok = load_v(j);
        }
        // Drain: the most recent chunk of every slot has landed before the CTA may exit.
        mbar_wait(&bars->q_full, 0, tmo, nullptr);
        for (int k = max(0, cnt - C::RING); k < cnt; ++k)
          mbar_wait(&bars->full[k % C::RING], (k / C::RING) & 1, tmo, nullptr);
      }
    } else if (warp == C::W_S || warp == C::W_PV) {
      // The issuer warps issue MMAs and nothing else.
      if constexpr (!C::DUAL) {
        // ------------------------------------------------------------------ one MMA issuer (d = 256)
        if (lane == 0 && warp == C::W_S) {
          constexpr uint32_t idesc_s = idesc_bf16_f32(128, BN, false);
          constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
          const uint64_t dq = sdesc_sw128(smem_u32(sQ), 16, 1024);
          const uint64_t dr_k = sdesc_sw128(smem_u32(sR), 16, 1024);       // K chunks: K-major
          const uint64_t dr_v = sdesc_sw128(smem_u32(sR), C::VK * 128, 1024);   // V chunks: MN-major
          int cnt = 0;
          bool ok = mbar_wait(&bars->q_full, 0, tmo, abort_flag);
          // S(j) into buffer j & 1 from K(j)'s chunks
          auto issue_s = [&](int j) -> bool {
            const uint32_t d_s = tmem + C::COL_S + (j & 1) * BN;
            for (int c = 0; c < C::KCH; ++c) {
              const int slot = cnt % C::RING;
              if (!mbar_wait(&bars->full[slot], (cnt / C::RING) & 1, tmo, abort_flag)) return false;
              tc_fence_after();
              const uint64_t bk = dr_k + (uint64_t)((slot * C::CHUNK) >> 4);
    #pragma unroll
              for (int k8 = 0; k8 < 8; ++k8) {                // 8 steps of 16 dims in this chunk
                const int kk = 8 * c + k8;
                const uint64_t aq = dq + (uint64_t)(((kk >> 2) * C::BM * 128 + (kk & 3) * 32) >> 4);
                const uint64_t bo = bk + (uint64_t)(((k8 >> 2) * BN * 128 + (k8 & 3) * 32) >> 4);
                umma_bf16_ss(d_s, aq, bo, idesc_s, kk > 0 ? 1u : 0u);
              }
              umma_commit(&bars->empty[slot]);
              ++cnt;
            }
            umma_commit(&bars->s_full[j & 1]);
            return true;
          };
          // O += P(j) V(j), P in the first 64 columns of S buffer j & 1
          uint32_t o_acc = 0u;
          auto issue_pv = [&](int j) -> bool {
            const uint32_t p_col = tmem + C::COL_S + (j & 1) * BN;
            for (int c = 0; c < C::VCH; ++c) {
              const int slot = cnt % C::RING;
              if (!mbar_wait(&bars->full[slot], (cnt / C::RING) & 1, tmo, abort_flag)) return false;
              tc_fence_after();
              const uint64_t bv = dr_v + (uint64_t)((slot * C::CHUNK) >> 4);
    #pragma unroll
              for (int k4 = 0; k4 < C::VK / 16; ++k4) {       // steps of 16 keys in this chunk
                const int kk = (C::VK / 16) * c + k4;
                umma_bf16_ts(tmem + C::COL_O, p_col + kk * 8, bv + (uint64_t)((k4 * 2048) >> 4), idesc_pv,
                             (o_acc | (uint32_t)k4) ? 1u : 0u);
              }
              o_acc = 1u;
              umma_commit(&bars->empty[slot]);
              ++cnt;
            }
            return true;
          };
          if (ok && n_tiles > 0) ok = issue_s(0);
          for (int j = 0; ok && j < n_tiles; ++j) {
            if (j + 1 < n_tiles && !(ok = issue_s(j + 1))) break;
            if (!(ok = mbar_wait(&bars->p_full[0][0], j & 1, tmo, abort_flag))) break;
            tc_fence_after();
            if (!(ok = issue_pv(j))) break;
            umma_commit(&bars->o_done);
            if (j + 1 == n_tiles) umma_commit(&bars->o_final);
          }
          // Drain: every MMA this thread issued has completed before TMEM can be released.
          umma_commit(&bars->mma_drain[0]);
          mbar_wait(&bars->mma_drain[0], 0, tmo, nullptr);
        }
      } else {
        // ------------------------------------------------------------------ MMA issuers (d = 128)
        // Both find their chunks in the ring from the producer's order: K(0), then K(j+1), V(j)
        // for j = 0, 1, ... (K(n) is not loaded), one chunk each.
        static_assert(C::KCH == 1 && C::VCH == 1 && C::VK == C::BN, "d = 128 chunk layout");
        if (lane == 0) {
          constexpr uint32_t idesc_s = idesc_bf16_f32(128, BN, false);
          constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
          const uint64_t dq = sdesc_sw128(smem_u32(sQ), 16, 1024);
          const uint64_t dr_k = sdesc_sw128(smem_u32(sR), 16, 1024);       // K chunks: K-major
          const uint64_t dr_v = sdesc_sw128(smem_u32(sR), C::VK * 128, 1024);   // V chunks: MN-major
          const int xi = warp - C::W_S;                    // 0: S issuer, 1: PV issuer
          auto kpos = [&](int j) { return j == 0 ? 0 : 2 * j - 1; };
          auto vpos = [&](int j) { return j + 1 < n_tiles ? 2 * j + 2 : 2 * j + 1; };
          bool ok = xi == 1 || mbar_wait(&bars->q_full, 0, tmo, abort_flag);
          for (int j = 0; ok && j < n_tiles; ++j) {
            const int buf = j & 1;
            if (xi == 0) {
              // S(j) into buffer j & 1, once PV(j-2) has read the P held there.  K(j) is waited
              // for first: it has usually landed long before, so only the PV wait is exposed.
              const int pos = kpos(j), slot = pos % C::RING;
              if (!(ok = mbar_wait(&bars->full[slot], (pos / C::RING) & 1, tmo, abort_flag))) break;
              if (j >= 2 && !(ok = mbar_wait(&bars->p_free[buf], ((j >> 1) - 1) & 1, tmo, abort_flag))) break;
              tc_fence_after();
              const uint32_t d_s = tmem + C::COL_S + buf * BN;
              const uint64_t bk = dr_k + (uint64_t)((slot * C::CHUNK) >> 4);
    #pragma unroll
              for (int kk = 0; kk < 8; ++kk) {                 // 8 steps of 16 dims
                const uint64_t aq = dq + (uint64_t)(((kk >> 2) * C::BM * 128 + (kk & 3) * 32) >> 4);
                const uint64_t bo = bk + (uint64_t)(((kk >> 2) * BN * 128 + (kk & 3) * 32) >> 4);
                umma_bf16_ss(d_s, aq, bo, idesc_s, kk > 0 ? 1u : 0u);
              }
              umma_commit(&bars->empty[slot]);
              umma_commit(&bars->s_full[buf]);
            } else {
              // O_(j&1) += P(j) V(j), P in the first 64 columns of S buffer j & 1.  The softmax
              // publishes P in two halves of 64 keys; the first half's MMAs run while the
              // second half is exponentiated.
              const int pos = vpos(j), slot = pos % C::RING;
              if (!(ok = mbar_wait(&bars->full[slot], (pos / C::RING) & 1, tmo, abort_flag))) break;
              const uint32_t p_col = tmem + C::COL_S + buf * BN;
              const uint32_t d_o = tmem + C::COL_O + buf * D;
              const uint64_t bv = dr_v + (uint64_t)((slot * C::CHUNK) >> 4);
              for (int half = 0; ok && half < 2; ++half) {
                if (!(ok = mbar_wait(&bars->p_full[buf][half], (j >> 1) & 1, tmo, abort_flag))) break;
                tc_fence_after();
    #pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {               // 4 steps of 16 keys
                  const int kk = 4 * half + k4;
                  umma_bf16_ts(d_o, p_col + kk * 8, bv + (uint64_t)((kk * 2048) >> 4), idesc_pv,
                               (j >= 2 || kk > 0) ? 1u : 0u);
                }
              }
              if (!ok) break;
              umma_commit(&bars->empty[slot]);
              umma_commit(&bars->p_free[buf]);
              if (j + 1 == n_tiles) umma_commit(&bars->o_final);
            }
          }
          // Drain: every MMA this thread issued has completed before TMEM can be released.
          umma_commit(&bars->mma_drain[xi]);
          mbar_wait(&bars->mma_drain[xi], 0, tmo, nullptr);
        }
      }
      __syncwarp();
  }
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    if constexpr (C::DUAL) regs_inc<C::SOFTMAX_REGS>();
    const int wg = warp >> 2;                         // key tiles wg, wg + NWG, wg + 2 NWG, ...
    const int row = threadIdx.x & 127;                // query row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_o = tmem + C::COL_O + wg * D + lane_off;
    const long long i = i_first + row;                // absolute position of this row
    const int lo = sh.window > 0 ? (int)max(0LL, i - sh.window + 1) : 0;
    const int hi = sh.causal ? (int)min((long long)Tk, i + 1) : Tk;
    const int lo_all = sh.window > 0 ? (int)max(0LL, i_last - sh.window + 1) : 0;
    const int hi_all = sh.causal ? (int)min((long long)Tk, i_first + 1) : Tk;
    const float scale_log2 = kLog2e / sqrtf((float)D);
    float m_run = -INFINITY, l_run = 0.0f;            // this warpgroup's share of the keys
    if (sh.sink && wg == 0) { m_run = sh.sink[h] * kLog2e; l_run = 1.0f; }

    for (int n = wg; n < n_tiles; n += C::NWG) {
      const int buf = n & 1;
      if (!warp_wait(&bars->s_full[buf], (n >> 1) & 1, tmo, abort_flag)) break;
      tc_fence_after();
      const uint32_t t_s = tmem + C::COL_S + buf * BN + lane_off;
      float sv[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
        tmem_ld32(t_s + 32 * c, *reinterpret_cast<float(*)[32]>(&sv[32 * c]));
      tmem_wait_ld();
      // keys of the two 64-column halves start at 64 ua and 64 ub
      int ua, ub;
      uint32_t pr;
      tile_units(n, ua, ub, pr);
      const int kb0 = 64 * ua, kb1 = 64 * ub;
      const bool interior = UNITS ? pr == 3u && kb0 >= lo_all && kb0 + 64 <= hi_all && kb1 >= lo_all && kb1 + 64 <= hi_all
                                  : kb0 >= lo_all && kb0 + BN <= hi_all;
      if (!interior) {
        const int lo0 = (pr & 1u) ? lo : 0x7fffffff, lo1 = (pr & 2u) ? lo : 0x7fffffff;   // absent half: no key
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const int jj = c < 64 ? kb0 + c : kb1 + (c - 64);
          sv[c] = (jj >= (c < 64 ? lo0 : lo1) && jj < hi) ? sv[c] : -INFINITY;
        }
      }
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
      auto rescale_o = [&]() {
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float o[32];
          tmem_ld32(t_o + c, o);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] *= alpha;
          tmem_st32(t_o + c, o);
        }
      };
      // d = 128: the accumulator's previous PV, PV(n-2), completed before S(n) was issued, so
      // the rescale can run before P is produced (PV(n) must see the rescaled accumulator).
      if constexpr (C::DUAL)
        if (n >= C::NWG && __any_sync(0xffffffffu, need)) rescale_o();
      float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32) {
        if constexpr (C::DUAL) {
          if (c0 == BN / 2) {                           // keys [0, 64) of P are in place
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_full[buf][0]);
          }
        }
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          float e0, e1, e2, e3;
          ffma2(e0, e1, sv[c0 + c], sv[c0 + c + 1], scale_log2, scale_log2, -m_use, -m_use);
          ffma2(e2, e3, sv[c0 + c + 2], sv[c0 + c + 3], scale_log2, scale_log2, -m_use, -m_use);
          const float p0 = ex2(e0), p1 = ex2(e1), p2 = ex2(e2), p3 = ex2(e3);
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
      if constexpr (!C::DUAL) {
        // d = 256: PV(n-1) may still accumulate into O, so the rescale waits for it (PV(n-2)
        // is complete) and runs last.
        if (n >= C::NWG && __any_sync(0xffffffffu, need)) {
          if (!warp_wait(&bars->o_done, (n - 1) & 1, tmo, abort_flag)) break;
          tc_fence_after();
          rescale_o();
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(C::DUAL ? &bars->p_full[buf][1] : &bars->p_full[0][0]);
    }

    // ---- epilogue: O / l from TMEM to global ------------------------------------------
    bool ok = __all_sync(0xffffffffu, *abort_flag == 0);
    if (ok && n_tiles > 0) ok = warp_wait(&bars->o_final, 0, tmo, abort_flag);
    tc_fence_after();
    const int t = t0 + row;
    const size_t orow_off = (((size_t)b * sh.n_heads + h) * sh.Tq + t) * D;
    __nv_bfloat16* orow = out + orow_off;
    auto store32 = [&](int c, const float (&o)[32], float s0) {
      if (row < rows) {
#pragma unroll
        for (int u = 0; u < 32; u += 8) {
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = o[u + e] * s0;
          if constexpr (EPI == 1) {
            float* dst = epi.out32 + orow_off + c + u;
            *reinterpret_cast<float4*>(dst) = make_float4(x[0], x[1], x[2], x[3]);
            *reinterpret_cast<float4*>(dst + 4) = make_float4(x[4], x[5], x[6], x[7]);
            continue;
          }
          if constexpr (EPI == 2) {
            const float* src = epi.sub + orow_off + c + u;
            const float4 a = *reinterpret_cast<const float4*>(src), b4 = *reinterpret_cast<const float4*>(src + 4);
            const float y[8] = {a.x, a.y, a.z, a.w, b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = fmaf(-epi.lam, x[e], y[e]);
          }
          uint4 pk;
          pk.x = pack_bf16x2(x[0], x[1]);
          pk.y = pack_bf16x2(x[2], x[3]);
          pk.z = pack_bf16x2(x[4], x[5]);
          pk.w = pack_bf16x2(x[6], x[7]);
          *reinterpret_cast<uint4*>(orow + c + u) = pk;
        }
      }
    };
    if constexpr (C::DUAL) {
      // Merge the warpgroups' partial results (running max m_w, sum l_w, accumulator O_w, all
      // relative to 2^m_w): out = sum_w 2^(m_w - M) O_w / sum_w 2^(m_w - M) l_w.  The warpgroups
      // swap (m, l) through shared memory; warpgroup w then writes columns [64 w, 64 w + 64).
      float2* xch = reinterpret_cast<float2*>(smem + C::OFF_XCH);
      if (ok) xch[wg * C::BM + row] = make_float2(m_run, l_run);
      asm volatile("bar.sync 1, 256;" ::: "memory");
      const float2 other = xch[(wg ^ 1) * C::BM + row];
      const float m0 = wg == 0 ? m_run : other.x, l0 = wg == 0 ? l_run : other.y;
      const float m1 = wg == 0 ? other.x : m_run, l1 = wg == 0 ? other.y : l_run;
      const float M = fmaxf(m0, m1);
      const float a0 = M == -INFINITY ? 0.0f : ex2(m0 - M);
      const float a1 = M == -INFINITY ? 0.0f : ex2(m1 - M);
      const float L = l0 * a0 + l1 * a1;
      const float inv_l = L > 0.0f ? 1.0f / L : 0.0f;
      const float s0 = a0 * inv_l, s1 = a1 * inv_l;
      if (ok) {
        const uint32_t t_o0 = tmem + C::COL_O + lane_off, t_o1 = t_o0 + D;
#pragma unroll 1
        for (int c = 64 * wg; c < 64 * wg + 64; c += 32) {
          float o0[32], o1[32];
          if (n_tiles > 0) tmem_ld32(t_o0 + c, o0);
          if (n_tiles > 1) tmem_ld32(t_o1 + c, o1);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const float x0 = n_tiles > 0 ? o0[u] : 0.0f, x1 = n_tiles > 1 ? o1[u] : 0.0f;
            o0[u] = fmaf(x0, s0, x1 * s1);
          }
          store32(c, o0, 1.0f);
        }
        if (lse && wg == 0 && row < rows)
          lse[((size_t)b * sh.n_heads + h) * sh.Tq + t] =
              L > 0.0f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
      }
    } else {
      const float inv_l = l_run > 0.0f ? 1.0f / l_run : 0.0f;
      if (ok) {
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float o[32];
          if (n_tiles > 0) {
            tmem_ld32(t_o + c, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int u = 0; u < 32; ++u) o[u] = 0.0f;
          }
          store32(c, o, inv_l);
        }
        if (lse && row < rows)
          lse[((size_t)b * sh.n_heads + h) * sh.Tq + t] =
              l_run > 0.0f ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == C::W_S) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace ga
