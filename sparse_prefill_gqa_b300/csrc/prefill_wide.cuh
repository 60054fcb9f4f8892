// prefill_wide.cuh -- bf16 attention prefill on the tensor cores, head dim 128 or 256: causal,
// window, sink, and block-sparse (a block mask over 64-key units).  A persistent kernel: one CTA
// per SM walks a fixed sequence of 128-row query tiles ("items").
//
// What it computes ("Attention in Code", "one function all designs use": scores q.k/sqrt(d),
// masked positions removed, optional sink logit in the normaliser, weighted sum of values;
// section 1 head grouping; the absolute-position causal rule; the sliding window of section 2),
// restricted to the selected key blocks when a block mask is given ("RBS-Attention review":
// attention is computed only over the blocks the selection keeps).
//
// Items are numbered heaviest causal tiles first, in blocks of query tiles whose items that
// share a kv head are numbered together (wide_item); a CTA's
// producer takes the next unclaimed item from a launch-wide counter, one item ahead of the one
// it loads (so the longest items start first and the CTAs finish together whatever the sequence
// lengths), and publishes it to the CTA's other roles.  The warps run decoupled across items:
// while the softmax
// warpgroups finish one item (the last tiles and the epilogue), the producer already loads the
// next item's Q and first K tiles and the S issuer computes its first scores, so a CTA's start
// and end are hidden behind the work of its neighbours in the sequence.  Every barrier phase and
// ring position is counted over the CTA's whole sequence, not per item.
//
// Block masks: the producer warp lists the selected 64-key units of the item's query tile, in
// key order, and pairs them into 128-key tiles; each half of a tile is loaded as its own 64-key
// box and masked from its own key base, so the work is proportional to the selected units and
// the MMAs stay full width.  It publishes each item's tile count with the item (item ring)
// and each tile's units (tile-info ring) to the other roles.  Launches without a block mask
// use the instantiation UNITS = false, where the tiles follow from the indices.
//
// d = 128 (12 warps): two softmax warpgroups split each item's key tiles between them, warpgroup
// w the tiles j of the item with j % 2 == w, each with its own running max and sum and its own
// output accumulator O_w in tensor memory; the epilogue merges the two partial results by the
// log-sum-exp rule (the same re-association as split-K decode).  The split depends on the item
// alone, never on which items the CTA ran before, so results do not depend on the scheduling.
// Tile j of an item uses S buffer j % 2 and accumulates into O_(j%2): buffer, accumulator and
// warpgroup go together, and each role counts the uses of each buffer (the barrier phases)
// across the CTA's items.
//   warps 0-3, 4-7  softmax: thread r of a warpgroup = query row r = TMEM lane r;
//   warp 8          producer: Q once per item, then K and V through a ring of 32 KB chunks
//                   (5 slots), K one tile ahead of V; lists the units of block-masked items;
//   warp 9          S issuer (one lane): S(j) = Q K(j)^T into S buffer j % 2;
//   warp 10         PV issuer (one lane): O_(j%2) += P(j) V(j), j the tile's index in its item;
//   warp 11         idle (completes the warpgroup whose registers move to the softmax).
// Tensor memory: O_0 [0,128), O_1 [128,256), S buffers [256,384) and [384,512).  P (bf16) is
// written over the first 64 columns of its tile's S buffer and read from there by the PV MMA, in
// two halves of 64 keys.  The next S into a buffer overwrites that P, so the S issuer waits for
// its PV first.  The first PV of an item into an accumulator waits until the previous item's
// epilogue has read it.
//
// d = 256 (6 warps): one softmax warpgroup takes every tile, warp 4 is the producer, warp 5
// alone issues S(J+1) before PV(J) (in-order completion makes S overwrite P only after PV read
// it).  Tensor memory: O [0,256), S buffers [256,384) and [384,512).  Ring of 4 slots.
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
  // d = 128: two softmax warpgroups on alternate key tiles, separate S and PV issuers.
  // d = 256 (O alone fills half of tensor memory): one softmax warpgroup, one issuer.
  static constexpr bool DUAL = D == 128;
  static constexpr int RING = DUAL ? 5 : 4;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = OFF_Q + Q_BYTES;
  static constexpr int OFF_BAR = OFF_RING + RING * CHUNK;
  static constexpr int BAR_BYTES = 512;
  static constexpr int OFF_XCH = OFF_BAR + BAR_BYTES;   // epilogue (m, l) exchange, two items (d = 128)
  static constexpr int TINFO = 8;                       // tile-info ring (block masks)
  static constexpr int OFF_TINFO = OFF_XCH + 2 * 2 * BM * 8;
  static constexpr int IINFO = 4;                       // item ring (block masks)
  static constexpr int OFF_IINFO = OFF_TINFO + TINFO * 16;        // IINFO x int2 (item, tiles)
  static constexpr int LIST_MAX = 2048;                 // block-mask tile list: tiles (2 units each)
  static constexpr int OFF_LIST = OFF_IINFO + 64;       // 2 x LIST_MAX 16-bit unit indices
  static constexpr int OFF_STAGE = (OFF_LIST + 2 * LIST_MAX * 2 + 127) / 128 * 128;   // epilogue: 2 KB a softmax warp
  static constexpr int SMEM_BYTES = OFF_STAGE + 8 * 2048 + 1024;
  static constexpr int NWG = DUAL ? 2 : 1;              // softmax warpgroups
  static constexpr int SM_THREADS = 128 * NWG;          // softmax threads
  static constexpr int W_PROD = 4 * NWG;                // producer warp
  static constexpr int W_S = W_PROD + 1;                // S issuer (the only issuer for d = 256)
  static constexpr int W_PV = W_PROD + 2;               // PV issuer (d = 128)
  static constexpr int THREADS = DUAL ? 384 : 192;
  static constexpr int ITEM_READERS = (DUAL ? 2 : 1) + 4 * NWG;   // issuers + softmax warps
  static constexpr uint32_t COL_O = 0, COL_S = 256;     // O_b at 128 b (d = 128); S_b at 256 + 128 b
  // register split (d = 128): launched at 168 a thread (384 threads, one CTA per SM)
  static constexpr int LAUNCH_REGS = 168, SOFTMAX_REGS = 200, OTHER_REGS = 96;
  static_assert(!DUAL || 256 * SOFTMAX_REGS + 128 * OTHER_REGS <= THREADS * LAUNCH_REGS, "register split");
  static_assert(D == 128 || D == 256, "head dim");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(NWG * D + 2 * BN <= 512 && COL_S == NWG * D, "tensor memory budget");
};

struct WideBars {
  uint64_t q_full, q_free;
  uint64_t full[6], empty[6];
  uint64_t s_full[2], p_full[2][2], p_free[2];
  uint64_t o_done, o_final, o_free, v_tail, mma_drain[2];
  uint64_t item_full[4], item_empty[4];
  uint64_t tinfo_full[8];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(WideBars) <= 512, "barrier area");

// The units of one 128-key tile (block-mask launches): key bases 64 ua and 64 ub of its two
// halves, and which halves hold keys of the item (bit 0: first half, bit 1: second).
struct WideTile {
  int ua, ub;
  uint32_t present;
  int pad;
};

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
constexpr uint16_t kUnitNone = 0xFFFFu;

// Launch-wide item counters.  Launch number e (host side, modulo kWideEpochs) claims items from
// g_wide_next[e] and counts its finished CTAs in g_wide_done[e]; the last CTA to finish sets
// both back to zero for the launch that reuses the slot.  Launches on one stream never share a
// slot while running; launches in flight at the same time on different streams share one only
// when kWideEpochs launches separate them.
constexpr int kWideEpochs = 64;
__device__ unsigned g_wide_next[kWideEpochs];
__device__ unsigned g_wide_done[kWideEpochs];

// One item: a 128-row query tile of one (query head, sequence), and its key range.
struct WideItem {
  int b, h, kvh, t0, rows, Tk;
  long long i_first, i_last;   // absolute positions of the tile's first and last rows
  int key_lo, key_hi;          // keys any row of the tile may use: [key_lo, key_hi)
  int kt_lo, n_dense;          // first 128-key tile and the number of contiguous tiles
};

// Item w of the launch.  The query tiles are taken in blocks of QB = sh.item_qt_block from the
// last (the heaviest causal tiles) to the first; within a block, sequence by sequence and kv head
// by kv head, and for each kv head its block's query tiles (last first) times its query heads.
// So the items that read the same keys and values (one kv head's query heads and, for QB > 1,
// neighbouring query tiles) are claimed together and stream them through L2 at about the same
// time, while the heaviest tiles still start first.  QB = 1 is the plain order: query tile, then
// sequence, then head.
// Every role of the CTA decodes each item it takes, on the path between two items; FAST (the
// d = 256 kernel, whose items are short under a window) turns the divisions by launch constants
// into multiply-shifts (FastDiv).  The d = 128 kernel keeps hardware divisions in the plain
// order: measured, the multiply-shift form made its main loop 2 % slower.
template <int BM, int BN, bool FAST>
__device__ __forceinline__ WideItem wide_item(const AttnShape& sh, int w) {
  WideItem it;
  const int n_qt = (sh.Tq + BM - 1) / BM;
  const int g = sh.n_heads / sh.n_kv, QB = sh.item_qt_block;
  int qt;
  if (QB == 1 && FAST) {
    const int qr = sh.fd_hb.div(w), rem = w - qr * (sh.n_heads * sh.batch);
    it.b = sh.fd_h.div(rem);
    it.h = rem - it.b * sh.n_heads;
    it.kvh = sh.fd_g.div(it.h);
    qt = n_qt - 1 - qr;
  } else if (QB == 1) {
    const int hb = sh.n_heads * sh.batch;
    const int qr = w / hb, rem = w - qr * hb;
    it.b = rem / sh.n_heads;
    it.h = rem - it.b * sh.n_heads;
    it.kvh = it.h / g;
    qt = n_qt - 1 - qr;
  } else {
    const int per_block = QB * sh.n_heads * sh.batch;           // items of a full block
    const int k = FAST ? sh.fd_pb.div(w) : w / per_block, rem = w - k * per_block;
    const int cnt = min(QB, n_qt - QB * k);                     // query tiles in block k
    const int grp = FAST ? (cnt == QB ? sh.fd_cg : sh.fd_cgl).div(rem) : rem / (cnt * g);
    const int r2 = rem - grp * (cnt * g);
    it.b = FAST ? sh.fd_nkv.div(grp) : grp / sh.n_kv;
    it.kvh = grp - it.b * sh.n_kv;
    const int qi = FAST ? sh.fd_g.div(r2) : r2 / g;
    it.h = it.kvh * g + (r2 - qi * g);
    qt = n_qt - 1 - (QB * k + qi);
  }
  it.Tk = seq_keys(sh.k_lens, it.b, sh.Tk_max);
  it.t0 = qt * BM;
  it.rows = min(BM, sh.Tq - it.t0);
  it.i_first = (long long)it.Tk - sh.Tq + it.t0;
  it.i_last = it.i_first + it.rows - 1;
  it.key_lo = sh.window > 0 ? (int)max(0LL, it.i_first - sh.window + 1) : 0;
  int key_hi = sh.causal ? (int)max(0LL, min((long long)it.Tk, it.i_last + 1)) : it.Tk;
  if (key_hi < it.key_lo) key_hi = it.key_lo;
  it.key_hi = key_hi;
  it.kt_lo = it.key_lo / BN;
  it.n_dense = key_hi > it.key_lo ? (key_hi + BN - 1) / BN - it.kt_lo : 0;
  return it;
}

// Number of items (query tiles over every head and sequence) of a launch.
__host__ __device__ inline long long wide_items(const AttnShape& sh) {
  return (long long)((sh.Tq + 127) / 128) * sh.n_heads * sh.batch;
}

// grid: min(items, SMs) CTAs; block: 384 threads (d = 128) or 192 (d = 256); 1 CTA per SM.
// Tensor maps (64-column SW128 boxes): tm_q 128 rows; tm_k 128 keys; tm_v 16384/d keys;
// tm_k64 and tm_v64 64 keys (the 64-key units of a block-masked tile).
// UNITS: the launch has a block mask (tiles are lists of 64-key units); without one the
// kernel compiles to contiguous 128-key tiles only.
// EPI: the epilogue's mode (WideEpi::mode), fixed at compile time so that plain launches carry
// none of the other modes' code.
// drop_chunk: test only -- every CTA's producer skips the load of its ring chunk number
// drop_chunk (counted over the CTA's sequence), so the waits on it run out; -1 (always, outside
// the failure-path test) loads every chunk.
template <int D_, bool UNITS, int EPI = 0>
__global__ void __launch_bounds__(WideCfg<D_>::THREADS, 1)
prefill_wide_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_k64,
                    const __grid_constant__ CUtensorMap tm_v64, __nv_bfloat16* __restrict__ out,
                    float* __restrict__ lse, AttnShape sh, WideEpi epi, int epoch, int drop_chunk) {
  using C = WideCfg<D_>;
  constexpr int D = C::D, BN = C::BN, BM = C::BM;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sQ = smem + C::OFF_Q;
  unsigned char* sR = smem + C::OFF_RING;
  WideBars* bars = reinterpret_cast<WideBars*>(smem + C::OFF_BAR);
  WideTile* tinfo = reinterpret_cast<WideTile*>(smem + C::OFF_TINFO);
  int2* iinfo = reinterpret_cast<int2*>(smem + C::OFF_IINFO);
  uint16_t* list_a = reinterpret_cast<uint16_t*>(smem + C::OFF_LIST);
  uint16_t* list_b = list_a + C::LIST_MAX;
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = (int)wide_items(sh);
  const uint64_t tmo = sh.timeout_ns;
  const bool masked = UNITS && sh.block_mask != nullptr;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_free, 1);
    for (int s = 0; s < C::RING; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->s_full[0], 1);
    mbar_init(&bars->s_full[1], 1);
    for (int b2 = 0; b2 < 4; ++b2) mbar_init(&bars->p_full[b2 >> 1][b2 & 1], 4);
    mbar_init(&bars->p_free[0], 1);
    mbar_init(&bars->p_free[1], 1);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->o_final, 1);
    mbar_init(&bars->o_free, 4 * C::NWG);
    mbar_init(&bars->v_tail, 1);
    mbar_init(&bars->mma_drain[0], 1);
    mbar_init(&bars->mma_drain[1], 1);
    for (int s = 0; s < C::IINFO; ++s) {
      mbar_init(&bars->item_full[s], 1);
      mbar_init(&bars->item_empty[s], C::ITEM_READERS);
    }
    for (int s = 0; s < C::TINFO; ++s) mbar_init(&bars->tinfo_full[s], 1);
    bars->abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == C::W_S) tmem_alloc(&bars->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  // Item number k of this CTA as the producer published it: the item index w (-1 after the
  // last one) and its tile count; the reader then releases the slot.  Returns false when the
  // wait gave up.
  auto item_get = [&](int k, bool warp_wide, int& w, int& n_tiles) -> bool {
    const int s = k % C::IINFO;
    const bool ok = warp_wide ? warp_wait(&bars->item_full[s], (k / C::IINFO) & 1, tmo, abort_flag)
                              : mbar_wait(&bars->item_full[s], (k / C::IINFO) & 1, tmo, abort_flag);
    if (!ok) return false;
    const int2 e = iinfo[s];
    w = e.x;
    n_tiles = e.y;
    if (warp_wide) __syncwarp();
    if (!warp_wide || lane == 0) mbar_arrive(&bars->item_empty[s]);
    return true;
  };

  if (warp >= C::W_PROD) {
    if constexpr (C::DUAL) regs_dec<C::OTHER_REGS>();
    if (warp == C::W_PROD) {
      // ------------------------------------------------------------------ producer
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
      }
      int cnt = 0, n_tail = 0, J = 0, qn = 0;          // chunks, tail chunks, tiles, Q loads
      bool ok = true;
      // Items are claimed one ahead (the heaviest one left each time), so that the next index is
      // known by the time this item's loads are issued.
      int w_next = n_items;
      if (lane == 0) w_next = (int)atomicAdd(&g_wide_next[epoch], 1u);
      for (int k_item = 0;; ++k_item) {
        int w = n_items;
        if (lane == 0 && ok) {
          w = w_next;
          if (w < n_items) w_next = (int)atomicAdd(&g_wide_next[epoch], 1u);
        }
        w = __shfl_sync(0xffffffffu, w, 0);
        const bool end = w >= n_items;
        const WideItem it = wide_item<BM, BN, D == 256>(sh, end ? 0 : w);
        int n_tiles = end ? 0 : it.n_dense;
        bool list = false;
        const uint8_t* mrow = masked
            ? sh.block_mask + (((size_t)it.b * sh.n_heads + it.h) * sh.nQb + it.t0 / sh.q_block) * sh.nKb
            : nullptr;
        // (unit indices are 16-bit: sequences of more than 64 * 65534 keys take the contiguous
        // tiles, masked per half)
        if (masked && n_tiles > 0 && (it.key_hi + 63) / 64 < (int)kUnitNone) {
          // the selected 64-key units in key order, paired into tiles (unit list_a[t] in the
          // first half of tile t, list_b[t] in the second), by the whole warp
          const int u_lo = it.key_lo / 64, u_hi = (it.key_hi + 63) / 64;
          const uint32_t lt = (1u << lane) - 1u;
          int run = 0;
          auto put = [&](int rank, int u) {
            if (rank < 2 * C::LIST_MAX) (rank & 1 ? list_b : list_a)[rank >> 1] = (uint16_t)u;
          };
          if (sh.k_block == 64) {
            // one mask byte per unit: the row is read as 16-byte words (the aligned words
            // covering units u_lo ... u_hi - 1; bytes outside that range are ignored), four
            // words a lane in flight, so a row of 2048 units is a single memory round trip
            const uintptr_t a0 = reinterpret_cast<uintptr_t>(mrow + u_lo) & ~uintptr_t(15);
            const int n_words = (int)((reinterpret_cast<uintptr_t>(mrow + u_hi) - a0 + 15) >> 4);
            const int u_a0 = (int)((intptr_t)a0 - reinterpret_cast<intptr_t>(mrow));   // unit of a0's byte 0
            for (int w0 = 0; w0 < n_words; w0 += 32 * 4) {
              uint4 wv[4];
#pragma unroll
              for (int r = 0; r < 4; ++r) {
                const int wi = w0 + 32 * r + lane;
                wv[r] = wi < n_words ? __ldg(reinterpret_cast<const uint4*>(a0) + wi) : make_uint4(0u, 0u, 0u, 0u);
              }
#pragma unroll
              for (int r = 0; r < 4; ++r) {
                const int ub = u_a0 + 16 * (w0 + 32 * r + lane);          // unit of this word's byte 0
                // bit j: byte j is nonzero (the top bit of each byte of __vcmpne4, gathered to
                // bits 28..31 by one multiply: the four partial products land on distinct bits)
                const uint32_t wd[4] = {wv[r].x, wv[r].y, wv[r].z, wv[r].w};
                uint32_t bits = 0;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                  bits |= (((__vcmpne4(wd[c], 0u) & 0x80808080u) * 0x00204081u) >> 28) << (4 * c);
                const int cut_lo = min(max(u_lo - ub, 0), 16), cut_hi = min(max(u_hi - ub, 0), 16);
                bits &= ((1u << cut_hi) - 1u) & ~((1u << cut_lo) - 1u);
                const int c = __popc(bits);
                int incl = c;                                  // inclusive prefix over the lanes
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                  const int t = __shfl_up_sync(0xffffffffu, incl, off);
                  if (lane >= off) incl += t;
                }
                int rank = run + incl - c;
                while (bits) {
                  put(rank++, ub + __ffs(bits) - 1);
                  bits &= bits - 1u;
                }
                run += __shfl_sync(0xffffffffu, incl, 31);
              }
            }
          } else {
            // several units per mask byte: 16 mask bytes per lane in flight at a time
            for (int base = u_lo; base < u_hi; base += 32 * 16) {
              bool sel[16];
#pragma unroll
              for (int r = 0; r < 16; ++r) {
                const int u = base + 32 * r + lane;
                sel[r] = u < u_hi && mrow[(64 * u) / sh.k_block] != 0;
              }
#pragma unroll
              for (int r = 0; r < 16; ++r) {
                const uint32_t bal = __ballot_sync(0xffffffffu, sel[r]);
                if (sel[r]) put(run + __popc(bal & lt), base + 32 * r + lane);
                run += __popc(bal);
              }
            }
          }
          if (run <= 2 * C::LIST_MAX) {     // else: contiguous tiles, masked per half
            list = true;
            if (lane == 0 && (run & 1)) list_b[run >> 1] = kUnitNone;
            n_tiles = (run + 1) / 2;
          }
          __syncwarp();
        }
        if (lane == 0 && ok) {                          // publish the item (or the end)
          const int s = k_item % C::IINFO;
          if (k_item >= C::IINFO) ok = mbar_wait(&bars->item_empty[s], ((k_item / C::IINFO) - 1) & 1, tmo, abort_flag);
          if (ok) {
            iinfo[s] = make_int2(end ? -1 : w, n_tiles);
            mbar_arrive(&bars->item_full[s]);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (end || !ok) break;
        {
          // The next item is already claimed: start moving its Q tile and its mask row into L2,
          // so that its list and its first scores are not held up by memory latency when this
          // item's loads are done.
          const int wn = __shfl_sync(0xffffffffu, w_next, 0);
          if (wn < n_items) {
            const WideItem nx = wide_item<BM, BN, D == 256>(sh, wn);
            if (lane == 0)
              for (int s = 0; s < D / 64; ++s)
                tma_prefetch_l2_3d(&tm_q, 64 * s, nx.t0, nx.b * sh.n_heads + nx.h);
            if (masked && nx.n_dense > 0) {
              const uint8_t* mr = sh.block_mask + (((size_t)nx.b * sh.n_heads + nx.h) * sh.nQb + nx.t0 / sh.q_block) * sh.nKb;
              const uintptr_t a0 = reinterpret_cast<uintptr_t>(mr + (64 * (nx.key_lo / 64)) / sh.k_block) & ~uintptr_t(127);
              const uintptr_t a1 = reinterpret_cast<uintptr_t>(mr + (64 * ((nx.key_hi + 63) / 64) - 1) / sh.k_block);
              for (uintptr_t a = a0 + 128 * lane; a <= a1; a += 128 * 32) prefetch_l2(reinterpret_cast<const void*>(a));
            }
          }
        }
        if (lane == 0 && ok && n_tiles > 0) {
          // Tile t's units; a lone unit is loaded into both halves, the second masked, so that
          // no half ever holds unloaded data.
          auto tile_units = [&](int t, int& ua, int& ub, uint32_t& present) {
            if (list) {
              const uint16_t lb = list_b[t];
              ua = (int)list_a[t];
              ub = lb == kUnitNone ? ua : (int)lb;
              present = lb == kUnitNone ? 1u : 3u;
            } else {
              ua = 2 * (it.kt_lo + t);
              ub = ua + 1;
              present = 3u;
              if (masked)
                present = (mrow[(64 * ua) / sh.k_block] ? 1u : 0u) |
                          ((64 * ub < sh.Tk_max && mrow[(64 * ub) / sh.k_block]) ? 2u : 0u);
            }
          };
          // ring slot of chunk number cnt: free once the chunk RING positions earlier was read
          auto slot_acquire = [&](int& slot) -> bool {
            slot = cnt % C::RING;
            return cnt < C::RING || mbar_wait(&bars->empty[slot], ((cnt / C::RING) + 1) & 1, tmo, abort_flag);
          };
          const int qz = it.b * sh.n_heads + it.h, kz = it.b * sh.n_kv + it.kvh;
          // Q, once the previous item's last S has read the buffer
          if (qn > 0) ok = mbar_wait(&bars->q_free, (qn - 1) & 1, tmo, abort_flag);
          if (ok) {
            mbar_arrive_expect_tx(&bars->q_full, C::Q_BYTES);
            for (int s = 0; s < D / 64; ++s)
              tma_load_3d(sQ + s * BM * 128, &tm_q, &bars->q_full, 64 * s, it.t0, qz);
          }
          ++qn;
          // With a block mask every half of a tile is a 64-key unit of its own (64-row boxes);
          // otherwise tile j is the contiguous keys 128 (kt_lo + j) ... (128-row boxes).
          auto load_k = [&](int j) -> bool {                 // K(j): chunks of 128 dims
            int ua, ub;
            uint32_t pr;
            tile_units(j, ua, ub, pr);
            if (masked) {                                    // the tile's units, for the softmax
              const int s = (J + j) % C::TINFO;
              tinfo[s].ua = ua;
              tinfo[s].ub = ub;
              tinfo[s].present = pr;
              mbar_arrive(&bars->tinfo_full[s]);
            }
            for (int c = 0; c < C::KCH; ++c) {
              int slot;
              if (!slot_acquire(slot)) return false;
              unsigned char* dst = sR + slot * C::CHUNK;
              if (cnt != drop_chunk) {
                mbar_arrive_expect_tx(&bars->full[slot], C::CHUNK);
                for (int s = 0; s < 2; ++s) {
                  if (!UNITS) {
                    tma_load_3d(dst + s * BN * 128, &tm_k, &bars->full[slot], 128 * c + 64 * s, (it.kt_lo + j) * BN, kz);
                  } else {
                    tma_load_3d(dst + s * BN * 128, &tm_k64, &bars->full[slot], 128 * c + 64 * s, 64 * ua, kz);
                    tma_load_3d(dst + s * BN * 128 + 64 * 128, &tm_k64, &bars->full[slot], 128 * c + 64 * s, 64 * ub, kz);
                  }
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
              for (int p = 0; p < PARTS; ++p) tail |= 64 * part_unit(p) + 64 > it.Tk;
              uint64_t* bar = tail ? &bars->v_tail : &bars->full[slot];
              const bool drop = cnt == drop_chunk;
              if (!drop) {
                mbar_arrive_expect_tx(bar, C::CHUNK);
                for (int s = 0; s < D / 64; ++s) {
                  if (!UNITS) {
                    tma_load_3d(dst + s * C::VK * 128, &tm_v, bar, 64 * s, (it.kt_lo + j) * BN + C::VK * c, kz);
                  } else {
                    for (int p = 0; p < PARTS; ++p)
                      tma_load_3d(dst + s * C::VK * 128 + p * 64 * 128, &tm_v64, bar, 64 * s, 64 * part_unit(p), kz);
                  }
                }
              }
              if (tail) {
                if (drop || !mbar_wait(&bars->v_tail, n_tail & 1, tmo, abort_flag)) return false;
                ++n_tail;
                for (int p = 0; p < PARTS; ++p)
                  for (int row = max(0, it.Tk - 64 * part_unit(p)); row < 64; ++row)
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
          if (ok) ok = load_k(0);
          for (int j = 0; ok && j < n_tiles; ++j) {
            if (j + 1 < n_tiles) ok = load_k(j + 1);
            if (ok) ok = load_v(j);
          }
          J += n_tiles;
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        __syncwarp();                                     // the list is rebuilt for the next item
        if (!ok) break;
      }
      // the launch's last CTA to finish resets its item counters
      if (lane == 0) {
        __threadfence();
        if (atomicAdd(&g_wide_done[epoch], 1u) == gridDim.x - 1) {
          g_wide_next[epoch] = 0u;
          g_wide_done[epoch] = 0u;
          __threadfence();
        }
      }
      // Drain: the last Q and the most recent chunk of every slot have landed before the CTA
      // may exit.
      if (lane == 0) {
        if (qn > 0) mbar_wait(&bars->q_full, (qn - 1) & 1, tmo, nullptr);
        for (int k = max(0, cnt - C::RING); k < cnt; ++k)
          mbar_wait(&bars->full[k % C::RING], (k / C::RING) & 1, tmo, nullptr);
      }
    } else if (warp == C::W_S || warp == C::W_PV) {
      // The issuer warps issue MMAs and nothing else.  Each runs its loop with all 32 lanes
      // converged (every wait, index and descriptor is the same in every lane) and one elected
      // lane executes each tcgen05 instruction: issued that way, with the descriptors of a
      // tile's MMAs a per-chunk base plus constants, one warp keeps pace with the tensor pipe
      // (64 cycles per 128x128x16 MMA); issued from a lone lane it cannot.
      {
        constexpr uint32_t idesc_s = idesc_bf16_f32(128, BN, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
        const uint64_t dq = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dr_k = sdesc_sw128(smem_u32(sR), 16, 1024);       // K chunks: K-major
        const uint64_t dr_v = sdesc_sw128(smem_u32(sR), C::VK * 128, 1024);   // V chunks: MN-major
        bool ok = true;
        if constexpr (!C::DUAL) {
          // ------------------------------------------------------------------ one MMA issuer (d = 256)
          // The chunks arrive in the producer's order, K(0), then K(j+1), V(j): the order in
          // which S(j+1) and PV(j) consume them.
          int cnt = 0, J = 0, qn = 0, k_item = 0;
          // S(J) into buffer J & 1 from the K chunks of tile j of the item
          auto issue_s = [&](int Jg) -> bool {
            const uint32_t d_s = tmem + C::COL_S + (Jg & 1) * BN;
            for (int c = 0; c < C::KCH; ++c) {
              const int slot = cnt % C::RING;
              if (!warp_wait(&bars->full[slot], (cnt / C::RING) & 1, tmo, abort_flag)) return false;
              tc_fence_after();
              const uint64_t bk = dr_k + (uint64_t)((slot * C::CHUNK) >> 4);
#pragma unroll
              for (int k8 = 0; k8 < 8; ++k8) {                // 8 steps of 16 dims in this chunk
                const int kk = 8 * c + k8;
                const uint64_t aq = dq + (uint64_t)(((kk >> 2) * BM * 128 + (kk & 3) * 32) >> 4);
                const uint64_t bo = bk + (uint64_t)(((k8 >> 2) * BN * 128 + (k8 & 3) * 32) >> 4);
                umma_bf16_ss_elect(d_s, aq, bo, idesc_s, kk > 0 ? 1u : 0u);
              }
              umma_commit_elect(&bars->empty[slot]);
              ++cnt;
            }
            umma_commit_elect(&bars->s_full[Jg & 1]);
            return true;
          };
          // O (+)= P(J) V(J), P in the first 64 columns of S buffer J & 1
          auto issue_pv = [&](int Jg, bool first) -> bool {
            const uint32_t p_col = tmem + C::COL_S + (Jg & 1) * BN;
            for (int c = 0; c < C::VCH; ++c) {
              const int slot = cnt % C::RING;
              if (!warp_wait(&bars->full[slot], (cnt / C::RING) & 1, tmo, abort_flag)) return false;
              tc_fence_after();
              const uint64_t bv = dr_v + (uint64_t)((slot * C::CHUNK) >> 4);
#pragma unroll
              for (int k4 = 0; k4 < C::VK / 16; ++k4) {       // steps of 16 keys in this chunk
                const int kk = (C::VK / 16) * c + k4;
                umma_bf16_ts_elect(tmem + C::COL_O, p_col + kk * 8, bv + (uint64_t)((k4 * 2048) >> 4), idesc_pv,
                             (!first || kk > 0) ? 1u : 0u);
              }
              umma_commit_elect(&bars->empty[slot]);
              ++cnt;
            }
            return true;
          };
          for (;; ++k_item) {
            int w, n_tiles;
            if (!(ok = item_get(k_item, true, w, n_tiles)) || w < 0) break;
            if (n_tiles == 0) continue;
            if (!(ok = warp_wait(&bars->q_full, qn & 1, tmo, abort_flag))) break;
            if (!(ok = issue_s(J))) break;
            for (int j = 0; ok && j < n_tiles; ++j) {
              const int Jg = J + j;
              if (j + 1 < n_tiles && !(ok = issue_s(Jg + 1))) break;
              if (j + 1 == n_tiles) umma_commit_elect(&bars->q_free);   // every S of the item issued
              if (!(ok = warp_wait(&bars->p_full[0][0], Jg & 1, tmo, abort_flag))) break;
              // the item's first PV overwrites O: the previous item's epilogue has read it
              if (j == 0 && qn > 0 && !(ok = warp_wait(&bars->o_free, (qn - 1) & 1, tmo, abort_flag))) break;
              tc_fence_after();
              if (!(ok = issue_pv(Jg, j == 0))) break;
              umma_commit_elect(&bars->o_done);
              if (j + 1 == n_tiles) umma_commit_elect(&bars->o_final);
            }
            J += n_tiles;
            ++qn;
          }
          // Drain: every MMA this thread issued has completed before TMEM can be released.
          umma_commit_elect(&bars->mma_drain[0]);
          warp_wait(&bars->mma_drain[0], 0, tmo, nullptr);
        } else {
          // ------------------------------------------------------------------ MMA issuers (d = 128)
          // Both find their chunks in the ring from the producer's order: per item K(0), then
          // K(j+1), V(j) for j = 0, 1, ... (K(n) is not loaded), one chunk each.
          static_assert(C::KCH == 1 && C::VCH == 1 && C::VK == C::BN, "d = 128 chunk layout");
          const int xi = warp - C::W_S;                    // 0: S issuer, 1: PV issuer
          int pos0 = 0, J = 0, qn = 0;
          int uses0 = 0, uses1 = 0;                        // S issuer: S per buffer; PV issuer: PV per buffer
          for (int k_item = 0;; ++k_item) {
            int w, n_tiles;
            if (!(ok = item_get(k_item, true, w, n_tiles)) || w < 0) break;
            if (n_tiles == 0) continue;
            auto kpos = [&](int j) { return pos0 + (j == 0 ? 0 : 2 * j - 1); };
            auto vpos = [&](int j) { return pos0 + (j + 1 < n_tiles ? 2 * j + 2 : 2 * j + 1); };
            if (xi == 0) {
              if (!(ok = warp_wait(&bars->q_full, qn & 1, tmo, abort_flag))) break;
              for (int j = 0; ok && j < n_tiles; ++j) {
                // S(j) into buffer j % 2, once the PV of the buffer's previous tile has read the P
                // held there.  K(j) is waited for first: it has usually landed long before, so
                // only the PV wait is exposed.
                const int buf = j & 1, u = buf ? uses1 : uses0;
                const int pos = kpos(j), slot = pos % C::RING;
                if (!(ok = warp_wait(&bars->full[slot], (pos / C::RING) & 1, tmo, abort_flag))) break;
                if (u >= 1 && !(ok = warp_wait(&bars->p_free[buf], (u - 1) & 1, tmo, abort_flag))) break;
                if (buf) ++uses1; else ++uses0;
                tc_fence_after();
                const uint32_t d_s = tmem + C::COL_S + buf * BN;
                const uint64_t bk = dr_k + (uint64_t)((slot * C::CHUNK) >> 4);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {                 // 8 steps of 16 dims
                  const uint64_t aq = dq + (uint64_t)(((kk >> 2) * BM * 128 + (kk & 3) * 32) >> 4);
                  const uint64_t bo = bk + (uint64_t)(((kk >> 2) * BN * 128 + (kk & 3) * 32) >> 4);
                  umma_bf16_ss_elect(d_s, aq, bo, idesc_s, kk > 0 ? 1u : 0u);
                }
                umma_commit_elect(&bars->empty[slot]);
                umma_commit_elect(&bars->s_full[buf]);
              }
              if (ok) umma_commit_elect(&bars->q_free);               // the item's last S read Q
            } else {
              // O_(j%2) += P(j) V(j), P in the first 64 columns of S buffer j % 2.  The softmax
              // publishes P in two halves of 64 keys; the first half's MMAs run while the
              // second half is exponentiated.
              for (int j = 0; ok && j < n_tiles; ++j) {
                const int buf = j & 1, u = buf ? uses1 : uses0;
                if (buf) ++uses1; else ++uses0;
                const int pos = vpos(j), slot = pos % C::RING;
                if (!(ok = warp_wait(&bars->full[slot], (pos / C::RING) & 1, tmo, abort_flag))) break;
                // the item's first PVs overwrite O_0 and O_1: the previous item's epilogue has
                // read them
                if (j == 0 && qn > 0 && !(ok = warp_wait(&bars->o_free, (qn - 1) & 1, tmo, abort_flag))) break;
                const uint32_t p_col = tmem + C::COL_S + buf * BN;
                const uint32_t d_o = tmem + C::COL_O + buf * D;
                const uint64_t bv = dr_v + (uint64_t)((slot * C::CHUNK) >> 4);
                for (int half = 0; ok && half < 2; ++half) {
                  if (!(ok = warp_wait(&bars->p_full[buf][half], u & 1, tmo, abort_flag))) break;
                  tc_fence_after();
#pragma unroll
                  for (int k4 = 0; k4 < 4; ++k4) {               // 4 steps of 16 keys
                    const int kk = 4 * half + k4;
                    umma_bf16_ts_elect(d_o, p_col + kk * 8, bv + (uint64_t)((kk * 2048) >> 4), idesc_pv,
                                 (j >= 2 || kk > 0) ? 1u : 0u);
                  }
                }
                if (!ok) break;
                umma_commit_elect(&bars->empty[slot]);
                umma_commit_elect(&bars->p_free[buf]);
                if (j + 1 == n_tiles) umma_commit_elect(&bars->o_final);
              }
            }
            pos0 += 2 * n_tiles;
            J += n_tiles;
            ++qn;
          }
          // Drain: every MMA this thread issued has completed before TMEM can be released.
          umma_commit_elect(&bars->mma_drain[xi]);
          warp_wait(&bars->mma_drain[xi], 0, tmo, nullptr);
        }
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    if constexpr (C::DUAL) regs_inc<C::SOFTMAX_REGS>();
    const int wg = warp >> 2;                         // tiles j of an item with j % NWG == wg
    const int row = threadIdx.x & 127;                // query row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float scale_log2 = kLog2e / sqrtf((float)D);
    float2* xch = reinterpret_cast<float2*>(smem + C::OFF_XCH);
    int J = 0, qn = 0;
    int own = 0;                                      // d = 128: tiles this warpgroup has taken (uses of S buffer wg)
    for (int k_item = 0;; ++k_item) {
      int w = -1, n_tiles = 0;
      bool ok = item_get(k_item, true, w, n_tiles);
      // every softmax warp takes the same branch: the next item, or out (the end, or a wait
      // that gave up somewhere)
      if (!named_all<1, C::SM_THREADS>(ok && w >= 0 && *abort_flag == 0)) break;
      const WideItem it = wide_item<BM, BN, D == 256>(sh, w);
      const long long i = it.i_first + row;           // absolute position of this row
      const int lo = sh.window > 0 ? (int)max(0LL, i - sh.window + 1) : 0;
      const int hi = sh.causal ? (int)max(0LL, min((long long)it.Tk, i + 1)) : it.Tk;
      const int lo_all = sh.window > 0 ? (int)max(0LL, it.i_last - sh.window + 1) : 0;
      const int hi_all = sh.causal ? (int)max(0LL, min((long long)it.Tk, it.i_first + 1)) : it.Tk;
      const uint32_t t_o = tmem + C::COL_O + wg * D + lane_off;
      float m_run = -INFINITY, l_run = 0.0f;          // this warpgroup's share of the item's keys
      if (sh.sink && wg == 0) { m_run = sh.sink[it.h] * kLog2e; l_run = 1.0f; }

      // this warpgroup's tiles of the item: j with j % NWG == wg
      const int j_first = C::DUAL ? wg : 0;
      for (int j = j_first; ok && j < n_tiles; j += C::NWG) {
        const int Jg = J + j;
        const int buf = C::DUAL ? wg : (Jg & 1);
        const uint32_t s_par = C::DUAL ? (uint32_t)(own & 1) : (uint32_t)((Jg >> 1) & 1);
        if (C::DUAL) ++own;
        if (!(ok = warp_wait(&bars->s_full[buf], s_par, tmo, abort_flag))) break;
        tc_fence_after();
        const uint32_t t_s = tmem + C::COL_S + buf * BN + lane_off;
        float sv[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
          tmem_ld32(t_s + 32 * c, *reinterpret_cast<float(*)[32]>(&sv[32 * c]));
        // keys of the two 64-column halves start at 64 ua and 64 ub
        int ua = 2 * (it.kt_lo + j), ub = ua + 1;
        uint32_t pr = 3u;
        if (masked) {
          const int s = Jg % C::TINFO;
          if (!(ok = warp_wait(&bars->tinfo_full[s], (Jg / C::TINFO) & 1, tmo, abort_flag))) {
            tmem_wait_ld();
            break;
          }
          ua = tinfo[s].ua;
          ub = tinfo[s].ub;
          pr = tinfo[s].present;
        }
        tmem_wait_ld();
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
        // d = 128: the accumulator's previous PV, PV(J-2), completed before S(J) was issued, so
        // the rescale can run before P is produced (PV(J) must see the rescaled accumulator).
        if constexpr (C::DUAL)
          if (j >= C::NWG && __any_sync(0xffffffffu, need)) rescale_o();
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
          // d = 256: PV(J-1) may still accumulate into O, so the rescale waits for it (PV(J-2)
          // is complete) and runs last.
          if (j >= C::NWG && __any_sync(0xffffffffu, need)) {
            if (!(ok = warp_wait(&bars->o_done, (Jg - 1) & 1, tmo, abort_flag))) break;
            tc_fence_after();
            rescale_o();
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(C::DUAL ? &bars->p_full[buf][1] : &bars->p_full[0][0]);
      }

      // ---- epilogue: O / l from TMEM to global --------------------------------------------
      if (ok && n_tiles > 0) ok = warp_wait(&bars->o_final, qn & 1, tmo, abort_flag);
      tc_fence_after();
      // The item's (m, l) of both warpgroups meet in shared memory (two buffers, by item
      // parity); the same barrier is the softmax threads' vote on whether every one of them
      // is still running, so all of them leave together if a wait gave up.
      float2* xb = xch + (k_item & 1) * 2 * BM;
      if (C::DUAL) xb[wg * BM + row] = make_float2(m_run, l_run);
      if (!named_all<1, C::SM_THREADS>(ok && *abort_flag == 0)) break;
      const int t = it.t0 + row;
      const size_t orow_off = (((size_t)it.b * sh.n_heads + it.h) * sh.Tq + t) * D;
      __nv_bfloat16* orow = out + orow_off;
      // Columns [c, c + 32) of this thread's row, times s0.  Plain bf16 output goes through the
      // warp's 2 KB staging area: each thread writes its row's 64 bytes there (16-byte pieces,
      // the piece index XOR (row / 2) % 4 so that no two of eight consecutive rows share banks),
      // then every store instruction of the warp covers 8 rows x 64 contiguous bytes instead of
      // 32 rows x 16 bytes.
      unsigned char* stage = smem + C::OFF_STAGE + (warp & 7) * 2048;
      auto store32 = [&](int c, const float (&o)[32], float s0) {
        if constexpr (EPI == 0) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(o[2 * e] * s0, o[2 * e + 1] * s0);
          const int sw = (lane >> 1) & 3;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(stage + lane * 64 + ((u ^ sw) << 4)) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int q = 32 * i + lane, r = q >> 2, u = q & 3;      // row r of the warp, piece u
            const uint4 v = *reinterpret_cast<const uint4*>(stage + r * 64 + ((u ^ ((r >> 1) & 3)) << 4));
            const int tr = 32 * (warp & 3) + r;                       // row of the query tile
            const size_t off = (((size_t)it.b * sh.n_heads + it.h) * sh.Tq + it.t0 + tr) * D + c + 8 * u;
            if (tr < it.rows && GA_BOUNDS(off + 8 <= (size_t)sh.batch * sh.n_heads * sh.Tq * D, 2, off))
              *reinterpret_cast<uint4*>(out + off) = v;
          }
          __syncwarp();
          return;
        }
        if (row < it.rows) {
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
            if (GA_BOUNDS(orow_off + c + u + 8 <= (size_t)sh.batch * sh.n_heads * sh.Tq * D, 2, orow_off + c + u))
              *reinterpret_cast<uint4*>(orow + c + u) = pk;
          }
        }
      };
      if constexpr (C::DUAL) {
        // Merge the warpgroups' partial results (running max m_w, sum l_w, accumulator O_w, all
        // relative to 2^m_w): out = sum_w 2^(m_w - M) O_w / sum_w 2^(m_w - M) l_w.  Warpgroup w
        // writes columns [64 w, 64 w + 64).  O_w holds this item's result only if warpgroup w
        // had a tile of the item.
        const float2 other = xb[(wg ^ 1) * BM + row];
        const float m0 = wg == 0 ? m_run : other.x, l0 = wg == 0 ? l_run : other.y;
        const float m1 = wg == 0 ? other.x : m_run, l1 = wg == 0 ? other.y : l_run;
        const float M = fmaxf(m0, m1);
        const float a0 = M == -INFINITY ? 0.0f : ex2(m0 - M);
        const float a1 = M == -INFINITY ? 0.0f : ex2(m1 - M);
        const float L = l0 * a0 + l1 * a1;
        const float inv_l = L > 0.0f ? 1.0f / L : 0.0f;
        const float s0 = a0 * inv_l, s1 = a1 * inv_l;
        const bool has0 = n_tiles >= 1, has1 = n_tiles >= 2;   // warpgroup w had a tile of the item
        const uint32_t t_o0 = tmem + C::COL_O + lane_off, t_o1 = t_o0 + D;
#pragma unroll 1
        for (int c = 64 * wg; c < 64 * wg + 64; c += 32) {
          float o0[32], o1[32];
          tmem_ld32(t_o0 + c, o0);              // both always: a select drops an unused one
          tmem_ld32(t_o1 + c, o1);
          tmem_wait_ld();
          if (c == 64 * wg + 32 && n_tiles > 0) {   // O is read: the next item's PVs may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->o_free);
          }
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const float x0 = has0 ? o0[u] : 0.0f, x1 = has1 ? o1[u] : 0.0f;
            o0[u] = fmaf(x0, s0, x1 * s1);
          }
          store32(c, o0, 1.0f);
        }
        if (lse && wg == 0 && row < it.rows && GA_BOUNDS(((size_t)it.b * sh.n_heads + it.h) * sh.Tq + t < (size_t)sh.batch * sh.n_heads * sh.Tq, 3, t))
          lse[((size_t)it.b * sh.n_heads + it.h) * sh.Tq + t] =
              L > 0.0f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
      } else {
        const float inv_l = l_run > 0.0f ? 1.0f / l_run : 0.0f;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float o[32];
          if (n_tiles > 0) {
            tmem_ld32(t_o + c, o);
            tmem_wait_ld();
            if (c == D - 32) {                  // O is read: the next item's PVs may overwrite it
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bars->o_free);
            }
          } else {
#pragma unroll
            for (int u = 0; u < 32; ++u) o[u] = 0.0f;
          }
          store32(c, o, inv_l);
        }
        if (lse && row < it.rows && GA_BOUNDS(((size_t)it.b * sh.n_heads + it.h) * sh.Tq + t < (size_t)sh.batch * sh.n_heads * sh.Tq, 3, t))
          lse[((size_t)it.b * sh.n_heads + it.h) * sh.Tq + t] =
              l_run > 0.0f ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
      }
      if (n_tiles > 0) ++qn;
      J += n_tiles;
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
