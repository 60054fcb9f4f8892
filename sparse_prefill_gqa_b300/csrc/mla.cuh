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
// Kernels: mla_absorb_kernel (q_lat, then q = [q_lat | q_rope] in bf16; one CTA per (head, 64
// latent rows) for every sequence, so each weight row is read once), mla_decode_kernel (two
// CTAs per SM, each taking an equal contiguous share of all sequences' 32-token tiles; the heads
// are the 16 rows of mma.sync m16n8k16) and mla_expand_kernel (the log-sum-exp re-association of
// a sequence's partials, then o_lat w_uv, per head, 64 output dims and 8 sequences).
#pragma once

#include "common.cuh"

namespace ga {

struct MlaCfg {
  static constexpr int R = 512, DR = 64, DN = 128, DV = 128;
  static constexpr int DK = R + DR;                     // 576 numbers per cached token
  static constexpr int SLABS = DK / 64;                 // 9 SW128 boxes of 64 columns
  static constexpr int TILE = 32;                       // tokens per stage (8 per compute warp)
  // The partition weighs each sequence as its tiles + SEQ_COST: starting a sequence inside a
  // share (publishing the previous partial, the next query tile, restarting the pipeline)
  // measured about as long as one tile (a cost of 1 ran 1.3 % faster than 2).
  static constexpr int SEQ_COST = 1;
  static constexpr int STAGES = 2;
  static constexpr int STAGE_BYTES = TILE * DK * 2;     // 36864
  static constexpr int QROW = DK * 2 + 16;              // padded row of the query tile (bytes)
  static constexpr int PROW = TILE * 2 + 16;            // padded row of the P tile (bytes)
  static constexpr int OFF_SX = STAGES * STAGE_BYTES;   // [4 warps][16][SXROW] partial scores
  static constexpr int SXROW = 40;                      // floats per head row of a partial-score tile
  static constexpr int OFF_P = OFF_SX + 4 * 16 * SXROW * 4;
  static constexpr int OFF_X = OFF_P + 16 * PROW;       // [4][16] float exchange
  static constexpr int OFF_BAR = OFF_X + 4 * 16 * 4;
  static constexpr int BAR_BYTES = 128;
  static constexpr int OFF_Q = OFF_BAR + BAR_BYTES;     // the next segment's query tile
  static constexpr int SMEM_BYTES = OFF_Q + 16 * QROW + 1024;
  static constexpr int THREADS = 160;
  static_assert(2 * SMEM_BYTES <= 232448, "shared memory: two CTAs per SM");
  // absorb: latent rows per CTA, sequences staged at a time; expand: output dims and sequences
  static constexpr int AB_ROWS = 64, AB_SEQ = 16, EX_DIMS = 64, EX_SEQ = 8;
  static constexpr int EX_WROW = EX_DIMS * 2 + 16;     // padded weight row (bytes): conflict-free matrix loads
  static constexpr int EX_LROW = R + 8;                 // padded latent row (floats)
  static constexpr int EX_SMEM = R * EX_WROW + EX_SEQ * EX_LROW * 4;   // weight slice, latent tile
  static_assert(8 * EX_SEQ * EX_DIMS * 4 <= EX_SEQ * EX_LROW * 4, "partial sums fit in the latent tile");
  static_assert(EX_SEQ == 8 && EX_DIMS % 16 == 0, "one sequence per warp, pairs of 8-dim output tiles");
};

struct MlaShape {
  int batch, n_heads, L_max;
  int n_cta;            // CTAs of the decode launch, each taking an equal share of all tiles
  int n_ids;            // partial slots per head: n_cta + batch - 1
  const int32_t* lens;
  int2* seg;            // per sequence: its first partial slot and slot count (decode -> expansion)
  uint64_t timeout_ns;
};

// grid: (R / 64, n_heads, ceil(batch / 16)); block: 128.  q[b, h] = [q_nope w_uk[h]^T (fp32
// sums, rounded to bf16) | q_rope] for latent rows 64 x .. 64 x + 63 of head h and 16 sequences,
// on the tensor cores: mma.sync m16n8k16 with the 16 sequences as M, the latent rows as N and
// the 128 nope dims as K; warp w takes latent rows 16 w .. 16 w + 15.  The 64 weight rows (16 KB)
// and the 16 query rows are staged in shared memory with 272-byte rows (conflict-free 8-row
// matrix loads); every weight row is read from global memory once per 16 sequences.
__global__ void __launch_bounds__(128)
mla_absorb_kernel(const __nv_bfloat16* __restrict__ q_nope, const __nv_bfloat16* __restrict__ q_rope,
                  const __nv_bfloat16* __restrict__ w_uk, __nv_bfloat16* __restrict__ q_abs, int n_heads,
                  int batch) {
  using C = MlaCfg;
  constexpr int RS = C::DN * 2 + 16;                    // staged row stride (bytes)
  __shared__ __align__(16) unsigned char w_s[C::AB_ROWS * RS];
  __shared__ __align__(16) unsigned char q_s[C::AB_SEQ * RS];
  const int rb = blockIdx.x, h = blockIdx.y, t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int b0 = blockIdx.z * C::AB_SEQ, nb = min(C::AB_SEQ, batch - b0);
  griddep_launch_dependents();                          // the decode may start streaming the cache
  const __nv_bfloat16* wsrc = w_uk + ((size_t)h * C::R + (size_t)rb * C::AB_ROWS) * C::DN;
  for (int e = t; e < C::AB_ROWS * C::DN / 8; e += 128) {    // 16-byte pieces, 16 per row
    const int row = e / (C::DN / 8), c = e % (C::DN / 8);
    *reinterpret_cast<uint4*>(w_s + row * RS + 16 * c) = *reinterpret_cast<const uint4*>(wsrc + 8 * e);
  }
  for (int e = t; e < C::AB_SEQ * C::DN / 8; e += 128) {
    const int bb = e / (C::DN / 8), c = e % (C::DN / 8);
    *reinterpret_cast<uint4*>(q_s + bb * RS + 16 * c) =
        bb < nb ? *reinterpret_cast<const uint4*>(q_nope + ((size_t)(b0 + bb) * n_heads + h) * C::DN + 8 * c)
                : make_uint4(0u, 0u, 0u, 0u);
  }
  if (rb == 0)                                          // the rope part of the sequences' queries
    for (int e = t; e < nb * (C::DR / 8); e += 128) {  // 16-byte pieces, 8 per row
      const size_t row = (size_t)(b0 + e / (C::DR / 8)) * n_heads + h;
      const int c = e % (C::DR / 8);
      if (GA_BOUNDS(row < (size_t)batch * n_heads, 9, row))
        *reinterpret_cast<uint4*>(q_abs + row * C::DK + C::R + 8 * c) =
            *reinterpret_cast<const uint4*>(q_rope + row * C::DR + 8 * c);
    }
  __syncthreads();
  const uint32_t qs = smem_u32(q_s), ws = smem_u32(w_s);
  const int mi = lane >> 3, rr = lane & 7;
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int kk = 0; kk < C::DN / 16; ++kk) {
    uint32_t a[4];
    ldmatrix_x4(qs + (lane & 15) * RS + (kk * 16 + (lane >> 4) * 8) * 2, a[0], a[1], a[2], a[3]);
    // matrices: (latent rows 16 w .. + 7, low 8 dims), (same rows, high 8), then rows + 8
    uint32_t b0_, b1_, b2_, b3_;
    ldmatrix_x4(ws + (16 * warp + ((mi >> 1) << 3) + rr) * RS + (kk * 16 + (mi & 1) * 8) * 2, b0_, b1_, b2_, b3_);
    mma_bf16_16816(acc[0], a, b0_, b1_);
    mma_bf16_16816(acc[1], a, b2_, b3_);
  }
  const int s_lo = lane >> 2, s_hi = s_lo + 8;          // sequences of the accumulator rows
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    const int r = rb * C::AB_ROWS + 16 * warp + 8 * n + 2 * (lane & 3);   // latent rows r, r + 1
    [[maybe_unused]] const size_t lim = (size_t)batch * n_heads * C::DK;
    const size_t o_lo = ((size_t)(b0 + s_lo) * n_heads + h) * C::DK + r, o_hi = ((size_t)(b0 + s_hi) * n_heads + h) * C::DK + r;
    if (s_lo < nb && GA_BOUNDS(o_lo + 2 <= lim && r + 2 <= C::R, 9, o_lo))
      *reinterpret_cast<uint32_t*>(q_abs + o_lo) = pack_bf16x2(acc[n][0], acc[n][1]);
    if (s_hi < nb && GA_BOUNDS(o_hi + 2 <= lim && r + 2 <= C::R, 9, o_hi))
      *reinterpret_cast<uint32_t*>(q_abs + o_hi) = pack_bf16x2(acc[n][2], acc[n][3]);
  }
}

struct MlaBars {
  uint64_t full[2], empty[2];
  int abort_flag;
  int b0;                                            // this CTA's first sequence
  long long p0;                                      // its first position in the weighted order
  long long wsum[MlaCfg::THREADS / 32];              // per-warp tile totals of the partition scan
};
static_assert(sizeof(MlaBars) <= MlaCfg::BAR_BYTES, "barrier block");

// 32-token tiles of sequence b.
__device__ __forceinline__ int mla_tiles(const MlaShape& s, int b) {
  return (seq_keys(s.lens, b, s.L_max) + MlaCfg::TILE - 1) / MlaCfg::TILE;
}

// Cached tokens of sequence b, 0 past the batch.
__device__ __forceinline__ int mla_keys(const MlaShape& s, int b) {
  return b < s.batch ? seq_keys(s.lens, b, s.L_max) : 0;
}

// AND of `ok` over the 128 consumer threads (named barrier 1): every consumer warp takes the
// same branch, so a wait that gave up in one warp can never leave another at a barrier.
__device__ __forceinline__ bool consumers_all(bool ok) {
  uint32_t res;
  asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
               "bar.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
               : "=r"(res) : "r"(ok ? 1u : 0u) : "memory");
  return res != 0;
}

// grid: n_cta (two per SM); block: 160 -- warps 0-3 compute, warp 4 loads 32-token tiles of the
// latent cache [batch, L_max, 576] by TMA (9 boxes of 64 columns, 128-byte swizzle).
// Partition: the sequences, in order, occupy consecutive positions, SEQ_COST for starting the
// sequence and then one per tile (an empty sequence none); the positions are cut into n_cta
// equal contiguous shares (per = ceil(total / n_cta)), and CTA c takes the tiles at positions
// c per .. c per + per - 1.  Every CTA has the same amount of work, so no SM is left with one
// CTA while others still hold two.  A share covers the end of one sequence, maybe whole short
// ones, and the start of another: one segment per (CTA, sequence) pair holding tiles, each
// publishing its partial (o, m, l) to slot c + b.  Along the order both c and b never decrease,
// so c + b is distinct for distinct segments and stays below n_cta + batch - 1.  The CTA holding
// a sequence's first tile records the sequence's first slot and slot count for the expansion.
// Per tile: warp w scores its 8 tokens for the 16 query rows (the heads; rows >= n_heads are
// zero), the warps agree on each row's tile maximum through shared memory, write their
// probabilities into a shared 16 x 32 P tile, and each accumulates latent dims 128 w .. 128 w +
// 127 of P c_kv over all 32 tokens.
__global__ void __launch_bounds__(MlaCfg::THREADS, 2)
mla_decode_kernel(const __grid_constant__ CUtensorMap tm_lat, const __nv_bfloat16* __restrict__ q_abs,
                  float* __restrict__ ws_o, float* __restrict__ ws_ml, MlaShape s) {
  using C = MlaCfg;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  MlaBars* bars = reinterpret_cast<MlaBars*>(smem + C::OFF_BAR);
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, H = s.n_heads;
  const uint64_t tmo = s.timeout_ns;
  griddep_launch_dependents();                       // the expansion may start its set-up

  // ---- this CTA's share: a block-wide scan of the sequences' tile counts ---------------------
  const int per_t = (s.batch + C::THREADS - 1) / C::THREADS;
  const int blo = min(s.batch, (int)threadIdx.x * per_t), bhi = min(s.batch, blo + per_t);
  auto weight = [&](int b) -> long long {
    const int nt = mla_tiles(s, b);
    return nt > 0 ? nt + C::SEQ_COST : 0;
  };
  long long mine = 0;
  for (int b = blo; b < bhi; ++b) mine += weight(b);
  long long incl = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) bars->wsum[warp] = incl;
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
  long long before = incl - mine, total = 0;
#pragma unroll
  for (int w = 0; w < C::THREADS / 32; ++w) {
    const long long x = bars->wsum[w];
    if (w < warp) before += x;
    total += x;
  }
  const long long per = (total + s.n_cta - 1) / s.n_cta;
  const long long start = (long long)c * per, end = min(start + per, total);
  if (start < end && before <= start && start < before + mine) {
    long long p = before;
    int b = blo;
    while (p + weight(b) <= start) p += weight(b++);   // the sequence holding position `start`
    bars->b0 = b;
    bars->p0 = p;
  }
  __syncthreads();
  if (start >= end) return;                          // nothing for this CTA (uniform)
  const int b_first = bars->b0;
  const long long p_first = bars->p0;

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_lat);
      int it = 0, issued = 0;
      bool ok = true;
      long long p = p_first;
      // the next sequence's length is read one sequence ahead, so that a segment boundary does
      // not wait on a load
      int L_cur = mla_keys(s, b_first), L_nxt = mla_keys(s, b_first + 1);
      for (int b = b_first; ok && p < end && b < s.batch; ++b, L_cur = L_nxt, L_nxt = mla_keys(s, b + 1)) {
        const int nt = (L_cur + C::TILE - 1) / C::TILE;
        if (nt == 0) continue;
        const long long r0 = p + C::SEQ_COST;        // position of tile 0 of sequence b
        const long long lo = max(start, r0), hi = min(end, r0 + nt);
        p = r0 + nt;
        const int j = (int)(lo - r0), take = (int)max(0LL, hi - lo);
        for (int u = 0; u < take; ++u, ++it) {
          const int st = it % C::STAGES, use = it / C::STAGES;
          if (it >= C::STAGES && !mbar_wait(&bars->empty[st], (use + 1) & 1, tmo, abort_flag)) {
            ok = false;
            break;
          }
          unsigned char* dst = smem + st * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&bars->full[st], C::STAGE_BYTES);
          ++issued;
          const int key0 = (j + u) * C::TILE;
          for (int sl = 0; sl < C::SLABS; ++sl)
            tma_load_3d(dst + sl * C::TILE * 128, &tm_lat, &bars->full[st], 64 * sl, key0, b);
        }
      }
      for (int k = max(0, issued - C::STAGES); k < issued; ++k)
        mbar_wait(&bars->full[k % C::STAGES], (k / C::STAGES) & 1, tmo, nullptr);
    }
    return;
  }

  // ---------------------------------------------------------------------- consumer warps
  const int r_lo = lane >> 2, r_hi = r_lo + 8;
  const float scale_log2 = kLog2e / sqrtf((float)(C::DN + C::DR));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t qs = sbase + C::OFF_Q, ps = sbase + C::OFF_P;
  float* xs = reinterpret_cast<float*>(smem + C::OFF_X);             // [4][16]
  float* sx = reinterpret_cast<float*>(smem + C::OFF_SX);            // [4 warps][16][SXROW]
  const int mi = lane >> 3, rr = lane & 7;
  constexpr int KW = C::DK / 16 / 4;                 // 16-dim steps per warp
  constexpr int QPR = C::DK / 8;                     // 16-byte pieces of a query row
  // The query tile of a segment's sequence is copied into shared memory while the previous
  // segment runs (16-byte asynchronous copies, one group); rows past the heads stay zero.
  auto fetch_q = [&](int b) {
    for (int e = threadIdx.x; e < H * QPR; e += 128) {
      const int r = e / QPR, ch = e % QPR;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                   :: "r"(qs + (uint32_t)(r * C::QROW + ch * 16)), "l"(q_abs + ((size_t)b * H + r) * C::DK + 8 * ch)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  for (int e = H * QPR + threadIdx.x; e < 16 * QPR; e += 128)
    *reinterpret_cast<uint4*>(smem + C::OFF_Q + (e / QPR) * C::QROW + (e % QPR) * 16) = make_uint4(0u, 0u, 0u, 0u);
  griddep_wait();                                    // q_lat is written by the absorption kernel
  fetch_q(b_first);
  int it = 0;                                        // tiles of the ring consumed so far
  bool dead = false;                                 // a wait gave up (uniform over the warps)
  long long p = p_first;
  int L = mla_keys(s, b_first), L_nxt = mla_keys(s, b_first + 1);   // read ahead, as in the producer
  for (int b = b_first; p < end && b < s.batch; ++b, L = L_nxt, L_nxt = mla_keys(s, b + 1)) {
    const int nt = (L + C::TILE - 1) / C::TILE;
    if (nt == 0) continue;                           // an empty sequence inside the share
    const long long r0 = p + C::SEQ_COST;            // position of tile 0 of sequence b
    const long long lo = max(start, r0), hi = min(end, r0 + nt);
    p = r0 + nt;
    if (hi <= lo) continue;                          // the share ends before the sequence's tiles
    const int j = (int)(lo - r0), take = (int)(hi - lo);
    const int kbeg = j * C::TILE, kend = min((j + take) * C::TILE, L);
    asm volatile("cp.async.wait_all;" ::: "memory");
    asm volatile("bar.sync 1, 128;" ::: "memory");   // sequence b's query tile has landed
    // Scores split over the dimensions: warp w takes the 16-dim steps 9 w .. 9 w + 8 for all 32
    // tokens of a tile, with its 9 query fragments held in registers for the whole segment (the
    // query tile is read from shared memory once); the four partial tiles meet in shared
    // memory, each warp summing its own 8 tokens' columns.
    uint32_t qa[KW][4];
#pragma unroll
    for (int i = 0; i < KW; ++i)
      ldmatrix_x4(qs + (lane & 15) * C::QROW + ((KW * warp + i) * 16 + (lane >> 4) * 8) * 2, qa[i][0], qa[i][1],
                  qa[i][2], qa[i][3]);
    asm volatile("bar.sync 1, 128;" ::: "memory");   // every warp has its fragments: the tile is free
    if (p + C::SEQ_COST < end) {                     // a next segment: the next sequence holding tiles
      int bn = b + 1;
      if (L_nxt == 0)
        while (bn < s.batch - 1 && mla_tiles(s, bn) == 0) ++bn;
      fetch_q(bn);
    }
    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.0f, 0.0f};

    for (int u = 0; u < take; ++u, ++it) {
      const int st = it % C::STAGES;
      if (!dead) dead = !consumers_all(warp_wait(&bars->full[st], (it / C::STAGES) & 1, tmo, abort_flag));
      if (dead) continue;
      const uint32_t kb = sbase + st * C::STAGE_BYTES;
      const int t0 = kbeg + u * C::TILE;               // first token of the tile
      // ---- partial scores over this warp's 144 dims, all 32 tokens ----------------------------
      {
        float sacc[4][4];
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) sacc[nb][0] = sacc[nb][1] = sacc[nb][2] = sacc[nb][3] = 0.0f;
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) {
          const int keyr = 8 * nb + rr;               // token row this lane addresses
#pragma unroll
          for (int i = 0; i < KW; i += 2) {
            // one 4-matrix load: matrices 0, 1 the low and high 8 dims of step i, 2, 3 those of
            // step i + 1 (the last, odd step loads its own dims twice)
            const int kk = KW * warp + i + ((mi >> 1) && i + 1 < KW ? 1 : 0);
            const int dchunk = 2 * kk + (mi & 1);
            const uint32_t addr = kb + (dchunk >> 3) * (C::TILE * 128) + keyr * 128 + (((dchunk & 7) ^ (keyr & 7)) << 4);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(addr, b0, b1, b2, b3);
            mma_bf16_16816(sacc[nb], qa[i], b0, b1);
            if (i + 1 < KW) mma_bf16_16816(sacc[nb], qa[i + 1], b2, b3);
          }
        }
        float* mine_sx = sx + warp * 16 * C::SXROW;
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) {
          const int col = 8 * nb + 2 * (lane & 3);
          *reinterpret_cast<float2*>(mine_sx + r_lo * C::SXROW + col) = make_float2(sacc[nb][0], sacc[nb][1]);
          *reinterpret_cast<float2*>(mine_sx + r_hi * C::SXROW + col) = make_float2(sacc[nb][2], sacc[nb][3]);
        }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory"); // the partial tiles are complete
      float sc[4];
      {
        const int col = 8 * warp + 2 * (lane & 3);     // this warp's tokens
        float2 lo = make_float2(0.f, 0.f), hi = make_float2(0.f, 0.f);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float2 x = *reinterpret_cast<const float2*>(sx + (w * 16 + r_lo) * C::SXROW + col);
          const float2 y = *reinterpret_cast<const float2*>(sx + (w * 16 + r_hi) * C::SXROW + col);
          lo.x += x.x; lo.y += x.y; hi.x += y.x; hi.y += y.y;
        }
        sc[0] = lo.x; sc[1] = lo.y; sc[2] = hi.x; sc[3] = hi.y;
      }
      float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int jj = t0 + 8 * warp + 2 * (lane & 3) + (e & 1);
        sc[e] = jj < kend ? sc[e] * scale_log2 : -INFINITY;
        mt[e >> 1] = fmaxf(mt[e >> 1], sc[e]);
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
      {
        float pr[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pr[e] = ex2(sc[e] - m_use[e >> 1]);
          l_part[e >> 1] += pr[e];
        }
        const int col = 8 * warp + 2 * (lane & 3);
        *reinterpret_cast<uint32_t*>(pb + r_lo * C::PROW + col * 2) = pack_bf16x2(pr[0], pr[1]);
        *reinterpret_cast<uint32_t*>(pb + r_hi * C::PROW + col * 2) = pack_bf16x2(pr[2], pr[3]);
      }
      if (alpha[0] != 1.0f || alpha[1] != 1.0f) {
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          o[n][0] *= alpha[0]; o[n][1] *= alpha[0];
          o[n][2] *= alpha[1]; o[n][3] *= alpha[1];
        }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory"); // the P tile is complete
      // ---- o += P c_kv over the tile's 32 tokens, latent dims 128 warp .. -----------------
      const int lim = kend - t0;                      // first tile row past the end
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
          if (tail) {                                 // latent rows past the end may hold anything
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
    // ---- row sums over the 4 warps' tokens, then this segment's partial -------------------
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      l_part[row] += __shfl_xor_sync(0xffffffffu, l_part[row], 1);
      l_part[row] += __shfl_xor_sync(0xffffffffu, l_part[row], 2);
    }
    if ((lane & 3) == 0) {
      xs[warp * 16 + r_lo] = l_part[0];
      xs[warp * 16 + r_hi] = l_part[1];
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    // a wait that ran out publishes an empty partial: max -inf and sum 0, which the
    // re-association skips, never what an earlier call left in the workspace
    float lsum[2];
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      const int r = row ? r_hi : r_lo;
      lsum[row] = dead ? 0.0f : (xs[r] + xs[16 + r]) + (xs[32 + r] + xs[48 + r]);
      if (dead) m_run[row] = -INFINITY;
    }
    const int id = c + b;                            // this segment's partial slot
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      const int h = row ? r_hi : r_lo;
      if (h >= H) continue;
      const size_t slot = (size_t)id * H + h;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        const int dim = 128 * warp + 8 * n + 2 * (lane & 3);
        if (GA_BOUNDS(slot < (size_t)s.n_ids * H && dim + 2 <= C::R, 10, slot))
          *reinterpret_cast<float2*>(ws_o + slot * C::R + dim) =
              dead ? make_float2(0.0f, 0.0f) : make_float2(o[n][2 * row], o[n][2 * row + 1]);
      }
      if (warp == 0 && (lane & 3) == 0 && GA_BOUNDS(slot < (size_t)s.n_ids * H, 10, slot)) {
        ws_ml[slot * 2 + 0] = m_run[row];
        ws_ml[slot * 2 + 1] = lsum[row];
      }
    }
    if (j == 0 && threadIdx.x == 0 && GA_BOUNDS(b < s.batch, 12, b)) {
      // the sequence's first tile is in this share: its slots are c + b .. c_last + b
      const long long c_last = (r0 + nt - 1) / per;
      s.seg[b] = make_int2(id, (int)(c_last - c + 1));
    }
  }
  // a share that holds only the start cost of a sequence never waited for its query tile
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// grid: (DV / 64, n_heads, ceil(batch / 8)); block: 256; dynamic shared memory EX_SMEM (88 KB).
// Head h, output dims 64 x .. 64 x + 63, 8 sequences:
//  1. the weight slice w_uv[h][:, 64 x ..] (512 x 64 bf16) is copied into shared memory (144-byte
//     rows) with 16-byte asynchronous copies before the wait on the decode (it does not depend on
//     it);
//  2. warp w re-associates the partials of sequence w (o_lat = sum_c 2^(m_c - M) o_c / sum_c
//     2^(m_c - M) l_c over the decode's segments of the sequence; lane l holds latent dims 4 l ..
//     4 l + 3 of every 128; the first two partials are loaded together with their (m, l)) into a
//     shared [8][512] fp32 tile;
//  3. out = o_lat w_uv[h] on the tensor cores, mma.sync m16n8k16: each fp32 o_lat value x is split
//     into bf16 hi = rn(x) and lo = rn(x - hi), rows 0-7 of A holding the 8 sequences' hi parts and
//     rows 8-15 their lo parts, so rows g and g + 8 of the product add up to o_lat w_uv with an
//     error of about 2^-16 relative to x (fp32 sums).  Warp w takes latent rows 64 w .. 64 w + 63
//     for all 64 output dims; the 8 warps' sums meet in shared memory.
__global__ void __launch_bounds__(256)
mla_expand_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_ml,
                  const __nv_bfloat16* __restrict__ w_uv, __nv_bfloat16* __restrict__ out, MlaShape s) {
  using C = MlaCfg;
  extern __shared__ __align__(16) unsigned char ex_smem[];
  float* lat = reinterpret_cast<float*>(ex_smem + C::R * C::EX_WROW);         // [EX_SEQ][EX_LROW]
  float* part = lat;                          // [8 warps][EX_SEQ][EX_DIMS], once the products are done
  const int xb = blockIdx.x, h = blockIdx.y, b0 = blockIdx.z * C::EX_SEQ;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int nb = min(C::EX_SEQ, s.batch - b0);
  const uint32_t wsm = smem_u32(ex_smem);
  {
    constexpr int PR = C::EX_DIMS / 8;                                       // 16-byte pieces per row
    const __nv_bfloat16* wsrc = w_uv + (size_t)h * C::R * C::DV + xb * C::EX_DIMS;
    for (int e = t; e < C::R * PR; e += 256) {
      const int r = e / PR, pc = e % PR;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                   :: "r"(wsm + (uint32_t)(r * C::EX_WROW + 16 * pc)), "l"(wsrc + (size_t)r * C::DV + 8 * pc)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  griddep_wait();                                    // the partials of the decode kernel
  {
    constexpr int U = C::R / 128;
    const int i = warp, b = b0 + i;
    // an empty sequence has no partial (and no record): zero row
    const int2 rec = i < nb && seq_keys(s.lens, b, s.L_max) > 0 ? s.seg[b] : make_int2(0, 0);
    const int n_used = rec.x >= 0 && rec.y > 0 && rec.x + rec.y <= s.n_ids ? rec.y : 0;
    auto slot_of = [&](int c) { return ((size_t)rec.x + c) * s.n_heads + h; };
    float2 ml[2] = {make_float2(-INFINITY, 0.0f), make_float2(-INFINITY, 0.0f)};
    float4 v[2][U];
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int u = 0; u < U; ++u) v[c][u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < 2; ++c)
      if (c < n_used) {
        ml[c] = *reinterpret_cast<const float2*>(ws_ml + slot_of(c) * 2);
        const float* src = ws_o + slot_of(c) * C::R + 4 * lane;
#pragma unroll
        for (int u = 0; u < U; ++u) v[c][u] = *reinterpret_cast<const float4*>(src + 128 * u);
      }
    float M = fmaxf(ml[0].x, ml[1].x);
    if (n_used > 2) {                                // a sequence over more than two shares
      float Mx = -INFINITY;
      for (int c = 2 + lane; c < n_used; c += 32) Mx = fmaxf(Mx, ws_ml[slot_of(c) * 2]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, off));
      M = fmaxf(M, Mx);
    }
    float4 o[U];
#pragma unroll
    for (int u = 0; u < U; ++u) o[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    float Lsum = 0.0f;
    if (M != -INFINITY) {
      auto add = [&](float2 mlc, const float4 (&vc)[U]) {
        const float f = mlc.x == -INFINITY ? 0.0f : ex2(mlc.x - M);
        Lsum = fmaf(f, mlc.y, Lsum);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          o[u].x = fmaf(f, vc[u].x, o[u].x); o[u].y = fmaf(f, vc[u].y, o[u].y);
          o[u].z = fmaf(f, vc[u].z, o[u].z); o[u].w = fmaf(f, vc[u].w, o[u].w);
        }
      };
      add(ml[0], v[0]);
      add(ml[1], v[1]);                              // zero weight when absent (m = -inf)
      for (int c = 2; c < n_used; ++c) {
        const float2 mlc = *reinterpret_cast<const float2*>(ws_ml + slot_of(c) * 2);
        float4 vc[U];
        const float* src = ws_o + slot_of(c) * C::R + 4 * lane;
#pragma unroll
        for (int u = 0; u < U; ++u) vc[u] = *reinterpret_cast<const float4*>(src + 128 * u);
        add(mlc, vc);
      }
    }
    const float inv = Lsum > 0.0f ? 1.0f / Lsum : 0.0f;
#pragma unroll
    for (int u = 0; u < U; ++u)
      *reinterpret_cast<float4*>(lat + i * C::EX_LROW + 128 * u + 4 * lane) =
          make_float4(o[u].x * inv, o[u].y * inv, o[u].z * inv, o[u].w * inv);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  const int g = lane >> 2, tq = lane & 3, mi = lane >> 3, rr = lane & 7;
  float acc[C::EX_DIMS / 8][4];
#pragma unroll
  for (int n = 0; n < C::EX_DIMS / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;
#pragma unroll
  for (int ks = 0; ks < C::R / 16 / 8; ++ks) {
    const int k0 = (C::R / 8) * warp + 16 * ks;
    const float2 x01 = *reinterpret_cast<const float2*>(lat + g * C::EX_LROW + k0 + 2 * tq);
    const float2 x23 = *reinterpret_cast<const float2*>(lat + g * C::EX_LROW + k0 + 2 * tq + 8);
    auto lo_of = [](float x) { return x - __bfloat162float(__float2bfloat16_rn(x)); };
    uint32_t a[4];
    a[0] = pack_bf16x2(x01.x, x01.y);                 // row g: hi parts
    a[1] = pack_bf16x2(lo_of(x01.x), lo_of(x01.y));   // row g + 8: lo parts
    a[2] = pack_bf16x2(x23.x, x23.y);
    a[3] = pack_bf16x2(lo_of(x23.x), lo_of(x23.y));
#pragma unroll
    for (int n = 0; n < C::EX_DIMS / 8; n += 2) {
      const int krow = k0 + ((mi & 1) << 3) + rr, chunk = n + (mi >> 1);
      uint32_t b0_, b1_, b2_, b3_;
      ldmatrix_x4_trans(wsm + (uint32_t)(krow * C::EX_WROW + chunk * 16), b0_, b1_, b2_, b3_);
      mma_bf16_16816(acc[n], a, b0_, b1_);
      mma_bf16_16816(acc[n + 1], a, b2_, b3_);
    }
  }
  __syncthreads();                                   // every read of the latent tile is done
#pragma unroll
  for (int n = 0; n < C::EX_DIMS / 8; ++n)
    *reinterpret_cast<float2*>(part + (warp * C::EX_SEQ + g) * C::EX_DIMS + 8 * n + 2 * tq) =
        make_float2(acc[n][0] + acc[n][2], acc[n][1] + acc[n][3]);
  __syncthreads();
  for (int q = t; q < C::EX_SEQ * C::EX_DIMS; q += 256) {
    const int i = q / C::EX_DIMS, d = q % C::EX_DIMS;
    if (i < nb) {
      float y = 0.0f;
#pragma unroll
      for (int w = 0; w < 8; ++w) y += part[(w * C::EX_SEQ + i) * C::EX_DIMS + d];
      const size_t off = ((size_t)(b0 + i) * s.n_heads + h) * C::DV + xb * C::EX_DIMS + d;
      if (GA_BOUNDS(off < (size_t)s.batch * s.n_heads * C::DV, 11, off)) out[off] = __float2bfloat16_rn(y);
    }
  }
}

}  // namespace ga
