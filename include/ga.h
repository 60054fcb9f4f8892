/*
 * ga.h -- C ABI of libga: grouped-query scaled-dot-product attention with an
 * absolute-position causal mask, an optional sliding window, an optional per-head sink,
 * split-K decode, and radius-bounded block-sparse prefill, for NVIDIA B300 (sm_103a).
 *
 * Sources (web pages, by title and section):
 *   "Attention in Code" (sotaaz.com/post/attention-in-code):
 *       "one function all designs use"   -- attend(q, k, v, mask, sink) and causal(Tq, Tk, window)
 *       section 1 (MHA, MQA, GQA)          -- query head h reads kv head h / (n_heads / n_kv)
 *       section 3 (attention sink)         -- one logit per head with no value behind it
 *   "Express note" (tilnote.io), "causal attention is a position problem"
 *                                          -- the causal rule uses absolute positions
 *   "Attention Masking" guide (devhandbook.co.kr), Example 6 -- per-sequence key lengths
 *   "RBS-Attention review" (patty.io)       -- block centroids, maximum key-block radius,
 *                                              mean-score and radius-rescue branches, union,
 *                                              block-sparse FlashAttention execution
 *
 * Conventions shared by every entry point
 *   - Tensors are dense, row-major, in device memory:
 *       q, out     [batch, n_heads, Tq, d]
 *       k, v       [batch, n_kv, Tk_max, d]
 *     Element type is given by `dtype` (GA_F32: float, GA_BF16: bfloat16); accumulation
 *     is always fp32.  Every tensor pointer must be 16-byte aligned.
 *   - Query row t of sequence b sits at absolute position i = Tk_b - Tq + t, where
 *     Tk_b = k_lens[b] (or Tk_max).  Key j may be used by that row when
 *       j < Tk_b  and  (!causal or j <= i)  and  (window == 0 or j > i - window)
 *       and (block_mask == NULL or block_mask[b, h, t / q_block, j / k_block] != 0).
 *     A chunk's own keys and values must already be written at positions
 *     Tk_b - Tq .. Tk_b - 1 of the cache.
 *   - Ownership: the caller owns every buffer, including workspaces.  The library never
 *     allocates device memory and never synchronises the stream, except in
 *     ga_read_device_status.  All launches go to `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and are asynchronous.
 *   - Errors: argument checks run on the host before any launch and return a negative
 *     ga_status without touching the GPU.  A failed launch returns GA_ERR_CUDA.  A device
 *     wait that runs past its time limit records GA_ERR_DEVICE_TIMEOUT in a sticky device
 *     status word, read (and cleared) by ga_read_device_status.
 */
#ifndef GA_H
#define GA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so that this header needs no CUDA headers. */
typedef struct CUstream_st* ga_stream_t;

typedef enum { GA_F32 = 0, GA_BF16 = 1 } ga_dtype;

typedef enum {
  GA_OK = 0,
  GA_ERR_INVALID_ARG = -1,     /* a size, pointer, alignment or combination is invalid   */
  GA_ERR_UNSUPPORTED = -2,     /* valid, but outside what the kernels implement          */
  GA_ERR_CUDA = -3,            /* a CUDA runtime or driver call failed                   */
  GA_ERR_DEVICE_TIMEOUT = -4,  /* a device-side wait ran past its limit (sticky status)  */
  GA_ERR_WORKSPACE = -5,       /* workspace pointer missing or smaller than required     */
  GA_ERR_SCRATCH_LIMIT = -6    /* needs more than the static scratch array holds         */
} ga_status;

/*
 * ga_attend -- out = softmax(q k^T / sqrt(d) + mask) v for every (b, h, t).
 * ("Attention in Code", "one function all designs use"; GQA from section 1.)
 *
 *   q, k, v, out   device tensors as above; out has q's shape and dtype.
 *   batch >= 1; n_heads >= 1; 1 <= n_kv <= n_heads with n_heads % n_kv == 0;
 *   d: head dimension, 1..256 (GA_F32) or one of 16, 32, 64, 128, 256 (GA_BF16);
 *   1 <= Tq <= Tk_max; every k_lens[b] must lie in [Tq, Tk_max] (not checked on the
 *   host when k_lens lives on the device: out-of-range lengths give undefined rows).
 *   k_lens       device int32 [batch], or NULL for "every sequence holds Tk_max keys".
 *   causal       1: absolute-position causal rule; 0: no causal rule (requires window == 0).
 *   window       0: no window; W >= 1: the W most recent positions including the query's
 *                own ("Attention in Code" causal(); "Attention Variants" window mask).
 *   sink         device float [n_heads] logits, or NULL.  A sink joins the softmax
 *                normaliser of every row of its query head and carries no value
 *                ("Attention in Code", section 3); it is not scaled by 1/sqrt(d).
 *   block_mask   device uint8 [batch, n_heads, ceil(Tq/q_block), ceil(Tk_max/k_block)],
 *                nonzero = the (query block, key block) pair may be used; or NULL.
 *                Key blocks that are zero are never loaded by the tensor-core kernels.
 *   q_block, k_block  block sizes of block_mask (ignored when it is NULL).  The tensor-core
 *                path takes q_block % 128 == 0 and k_block % 64 == 0; other values run on the
 *                CUDA-core path.
 *   lse          optional device float [batch, n_heads, Tq]: natural-log normaliser
 *                ln(sum_allowed e^s + e^sink); -inf for a row with no allowed key and no sink.
 *   A row with no allowed key gets out = 0.
 *   workspace    device scratch of at least ga_workspace_size(...) bytes (may be NULL when
 *                that size is 0).  Must not be used by another call in flight.
 */
int ga_attend(const void* q, const void* k, const void* v, void* out,
              int batch, int n_heads, int n_kv, int d, int Tq, int Tk_max,
              const int32_t* k_lens, int causal, int window, const float* sink,
              const uint8_t* block_mask, int q_block, int k_block, float* lse,
              ga_dtype dtype, void* workspace, size_t workspace_bytes, ga_stream_t stream);

/* Bytes of workspace ga_attend needs for these sizes (0 when it needs none); SIZE_MAX
 * when the sizes are invalid.  Only the split-K decode path (Tq * n_heads / n_kv <= 16,
 * bf16) uses workspace: per (b, h, query row, key chunk) one fp32 partial output row plus
 * its running max and sum. */
size_t ga_workspace_size(int batch, int n_heads, int n_kv, int d, int Tq, int Tk_max,
                         ga_dtype dtype);

/* Size of the device array that ga_attend_decode_static uses as its scratch (16 MiB). */
#define GA_DECODE_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * ga_attend_decode_static -- the split-K decode of ga_attend, for callers that cannot
 * allocate device memory.  (No counterpart on the pages: this entry point exists only for
 * such callers.)  Examples: a plugin that runs inside an engine which owns all device
 * memory through its own pool and forbids outside allocations, and a latency-bound loop
 * where cudaMalloc/cudaFree are off limits because they can synchronise the device.  Such a
 * caller has no workspace to pass, so this call keeps its partial results in a
 * library-owned array instead.
 *
 * Computes exactly what ga_attend computes with dtype GA_BF16, block_mask NULL and a
 * workspace, for shapes on the split-K decode path: d = 64, 128 or 256 and
 * (n_heads / n_kv) * Tq <= 16.  Other shapes return GA_ERR_UNSUPPORTED.  The other
 * arguments, layouts and errors are those of ga_attend.
 *
 * Scratch: a file-scope __device__ array of GA_DECODE_STATIC_SCRATCH_BYTES, which every GPU
 * that loads the library holds until the process exits.  Shapes that would need more than
 * that (ga_workspace_size(...) > GA_DECODE_STATIC_SCRATCH_BYTES) return
 * GA_ERR_SCRATCH_LIMIT before any CUDA call.
 *   - The first call on a device does its set-up with that device current: it looks up
 *     the array's device address and sets the decode kernels' shared-memory limit.  Make
 *     that first call before any stream capture.
 *   - Every call shares the one array, which keeps the last call's contents.  Nothing in it
 *     needs to start at zero: each call writes every scratch slot it reads before reading it
 *     (a key chunk whose wait ran out writes an empty partial, which the combine skips).
 *   - Calls that overlap on the GPU race on the array: on different streams, or from host
 *     threads with no ordering between them.  Order such calls on one stream or with events.
 *   - It allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
int ga_attend_decode_static(const void* q, const void* k, const void* v, void* out,
                            int batch, int n_heads, int n_kv, int d, int Tq, int Tk_max,
                            const int32_t* k_lens, int causal, int window, const float* sink,
                            float* lse, ga_stream_t stream);

/*
 * ga_attend_diff -- differential attention, out = (A1 - lam * A2) v.
 * ("Attention Variants", differential attention: two attention maps from two query/key
 * pairs over the same values, the second scaled by a mixing coefficient and subtracted.)
 *
 *   A1 = softmax(q1 k1^T / sqrt(d) + mask), A2 = softmax(q2 k2^T / sqrt(d) + mask), the mask
 *   being ga_attend's (k_lens, causal, window) applied to both maps.
 *   q1, q2, out     device bf16 [batch, n_heads, Tq, d];  k1, k2, v: [batch, n_kv, Tk_max, d].
 *   lam             the mixing coefficient (finite).
 *   workspace       device scratch of at least batch * n_heads * Tq * d * 4 bytes, 16-byte
 *                   aligned: A1 v in fp32.  The difference is formed in fp32 and rounded to
 *                   bf16 once (the two terms may nearly cancel).
 *   d: 128 or 256 (the tensor-core path); other shapes GA_ERR_UNSUPPORTED.  Other arguments
 *   and errors as in ga_attend.
 */
int ga_attend_diff(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                   void* out, int batch, int n_heads, int n_kv, int d, int Tq, int Tk_max,
                   const int32_t* k_lens, int causal, int window, float lam, void* workspace,
                   size_t workspace_bytes, ga_stream_t stream);

/*
 * Token top-k sparse attention for decode ("Attention in Code", section 5): a small indexer
 * scores every cached token for the current query, and attention reads only the k tokens with
 * the highest scores; the cache keeps every token.  Decode form: one query per sequence at
 * position lens[b] - 1, which may see every cached token.  Three calls, in order:
 *
 * ga_dsa_indexer -- scores[b, s] = sum_j wi[b, j] * relu(qi[b, j] . ki[b, s]) for s < lens[b],
 *   -inf for lens[b] <= s < L_max.
 *   qi      device bf16 [batch, n_idx_heads, di]: the indexer's query heads.
 *   wi      device float [batch, n_idx_heads]: their weights.
 *   ki      device bf16 [batch, L_max, di]: one indexer key per cached token.
 *   lens    device int32 [batch] (tokens cached; clamped to [0, L_max]) or NULL (= L_max).
 *   scores  device float out [batch, L_max] (fp32 dot products and sums).
 *   di: 64 or 128; n_idx_heads a power of two <= di / 8; others GA_ERR_UNSUPPORTED.
 */
int ga_dsa_indexer(const void* qi, const float* wi, const void* ki, const int32_t* lens, int batch,
                   int n_idx_heads, int di, int L_max, float* scores, ga_stream_t stream);

/*
 * ga_topk_indices -- per sequence, the min(topk, lens[b]) positions with the highest scores,
 *   in increasing position order; among equal scores at the boundary the lower positions are
 *   kept.  idx device int32 out [batch, topk] (-1 past the count); n_sel device int32 out
 *   [batch]: the count.  scores as produced by ga_dsa_indexer (NaN scores: undefined order).
 */
int ga_topk_indices(const float* scores, const int32_t* lens, int batch, int L_max, int topk,
                    int32_t* idx, int32_t* n_sel, ga_stream_t stream);

/* Bytes of workspace ga_attend_gather needs (SIZE_MAX for invalid sizes): the split-K decode's
 * partial results over topk keys; 0 when the decode runs as one chunk (workspace may be NULL). */
size_t ga_attend_gather_workspace_size(int batch, int n_heads, int n_kv, int d, int topk);

/*
 * ga_attend_gather -- decode attention of q [batch, n_heads, 1, d] over the cached tokens
 *   idx[b, 0 .. n_sel[b]-1] of k, v [batch, n_kv, Tk_max, d] (bf16): softmax over exactly
 *   those keys (plus the optional sink), for every head of the sequence.  The split-K decode
 *   reads the selected rows straight from the cache; no compact copy is made.  n_sel[b] = 0
 *   (an empty cache) gives a zero row, and lse = the sink's logit or -inf.  idx entries must
 *   lie in [0, Tk_max) (others are clamped into it); idx 4-byte aligned, n_sel, lse and sink
 *   16-byte aligned.
 *   d: 64, 128 or 256; n_heads / n_kv <= 16; batch * n_kv * Tk_max < 2^31 (GA_ERR_UNSUPPORTED
 *   otherwise).  sink, lse as in ga_attend.
 */
int ga_attend_gather(const void* q, const void* k, const void* v, void* out, int batch,
                     int n_heads, int n_kv, int d, int Tk_max, const int32_t* idx,
                     const int32_t* n_sel, int topk, const float* sink, float* lse,
                     void* workspace, size_t workspace_bytes, ga_stream_t stream);

/*
 * ga_mla_decode -- multi-head latent attention, absorbed form, one new token per sequence.
 * ("Attention in Code", section 4: store only the latent vectors and move the weights to the
 * query side.)  With DeepSeek-V2-Lite's sizes: latent r = 512, rope key dr = 64, head dims
 * dn = dv = 128, up to 16 heads sharing the latent cache:
 *   q_lat = q_nope w_uk[h]^T, s_j = (q_lat . c_kv_j + q_rope . k_rope_j) / sqrt(dn + dr),
 *   out   = (softmax(s) c_kv) w_uv[h], over every cached token j < lens[b].
 *   q_nope   device bf16 [batch, n_heads, 128];  q_rope: [batch, n_heads, 64].
 *   latent   device bf16 [batch, L_max, 576]: per token c_kv (512) then k_rope (64).
 *   w_uk     device bf16 [n_heads, 512, 128];  w_uv: [n_heads, 512, 128].
 *   lens     device int32 [batch]: tokens cached, the new token's latent included, so
 *            1..L_max (larger values are clamped to L_max; 0, an empty cache, gives a zero
 *            row); or NULL (= L_max).
 *   out      device bf16 [batch, n_heads, 128].
 *   workspace of ga_mla_decode_workspace_size(batch, n_heads, L_max) bytes, 16-byte aligned:
 *            four parts, each rounded up to 256 bytes -- q_lat bf16 [batch, n_heads, 576], the
 *            decode's partial latents fp32 [n_ids, n_heads, 512] and their (max, sum) fp32
 *            [n_ids, n_heads, 2] with n_ids = 384 + batch - 1 (one slot per (CTA, sequence)
 *            segment of up to 384 decode CTAs), and per sequence its first slot and slot count,
 *            int32 [batch, 2].  The size does not depend on L_max.
 *   n_heads <= 16 (GA_ERR_UNSUPPORTED otherwise).  q_lat is rounded to bf16 before the scores.
 */
size_t ga_mla_decode_workspace_size(int batch, int n_heads, int L_max);
int ga_mla_decode(const void* q_nope, const void* q_rope, const void* latent, const void* w_uk,
                  const void* w_uv, const int32_t* lens, void* out, int batch, int n_heads,
                  int L_max, void* workspace, size_t workspace_bytes, ga_stream_t stream);

/*
 * ga_ring_append -- write one new token per sequence into a sliding-window ring cache.
 * ("Attention in Code", section 2: a layer that only looks at the last W tokens keeps a
 * cache of W slots per kv head; token number n, counting from 0, goes to slot n mod W and
 * overwrites the oldest token once the cache is full.)
 *
 *   k_ring, v_ring  device bf16 [batch, n_kv, W, d], caller-owned, updated in place.
 *   k_new, v_new    device bf16 [batch, n_kv, d]: the new token's key and value per kv head.
 *   n_seen          device int32 [batch]: tokens written so far.  Slot n_seen[b] mod W of
 *                   every kv head of sequence b receives the new token, then n_seen[b] is
 *                   incremented.  Must be >= 0 (not checked on the host; a negative value
 *                   writes nothing and leaves the counter unchanged).
 *   batch >= 1, n_kv >= 1, W >= 1, d a multiple of 8 in 8..256; the rings and new tokens
 *   16-byte aligned, n_seen 4-byte aligned.
 *   Asynchronous on stream; allocates nothing.  Calls that touch the same sequences must be
 *   ordered (one stream or events): each reads and increments the counter.
 */
int ga_ring_append(void* k_ring, void* v_ring, const void* k_new, const void* v_new,
                   int32_t* n_seen, int batch, int n_kv, int d, int W, ga_stream_t stream);

/*
 * ga_attend_ring -- decode attention of one query token per sequence over a ring cache.
 * ("Attention in Code", section 2.)  For the query at absolute position n_seen[b] - 1 with a
 * window of W positions, the keys it may use are exactly the min(n_seen[b], W) filled slots
 * of the ring; their order in the ring does not matter, because a softmax over a set of keys
 * does not depend on the order of the keys.  The result equals ga_attend with causal = 1 and
 * window = W over the whole key sequence.
 *
 *   q, out          device bf16 [batch, n_heads, 1, d].
 *   k_ring, v_ring  as in ga_ring_append, after the query token's own key and value were
 *                   appended.
 *   n_seen          device int32 [batch], >= 1 (values above W use all W slots).
 *   sink, lse       as in ga_attend.
 *   workspace       device scratch of ga_workspace_size(batch, n_heads, n_kv, d, 1, W,
 *                   GA_BF16) bytes (may be NULL when that is 0).
 *   d: 64, 128 or 256; n_heads / n_kv <= 16; other arguments and errors as in ga_attend.
 */
int ga_attend_ring(const void* q, const void* k_ring, const void* v_ring, void* out,
                   int batch, int n_heads, int n_kv, int d, int W, const int32_t* n_seen,
                   const float* sink, float* lse, void* workspace, size_t workspace_bytes,
                   ga_stream_t stream);

/*
 * ga_block_stats -- centroid and maximum radius of every key block.
 * ("RBS-Attention review": blocks represented by their centroid; the maximum key-block
 * radius is the distance from the centroid to the farthest key of the block.)
 *
 *   k          device [batch, n_kv, Tk_max, d], GA_BF16 or GA_F32.
 *   k_lens     device int32 [batch] or NULL (= Tk_max for every sequence).
 *   k_block    keys per block, 1..1024.
 *   centroid   device float [batch, n_kv, nKb, d], nKb = ceil(Tk_max / k_block):
 *              (1/n) sum of the n keys present in the block.
 *   radius     device float [batch, n_kv, nKb]: max over the block's keys of the
 *              Euclidean distance to the centroid.
 *   Blocks with no key present (j >= k_lens[b]) get a zero centroid and zero radius.
 *   d: 1..256.
 */
int ga_block_stats(const void* k, const int32_t* k_lens, int batch, int n_kv, int d,
                   int Tk_max, int k_block, float* centroid, float* radius, ga_dtype dtype,
                   ga_stream_t stream);

/*
 * ga_select_blocks -- block mask for radius-bounded sparse prefill.
 * ("RBS-Attention review": mean score of a query block against key-block centroids, a
 * radius-rescue branch judged against the head's own radius distribution, each with its
 * own threshold, joined by a union.)
 *
 * For query block alpha (rows alpha*q_block .. min(Tq, (alpha+1)*q_block) - 1, absolute
 * positions i_first .. i_last = Tk - Tq + those rows) of query head h, kv head
 * kvh = h / (n_heads / n_kv):
 *   visible(beta)  key block beta holds a key some row of the block may use under the
 *                  causal rule and window (all blocks when causal == 0);
 *   s(beta)        = mean_rows(q) . centroid[beta] / sqrt(d)             (fp32 operands; the
 *                  products on the tensor cores as three TF32 products of the operands'
 *                  high and low parts, accumulated in fp32: within about 2^-20 of each
 *                  product, rounding order aside)
 *   mean branch    s(beta) >= max_{visible} s - tau_mean                 (INFINITY = dense)
 *   radius branch  (radius[beta] - mu) / sigma >= lambda_radius, mu and sigma (population)
 *                  over the radii of all ceil(Tk/k_block) blocks of (b, kvh), in fp64;
 *                  nothing is rescued when sigma == 0
 *   diagonal       key blocks overlapping [i_first, i_last] are always kept
 *   block_mask[b, h, alpha, beta] = visible && (mean || radius || diagonal)
 * Key blocks beta >= ceil(Tk/k_block) of a row are written as 0 up to nKb_out.
 *
 *   q          device [batch, n_heads, Tq, d] (GA_BF16 or GA_F32).
 *   centroid, radius  as produced by ga_block_stats for the same k_block (row stride nKb_out).
 *   Tk         keys present in every sequence (Tq <= Tk); nKb_out = ceil(Tk_max/k_block) is
 *              the row length of block_mask, centroid and radius (nKb_out >= ceil(Tk/k_block)).
 *   block_mask device uint8 out [batch, n_heads, ceil(Tq/q_block), nKb_out].
 *   n_selected device int32 out [batch, n_heads, ceil(Tq/q_block)], or NULL.
 *   workspace  device scratch of ga_select_workspace_size(...) bytes, 256-byte aligned
 *              (GA_ERR_WORKSPACE otherwise): the mean query row of every query block and the
 *              centroids, each split into high and low parts, the rows' norms, the row maxima,
 *              the rescue flags and every mean-branch score, each computed once per call.
 *              Must not be used by another call in flight.
 *   d: 1..256; q_block: 1..4096; ceil(Tk/k_block) <= 32768.
 */
int ga_select_blocks(const void* q, const float* centroid, const float* radius,
                     int batch, int n_heads, int n_kv, int d, int Tq, int Tk, int nKb_out,
                     int q_block, int k_block, int causal, int window,
                     float tau_mean, float lambda_radius,
                     uint8_t* block_mask, int32_t* n_selected, ga_dtype dtype,
                     void* workspace, size_t workspace_bytes, ga_stream_t stream);

/* Bytes of workspace ga_select_blocks / ga_select_blocks_ex need (SIZE_MAX for invalid sizes):
 * batch * P * ceil(Tq/q_block) * (2 D + 2 + S) floats, batch * n_kv * ceil(Tk/k_block) * 2 D
 * floats and batch * n_kv * ceil(Tk/k_block) bytes, each of the seven parts rounded to 256
 * bytes, with P = n_kv when group_shared is 1 and n_heads otherwise, D = d rounded up to a
 * multiple of 32, and S = ceil(Tk/k_block) rounded up to a multiple of 128 (one score per key
 * block). */
size_t ga_select_workspace_size(int batch, int n_heads, int n_kv, int d, int Tq, int Tk, int q_block,
                                int k_block, int group_shared);

/* Radius rules of ga_select_blocks_ex. */
typedef enum {
  GA_RADIUS_ZSCORE = 0,   /* (r - mean) / population std, as ga_select_blocks */
  GA_RADIUS_MAD = 1       /* (r - median) / (1.4826 * median |r - median|): a few very large
                             radii cannot inflate the scale and hide themselves */
} ga_radius_rule;

/*
 * ga_select_blocks_ex -- ga_select_blocks with a choice of radius rule and a third branch.
 * ("RBS-Attention review": the radius is judged against the head's own radius
 * distribution; the method's name, radius-bounded, and the maximum key-block radius.)
 *
 *   radius_rule  GA_RADIUS_ZSCORE: the radius branch of ga_select_blocks.
 *                GA_RADIUS_MAD: z = (r - median) / (1.4826 * MAD) over the radii of the
 *                ceil(Tk/k_block) blocks of (b, kvh), median and MAD (median absolute
 *                deviation) of an even count being the mean of the two middle values, fp64;
 *                nothing is rescued when MAD == 0.  Needs ceil(Tk/k_block) <= 16384.
 *   tau_bound    bound branch: keep beta if
 *                  (mean_rows(q) . centroid[beta] + |mean_rows(q)| * radius[beta]) / sqrt(d)
 *                    >= max_{visible} s - tau_bound.
 *                The left side bounds the pooled query's score over every key of the block
 *                (Cauchy-Schwarz: |k - c| <= radius), so a block whose keys could score that
 *                high is kept however low its mean is.  -INFINITY: no bound branch.
 *   group_shared 1: one selection per kv head, from the query rows of its n_heads / n_kv heads
 *                pooled together (mean_rows above is then the mean over those heads' rows);
 *                every head of the group receives that mask and count (the heads of a group
 *                then read the same key blocks).  0: per query head.
 *   block_mask = visible && (mean || bound || radius || diagonal).  Everything else as in
 *   ga_select_blocks; NaN thresholds and unknown rules give GA_ERR_INVALID_ARG.
 */
int ga_select_blocks_ex(const void* q, const float* centroid, const float* radius,
                        int batch, int n_heads, int n_kv, int d, int Tq, int Tk, int nKb_out,
                        int q_block, int k_block, int causal, int window,
                        float tau_mean, float lambda_radius, int radius_rule, float tau_bound,
                        int group_shared, uint8_t* block_mask, int32_t* n_selected,
                        ga_dtype dtype, void* workspace, size_t workspace_bytes,
                        ga_stream_t stream);

/* Synchronises `stream`, then returns and clears the sticky device status of the device
 * current in the calling thread (each device has its own status word; make the device whose
 * kernels are to be checked current first, and pass a stream of that device): GA_OK, or
 * GA_ERR_DEVICE_TIMEOUT when some kernel on that device gave up on a wait since the last read.
 * Returns GA_ERR_CUDA when the synchronisation itself fails. */
int ga_read_device_status(ga_stream_t stream);

/* The debug build (the same sources compiled with GA_DEBUG defined: libga_debug.so) checks, in
 * the kernels, the offsets of its output stores against the outputs' extents and the coordinates
 * of its TMA copies, skips an access that fails and records the device's first failure in a
 * sticky word.  Synchronises `stream`, then stores and clears that word in *first: 0 when no
 * check failed, else (site << 48) | offset (sites: 1 TMA coordinate or destination, 2 prefill
 * output, 3 prefill lse, 4 decode partials, 5 decode output, 6 top-k indices, 7 selection
 * scores, 8 block mask, 9 MLA q_lat, 10 MLA partials, 11 MLA output, 12 MLA per-sequence slot
 * records).  Returns GA_OK, or
 * GA_ERR_UNSUPPORTED from the ordinary build (no checks compiled), GA_ERR_CUDA on a failed
 * synchronisation. */
int ga_debug_violation(uint64_t* first, ga_stream_t stream);

/* Time limit for every device-side wait, in nanoseconds (default 2e9; minimum 1e5).
 * Applies to launches made after the call. */
void ga_set_wait_timeout_ns(uint64_t ns);

/* Launches one small kernel that waits on a flag nothing ever sets, with the bounded wait
 * every kernel of the library uses, and returns the launch status.  The wait gives up
 * after `timeout_ns` and records GA_ERR_DEVICE_TIMEOUT, which ga_read_device_status then
 * reports.  Used to test the failure path without faulting or hanging the GPU. */
int ga_selftest_wait_timeout(uint64_t timeout_ns, ga_stream_t stream);

/* Test only (the failure-path test of the pipeline waits): from the next call on, the
 * tensor-core prefill's producer in every CTA skips the load of ring chunk number `chunk`
 * (counted over that CTA's work, from 0), so every wait on that chunk runs out after the wait
 * limit and the launch ends with GA_ERR_DEVICE_TIMEOUT in the status word, its other loads and
 * MMAs drained and its tensor memory freed.  -1 (the default) turns it off again; nothing else
 * in the library reads it.  Not for concurrent use with other calls. */
void ga_selftest_drop_prefill_chunk(int chunk);

/* Human-readable name of a ga_status value (a static string). */
const char* ga_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int ga_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GA_H */
