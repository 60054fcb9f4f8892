"""Oracle: a plain, slow, float64 CPU statement of what the attention path computes.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call, link or execute
anything under ``oracle/``; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` do.  The oracle shares no code
with the CUDA library (no kernels, headers, helpers or constants); both are fed from the
seeded generators in ``workloads/``, which hold none of the method's arithmetic.

Sources (web pages, cited by title and section):
  * "Attention in Code" (sotaaz.com/post/attention-in-code): the ``attend`` / ``causal``
    pair in "one function all designs use", grouped-query heads in section 1, the sliding
    ring cache in section 2, the sink in section 3.
  * "RBS-Attention review" (patty.io): block centroid scoring, mean dilution, the maximum
    key-block radius judged against its own distribution, two thresholded branches joined
    by a union, block-sparse FlashAttention execution.
  * "Attention Variants" lesson (factory.pai-world.com): the causal sliding-window mask and
    its W=4 diagram.
  * "Attention Masking" guide (devhandbook.co.kr): per-sequence length (padding) masks.
  * "Attention Variants" lesson: differential attention, (A1 - lambda A2) V.
  * "Attention in Code" section 5: an indexer scores every cached token, attention reads the top k.

Modules:
  attention  -- attend (dense / windowed / sink / block-masked / ragged), visibility rule
  blocks     -- block centroids and radii, mean-score + radius-rescue block selection
  ring       -- W-slot ring-buffer decode (the windowed cache of "Attention in Code" s.2)
  variants   -- differential attention ("Attention Variants", differential attention)
  dsa        -- token top-k sparse attention with a lightning-style indexer ("Attention in Code" s.5)
  mla        -- multi-head latent attention, naive and absorbed ("Attention in Code" s.4)
"""
from .attention import attend, positions, visible
from .blocks import allowed_blocks, block_stats, radius_zscores, select_blocks
from .ring import ring_contents, ring_decode
from .variants import attention_weights, diff_attend
from .dsa import dsa_decode, indexer_scores, sparse_attend, topk_indices

__all__ = ["attend", "positions", "visible", "allowed_blocks", "block_stats",
           "radius_zscores", "select_blocks", "ring_contents", "ring_decode", "attention_weights", "diff_attend",
           "dsa_decode", "indexer_scores", "sparse_attend", "topk_indices"]
