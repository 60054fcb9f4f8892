"""Seeded generators for q, k, v, sinks, sequence lengths, planted outlier keys and sampled rows.

Every [B, H, T, d] tensor is drawn one (b, h) slice at a time from its own PCG64 stream,
keyed by (seed, tensor tag, b, h).  A slice can therefore be regenerated on its own (the
oracle checks at full size need only a few slices) and the result does not depend on how
many threads drew it.  Values are drawn in float32 and, for bf16 workloads, cast to bf16 on
the host with round-to-nearest-even; both the CUDA path and the oracle receive exactly those
bf16 values (the oracle upcasts them to float64).
"""
from __future__ import annotations

import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = [
    "f32_to_bf16_bits", "bf16_bits_to_f32", "slice_rng", "normal_slices", "randn_bhtd",
    "uniform_lengths", "planted_outliers", "sample_rows",
]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even cast of finite float32 values to bfloat16 bit patterns (uint16)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns (uint16) to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _tag_id(tag: str) -> int:
    return zlib.crc32(tag.encode("ascii")) & 0x7FFFFFFF


def slice_rng(seed: int, tag: str, *idx: int) -> np.random.Generator:
    """Independent PCG64 stream for one slice of one tensor of one workload."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _tag_id(tag), *idx])))


def normal_slices(seed: int, tag: str, b: int, h: int, rows: int, d: int,
                  dtype: str = "bf16") -> np.ndarray:
    """One [rows, d] slice of N(0, 1) draws: uint16 bf16 bits for dtype 'bf16', else float32."""
    x = slice_rng(seed, tag, b, h).standard_normal((rows, d), dtype=np.float32)
    return f32_to_bf16_bits(x) if dtype == "bf16" else x


def randn_bhtd(seed: int, tag: str, shape, dtype: str = "bf16", lengths=None,
               threads: int | None = None) -> np.ndarray:
    """[B, H, T, d] tensor of N(0, 1) draws, slice (b, h) from its own stream.

    With ``lengths`` (one per batch entry), only rows t < lengths[b] are drawn; the rest of
    the slice is left zero.  Returns uint16 bf16 bits for dtype 'bf16', float32 otherwise.
    """
    B, H, T, d = (int(s) for s in shape)
    out = np.zeros((B, H, T, d), dtype=np.uint16 if dtype == "bf16" else np.float32)

    def work(bh):
        b, h = divmod(bh, H)
        n = T if lengths is None else int(lengths[b])
        if n > 0:
            out[b, h, :n] = normal_slices(seed, tag, b, h, n, d, dtype)

    nthreads = threads or min(32, os.cpu_count() or 1)
    if B * H == 1 or nthreads == 1:
        for bh in range(B * H):
            work(bh)
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(work, range(B * H)))
    return out


def uniform_lengths(seed: int, batch: int, lo: int, hi: int) -> np.ndarray:
    """Per-sequence lengths drawn uniformly from the integers lo..hi inclusive (int32)."""
    return slice_rng(seed, "k_lens").integers(lo, hi + 1, size=batch).astype(np.int32)


def planted_outliers(seed: int, n_kv: int, T: int, d: int, k_block: int,
                     fraction: float = 0.05, scale: float | None = None):
    """Choose the key blocks that hold one planted outlier key, and the key itself.

    Per kv head, round(fraction * n_blocks) blocks are drawn without replacement; in each,
    one slot is drawn uniformly and its key is replaced by ``scale * u`` with u uniform on
    the unit sphere (a normalised N(0, I_d) draw).  ``scale`` defaults to 8 * sqrt(d).
    Returns a list of (kvh, block, token_index, float32 vector[d]).
    """
    n_blocks = -(-T // k_block)
    n_plant = int(round(fraction * n_blocks))
    s = 8.0 * np.sqrt(d) if scale is None else float(scale)
    planted = []
    for kvh in range(n_kv):
        rng = slice_rng(seed, "planted", kvh)
        blocks = np.sort(rng.choice(n_blocks, size=n_plant, replace=False))
        for blk in blocks:
            size = min(k_block, T - int(blk) * k_block)
            slot = int(rng.integers(0, size))
            z = rng.standard_normal(d).astype(np.float64)
            u = z / np.linalg.norm(z)
            planted.append((kvh, int(blk), int(blk) * k_block + slot, (s * u).astype(np.float32)))
    return planted


def sample_rows(Tq: int, n: int = 256, seed: int = 0, q_block: int = 128, window: int = 0,
                Tk: int | None = None, extra=()) -> np.ndarray:
    """Sorted distinct query rows for sampled oracle checks at full size.

    Always includes the first and last rows, the rows on each side of every query-block
    boundary (up to a cap), the rows whose absolute position sits at the window edge, and
    any ``extra`` rows; the remainder is a seeded uniform draw.
    """
    Tk = Tq if Tk is None else Tk
    must = {0, Tq - 1}
    for a in range(q_block, Tq, q_block)[:16]:
        must.update((a - 1, a))
    if window:
        off = Tk - Tq
        for i in (window - 1, window, window + 1):
            t = i - off
            if 0 <= t < Tq:
                must.add(t)
    must.update(int(t) for t in extra if 0 <= int(t) < Tq)
    must = sorted(must)
    if len(must) >= min(n, Tq):
        return np.array(must[:max(n, len(must))], dtype=np.int64)
    rng = slice_rng(seed, "rows")
    pool = np.setdiff1d(np.arange(Tq), np.array(must))
    fill = rng.choice(pool, size=min(n, Tq) - len(must), replace=False)
    return np.sort(np.concatenate([np.array(must), fill])).astype(np.int64)
