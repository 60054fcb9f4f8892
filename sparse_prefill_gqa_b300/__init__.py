"""Python binding of libga (include/ga.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does nothing but check
tensors, allocate outputs and workspace through PyTorch (device memory is PyTorch's job),
and pass pointers, sizes and the current CUDA stream to the library.  All arithmetic runs in
the library's CUDA kernels; there is no fallback of any kind: if ``libga.so`` is missing or
fails to load, every call raises.

Layouts (row-major, contiguous, on one CUDA device):
    q, out   [batch, n_heads, Tq, d]
    k, v     [batch, n_kv, Tk_max, d]
    dtype    torch.float32 or torch.bfloat16 (accumulation is fp32 either way)
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

__all__ = [
    "GAError", "lib", "library_path", "ga_attend", "ga_workspace_size", "ga_block_stats",
    "ga_select_blocks", "ga_read_device_status", "ga_set_wait_timeout_ns",
    "ga_selftest_wait_timeout", "ga_selftest_drop_prefill_chunk", "ga_status_string", "ga_version", "GA_OK", "GA_ERR_INVALID_ARG",
    "GA_ERR_UNSUPPORTED", "GA_ERR_CUDA", "GA_ERR_DEVICE_TIMEOUT", "GA_ERR_WORKSPACE",
    "GA_ERR_SCRATCH_LIMIT", "GA_DECODE_STATIC_SCRATCH_BYTES", "ga_attend_decode_static",
    "ga_ring_append", "ga_attend_ring", "ga_attend_diff", "ga_dsa_indexer", "ga_topk_indices",
    "ga_attend_gather", "dsa_decode", "ga_mla_decode", "GA_RADIUS_ZSCORE", "GA_RADIUS_MAD",
]

GA_OK, GA_ERR_INVALID_ARG, GA_ERR_UNSUPPORTED = 0, -1, -2
GA_ERR_CUDA, GA_ERR_DEVICE_TIMEOUT, GA_ERR_WORKSPACE = -3, -4, -5
GA_ERR_SCRATCH_LIMIT = -6
GA_DECODE_STATIC_SCRATCH_BYTES = 16 * 1024 * 1024
GA_RADIUS_ZSCORE, GA_RADIUS_MAD = 0, 1
_DTYPES = {torch.float32: 0, torch.bfloat16: 1}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


class GAError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {ga_status_string(status)} ({status})")
        self.status = status


def library_path() -> str:
    """The in-tree libga.so, or the library the GA_LIBRARY environment variable names (another
    build of the same sources, e.g. one with in-kernel checks)."""
    return os.environ.get("GA_LIBRARY") or os.path.join(_HERE, "libga.so")


def lib() -> ctypes.CDLL:
    """The loaded libga.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run `python -m sparse_prefill_gqa_b300.build`")
    L = ctypes.CDLL(path)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.ga_attend.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, i32, i32, vp, vp, i32,
                            i32, vp, i32, vp, sz, vp]
    L.ga_attend.restype = i32
    L.ga_attend_decode_static.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, i32, i32,
                                          vp, vp, vp]
    L.ga_attend_decode_static.restype = i32
    L.ga_dsa_indexer.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp]
    L.ga_dsa_indexer.restype = i32
    L.ga_topk_indices.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp]
    L.ga_topk_indices.restype = i32
    L.ga_attend_gather_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.ga_attend_gather_workspace_size.restype = sz
    L.ga_attend_gather.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, i32, vp, vp, vp, sz, vp]
    L.ga_attend_gather.restype = i32
    L.ga_mla_decode_workspace_size.argtypes = [i32, i32, i32]
    L.ga_mla_decode_workspace_size.restype = sz
    L.ga_mla_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, sz, vp]
    L.ga_mla_decode.restype = i32
    L.ga_attend_diff.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, i32, i32, f32,
                                 vp, sz, vp]
    L.ga_attend_diff.restype = i32
    L.ga_ring_append.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]
    L.ga_ring_append.restype = i32
    L.ga_attend_ring.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, sz, vp]
    L.ga_attend_ring.restype = i32
    L.ga_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    L.ga_workspace_size.restype = sz
    L.ga_block_stats.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, i32, vp]
    L.ga_block_stats.restype = i32
    L.ga_select_blocks.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                   f32, f32, vp, vp, i32, vp, sz, vp]
    L.ga_select_blocks.restype = i32
    L.ga_select_blocks_ex.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                      f32, f32, i32, f32, i32, vp, vp, i32, vp, sz, vp]
    L.ga_select_blocks_ex.restype = i32
    L.ga_select_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32]
    L.ga_select_workspace_size.restype = sz
    L.ga_read_device_status.argtypes = [vp]
    L.ga_read_device_status.restype = i32
    L.ga_debug_violation.argtypes = [ctypes.POINTER(ctypes.c_uint64), vp]
    L.ga_debug_violation.restype = i32
    L.ga_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    L.ga_set_wait_timeout_ns.restype = None
    L.ga_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    L.ga_selftest_wait_timeout.restype = i32
    L.ga_selftest_drop_prefill_chunk.argtypes = [i32]
    L.ga_selftest_drop_prefill_chunk.restype = None
    L.ga_status_string.argtypes = [i32]
    L.ga_status_string.restype = ctypes.c_char_p
    L.ga_version.argtypes = []
    L.ga_version.restype = i32
    _LIB = L
    return L


def ga_status_string(status: int) -> str:
    return lib().ga_status_string(int(status)).decode()


def ga_version() -> int:
    return int(lib().ga_version())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device=None):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _one_device(tensors, stream=None):
    """The one CUDA device that every given tensor (None entries skipped) and the explicit
    stream, if any, live on.  The library launches on the device current in the calling
    thread, with that device's static scratch and stream, so tensors on another device would
    reach a kernel as foreign pointers: mixed devices are refused here."""
    devs = {t.device for t in tensors if t is not None}
    if stream is not None:
        devs.add(torch.device(stream.device))
    if len(devs) != 1:
        raise ValueError("all tensors (and the stream) must be on one CUDA device, got "
                         + ", ".join(sorted(str(d) for d in devs)))
    return devs.pop()


def _check(status: int, what: str):
    if status != GA_OK:
        raise GAError(status, what)


def _need(t, name, dtype=None, dims=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dimensions")


def _need_size(t, name, n):
    """The kernels index ``t`` up to ``n`` elements: a shorter tensor is refused."""
    if t.numel() < n:
        raise ValueError(f"{name} must hold at least {n} elements (it holds {t.numel()})")


def _need_out(t, name, dtype, shape):
    _need(t, name, dtype, len(shape))
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}")


def _need_ws(t):
    if t is not None:
        _need(t, "workspace")


def ga_workspace_size(batch, n_heads, n_kv, d, Tq, Tk_max, dtype) -> int:
    return int(lib().ga_workspace_size(batch, n_heads, n_kv, d, Tq, Tk_max, _DTYPES[dtype]))


def ga_attend(q, k, v, out=None, *, k_lens=None, causal=True, window=0, sink=None,
              block_mask=None, q_block=128, k_block=64, lse=None, workspace=None, stream=None):
    """softmax(q k^T / sqrt(d) + mask) v with GQA heads; returns ``out`` (allocated if None).

    k_lens: int32 [batch] keys present per sequence; sink: float32 [n_heads];
    block_mask: uint8 [batch, n_heads, ceil(Tq/q_block), ceil(Tk_max/k_block)];
    lse: optional float32 [batch, n_heads, Tq] output; workspace: uint8 scratch of at least
    ga_workspace_size(...) bytes (allocated here if None and needed).
    """
    L = lib()
    if q.dtype not in _DTYPES:
        raise ValueError("q must be float32 or bfloat16")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, 4)
    B, H, Tq, d = q.shape
    n_kv, Tk_max = k.shape[1], k.shape[2]
    if k.shape != (B, n_kv, Tk_max, d) or v.shape != k.shape:
        raise ValueError("k and v must be [batch, n_kv, Tk_max, d] matching q")
    if out is None:
        out = torch.empty_like(q)
    _need_out(out, "out", q.dtype, q.shape)
    if k_lens is not None:
        _need(k_lens, "k_lens", torch.int32, 1)
        _need_size(k_lens, "k_lens", B)
    if sink is not None:
        _need(sink, "sink", torch.float32, 1)
        _need_size(sink, "sink", H)
    if block_mask is not None:
        _need(block_mask, "block_mask", torch.uint8, 4)
        _need_size(block_mask, "block_mask", B * H * -(-Tq // max(1, q_block)) * -(-Tk_max // max(1, k_block)))
    if lse is not None:
        _need(lse, "lse", torch.float32, 3)
        _need_size(lse, "lse", B * H * Tq)
    _need_ws(workspace)
    need = ga_workspace_size(B, H, n_kv, d, Tq, Tk_max, q.dtype) if H % max(n_kv, 1) == 0 else 0
    if need == 2 ** 64 - 1:
        need = 0
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dev = _one_device([q, k, v, out, k_lens, sink, block_mask, lse, workspace], stream)
    with torch.cuda.device(dev):
        st = L.ga_attend(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, n_kv, d, Tq, Tk_max, _ptr(k_lens),
                         int(bool(causal)), int(window), _ptr(sink), _ptr(block_mask), int(q_block),
                         int(k_block), _ptr(lse), _DTYPES[q.dtype], _ptr(workspace), ws_bytes,
                         _stream(stream, dev))
    _check(st, "ga_attend")
    return out


def ga_attend_decode_static(q, k, v, out=None, *, k_lens=None, causal=True, window=0, sink=None,
                            lse=None, stream=None):
    """Split-K decode (bf16) that allocates no device memory of its own: its scratch is the
    library's static array of GA_DECODE_STATIC_SCRATCH_BYTES, shared by every call.  For
    callers that cannot allocate (or pass) a workspace.  Calls that overlap on the GPU race
    on that array; the first call on a device should come before any stream capture.
    ``out`` is allocated here when None; pass it to allocate nothing at all."""
    L = lib()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    B, H, Tq, d = q.shape
    n_kv, Tk_max = k.shape[1], k.shape[2]
    if k.shape != (B, n_kv, Tk_max, d) or v.shape != k.shape:
        raise ValueError("k and v must be [batch, n_kv, Tk_max, d] matching q")
    if out is None:
        out = torch.empty_like(q)
    _need_out(out, "out", torch.bfloat16, q.shape)
    if k_lens is not None:
        _need(k_lens, "k_lens", torch.int32, 1)
        _need_size(k_lens, "k_lens", B)
    if sink is not None:
        _need(sink, "sink", torch.float32, 1)
        _need_size(sink, "sink", H)
    if lse is not None:
        _need(lse, "lse", torch.float32, 3)
        _need_size(lse, "lse", B * H * Tq)
    dev = _one_device([q, k, v, out, k_lens, sink, lse], stream)
    with torch.cuda.device(dev):
        st = L.ga_attend_decode_static(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, n_kv, d, Tq, Tk_max,
                                       _ptr(k_lens), int(bool(causal)), int(window), _ptr(sink), _ptr(lse),
                                       _stream(stream, dev))
    _check(st, "ga_attend_decode_static")
    return out


def ga_attend_diff(q1, k1, q2, k2, v, lam, out=None, *, k_lens=None, causal=True, window=0,
                   workspace=None, stream=None):
    """Differential attention (A1 - lam A2) v with A_i = softmax(q_i k_i^T / sqrt(d) + mask);
    bf16, d = 128 or 256.  workspace: >= batch * n_heads * Tq * d * 4 bytes (allocated here if
    None): the first map's result in fp32."""
    L = lib()
    for t, n in ((q1, "q1"), (k1, "k1"), (q2, "q2"), (k2, "k2"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    B, H, Tq, d = q1.shape
    n_kv, Tk_max = k1.shape[1], k1.shape[2]
    if q2.shape != q1.shape or k1.shape != (B, n_kv, Tk_max, d) or k2.shape != k1.shape or v.shape != k1.shape:
        raise ValueError("q1, q2 [B, H, Tq, d]; k1, k2, v [B, n_kv, Tk_max, d]")
    if out is None:
        out = torch.empty_like(q1)
    _need_out(out, "out", torch.bfloat16, q1.shape)
    if k_lens is not None:
        _need(k_lens, "k_lens", torch.int32, 1)
        _need_size(k_lens, "k_lens", B)
    _need_ws(workspace)
    need = B * H * Tq * d * 4
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q1.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    dev = _one_device([q1, k1, q2, k2, v, out, k_lens, workspace], stream)
    with torch.cuda.device(dev):
        st = L.ga_attend_diff(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v), _ptr(out), B, H, n_kv, d, Tq,
                              Tk_max, _ptr(k_lens), int(bool(causal)), int(window), float(lam), _ptr(workspace),
                              ws_bytes, _stream(stream, dev))
    _check(st, "ga_attend_diff")
    return out


def ga_dsa_indexer(qi, wi, ki, lens=None, scores=None, *, stream=None):
    """Indexer scores [B, L_max] (float32): sum_j wi[b, j] relu(qi[b, j] . ki[b, s]); -inf past
    lens[b].  qi [B, Hi, di] and ki [B, L_max, di] bf16, wi [B, Hi] float32."""
    L = lib()
    _need(qi, "qi", torch.bfloat16, 3)
    _need(ki, "ki", torch.bfloat16, 3)
    _need(wi, "wi", torch.float32, 2)
    B, Hi, di = qi.shape
    L_max = ki.shape[1]
    if ki.shape != (B, L_max, di) or wi.shape != (B, Hi):
        raise ValueError("qi [B, Hi, di], ki [B, L_max, di], wi [B, Hi]")
    if lens is not None:
        _need(lens, "lens", torch.int32, 1)
        _need_size(lens, "lens", B)
    if scores is None:
        scores = torch.empty(B, L_max, dtype=torch.float32, device=qi.device)
    _need_out(scores, "scores", torch.float32, (B, L_max))
    dev = _one_device([qi, wi, ki, lens, scores], stream)
    with torch.cuda.device(dev):
        _check(L.ga_dsa_indexer(_ptr(qi), _ptr(wi), _ptr(ki), _ptr(lens), B, Hi, di, L_max, _ptr(scores),
                                _stream(stream, dev)), "ga_dsa_indexer")
    return scores


def ga_topk_indices(scores, topk, lens=None, idx=None, n_sel=None, *, stream=None):
    """Per sequence the min(topk, lens[b]) highest-scoring positions (increasing order, ties to
    the lower position): (idx int32 [B, topk] with -1 padding, n_sel int32 [B])."""
    L = lib()
    _need(scores, "scores", torch.float32, 2)
    B, L_max = scores.shape
    if lens is not None:
        _need(lens, "lens", torch.int32, 1)
        _need_size(lens, "lens", B)
    if idx is None:
        idx = torch.empty(B, topk, dtype=torch.int32, device=scores.device)
    if n_sel is None:
        n_sel = torch.empty(B, dtype=torch.int32, device=scores.device)
    _need_out(idx, "idx", torch.int32, (B, int(topk)))
    _need(n_sel, "n_sel", torch.int32, 1)
    _need_size(n_sel, "n_sel", B)
    dev = _one_device([scores, lens, idx, n_sel], stream)
    with torch.cuda.device(dev):
        _check(L.ga_topk_indices(_ptr(scores), _ptr(lens), B, L_max, int(topk), _ptr(idx), _ptr(n_sel),
                                 _stream(stream, dev)), "ga_topk_indices")
    return idx, n_sel


def ga_attend_gather(q, k, v, idx, n_sel, out=None, *, sink=None, lse=None, workspace=None, stream=None):
    """Decode attention of q [B, H, 1, d] over the tokens idx[b, :n_sel[b]] of k, v."""
    L = lib()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    _need(idx, "idx", torch.int32, 2)
    _need(n_sel, "n_sel", torch.int32, 1)
    B, H, Tq, d = q.shape
    n_kv, Tk_max = k.shape[1], k.shape[2]
    topk = idx.shape[1]
    if Tq != 1 or v.shape != k.shape or idx.shape[0] != B:
        raise ValueError("q [B, H, 1, d], k, v [B, n_kv, Tk_max, d], idx [B, topk]")
    _need_size(n_sel, "n_sel", B)
    if out is None:
        out = torch.empty_like(q)
    _need_out(out, "out", torch.bfloat16, q.shape)
    if sink is not None:
        _need(sink, "sink", torch.float32, 1)
        _need_size(sink, "sink", H)
    if lse is not None:
        _need(lse, "lse", torch.float32, 3)
        _need_size(lse, "lse", B * H)
    _need_ws(workspace)
    need = int(L.ga_attend_gather_workspace_size(B, H, n_kv, d, topk))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    dev = _one_device([q, k, v, idx, n_sel, out, sink, lse, workspace], stream)
    with torch.cuda.device(dev):
        _check(L.ga_attend_gather(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, n_kv, d, Tk_max, _ptr(idx),
                                  _ptr(n_sel), topk, _ptr(sink), _ptr(lse), _ptr(workspace), ws_bytes,
                                  _stream(stream, dev)), "ga_attend_gather")
    return out


def dsa_decode(q, k, v, qi, wi, ki, topk, lens=None, *, sink=None, stream=None):
    """Indexer, top-k and gathered decode in order; returns (out, idx, n_sel, scores)."""
    scores = ga_dsa_indexer(qi, wi, ki, lens, stream=stream)
    idx, n_sel = ga_topk_indices(scores, topk, lens, stream=stream)
    out = ga_attend_gather(q, k, v, idx, n_sel, sink=sink, stream=stream)
    return out, idx, n_sel, scores


def ga_mla_decode(q_nope, q_rope, latent, w_uk, w_uv, lens=None, out=None, *, workspace=None, stream=None):
    """MLA decode, absorbed form: q_nope [B, H, 128], q_rope [B, H, 64], latent [B, L_max, 576]
    (c_kv | k_rope per token), w_uk and w_uv [H, 512, 128], all bf16; returns out [B, H, 128]."""
    L = lib()
    _need(q_nope, "q_nope", torch.bfloat16, 3)
    _need(q_rope, "q_rope", torch.bfloat16, 3)
    _need(latent, "latent", torch.bfloat16, 3)
    _need(w_uk, "w_uk", torch.bfloat16, 3)
    _need(w_uv, "w_uv", torch.bfloat16, 3)
    B, H, _ = q_nope.shape
    L_max = latent.shape[1]
    if q_nope.shape != (B, H, 128) or q_rope.shape != (B, H, 64) or latent.shape != (B, L_max, 576) \
            or w_uk.shape != (H, 512, 128) or w_uv.shape != (H, 512, 128):
        raise ValueError("MLA shapes: q_nope [B,H,128], q_rope [B,H,64], latent [B,L,576], w_uk/w_uv [H,512,128]")
    if lens is not None:
        _need(lens, "lens", torch.int32, 1)
        _need_size(lens, "lens", B)
    if out is None:
        out = torch.empty(B, H, 128, dtype=torch.bfloat16, device=q_nope.device)
    _need_out(out, "out", torch.bfloat16, (B, H, 128))
    _need_ws(workspace)
    need = int(L.ga_mla_decode_workspace_size(B, H, L_max))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_nope.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    dev = _one_device([q_nope, q_rope, latent, w_uk, w_uv, lens, out, workspace], stream)
    with torch.cuda.device(dev):
        _check(L.ga_mla_decode(_ptr(q_nope), _ptr(q_rope), _ptr(latent), _ptr(w_uk), _ptr(w_uv), _ptr(lens), _ptr(out),
                               B, H, L_max, _ptr(workspace), ws_bytes, _stream(stream, dev)), "ga_mla_decode")
    return out


def ga_ring_append(k_ring, v_ring, k_new, v_new, n_seen, *, stream=None):
    """Write one token per sequence into the W-slot ring caches: k_new, v_new [B, n_kv, d]
    go to slot n_seen[b] % W of k_ring, v_ring [B, n_kv, W, d]; n_seen [B] (int32) is then
    incremented on the device."""
    L = lib()
    for t, n in ((k_ring, "k_ring"), (v_ring, "v_ring")):
        _need(t, n, torch.bfloat16, 4)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, n, torch.bfloat16, 3)
    _need(n_seen, "n_seen", torch.int32, 1)
    B, n_kv, W, d = k_ring.shape
    if v_ring.shape != k_ring.shape or k_new.shape != (B, n_kv, d) or v_new.shape != k_new.shape \
            or n_seen.shape != (B,):
        raise ValueError("ring shapes: rings [B, n_kv, W, d], new tokens [B, n_kv, d], n_seen [B]")
    dev = _one_device([k_ring, v_ring, k_new, v_new, n_seen], stream)
    with torch.cuda.device(dev):
        st = L.ga_ring_append(_ptr(k_ring), _ptr(v_ring), _ptr(k_new), _ptr(v_new), _ptr(n_seen),
                              B, n_kv, d, W, _stream(stream, dev))
    _check(st, "ga_ring_append")


def ga_attend_ring(q, k_ring, v_ring, n_seen, out=None, *, sink=None, lse=None, workspace=None,
                   stream=None):
    """Decode attention of the newest token of every sequence (q [B, n_heads, 1, d]) over its
    ring cache: the min(n_seen[b], W) filled slots, after that token was appended."""
    L = lib()
    for t, n in ((q, "q"), (k_ring, "k_ring"), (v_ring, "v_ring")):
        _need(t, n, torch.bfloat16, 4)
    _need(n_seen, "n_seen", torch.int32, 1)
    B, H, Tq, d = q.shape
    n_kv, W = k_ring.shape[1], k_ring.shape[2]
    if Tq != 1 or k_ring.shape != (B, n_kv, W, d) or v_ring.shape != k_ring.shape or n_seen.shape != (B,):
        raise ValueError("q [B, n_heads, 1, d], rings [B, n_kv, W, d], n_seen [B]")
    if out is None:
        out = torch.empty_like(q)
    _need_out(out, "out", torch.bfloat16, q.shape)
    if sink is not None:
        _need(sink, "sink", torch.float32, 1)
        _need_size(sink, "sink", H)
    if lse is not None:
        _need(lse, "lse", torch.float32, 3)
        _need_size(lse, "lse", B * H)
    _need_ws(workspace)
    need = ga_workspace_size(B, H, n_kv, d, 1, W, q.dtype) if H % max(n_kv, 1) == 0 else 0
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dev = _one_device([q, k_ring, v_ring, out, n_seen, sink, lse, workspace], stream)
    with torch.cuda.device(dev):
        st = L.ga_attend_ring(_ptr(q), _ptr(k_ring), _ptr(v_ring), _ptr(out), B, H, n_kv, d, W, _ptr(n_seen),
                              _ptr(sink), _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream, dev))
    _check(st, "ga_attend_ring")
    return out


def ga_block_stats(k, k_block=64, *, k_lens=None, centroid=None, radius=None, stream=None):
    """Centroid [B, n_kv, nKb, d] and maximum radius [B, n_kv, nKb] of every key block."""
    L = lib()
    _need(k, "k", None, 4)
    if k.dtype not in _DTYPES:
        raise ValueError("k must be float32 or bfloat16")
    B, n_kv, Tk_max, d = k.shape
    nKb = -(-Tk_max // k_block)
    if centroid is None:
        centroid = torch.empty(B, n_kv, nKb, d, dtype=torch.float32, device=k.device)
    if radius is None:
        radius = torch.empty(B, n_kv, nKb, dtype=torch.float32, device=k.device)
    _need(centroid, "centroid", torch.float32, 4)
    _need_size(centroid, "centroid", B * n_kv * nKb * d)
    _need(radius, "radius", torch.float32, 3)
    _need_size(radius, "radius", B * n_kv * nKb)
    if k_lens is not None:
        _need(k_lens, "k_lens", torch.int32, 1)
        _need_size(k_lens, "k_lens", B)
    dev = _one_device([k, k_lens, centroid, radius], stream)
    with torch.cuda.device(dev):
        st = L.ga_block_stats(_ptr(k), _ptr(k_lens), B, n_kv, d, Tk_max, int(k_block), _ptr(centroid),
                              _ptr(radius), _DTYPES[k.dtype], _stream(stream, dev))
    _check(st, "ga_block_stats")
    return centroid, radius


def ga_select_blocks(q, centroid, radius, *, Tk=None, q_block=128, k_block=64, causal=True,
                     window=0, tau_mean=math.inf, lambda_radius=3.0, block_mask=None,
                     n_selected=None, n_kv=None, radius_rule="z", tau_bound=None, group_shared=False,
                     workspace=None, stream=None):
    """Block mask (uint8 [B, H, nQb, nKb]) and per-row counts (int32 [B, H, nQb]).

    radius_rule: "z" (mean and population std) or "mad" (median and 1.4826 * MAD);
    tau_bound: threshold of the Cauchy-Schwarz bound branch, None for no bound branch;
    group_shared: one selection per kv head from its heads' pooled query rows;
    workspace: uint8 scratch of ga_select_workspace_size(...) bytes (allocated here if None)."""
    L = lib()
    _need(q, "q", None, 4)
    if q.dtype not in _DTYPES:
        raise ValueError("q must be float32 or bfloat16")
    _need(centroid, "centroid", torch.float32, 4)
    _need(radius, "radius", torch.float32, 3)
    B, H, Tq, d = q.shape
    n_kv = centroid.shape[1] if n_kv is None else n_kv
    nKb_out = centroid.shape[2]
    Tk = nKb_out * k_block if Tk is None else Tk
    nQb = -(-Tq // q_block)
    _need_size(centroid, "centroid", B * n_kv * nKb_out * d)
    _need_size(radius, "radius", B * n_kv * nKb_out)
    if block_mask is None:
        block_mask = torch.empty(B, H, nQb, nKb_out, dtype=torch.uint8, device=q.device)
    if n_selected is None:
        n_selected = torch.empty(B, H, nQb, dtype=torch.int32, device=q.device)
    _need(block_mask, "block_mask", torch.uint8, 4)
    _need_size(block_mask, "block_mask", B * H * nQb * nKb_out)
    _need(n_selected, "n_selected", torch.int32, 3)
    _need_size(n_selected, "n_selected", B * H * nQb)
    rule = {"z": GA_RADIUS_ZSCORE, "mad": GA_RADIUS_MAD}[radius_rule]
    tb = -math.inf if tau_bound is None else float(tau_bound)
    _need_ws(workspace)
    need = int(L.ga_select_workspace_size(B, H, n_kv, d, Tq, int(Tk), int(q_block), int(k_block),
                                          int(bool(group_shared))))
    if need == 2 ** 64 - 1:
        need = 0
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dev = _one_device([q, centroid, radius, block_mask, n_selected, workspace], stream)
    with torch.cuda.device(dev):
        st = L.ga_select_blocks_ex(_ptr(q), _ptr(centroid), _ptr(radius), B, H, n_kv, d, Tq, int(Tk),
                                   nKb_out, int(q_block), int(k_block), int(bool(causal)), int(window),
                                   float(tau_mean), float(lambda_radius), rule, tb, int(bool(group_shared)),
                                   _ptr(block_mask),
                                   _ptr(n_selected), _DTYPES[q.dtype], _ptr(workspace), ws_bytes,
                                   _stream(stream, dev))
    _check(st, "ga_select_blocks")
    return block_mask, n_selected


def ga_read_device_status(stream=None) -> int:
    return int(lib().ga_read_device_status(_stream(stream)))


def ga_debug_violation(stream=None):
    """The debug build's first failed in-kernel bounds check since the last read (0: none), read
    and cleared; None from the ordinary build, which compiles no checks."""
    v = ctypes.c_uint64(0)
    st = int(lib().ga_debug_violation(ctypes.byref(v), _stream(stream)))
    if st == GA_ERR_UNSUPPORTED:
        return None
    if st != GA_OK:
        raise GAError(st, "ga_debug_violation")
    return int(v.value)


def ga_set_wait_timeout_ns(ns: int) -> None:
    lib().ga_set_wait_timeout_ns(int(ns))


def ga_selftest_wait_timeout(timeout_ns: int, stream=None) -> int:
    return int(lib().ga_selftest_wait_timeout(int(timeout_ns), _stream(stream)))


def ga_selftest_drop_prefill_chunk(chunk: int) -> None:
    """Test only: every CTA of the tensor-core prefill skips loading its ring chunk ``chunk``
    from the next call on, so its pipeline waits run out (-1 turns it off)."""
    lib().ga_selftest_drop_prefill_chunk(int(chunk))
