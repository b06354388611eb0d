"""Thin Python binding of librq.so (include/rq.h).

Argument marshalling only: every step of quantize-append and attention runs in the CUDA
kernels of librq.so.  PyTorch tensors supply device memory and the current CUDA stream.
There is no CPU fallback: if the library cannot be built or loaded, every call raises.

Low-level functions carry the C names (rq_create, rq_quantize_append, rq_decode_attention,
rq_verify_attention, rq_free, ...); `KVCache` bundles a context with its page pool.
"""
from __future__ import annotations

import ctypes
import threading

import numpy as np
import torch

from . import build as _build

RQ_OK, RQ_ERR_INVALID, RQ_ERR_UNSUPPORTED, RQ_ERR_CUDA, RQ_ERR_CAPACITY = 0, 1, 2, 3, 4
RQ_STATUS_BAD_PAGE, RQ_STATUS_BAD_SLOT, RQ_STATUS_BAD_LEN, RQ_STATUS_NORM_OVERFLOW, RQ_STATUS_TIMEOUT = 1, 2, 4, 8, 16
RQ_PLANAR, RQ_ISO, RQ_DENSE = 0, 1, 2
HEAD_DIM = 128

EXPORTS = ["rq_create", "rq_free", "rq_page_bytes", "rq_lloyd_max_codebook", "rq_get_codebook",
           "rq_quantize_append", "rq_decode_attention", "rq_verify_attention", "rq_set_profile_events",
           "rq_decode_attention_noalloc", "rq_tree_verify_attention", "rq_decode_step", "rq_extend_attention", "rq_status_string"]


class RQError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {status_string(code)} ({code})")
        self.code = code


class rq_config(ctypes.Structure):
    _fields_ = [
        ("head_dim", ctypes.c_int), ("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
        ("bits", ctypes.c_int), ("mode", ctypes.c_int), ("page_size", ctypes.c_int), ("num_pages", ctypes.c_int),
        ("max_batch", ctypes.c_int), ("max_query_tokens", ctypes.c_int), ("max_pages_per_seq", ctypes.c_int),
        ("rot_k", ctypes.POINTER(ctypes.c_float)), ("rot_v", ctypes.POINTER(ctypes.c_float)),
        ("codebook", ctypes.POINTER(ctypes.c_float)), ("sm_scale", ctypes.c_float), ("device", ctypes.c_int),
    ]


_lock = threading.Lock()
_lib = None


def lib(path: str | None = None) -> ctypes.CDLL:
    """Load librq.so (building it with nvcc first if it is missing or stale)."""
    global _lib
    if _lib is not None and path is None:  # loaded: no lock on the call path
        return _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(path or _build.build())
            vp, i32p, fp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_float)
            L.rq_create.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(rq_config)]
            L.rq_create.restype = ctypes.c_int
            L.rq_free.argtypes = [vp]
            L.rq_free.restype = None
            L.rq_page_bytes.argtypes = [vp]
            L.rq_page_bytes.restype = ctypes.c_size_t
            L.rq_lloyd_max_codebook.argtypes = [ctypes.c_int, ctypes.c_int, fp]
            L.rq_lloyd_max_codebook.restype = ctypes.c_int
            L.rq_get_codebook.argtypes = [vp, fp, fp]
            L.rq_get_codebook.restype = ctypes.c_int
            L.rq_quantize_append.argtypes = [vp, vp, vp, vp, ctypes.c_int, vp, vp, vp]
            L.rq_quantize_append.restype = ctypes.c_int
            L.rq_decode_attention.argtypes = [vp, vp, vp, vp, ctypes.c_int, vp, ctypes.c_int, vp, vp, vp]
            L.rq_decode_attention.restype = ctypes.c_int
            L.rq_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, ctypes.c_int, vp, vp, vp]
            L.rq_decode_step.restype = ctypes.c_int
            L.rq_extend_attention.argtypes = [vp, vp, ctypes.c_int, vp, vp, ctypes.c_int, vp, ctypes.c_int, vp, vp, vp]
            L.rq_extend_attention.restype = ctypes.c_int
            L.rq_verify_attention.argtypes = [vp, vp, ctypes.c_int, vp, vp, ctypes.c_int, vp, ctypes.c_int, vp, vp,
                                              vp]
            L.rq_verify_attention.restype = ctypes.c_int
            L.rq_tree_verify_attention.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, ctypes.c_int, vp, ctypes.c_int,
                                                   vp, vp, vp]
            L.rq_tree_verify_attention.restype = ctypes.c_int
            L.rq_decode_attention_noalloc.argtypes = [ctypes.POINTER(rq_config), vp, vp, vp, vp, vp, vp,
                                                      ctypes.c_int, vp, ctypes.c_int, vp, vp, vp]
            L.rq_decode_attention_noalloc.restype = ctypes.c_int
            L.rq_set_profile_events.argtypes = [vp, vp, vp]
            L.rq_set_profile_events.restype = ctypes.c_int
            L.rq_status_string.argtypes = [ctypes.c_int]
            L.rq_status_string.restype = ctypes.c_char_p
            _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().rq_status_string(int(code)).decode()


def _check(fn: str, code: int):
    if code != RQ_OK:
        raise RQError(fn, code)


def _ptr(t):
    """An address for a c_void_p argument (ctypes converts the int itself)."""
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr()
    return int(t)


def _stream(stream, device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream if hasattr(s, "cuda_stream") else int(s)


def rq_lloyd_max_codebook(bits: int, head_dim: int = HEAD_DIM) -> np.ndarray:
    out = np.zeros(1 << bits, np.float32)
    _check("rq_lloyd_max_codebook",
           lib().rq_lloyd_max_codebook(bits, head_dim, out.ctypes.data_as(ctypes.POINTER(ctypes.c_float))))
    return out


def rq_create(mode: int, bits: int, num_q_heads: int, num_kv_heads: int, page_size: int, num_pages: int,
              rot_k, rot_v, max_batch: int, max_query_tokens: int = 1, max_pages_per_seq: int = 1,
              codebook=None, sm_scale: float = 0.0, device: int = -1) -> ctypes.c_void_p:
    rk = np.ascontiguousarray(rot_k, np.float32).reshape(-1)
    rv = np.ascontiguousarray(rot_v, np.float32).reshape(-1)
    want = num_kv_heads * HEAD_DIM * (HEAD_DIM if mode == RQ_DENSE else 1)
    if rk.size != want or rv.size != want:  # the library reads exactly `want` floats of each
        raise RQError("rq_create", RQ_ERR_INVALID)
    cb = None if codebook is None else np.ascontiguousarray(codebook, np.float32)
    fp = ctypes.POINTER(ctypes.c_float)
    cfg = rq_config(HEAD_DIM, num_q_heads, num_kv_heads, bits, mode, page_size, num_pages, max_batch,
                    max_query_tokens, max_pages_per_seq, rk.ctypes.data_as(fp), rv.ctypes.data_as(fp),
                    cb.ctypes.data_as(fp) if cb is not None else fp(), float(sm_scale), int(device))
    ctx = ctypes.c_void_p()
    _check("rq_create", lib().rq_create(ctypes.byref(ctx), ctypes.byref(cfg)))
    return ctx


def rq_free(ctx) -> None:
    lib().rq_free(ctx)


def rq_page_bytes(ctx) -> int:
    return int(lib().rq_page_bytes(ctx))


def rq_get_codebook(ctx, bits: int):
    c = np.zeros(1 << bits, np.float32)
    b = np.zeros((1 << bits) - 1, np.float32)
    fp = ctypes.POINTER(ctypes.c_float)
    _check("rq_get_codebook", lib().rq_get_codebook(ctx, c.ctypes.data_as(fp), b.ctypes.data_as(fp)))
    return c, b


def rq_quantize_append(ctx, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, kv_pages: torch.Tensor,
                       status: torch.Tensor | None = None, stream=None) -> None:
    """k, v: fp16 [n][Hkv][128] on the device; slot_mapping int32 [n]."""
    n = slot_mapping.numel()
    if n:
        assert k.dtype == torch.float16 and v.dtype == torch.float16 and slot_mapping.dtype == torch.int32
        assert k.is_contiguous() and v.is_contiguous() and slot_mapping.is_contiguous()
    _check("rq_quantize_append",
           lib().rq_quantize_append(ctx, _ptr(k), _ptr(v), _ptr(slot_mapping), n, _ptr(kv_pages), _ptr(status),
                                    _stream(stream, kv_pages.device)))


def rq_decode_attention(ctx, q: torch.Tensor, kv_pages: torch.Tensor, block_table: torch.Tensor,
                        seq_lens: torch.Tensor, out: torch.Tensor, status: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """q, out: fp16 [B][Hq][128]; block_table int32 [B][max_pages]; seq_lens int32 [B]."""
    B = seq_lens.numel()
    assert q.dtype == torch.float16 and out.dtype == torch.float16 and q.is_contiguous() and out.is_contiguous()
    assert block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32 and block_table.is_contiguous()
    _check("rq_decode_attention",
           lib().rq_decode_attention(ctx, _ptr(q), _ptr(kv_pages), _ptr(block_table), block_table.shape[-1],
                                     _ptr(seq_lens), B, _ptr(out), _ptr(status), _stream(stream, q.device)))
    return out


def rq_decode_step(ctx, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, kv_pages: torch.Tensor,
                   block_table: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor,
                   status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One decode step: append k_new / v_new (fp16 [B][Hkv][128]) at position seq_lens[b] - 1 of
    each sequence, then decode attention; q, out fp16 [B][Hq][128]."""
    B = seq_lens.numel()
    for t in (q, out, k_new, v_new):
        assert t.dtype == torch.float16 and t.is_contiguous()
    assert block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32 and block_table.is_contiguous()
    _check("rq_decode_step",
           lib().rq_decode_step(ctx, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kv_pages), _ptr(block_table),
                                block_table.shape[-1], _ptr(seq_lens), B, _ptr(out), _ptr(status),
                                _stream(stream, q.device)))
    return out


def rq_extend_attention(ctx, q: torch.Tensor, kv_pages: torch.Tensor, block_table: torch.Tensor,
                        seq_lens: torch.Tensor, out: torch.Tensor, status: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """Extend (prefill) attention: q, out fp16 [B][T][Hq][128]; row j sees positions <= len - T + j."""
    B, T = q.shape[0], q.shape[1]
    assert q.dtype == torch.float16 and out.dtype == torch.float16 and q.is_contiguous() and out.is_contiguous()
    assert block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32 and block_table.is_contiguous()
    _check("rq_extend_attention",
           lib().rq_extend_attention(ctx, _ptr(q), T, _ptr(kv_pages), _ptr(block_table), block_table.shape[-1],
                                     _ptr(seq_lens), B, _ptr(out), _ptr(status), _stream(stream, q.device)))
    return out


def rq_verify_attention(ctx, q: torch.Tensor, kv_pages: torch.Tensor, block_table: torch.Tensor,
                        seq_lens: torch.Tensor, out: torch.Tensor, status: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """q, out: fp16 [B][T][Hq][128]."""
    B, T = q.shape[0], q.shape[1]
    assert q.dtype == torch.float16 and out.dtype == torch.float16 and q.is_contiguous() and out.is_contiguous()
    assert block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32 and block_table.is_contiguous()
    _check("rq_verify_attention",
           lib().rq_verify_attention(ctx, _ptr(q), T, _ptr(kv_pages), _ptr(block_table), block_table.shape[-1],
                                     _ptr(seq_lens), B, _ptr(out), _ptr(status), _stream(stream, q.device)))
    return out


def rq_tree_verify_attention(ctx, q: torch.Tensor, tree_mask: torch.Tensor, kv_pages: torch.Tensor,
                             block_table: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor,
                             status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """q, out: fp16 [B][T][Hq][128]; tree_mask int64/uint64 [B][T] (bit i of row j: draft i visible)."""
    B, T = q.shape[0], q.shape[1]
    assert q.dtype == torch.float16 and out.dtype == torch.float16 and q.is_contiguous() and out.is_contiguous()
    assert tree_mask.dtype in (torch.int64, torch.uint64) and tree_mask.is_contiguous() and tuple(tree_mask.shape) == (B, T)
    assert block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32 and block_table.is_contiguous()
    _check("rq_tree_verify_attention",
           lib().rq_tree_verify_attention(ctx, _ptr(q), T, _ptr(tree_mask), _ptr(kv_pages), _ptr(block_table),
                                          block_table.shape[-1], _ptr(seq_lens), B, _ptr(out), _ptr(status),
                                          _stream(stream, q.device)))
    return out


def rq_decode_attention_noalloc(mode: int, bits: int, num_q_heads: int, num_kv_heads: int, page_size: int,
                                num_pages: int, d_rot_k: torch.Tensor, d_rot_v: torch.Tensor,
                                d_centroids: torch.Tensor, q: torch.Tensor, kv_pages: torch.Tensor,
                                block_table: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor,
                                status: torch.Tensor | None = None, sm_scale: float = 0.0,
                                stream=None) -> torch.Tensor:
    """Decode attention with no allocation: tables as device float32 tensors, scratch in the
    library's fixed device array (see include/rq.h)."""
    for t in (d_rot_k, d_rot_v, d_centroids):
        assert t.dtype == torch.float32 and t.is_contiguous() and t.is_cuda
    assert q.dtype == torch.float16 and out.dtype == torch.float16 and q.is_contiguous() and out.is_contiguous()
    assert block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32 and block_table.is_contiguous()
    cfg = rq_config(HEAD_DIM, num_q_heads, num_kv_heads, bits, mode, page_size, num_pages, 0, 0, 0,
                    ctypes.POINTER(ctypes.c_float)(), ctypes.POINTER(ctypes.c_float)(),
                    ctypes.POINTER(ctypes.c_float)(), float(sm_scale), -1)
    _check("rq_decode_attention_noalloc",
           lib().rq_decode_attention_noalloc(ctypes.byref(cfg), _ptr(d_rot_k), _ptr(d_rot_v), _ptr(d_centroids),
                                             _ptr(q), _ptr(kv_pages), _ptr(block_table), block_table.shape[-1],
                                             _ptr(seq_lens), seq_lens.numel(), _ptr(out), _ptr(status),
                                             _stream(stream, q.device)))
    return out


def rq_set_profile_events(ctx, ev_start=None, ev_end=None) -> None:
    """Record torch.cuda.Event pairs around the split-K attention kernel of later calls."""
    a = ctypes.c_void_p(ev_start.cuda_event) if ev_start is not None else None
    b = ctypes.c_void_p(ev_end.cuda_event) if ev_end is not None else None
    _check("rq_set_profile_events", lib().rq_set_profile_events(ctx, a, b))


class KVCache:
    """A context plus its device page pool ([num_pages][Hkv][page_bytes] uint8) and status word."""

    def __init__(self, mode, bits, num_q_heads, num_kv_heads, page_size, num_pages, rot_k, rot_v, max_batch,
                 max_query_tokens=1, max_pages_per_seq=None, codebook=None, sm_scale=0.0, device="cuda"):
        self.device = torch.device(device)
        if self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.mode, self.bits = mode, bits
        self.num_q_heads, self.num_kv_heads = num_q_heads, num_kv_heads
        self.page_size, self.num_pages = page_size, num_pages
        if max_pages_per_seq is None:
            max_pages_per_seq = num_pages
        self.ctx = rq_create(mode, bits, num_q_heads, num_kv_heads, page_size, num_pages, rot_k, rot_v, max_batch,
                             max_query_tokens, max_pages_per_seq, codebook, sm_scale, self.device.index)
        self.page_bytes = rq_page_bytes(self.ctx)
        self.pages = torch.zeros((num_pages, num_kv_heads, self.page_bytes), dtype=torch.uint8, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)

    def codebook(self):
        return rq_get_codebook(self.ctx, self.bits)

    def append(self, k, v, slot_mapping, stream=None):
        rq_quantize_append(self.ctx, k, v, slot_mapping, self.pages, self.status, stream)

    def decode(self, q, block_table, seq_lens, out=None, stream=None):
        if out is None:
            out = torch.empty_like(q)
        return rq_decode_attention(self.ctx, q, self.pages, block_table, seq_lens, out, self.status, stream)

    def decode_step(self, q, k_new, v_new, block_table, seq_lens, out=None, stream=None):
        if out is None:
            out = torch.empty_like(q)
        return rq_decode_step(self.ctx, q, k_new, v_new, self.pages, block_table, seq_lens, out, self.status, stream)

    def extend(self, q, block_table, seq_lens, out=None, stream=None):
        if out is None:
            out = torch.empty_like(q)
        return rq_extend_attention(self.ctx, q, self.pages, block_table, seq_lens, out, self.status, stream)

    def verify(self, q, block_table, seq_lens, out=None, stream=None):
        if out is None:
            out = torch.empty_like(q)
        return rq_verify_attention(self.ctx, q, self.pages, block_table, seq_lens, out, self.status, stream)

    def tree_verify(self, q, tree_mask, block_table, seq_lens, out=None, stream=None):
        if out is None:
            out = torch.empty_like(q)
        return rq_tree_verify_attention(self.ctx, q, tree_mask, self.pages, block_table, seq_lens, out, self.status,
                                        stream)

    def close(self):
        if self.ctx is not None:
            torch.cuda.synchronize(self.device)
            rq_free(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
