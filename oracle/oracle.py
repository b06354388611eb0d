"""Python wrapper of the fp64 CPU oracle (``rq_oracle.c``).

TEST INFRASTRUCTURE ONLY: ``tests/``, the smoke check in ``__graft_entry__.py`` and the
``cpu_baseline`` leg of ``bench.py`` may import this module.  It never imports the CUDA
library or its Python binding, and the CUDA path never imports it.

Every function marshals numpy arrays into the C oracle; the arithmetic lives in
``rq_oracle.c`` (see its header for what each step follows on the "SGLang 1-Bit Turbo"
README, section "RotorQuant KV Cache Compression").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

PLANAR, ISO, DENSE = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile rq_oracle.c into a shared library with plain gcc (no target-specific flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(arr, ctype):
    return arr.ctypes.data_as(ctypes.POINTER(ctype))


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            c_int, c_dbl, c_sz = ctypes.c_int, ctypes.c_double, ctypes.c_size_t
            P = ctypes.POINTER
            L.rqo_half_to_double.argtypes = [ctypes.c_uint16]
            L.rqo_half_to_double.restype = c_dbl
            L.rqo_double_to_half.argtypes = [c_dbl]
            L.rqo_double_to_half.restype = ctypes.c_uint16
            L.rqo_lloyd_max_normal.argtypes = [c_int, P(c_dbl), P(c_dbl), P(c_dbl)]
            L.rqo_lloyd_max_normal.restype = c_int
            L.rqo_codebook.argtypes = [c_int, c_int, P(ctypes.c_float), P(ctypes.c_float)]
            L.rqo_codebook.restype = None
            L.rqo_rotate.argtypes = [c_int, P(ctypes.c_float), c_int, P(c_dbl), P(c_dbl), c_int]
            L.rqo_rotate.restype = ctypes.c_long
            L.rqo_rotation_matrix.argtypes = [c_int, P(ctypes.c_float), c_int, P(c_dbl)]
            L.rqo_rotation_matrix.restype = None
            L.rqo_matvec.argtypes = [P(c_dbl), c_int, P(c_dbl), P(c_dbl), c_int]
            L.rqo_matvec.restype = ctypes.c_long
            L.rqo_encode.argtypes = [c_int, c_int, c_int, P(ctypes.c_float), P(ctypes.c_float),
                                     P(ctypes.c_uint16), P(ctypes.c_uint8), P(ctypes.c_uint16), P(c_dbl)]
            L.rqo_encode.restype = None
            L.rqo_vector_bytes.argtypes = [c_int, c_int]
            L.rqo_vector_bytes.restype = c_sz
            L.rqo_pack.argtypes = [c_int, c_int, P(ctypes.c_uint8), P(ctypes.c_uint8)]
            L.rqo_pack.restype = None
            L.rqo_unpack.argtypes = [c_int, c_int, P(ctypes.c_uint8), P(ctypes.c_uint8)]
            L.rqo_unpack.restype = None
            L.rqo_dequant.argtypes = [c_int, c_int, c_int, P(ctypes.c_float), P(ctypes.c_float),
                                      P(ctypes.c_uint8), ctypes.c_uint16, P(c_dbl)]
            L.rqo_dequant.restype = None
            L.rqo_v_unit_offset.argtypes = [c_int, c_int, c_int, c_int]
            L.rqo_v_unit_offset.restype = c_sz
            L.rqo_v_unit_bytes.argtypes = [c_int, c_int]
            L.rqo_v_unit_bytes.restype = c_int
            L.rqo_page_bytes.argtypes = [c_int, c_int, c_int]
            L.rqo_page_bytes.restype = c_sz
            L.rqo_append.argtypes = [c_int, c_int, c_int, c_int, c_int, P(ctypes.c_float), P(ctypes.c_float),
                                     P(ctypes.c_float), P(ctypes.c_uint16), P(ctypes.c_uint16),
                                     P(ctypes.c_int32), c_int, P(ctypes.c_uint8), P(c_dbl), P(c_dbl)]
            L.rqo_append.restype = None
            L.rqo_attention.argtypes = [c_int, c_int, c_int, c_int, c_int, c_int, P(ctypes.c_float),
                                        P(ctypes.c_float), P(ctypes.c_float), c_dbl, P(ctypes.c_uint16), c_int,
                                        P(ctypes.c_uint8), P(ctypes.c_int32), c_int, P(ctypes.c_int32), c_int,
                                        P(c_dbl)]
            L.rqo_attention.restype = c_int
            L.rqo_tree_attention.argtypes = [c_int, c_int, c_int, c_int, c_int, c_int, P(ctypes.c_float),
                                             P(ctypes.c_float), P(ctypes.c_float), c_dbl, P(ctypes.c_uint16), c_int,
                                             P(ctypes.c_uint64), P(ctypes.c_uint8), P(ctypes.c_int32), c_int,
                                             P(ctypes.c_int32), c_int, P(c_dbl)]
            L.rqo_tree_attention.restype = c_int
            L.rqo_attention_dense.argtypes = [c_int, c_int, c_int, c_dbl, P(ctypes.c_uint16), c_int,
                                              P(ctypes.c_uint16), P(ctypes.c_uint16), c_int, P(ctypes.c_int32),
                                              c_int, P(c_dbl)]
            L.rqo_attention_dense.restype = c_int
            _lib = L
    return _lib


def _f16bits(x) -> np.ndarray:
    """fp16 array (numpy float16 or uint16 bit patterns) -> contiguous uint16 bit patterns."""
    a = np.asarray(x)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return np.ascontiguousarray(a)


# ---------------------------------------------------------------------------------------
# fp16
# ---------------------------------------------------------------------------------------
def half_to_double(h: int) -> float:
    return lib().rqo_half_to_double(int(h))


def double_to_half(x: float) -> int:
    return lib().rqo_double_to_half(float(x))


# ---------------------------------------------------------------------------------------
# Lloyd-Max and codebook
# ---------------------------------------------------------------------------------------
def lloyd_max_normal(levels: int):
    """Levels (ascending), thresholds and MSE of the Lloyd-Max quantizer for N(0, 1)."""
    c = np.zeros(levels, np.float64)
    t = np.zeros(max(levels - 1, 1), np.float64)
    mse = ctypes.c_double(0.0)
    it = lib().rqo_lloyd_max_normal(levels, _p(c, ctypes.c_double), _p(t, ctypes.c_double), ctypes.byref(mse))
    if it < 0:
        raise ValueError("levels out of range")
    return c, t[: levels - 1], mse.value, it


def codebook(bits: int, head_dim: int = 128):
    """(centroids fp32 [2^bits], boundaries fp32 [2^bits - 1]) for coordinates ~ N(0, 1/head_dim)."""
    L = 1 << bits
    c = np.zeros(L, np.float32)
    b = np.zeros(L - 1, np.float32)
    lib().rqo_codebook(bits, head_dim, _p(c, ctypes.c_float), _p(b, ctypes.c_float))
    return c, b


# ---------------------------------------------------------------------------------------
# Rotations
# ---------------------------------------------------------------------------------------
def rotate(mode: int, params, x, inverse: bool = False):
    """Apply one head's structured rotation to a vector; returns (y, fma_count)."""
    params = np.ascontiguousarray(params, np.float32).reshape(-1)
    x = np.ascontiguousarray(x, np.float64)
    d = x.shape[0]
    y = np.zeros(d, np.float64)
    n = lib().rqo_rotate(mode, _p(params, ctypes.c_float), d, _p(x, ctypes.c_double),
                         _p(y, ctypes.c_double), int(inverse))
    return y, n


def rotation_matrix(mode: int, params, d: int):
    params = np.ascontiguousarray(params, np.float32).reshape(-1)
    R = np.zeros((d, d), np.float64)
    lib().rqo_rotation_matrix(mode, _p(params, ctypes.c_float), d, _p(R, ctypes.c_double))
    return R


def matvec(R, x, transpose: bool = False):
    R = np.ascontiguousarray(R, np.float64)
    x = np.ascontiguousarray(x, np.float64)
    y = np.zeros(R.shape[0], np.float64)
    n = lib().rqo_matvec(_p(R, ctypes.c_double), R.shape[0], _p(x, ctypes.c_double), _p(y, ctypes.c_double),
                         int(transpose))
    return y, n


# ---------------------------------------------------------------------------------------
# Codec
# ---------------------------------------------------------------------------------------
def encode(mode: int, bits: int, rot_head, boundaries, x16):
    """Encode one vector: (codes uint8 [d], n16 uint16, margins float64 [d])."""
    x16 = _f16bits(x16)
    d = x16.shape[0]
    rot_head = np.ascontiguousarray(rot_head, np.float32).reshape(-1)
    boundaries = np.ascontiguousarray(boundaries, np.float32)
    codes = np.zeros(d, np.uint8)
    n16 = ctypes.c_uint16(0)
    margin = np.zeros(d, np.float64)
    lib().rqo_encode(mode, bits, d, _p(rot_head, ctypes.c_float), _p(boundaries, ctypes.c_float),
                     _p(x16, ctypes.c_uint16), _p(codes, ctypes.c_uint8), ctypes.byref(n16),
                     _p(margin, ctypes.c_double))
    return codes, n16.value, margin


def vector_bytes(bits: int, d: int = 128) -> int:
    return int(lib().rqo_vector_bytes(bits, d))


def pack(bits: int, codes):
    codes = np.ascontiguousarray(codes, np.uint8)
    out = np.zeros(vector_bytes(bits, codes.shape[0]), np.uint8)
    lib().rqo_pack(bits, codes.shape[0], _p(codes, ctypes.c_uint8), _p(out, ctypes.c_uint8))
    return out


def unpack(bits: int, packed, d: int = 128):
    packed = np.ascontiguousarray(packed, np.uint8)
    codes = np.zeros(d, np.uint8)
    lib().rqo_unpack(bits, d, _p(packed, ctypes.c_uint8), _p(codes, ctypes.c_uint8))
    return codes


def dequant(mode: int, bits: int, rot_head, centroids, codes, n16: int):
    codes = np.ascontiguousarray(codes, np.uint8)
    d = codes.shape[0]
    rot_head = np.ascontiguousarray(rot_head, np.float32).reshape(-1)
    centroids = np.ascontiguousarray(centroids, np.float32)
    out = np.zeros(d, np.float64)
    lib().rqo_dequant(mode, bits, d, _p(rot_head, ctypes.c_float), _p(centroids, ctypes.c_float),
                      _p(codes, ctypes.c_uint8), int(n16), _p(out, ctypes.c_double))
    return out


# ---------------------------------------------------------------------------------------
# Paged cache and attention
# ---------------------------------------------------------------------------------------
def v_unit_offset(bits: int, off: int, unit: int, d: int = 128) -> int:
    """Byte offset of 8-byte unit `unit` of V token `off` inside a chunk's V-codes section."""
    return int(lib().rqo_v_unit_offset(bits, d, off, unit))


def v_unit_bytes(bits: int, d: int = 128) -> int:
    return int(lib().rqo_v_unit_bytes(bits, d))


def v_codes_of(bits: int, chunk: np.ndarray, page_size: int, off: int, d: int = 128) -> np.ndarray:
    """The packed codes of V token `off` gathered from a chunk."""
    vb = vector_bytes(bits, d)
    ub = v_unit_bytes(bits, d)
    base = page_size * vb
    return np.concatenate([chunk[base + v_unit_offset(bits, off, u, d):base + v_unit_offset(bits, off, u, d) + ub]
                           for u in range(vb // ub)])


def page_bytes(bits: int, page_size: int, d: int = 128) -> int:
    return int(lib().rqo_page_bytes(bits, page_size, d))


class Cache:
    """The oracle's own paged cache: geometry, rotation tables, codebook and the byte pool."""

    def __init__(self, mode, bits, num_q_heads, num_kv_heads, page_size, num_pages, rot_k, rot_v,
                 head_dim=128, sm_scale=None):
        self.mode, self.bits = int(mode), int(bits)
        self.hq, self.hkv, self.P, self.d = int(num_q_heads), int(num_kv_heads), int(page_size), int(head_dim)
        self.num_pages = int(num_pages)
        per_head = self.d * self.d if self.mode == DENSE else self.d
        self.rot_k = np.ascontiguousarray(rot_k, np.float32).reshape(self.hkv, per_head)
        self.rot_v = np.ascontiguousarray(rot_v, np.float32).reshape(self.hkv, per_head)
        self.centroids, self.boundaries = codebook(self.bits, self.d)
        self.sm_scale = float(sm_scale) if sm_scale else 1.0 / np.sqrt(self.d)
        self.page_bytes = page_bytes(self.bits, self.P, self.d)
        self.pages = np.zeros(self.num_pages * self.hkv * self.page_bytes, np.uint8)

    def append(self, k16, v16, slots, with_margins=False):
        """k16, v16: fp16 [n][Hkv][d]; slots int32 [n].  Returns (margin_k, margin_v) or None."""
        k16, v16 = _f16bits(k16), _f16bits(v16)
        slots = np.ascontiguousarray(slots, np.int32)
        n = slots.shape[0]
        assert k16.size == n * self.hkv * self.d and v16.size == k16.size
        mk = mv = None
        if with_margins:
            mk = np.zeros((n, self.hkv, self.d), np.float64)
            mv = np.zeros((n, self.hkv, self.d), np.float64)
        P = ctypes.POINTER(ctypes.c_double)
        lib().rqo_append(self.mode, self.bits, self.d, self.hkv, self.P, _p(self.rot_k, ctypes.c_float),
                         _p(self.rot_v, ctypes.c_float), _p(self.boundaries, ctypes.c_float),
                         _p(k16, ctypes.c_uint16), _p(v16, ctypes.c_uint16), _p(slots, ctypes.c_int32), n,
                         _p(self.pages, ctypes.c_uint8),
                         _p(mk, ctypes.c_double) if mk is not None else P(),
                         _p(mv, ctypes.c_double) if mv is not None else P())
        return (mk, mv) if with_margins else None

    def attention(self, q16, block_table, seq_lens, T=1):
        """q16: fp16 [B][T][Hq][d] (or [B][Hq][d] for T=1) -> float64 [B][T][Hq][d]."""
        q16 = _f16bits(q16)
        bt = np.ascontiguousarray(block_table, np.int32)
        sl = np.ascontiguousarray(seq_lens, np.int32)
        B, max_pages = bt.shape
        out = np.zeros((B, T, self.hq, self.d), np.float64)
        rc = lib().rqo_attention(self.mode, self.bits, self.d, self.hq, self.hkv, self.P,
                                 _p(self.rot_k, ctypes.c_float), _p(self.rot_v, ctypes.c_float),
                                 _p(self.centroids, ctypes.c_float), self.sm_scale, _p(q16, ctypes.c_uint16), T,
                                 _p(self.pages, ctypes.c_uint8), _p(bt, ctypes.c_int32), max_pages,
                                 _p(sl, ctypes.c_int32), B, _p(out, ctypes.c_double))
        if rc != 0:
            raise MemoryError("oracle attention: allocation failed")
        return out

    def tree_attention(self, q16, tree_mask, block_table, seq_lens):
        """Tree verify: q16 fp16 [B][T][Hq][d]; tree_mask uint64 [B][T] (bit i of row j: query j
        sees draft i, the draft being position len - T + i) -> float64 [B][T][Hq][d]."""
        q16 = _f16bits(q16)
        mask = np.ascontiguousarray(tree_mask, np.uint64)
        bt = np.ascontiguousarray(block_table, np.int32)
        sl = np.ascontiguousarray(seq_lens, np.int32)
        B, max_pages = bt.shape
        T = mask.shape[1]
        out = np.zeros((B, T, self.hq, self.d), np.float64)
        rc = lib().rqo_tree_attention(self.mode, self.bits, self.d, self.hq, self.hkv, self.P,
                                      _p(self.rot_k, ctypes.c_float), _p(self.rot_v, ctypes.c_float),
                                      _p(self.centroids, ctypes.c_float), self.sm_scale, _p(q16, ctypes.c_uint16), T,
                                      _p(mask, ctypes.c_uint64), _p(self.pages, ctypes.c_uint8),
                                      _p(bt, ctypes.c_int32), max_pages, _p(sl, ctypes.c_int32), B,
                                      _p(out, ctypes.c_double))
        if rc != 0:
            raise ValueError("oracle tree attention failed (T must be 1..64)")
        return out

    def chunk(self, page: int, head: int) -> np.ndarray:
        o = (page * self.hkv + head) * self.page_bytes
        return self.pages[o:o + self.page_bytes]


def attention_dense(q16, k16, v16, seq_lens, num_q_heads, num_kv_heads, T=1, sm_scale=None):
    """Attention over unquantised fp16 K/V [B][L][Hkv][d] (fidelity reference)."""
    q16, k16, v16 = _f16bits(q16), _f16bits(k16), _f16bits(v16)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    B, L, hkv, d = k16.shape
    scale = float(sm_scale) if sm_scale else 1.0 / np.sqrt(d)
    out = np.zeros((B, T, num_q_heads, d), np.float64)
    rc = lib().rqo_attention_dense(d, num_q_heads, num_kv_heads, scale, _p(q16, ctypes.c_uint16), T,
                                   _p(k16, ctypes.c_uint16), _p(v16, ctypes.c_uint16), L, _p(sl, ctypes.c_int32),
                                   B, _p(out, ctypes.c_double))
    if rc != 0:
        raise MemoryError("oracle dense attention: allocation failed")
    return out
