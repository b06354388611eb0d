"""The C-ABI library on a host without a GPU: it loads, exports every symbol include/rq.h
declares, rejects bad arguments before touching CUDA, and its default codebook is the
Lloyd-Max codebook the oracle derives independently."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import oracle as O
from rotation_quantized_kv_rq_gb300 import rq

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "rq.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rq_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert set(names) == set(rq.EXPORTS), names
    L = rq.lib()
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_null_safety():
    assert rq.status_string(0) == "ok"
    assert rq.status_string(4) == "above the context's capacity"
    assert rq.status_string(999) == "unknown status"
    L = rq.lib()
    L.rq_free(None)
    assert L.rq_page_bytes(None) == 0
    assert L.rq_get_codebook(None, None, None) == rq.RQ_ERR_INVALID


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_default_codebook_equals_oracle(bits):
    lib_c = rq.rq_lloyd_max_codebook(bits, 128)
    or_c, _ = O.codebook(bits, 128)
    assert np.array_equal(lib_c, or_c)


def _cfg(**over):
    rk = np.zeros((8, 128), np.float32)
    rk[:, 0::2] = 1.0
    base = dict(head_dim=128, num_q_heads=32, num_kv_heads=8, bits=4, mode=0, page_size=16, num_pages=64,
                max_batch=4, max_query_tokens=1, max_pages_per_seq=8)
    base.update(over)
    fp = ctypes.POINTER(ctypes.c_float)
    keep = [rk]
    cfg = rq.rq_config(base["head_dim"], base["num_q_heads"], base["num_kv_heads"], base["bits"], base["mode"],
                       base["page_size"], base["num_pages"], base["max_batch"], base["max_query_tokens"],
                       base["max_pages_per_seq"], rk.ctypes.data_as(fp), rk.ctypes.data_as(fp), fp(),
                       float(over.get("sm_scale", 0.0)), -1)
    return cfg, keep


@pytest.mark.parametrize("over,code", [
    (dict(head_dim=64), rq.RQ_ERR_UNSUPPORTED),
    (dict(bits=1), rq.RQ_ERR_UNSUPPORTED),
    (dict(bits=5), rq.RQ_ERR_UNSUPPORTED),
    (dict(bits=8), rq.RQ_ERR_UNSUPPORTED),
    (dict(page_size=24), rq.RQ_ERR_UNSUPPORTED),
    (dict(page_size=512), rq.RQ_ERR_UNSUPPORTED),
    (dict(num_q_heads=30), rq.RQ_ERR_INVALID),
    (dict(num_kv_heads=0), rq.RQ_ERR_INVALID),
    (dict(mode=3), rq.RQ_ERR_INVALID),
    (dict(mode=-1), rq.RQ_ERR_INVALID),
    (dict(num_pages=0), rq.RQ_ERR_INVALID),
    (dict(max_batch=-1), rq.RQ_ERR_INVALID),
    (dict(sm_scale=-1.0), rq.RQ_ERR_INVALID),
])
def test_create_rejects_bad_configs_without_cuda(over, code):
    cfg, keep = _cfg(**over)
    ctx = ctypes.c_void_p(1)
    rc = rq.lib().rq_create(ctypes.byref(ctx), ctypes.byref(cfg))
    assert rc == code
    assert ctx.value is None


def test_calls_reject_null_context():
    L = rq.lib()
    assert L.rq_quantize_append(None, None, None, None, 1, None, None, None) == rq.RQ_ERR_INVALID
    assert L.rq_decode_attention(None, None, None, None, 1, None, 1, None, None, None) == rq.RQ_ERR_INVALID
    assert L.rq_decode_step(None, None, None, None, None, None, 1, None, 1, None, None, None) == rq.RQ_ERR_INVALID
    assert L.rq_extend_attention(None, None, 2, None, None, 1, None, 1, None, None, None) == rq.RQ_ERR_INVALID
    assert L.rq_verify_attention(None, None, 2, None, None, 1, None, 1, None, None, None) == rq.RQ_ERR_INVALID


def test_binding_checks_rotation_table_size():
    """A dense context reads Hkv x 128 x 128 floats per table; the binding refuses a wrong size
    before the library could read past the caller's array."""
    rk = np.zeros((8, 128), np.float32)
    with pytest.raises(rq.RQError) as e:
        rq.rq_create(rq.RQ_DENSE, 4, 32, 8, 16, 64, rk, rk, max_batch=1)
    assert e.value.code == rq.RQ_ERR_INVALID
    dense = np.zeros((8, 128, 128), np.float32)
    with pytest.raises(rq.RQError) as e:
        rq.rq_create(rq.RQ_PLANAR, 4, 32, 8, 16, 64, dense, dense, max_batch=1)
    assert e.value.code == rq.RQ_ERR_INVALID


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="host-side check only; fake pointers")
@pytest.mark.parametrize("which", ["q", "kv_pages", "out"])
def test_noalloc_rejects_misaligned_pointers_before_cuda(which):
    """The bulk copies and vector loads of the decode kernel need 16-byte aligned q, kv_pages
    and out; a misaligned one is refused on the host, before any CUDA call."""
    cfg, keep = _cfg()
    ptr = {"q": 0x10000, "kv_pages": 0x20000, "out": 0x30000}
    ptr[which] += 8
    rc = rq.lib().rq_decode_attention_noalloc(ctypes.byref(cfg), 0x40000, 0x40000, 0x40000, ptr["q"],
                                               ptr["kv_pages"], 0x50000, 1, 0x60000, 1, ptr["out"], None, None)
    assert rc == rq.RQ_ERR_INVALID
