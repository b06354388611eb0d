"""Shared helpers of the GPU parity tests: run the CUDA library and the CPU oracle on the same
seeded inputs and compare.  Test infrastructure: imports both sides, used only by tests/,
the smoke check and bench.py's oracle legs."""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as O
from rotation_quantized_kv_rq_gb300 import synth

ATOL, RTOL = 2e-3, 1e-3          # attention output tolerance (fp16 output vs fp64 oracle)
BOUNDARY_BAND = 1e-6             # codes within this distance of a bin boundary may differ


def oracle_cache(wl: synth.Workload, num_pages=None) -> O.Cache:
    s = wl.spec
    return O.Cache(s.mode, s.bits, s.num_q_heads, s.num_kv_heads, s.page_size,
                   num_pages if num_pages is not None else wl.num_pages, wl.rot_k, wl.rot_v)


def positions_slots(wl: synth.Workload, b: int, start: int, count: int) -> np.ndarray:
    return synth.slots_for(wl.block_table, b, np.arange(start, start + count), wl.spec.page_size)


def compare_chunks(gpu_pages: np.ndarray, ocache: O.Cache, tokens, margins=None, inputs=None, flips=None):
    """Compare the packed codes and norms of the given (page, offset, head, token-index) tuples.

    gpu_pages: uint8 [num_pages][Hkv][page_bytes] copied from the device.  margins: dict
    token-index -> (margin_k [Hkv][d], margin_v [Hkv][d]) from the oracle's append; inputs:
    (K, V) fp16 numpy [n][Hkv][d] indexed by token-index, to locate fp16 rounding midpoints.
    Returns (n_codes_compared, n_mismatch_in_band); `flips`, if a set, receives the
    (token-index, kv head) of every in-band difference.  Raises AssertionError on any mismatch
    outside the band or any norm mismatch that is not at an fp16 rounding midpoint."""
    bits, P = ocache.bits, ocache.P
    vb = O.vector_bytes(bits)
    compared = in_band = 0
    for (page, off, h, ti) in tokens:
        g_ch = gpu_pages[page, h]
        o_ch = ocache.chunk(page, h)
        for kv in (0, 1):
            if kv == 0:
                gb, ob = g_ch[off * vb:(off + 1) * vb], o_ch[off * vb:(off + 1) * vb]
            else:
                gb, ob = O.v_codes_of(bits, g_ch, P, off), O.v_codes_of(bits, o_ch, P, off)
            compared += 128
            if not np.array_equal(gb, ob):
                gc, oc = O.unpack(bits, gb), O.unpack(bits, ob)
                bad = np.nonzero(gc != oc)[0]
                assert margins is not None, f"code mismatch page {page} off {off} head {h} kv {kv} dims {bad}"
                m = margins[ti][kv][h]
                assert np.all(m[bad] < BOUNDARY_BAND), (page, off, h, kv, bad, m[bad], gc[bad], oc[bad])
                in_band += len(bad)
                if flips is not None:
                    flips.add((ti, h))
            no = 2 * P * vb + kv * 2 * P + 2 * off
            gn = int(g_ch[no]) | int(g_ch[no + 1]) << 8
            on = int(o_ch[no]) | int(o_ch[no + 1]) << 8
            if gn != on:
                # allowed only when the exact norm is within 1e-6 (relative) of the fp16 rounding
                # midpoint between the two stored values
                assert inputs is not None, ("norm mismatch", page, off, h, kv, gn, on)
                exact = float(np.linalg.norm(inputs[kv][ti][h].astype(np.float64)))
                a, b = O.half_to_double(gn), O.half_to_double(on)
                mid = 0.5 * (a + b)
                assert abs(exact - mid) <= 1e-6 * exact, ("norm mismatch", page, off, h, kv, gn, on, exact)
                in_band += 1
                if flips is not None:
                    flips.add((ti, h))
    return compared, in_band


def assert_close(gpu: np.ndarray, ref: np.ndarray, what=""):
    gpu = gpu.astype(np.float64)
    err = np.abs(gpu - ref)
    lim = ATOL + RTOL * np.abs(ref)
    bad = err > lim
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside {ATOL} + {RTOL}|ref|; "
                           f"max abs err {err.max():.3g} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max())


def assert_close_except(gpu: np.ndarray, ref: np.ndarray, group: int, allowed, what=""):
    """assert_close over [B][T][Hq][d], except that (sequence, kv head) groups in `allowed` may
    miss: there a near-boundary code was decided the other way, also a correct decision, and one
    such code of a dominant token can move the output by more than the tolerance.  Returns the
    (sequence, kv head) groups that missed."""
    miss = np.abs(gpu.astype(np.float64) - ref) > ATOL + RTOL * np.abs(ref)
    groups = {(int(b), int(hq) // group) for b, _, hq in np.argwhere(miss.any(axis=3))}
    assert groups <= set(allowed), (what, sorted(groups - set(allowed)))
    return sorted(groups)


def cosine_per_head(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    a = a.reshape(-1, a.shape[-1]).astype(np.float64)
    b = b.reshape(-1, b.shape[-1]).astype(np.float64)
    na, nb = np.linalg.norm(a, axis=1), np.linalg.norm(b, axis=1)
    ok = (na > 0) & (nb > 0)
    return (a[ok] * b[ok]).sum(1) / (na[ok] * nb[ok])


def to_dev(x, device="cuda"):
    if isinstance(x, np.ndarray):
        x = torch.from_numpy(np.ascontiguousarray(x))
    return x.to(device).contiguous()
