"""Negative controls of the parity harness, on the CPU: the comparisons that the GPU tests rely
on (tests/parity.py) must FAIL when one mistake is planted in one of the two sides compared --
the discipline of a perturbed build that must differ.  Both sides here are the oracle; the
planted mistake sits in one copy of it, on the CPU."""
import numpy as np
import pytest

from oracle import oracle as O
from rotation_quantized_kv_rq_gb300 import synth
from tests import parity as PT


def _case(mode=synth.ISO, bits=4, lens=(200, 77), hq=32, hkv=8, P=16, seed=41):
    lens = np.asarray(lens, np.int32)
    spec = synth.Spec("neg", mode, bits, len(lens), int(lens.max()), hq, hkv, P, seed=seed)
    rng = np.random.default_rng(seed)
    rk = synth.rotation_params(mode, hkv, rng)
    rv = synth.rotation_params(mode, hkv, rng)
    bt, total = synth.block_table(spec, lens)
    wl = synth.Workload(spec, rk, rv, lens, bt, total)
    kv = [tuple(x.numpy() for x in synth.kv_tokens(spec, b, 0, int(L))) for b, L in enumerate(lens)]
    q = synth.queries(spec).numpy()
    return wl, kv, q


def _fill(oc, wl, kv, margins=False):
    tokens, mg, ti, K, V = [], {}, 0, [], []
    for b, (k, v) in enumerate(kv):
        slots = PT.positions_slots(wl, b, 0, k.shape[0])
        m = oc.append(k, v, slots, with_margins=margins)
        for t in range(k.shape[0]):
            if margins:
                mg[ti + t] = (m[0][t], m[1][t])
            for h in range(wl.spec.num_kv_heads):
                tokens.append((int(slots[t]) // wl.spec.page_size, int(slots[t]) % wl.spec.page_size, h, ti + t))
        ti += k.shape[0]
        K.append(k)
        V.append(v)
    return tokens, mg, (np.concatenate(K), np.concatenate(V))


def test_faithful_copies_agree():
    wl, kv, q = _case()
    a, b = PT.oracle_cache(wl), PT.oracle_cache(wl)
    tokens, mg, inputs = _fill(a, wl, kv, margins=True)
    _fill(b, wl, kv)
    compared, in_band = PT.compare_chunks(b.pages.reshape(wl.num_pages, wl.spec.num_kv_heads, -1), a, tokens, mg,
                                          inputs)
    assert in_band == 0 and compared > 0
    PT.assert_close(b.attention(q, wl.block_table, wl.seq_lens), a.attention(q, wl.block_table, wl.seq_lens))


@pytest.mark.parametrize("plant", ["rotation", "boundary", "norm_byte", "code_byte"])
def test_planted_encoding_mistake_fails_the_code_comparison(plant):
    wl, kv, q = _case()
    a, b = PT.oracle_cache(wl), PT.oracle_cache(wl)
    b.rot_k, b.rot_v = b.rot_k.copy(), b.rot_v.copy()  # the cache views the workload's tables
    tokens, mg, inputs = _fill(a, wl, kv, margins=True)
    if plant == "rotation":
        b.rot_k[2, 4:8] = b.rot_k[2, [5, 4, 7, 6]]       # one quaternion block of head 2
    elif plant == "boundary":
        j = len(b.boundaries) // 2 - 3
        b.boundaries[j] = np.float32(0.5 * (b.boundaries[j] + b.boundaries[j - 1]))
    _fill(b, wl, kv)
    got = b.pages.reshape(wl.num_pages, wl.spec.num_kv_heads, -1).copy()
    page, off, h, _ = tokens[len(tokens) // 3]
    vb = O.vector_bytes(wl.spec.bits)
    if plant == "norm_byte":
        got[page, h, 2 * wl.spec.page_size * vb + 2 * off] ^= 1        # K norm's low bit
    elif plant == "code_byte":
        got[page, h, off * vb + 5] ^= 0x10                              # one K code
    with pytest.raises(AssertionError):
        PT.compare_chunks(got, a, tokens, mg, inputs)


@pytest.mark.parametrize("plant", ["rot_v", "rot_k", "centroid", "sm_scale", "one_token"])
def test_planted_attention_mistake_fails_the_output_comparison(plant):
    wl, kv, q = _case()
    a, b = PT.oracle_cache(wl), PT.oracle_cache(wl)
    b.rot_k, b.rot_v = b.rot_k.copy(), b.rot_v.copy()  # the cache views the workload's tables
    _fill(a, wl, kv)
    b.pages[:] = a.pages
    if plant == "rot_v":
        b.rot_v[5, 0:4] = b.rot_v[5, [1, 0, 3, 2]]
    elif plant == "rot_k":
        b.rot_k[1, 1:4] = -b.rot_k[1, 1:4]               # the inverse rotation of one block
    elif plant == "centroid":
        b.centroids[9] = np.float32(b.centroids[9] * 1.02)
    elif plant == "sm_scale":
        b.sm_scale *= 1.01
    else:
        lens = wl.seq_lens.copy()
        lens[0] -= 1                                      # one token left out of sequence 0
        with pytest.raises(AssertionError):
            PT.assert_close(b.attention(q, wl.block_table, lens), a.attention(q, wl.block_table, wl.seq_lens))
        return
    with pytest.raises(AssertionError):
        PT.assert_close(b.attention(q, wl.block_table, wl.seq_lens), a.attention(q, wl.block_table, wl.seq_lens))
