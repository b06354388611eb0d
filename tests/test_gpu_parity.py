"""GPU parity on small cases: the CUDA library (through the C ABI) against the fp64 oracle on
the same seeded inputs.  Codes and norms bit-exact (near-boundary exceptions counted and
bounded); attention within 2e-3 + 1e-3|ref| of the oracle's fp64 attention over the
dequantised cache."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from rotation_quantized_kv_rq_gb300 import rq, synth
from tests import parity as PT

pytestmark = pytest.mark.gpu

PLANAR, ISO, DENSE = synth.PLANAR, synth.ISO, synth.DENSE
MODE_NAMES = {PLANAR: 'planar', ISO: 'iso', DENSE: 'dense'}


def make_case(mode, bits, hq, hkv, P, lens, T=1, seed=7, zero_tokens=(), permuted=True):
    lens = np.asarray(lens, np.int32)
    spec = synth.Spec("case", mode, bits, len(lens), int(max(lens.max(), 1)), hq, hkv, P, permuted=permuted,
                      query_tokens=T, seed=seed)
    rng = np.random.default_rng(seed)
    rk = synth.rotation_params(mode, hkv, rng)
    rv = synth.rotation_params(mode, hkv, rng)
    bt, total = synth.block_table(spec, lens, extra_pages=3)
    wl = synth.Workload(spec, rk, rv, lens, bt, total)
    kv = []
    for b, L in enumerate(lens):
        if L == 0:
            kv.append((np.zeros((0, hkv, 128), np.float16), np.zeros((0, hkv, 128), np.float16)))
            continue
        k, v = synth.kv_tokens(spec, b, 0, int(L))
        k, v = k.numpy(), v.numpy()
        for (zb, zt) in zero_tokens:
            if zb == b and zt < L:
                k[zt] = 0
                v[zt] = 0
        kv.append((k, v))
    q = synth.queries(spec).numpy()
    return wl, kv, q


def with_codebook(oc, codebook):
    """The oracle cache with a caller's codebook instead of the default: its centroids, and the
    midpoints between them as the boundaries (the nearest-centroid rule)."""
    if codebook is not None:
        c = np.asarray(codebook, np.float32)
        oc.centroids = c.copy()
        oc.boundaries = (0.5 * (c[:-1].astype(np.float64) + c[1:].astype(np.float64))).astype(np.float32)
    return oc


def run_both(wl, kv, q, codebook=None):
    s = wl.spec
    oc = with_codebook(PT.oracle_cache(wl), codebook)
    margins, tokens, seq_of = {}, [], {}
    flat_k, flat_v, flat_slots = [], [], []
    ti = 0
    for b, (k, v) in enumerate(kv):
        L = k.shape[0]
        if L == 0:
            continue
        slots = PT.positions_slots(wl, b, 0, L)
        mk, mv = oc.append(k, v, slots, with_margins=True)
        for t in range(L):
            margins[ti + t] = (mk[t], mv[t])
            seq_of[ti + t] = b
            for h in range(s.num_kv_heads):
                tokens.append((int(slots[t]) // s.page_size, int(slots[t]) % s.page_size, h, ti + t))
        flat_k.append(k)
        flat_v.append(v)
        flat_slots.append(slots)
        ti += L
    T = s.query_tokens
    ref = oc.attention(q, wl.block_table, wl.seq_lens, T=T)

    cache = rq.KVCache(s.mode, s.bits, s.num_q_heads, s.num_kv_heads, s.page_size, wl.num_pages, wl.rot_k, wl.rot_v,
                       max_batch=s.batch, max_query_tokens=T, max_pages_per_seq=wl.block_table.shape[1],
                       codebook=codebook)
    K = np.concatenate(flat_k)
    V = np.concatenate(flat_v)
    cache.append(PT.to_dev(K), PT.to_dev(V), PT.to_dev(np.concatenate(flat_slots)))
    bt, sl = PT.to_dev(wl.block_table), PT.to_dev(wl.seq_lens)
    qd = PT.to_dev(q)
    if T == 1:
        out = cache.decode(qd[:, 0].contiguous(), bt, sl).unsqueeze(1)
    else:
        out = cache.verify(qd, bt, sl)
    torch.cuda.synchronize()
    gpu_pages = cache.pages.cpu().numpy()
    status = int(cache.status.item())
    out = out.cpu().numpy()

    # the oracle's attention over the GPU's own packed bytes: whatever codes the GPU decided,
    # its attention over them must match this strictly
    og = with_codebook(PT.oracle_cache(wl), codebook)
    og.pages[:] = gpu_pages.reshape(-1)
    ref_own = og.attention(q, wl.block_table, wl.seq_lens, T=T)

    # decode alone, over the oracle's own packed bytes
    cache.pages.copy_(torch.from_numpy(oc.pages.reshape(cache.pages.shape)))
    out2 = (cache.decode(qd[:, 0].contiguous(), bt, sl).unsqueeze(1) if T == 1 else cache.verify(qd, bt, sl))
    out2 = out2.cpu().numpy()
    cache.close()
    return dict(oc=oc, ref=ref, ref_own=ref_own, out=out, out_on_oracle_pages=out2, gpu_pages=gpu_pages,
                tokens=tokens, margins=margins, inputs=(K, V), status=status, seq_of=seq_of)


CASES = [
    # mode, bits, Hq, Hkv, P, lens, T
    (PLANAR, 4, 32, 8, 16, [1024], 1),
    (PLANAR, 3, 32, 8, 16, [37, 16, 1, 160, 0, 15, 17, 33], 1),
    (ISO, 4, 64, 8, 16, [300, 511, 129, 2], 1),
    (ISO, 3, 32, 8, 16, [70, 100, 6, 7], 6),
    (PLANAR, 3, 64, 8, 64, [200, 64, 65, 63], 1),
    (ISO, 4, 16, 2, 32, [95, 1], 1),
    (PLANAR, 4, 8, 8, 16, [40, 41], 1),
    (ISO, 3, 24, 2, 16, [90, 33], 1),
    (PLANAR, 4, 12, 4, 16, [48, 20], 3),
    (ISO, 4, 32, 8, 16, [5000], 1),
    (PLANAR, 3, 32, 8, 128, [700, 129], 2),
    (PLANAR, 3, 32, 8, 48, [100, 47, 200], 1),  # a page size that is not a power of two
    # 2-bit codes and the dense (TurboQuant) rotation
    (PLANAR, 2, 32, 8, 16, [200, 33, 1], 1),
    (ISO, 2, 64, 8, 64, [300, 65], 1),
    (DENSE, 4, 32, 8, 16, [300, 17, 1024], 1),
    (DENSE, 3, 64, 8, 16, [129, 1000, 5], 1),
    (DENSE, 2, 32, 8, 16, [70, 100, 6, 7], 6),
    (DENSE, 4, 24, 2, 32, [95, 3], 2),
    (DENSE, 3, 40, 2, 16, [50, 200], 1),
    (DENSE, 2, 8, 8, 16, [16, 48], 1),
    (DENSE, 4, 32, 8, 48, [130, 49], 1),
    # units of several n-tiles: group 16 decode (2 n-tiles per unit), 6 drafts x group 8 verify
    # (48 rows: two units of 3 n-tiles per kv head) with a sequence long enough to split units
    # across CTAs, and a dense 2-n-tile verify
    (ISO, 4, 128, 8, 16, [300, 1500], 1),
    (PLANAR, 3, 64, 8, 16, [400, 9000, 7], 6),
    (ISO, 2, 48, 8, 64, [3000, 65], 4),
    (DENSE, 3, 64, 8, 16, [700, 33], 2),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{MODE_NAMES[c[0]]}{c[1]}_G{c[2] // c[3]}_P{c[4]}_T{c[6]}_n{len(c[5])}")
def test_append_and_attention_match_oracle(case, capsys):
    mode, bits, hq, hkv, P, lens, T = case
    wl, kv, q = make_case(mode, bits, hq, hkv, P, lens, T, zero_tokens=[(0, 3)])
    r = run_both(wl, kv, q)
    assert r["status"] == 0
    flips = set()
    compared, in_band = PT.compare_chunks(r["gpu_pages"], r["oc"], r["tokens"], r["margins"], r["inputs"], flips)
    with capsys.disabled():
        print(f" [{compared} codes, {in_band} within 1e-6 of a boundary]", end="")
    assert in_band <= max(2, compared // 100000), (in_band, compared)
    PT.assert_close(r["out_on_oracle_pages"], r["ref"], "attention over the oracle's pages")
    PT.assert_close(r["out"], r["ref_own"], "append + attention, against the oracle over the GPU's own pages")
    allowed = {(r["seq_of"][ti], h) for ti, h in flips}
    PT.assert_close_except(r["out"], r["ref"], hq // hkv, allowed, "append + attention")


def test_dense_append_with_boundaries_closer_than_a_table_bin(capsys):
    """A codebook whose two middle boundaries (0 and 2e-4) fall in one bin of the binned code
    table (bins 1/2048 wide): the context keeps no table, the dense append decides every code by
    the select tree, and codes and attention still match the oracle's."""
    cents, _ = O.codebook(3, 128)
    c = cents.astype(np.float64)
    c[3], c[4], c[5] = -1e-4, 1e-4, 3e-4
    assert np.all(np.diff(c) > 0)
    wl, kv, q = make_case(DENSE, 3, 32, 8, 16, [300, 77], 1, seed=11)
    r = run_both(wl, kv, q, codebook=c.astype(np.float32))
    assert r["status"] == 0
    flips = set()
    compared, in_band = PT.compare_chunks(r["gpu_pages"], r["oc"], r["tokens"], r["margins"], r["inputs"], flips)
    with capsys.disabled():
        print(f" [{compared} codes, {in_band} within 1e-6 of a boundary]", end="")
    assert in_band <= max(2, compared // 100000), (in_band, compared)
    PT.assert_close(r["out_on_oracle_pages"], r["ref"], "attention over the oracle's pages")
    PT.assert_close(r["out"], r["ref_own"], "append + attention, against the oracle over the GPU's own pages")


@pytest.mark.parametrize("plant", ["rot_v", "rot_k", "boundary", "centroid"])
def test_negative_control_planted_in_the_oracle(plant):
    """The comparison has teeth: with one mistake planted in the ORACLE (on the CPU) -- a rotation
    parameter of one head nudged, one bin boundary moved, one centroid changed -- the GPU's
    output or codes must fail the same checks that pass against the faithful oracle."""
    wl, kv, q = make_case(ISO, 4, 32, 8, 16, [300, 129], 1, seed=31)
    r = run_both(wl, kv, q)
    assert r["status"] == 0
    bad = PT.oracle_cache(wl)
    bad.rot_k, bad.rot_v = bad.rot_k.copy(), bad.rot_v.copy()  # the cache views the workload's tables
    if plant == "rot_v":
        bad.rot_v[3, 8:12] = bad.rot_v[3, [9, 8, 11, 10]]  # one quaternion block of head 3, permuted
    elif plant == "rot_k":
        bad.rot_k[0, 1:4] = -bad.rot_k[0, 1:4]            # one block of head 0: the inverse rotation
    elif plant == "boundary":
        j = len(bad.boundaries) // 2 + 2
        bad.boundaries[j] = np.float32((bad.boundaries[j] + bad.boundaries[j + 1]) / 2)
    else:
        bad.centroids[5] = np.float32(bad.centroids[5] * 1.02)
    if plant == "boundary":
        # the codes: re-encoding with the planted boundary disagrees with the GPU's bytes
        for b, (k, v) in enumerate(kv):
            bad.append(k, v, PT.positions_slots(wl, b, 0, k.shape[0]))
        with pytest.raises(AssertionError):
            PT.compare_chunks(r["gpu_pages"], bad, r["tokens"])
        return
    bad.pages[:] = r["gpu_pages"].reshape(-1)
    ref_bad = bad.attention(q, wl.block_table, wl.seq_lens)
    with pytest.raises(AssertionError):
        PT.assert_close(r["out"], ref_bad, "planted")


def test_zero_length_sequences_give_zeros():
    wl, kv, q = make_case(PLANAR, 4, 32, 8, 16, [0, 50, 0])
    r = run_both(wl, kv, q)
    assert not r["out"][0].any() and not r["out"][2].any()
    PT.assert_close(r["out"], r["ref"])


@pytest.mark.parametrize("mode", [ISO, DENSE], ids=["iso", "dense"])
def test_status_flags_and_clamping(mode):
    """Out-of-range inputs set status bits instead of faulting; other sequences are unaffected."""
    wl, kv, q = make_case(mode, 3, 32, 8, 16, [40, 40])
    s = wl.spec
    cache = rq.KVCache(s.mode, s.bits, s.num_q_heads, s.num_kv_heads, s.page_size, wl.num_pages, wl.rot_k,
                       wl.rot_v, max_batch=2, max_pages_per_seq=wl.block_table.shape[1])
    k, v = kv[0]
    bad_slot = np.array([wl.num_pages * s.page_size + 5], np.int32)
    cache.append(PT.to_dev(k[:1]), PT.to_dev(v[:1]), PT.to_dev(bad_slot))
    torch.cuda.synchronize()
    assert cache.status.item() & rq.RQ_STATUS_BAD_SLOT
    assert not cache.pages.any()                      # nothing written
    cache.status.zero_()
    skip = np.array([-1], np.int32)
    cache.append(PT.to_dev(k[:1]), PT.to_dev(v[:1]), PT.to_dev(skip))
    torch.cuda.synchronize()
    assert cache.status.item() == 0 and not cache.pages.any()
    bt = wl.block_table.copy()
    bt[1, 1] = wl.num_pages + 100                     # bad page id in sequence 1
    out = cache.decode(PT.to_dev(q[:, 0]), PT.to_dev(bt), PT.to_dev(wl.seq_lens))
    torch.cuda.synchronize()
    assert cache.status.item() & rq.RQ_STATUS_BAD_PAGE
    cache.status.zero_()
    lens = wl.seq_lens.copy()
    lens[0] = bt.shape[1] * s.page_size + 1           # longer than its block-table row
    cache.decode(PT.to_dev(q[:, 0]), PT.to_dev(wl.block_table), PT.to_dev(lens), out=out)
    torch.cuda.synchronize()
    assert cache.status.item() & rq.RQ_STATUS_BAD_LEN
    cache.close()


def test_capacity_and_argument_errors():
    wl, kv, q = make_case(PLANAR, 4, 32, 8, 16, [20])
    s = wl.spec
    cache = rq.KVCache(s.mode, s.bits, s.num_q_heads, s.num_kv_heads, s.page_size, wl.num_pages, wl.rot_k,
                       wl.rot_v, max_batch=1, max_pages_per_seq=wl.block_table.shape[1])
    q2 = PT.to_dev(np.concatenate([q, q])[:, 0])
    bt2 = PT.to_dev(np.concatenate([wl.block_table] * 2))
    with pytest.raises(rq.RQError) as e:
        cache.decode(q2, bt2, PT.to_dev(np.array([20, 20], np.int32)))
    assert e.value.code == rq.RQ_ERR_CAPACITY
    with pytest.raises(rq.RQError) as e:
        cache.verify(PT.to_dev(np.repeat(q, 2, axis=1)), PT.to_dev(wl.block_table), PT.to_dev(wl.seq_lens))
    assert e.value.code == rq.RQ_ERR_CAPACITY
    cache.close()


def test_repeated_calls_are_deterministic():
    """Relaunching on the same inputs gives bitwise the same outputs (no races in the merges)."""
    wl, kv, q = make_case(ISO, 4, 64, 8, 16, [3000, 1700, 20])
    s = wl.spec
    cache = rq.KVCache(s.mode, s.bits, s.num_q_heads, s.num_kv_heads, s.page_size, wl.num_pages, wl.rot_k,
                       wl.rot_v, max_batch=3, max_pages_per_seq=wl.block_table.shape[1])
    for b, (k, v) in enumerate(kv):
        cache.append(PT.to_dev(k), PT.to_dev(v), PT.to_dev(PT.positions_slots(wl, b, 0, k.shape[0])))
    qd, bt, sl = PT.to_dev(q[:, 0]), PT.to_dev(wl.block_table), PT.to_dev(wl.seq_lens)
    first = cache.decode(qd, bt, sl).clone()
    for _ in range(20):
        again = cache.decode(qd, bt, sl)
        assert torch.equal(first.view(torch.int16), again.view(torch.int16))
    cache.close()


def _tree_masks(rng, B, T):
    """Ancestor masks of random draft trees (parent = the prefix or an earlier draft)."""
    masks = np.zeros((B, T), np.uint64)
    for b in range(B):
        parent = [-1] + [int(rng.integers(-1, i)) for i in range(1, T)]
        for i in range(T):
            m, j = 0, i
            while j >= 0:
                m |= 1 << j
                j = parent[j]
            masks[b, i] = m
    return masks


@pytest.mark.parametrize("mode,bits,hq,hkv,P,lens,T", [
    (ISO, 3, 32, 8, 16, [300, 6, 90], 6),
    (PLANAR, 4, 64, 8, 16, [513, 40], 8),
    (ISO, 4, 24, 2, 64, [200, 3], 3),
])
def test_tree_verify_matches_oracle(mode, bits, hq, hkv, P, lens, T):
    wl, kv, q = make_case(mode, bits, hq, hkv, P, lens, T, seed=23)
    s = wl.spec
    oc = PT.oracle_cache(wl)
    cache = rq.KVCache(s.mode, s.bits, s.num_q_heads, s.num_kv_heads, s.page_size, wl.num_pages, wl.rot_k, wl.rot_v,
                       max_batch=s.batch, max_query_tokens=T, max_pages_per_seq=wl.block_table.shape[1])
    for b, (k, v) in enumerate(kv):
        slots = PT.positions_slots(wl, b, 0, k.shape[0])
        oc.append(k, v, slots)
        cache.append(PT.to_dev(k), PT.to_dev(v), PT.to_dev(slots))
    rng = np.random.default_rng(5)
    masks = _tree_masks(rng, s.batch, T)
    qd, bt, sl = PT.to_dev(q), PT.to_dev(wl.block_table), PT.to_dev(wl.seq_lens)
    dmask = torch.from_numpy(masks.view(np.int64)).cuda()
    got = cache.tree_verify(qd, dmask, bt, sl).cpu().numpy()
    ref = oc.tree_attention(q, masks, wl.block_table, wl.seq_lens)
    PT.assert_close(got, ref, "tree verify")
    chain = torch.tensor([[(1 << (j + 1)) - 1 for j in range(T)]] * s.batch, dtype=torch.int64).cuda()
    a = cache.tree_verify(qd, chain, bt, sl)
    b2 = cache.verify(qd, bt, sl)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b2.view(torch.int16))
    assert int(cache.status.item()) == 0
    cache.close()


STEP_CASES = [
    # mode, bits, Hq, Hkv, P, lens (each sequence's last token arrives with the step)
    (PLANAR, 3, 32, 8, 16, [300, 17, 1, 64]),
    (ISO, 4, 64, 8, 64, [200, 129, 64]),
    (PLANAR, 4, 96, 8, 16, [100, 33]),     # group 12: two n-tiles per kv head write the token
    (ISO, 2, 32, 8, 16, [50, 16, 2049]),
    # 344 rounds over the CTAs: ranges cross unit boundaries, so tokens land in a CTA's second
    # fragment and in units split across CTAs
    (PLANAR, 3, 32, 8, 16, [5000, 3000, 777, 12345]),
    # dense rotation: the tokens are coded by the launch that rotates the queries
    (DENSE, 3, 32, 8, 16, [300, 17, 1, 64]),
    (DENSE, 4, 64, 8, 64, [200, 2049, 129]),
    (DENSE, 2, 96, 8, 16, [100, 33]),
]


@pytest.mark.parametrize("case", STEP_CASES, ids=lambda c: f"{MODE_NAMES[c[0]]}{c[1]}_G{c[2] // c[3]}_P{c[4]}")
def test_decode_step_appends_then_attends(case, capsys):
    """rq_decode_step (append folded into the split-K kernel) writes the same bytes as
    rq_quantize_append and returns the same output as append + rq_decode_attention; both match
    the oracle."""
    mode, bits, hq, hkv, P, lens = case
    wl, kv, q = make_case(mode, bits, hq, hkv, P, lens, seed=17)
    s = wl.spec
    oc = PT.oracle_cache(wl)
    margins, tokens, seq_of, flat = {}, [], {}, ([], [])
    ti = 0
    for b, (k, v) in enumerate(kv):
        L = k.shape[0]
        slots = PT.positions_slots(wl, b, 0, L)
        mk, mv = oc.append(k, v, slots, with_margins=True)
        for t in range(L):
            margins[ti + t] = (mk[t], mv[t])
            seq_of[ti + t] = b
            for h in range(hkv):
                tokens.append((int(slots[t]) // P, int(slots[t]) % P, h, ti + t))
        flat[0].append(k)
        flat[1].append(v)
        ti += L
    ref = oc.attention(q, wl.block_table, wl.seq_lens)
    bt, sl, qd = PT.to_dev(wl.block_table), PT.to_dev(wl.seq_lens), PT.to_dev(q[:, 0])
    k_new = PT.to_dev(np.stack([k[-1] for k, _ in kv]))
    v_new = PT.to_dev(np.stack([v[-1] for _, v in kv]))

    outs, pages = [], []
    for fused in (True, False):
        cache = rq.KVCache(mode, bits, hq, hkv, P, wl.num_pages, wl.rot_k, wl.rot_v, max_batch=s.batch,
                           max_pages_per_seq=wl.block_table.shape[1])
        for b, (k, v) in enumerate(kv):  # everything but the step's token
            if k.shape[0] > 1:
                cache.append(PT.to_dev(k[:-1]), PT.to_dev(v[:-1]),
                             PT.to_dev(PT.positions_slots(wl, b, 0, k.shape[0] - 1)))
        if fused:
            out = cache.decode_step(qd, k_new, v_new, bt, sl)
        else:
            last = np.array([PT.positions_slots(wl, b, k.shape[0] - 1, 1)[0] for b, (k, _) in enumerate(kv)], np.int32)
            cache.append(k_new, v_new, PT.to_dev(last))
            out = cache.decode(qd, bt, sl)
        torch.cuda.synchronize()
        assert int(cache.status.item()) == 0
        outs.append(out.cpu().numpy())
        pages.append(cache.pages.cpu().numpy())
        cache.close()
    assert np.array_equal(pages[0], pages[1]), "decode step and append wrote different bytes"
    assert np.array_equal(outs[0], outs[1]), "decode step and append + decode differ"
    flips = set()
    compared, in_band = PT.compare_chunks(pages[0], oc, tokens, margins,
                                          (np.concatenate(flat[0]), np.concatenate(flat[1])), flips)
    with capsys.disabled():
        print(f" [{compared} codes, {in_band} within 1e-6 of a boundary]", end="")
    og = PT.oracle_cache(wl)
    og.pages[:] = pages[0].reshape(-1)
    PT.assert_close(outs[0][:, None], og.attention(q, wl.block_table, wl.seq_lens), "decode step, over its own pages")
    allowed = {(seq_of[t], h) for t, h in flips}
    PT.assert_close_except(outs[0][:, None], ref, hq // hkv, allowed, "decode step")


EXTEND_CASES = [
    # mode, bits, Hq, Hkv, P, lens (after the new tokens), T
    (PLANAR, 4, 32, 8, 16, [300, 1000], 64),
    (ISO, 3, 64, 8, 64, [200, 513], 100),
    (PLANAR, 2, 32, 8, 16, [17, 50, 33], 17),
    (ISO, 4, 24, 2, 32, [129, 70], 70),      # group 12: 64-row blocks cut through a draft's heads
    (PLANAR, 3, 8, 8, 16, [2048], 256),
    (ISO, 2, 32, 8, 16, [0, 130, 64], 64),  # an empty sequence (zeros) and one of only new tokens
    # dense rotation: queries rotated before the launch, R_v^T per row at the end
    (DENSE, 3, 32, 8, 16, [300, 1000], 64),
    (DENSE, 2, 64, 8, 64, [200, 513], 100),
    (DENSE, 4, 24, 2, 32, [0, 129, 70], 70),
]


@pytest.mark.parametrize("case", EXTEND_CASES, ids=lambda c: f"{MODE_NAMES[c[0]]}{c[1]}_G{c[2] // c[3]}_P{c[4]}_T{c[6]}")
def test_extend_attention_matches_oracle(case):
    """rq_extend_attention (causal attention of T new tokens over the packed cache) against the
    oracle's chain attention over the same pages, and against rq_verify_attention."""
    mode, bits, hq, hkv, P, lens, T = case
    wl, kv, q = make_case(mode, bits, hq, hkv, P, lens, T=T, seed=23)
    s = wl.spec
    oc = PT.oracle_cache(wl)
    for b, (k, v) in enumerate(kv):
        oc.append(k, v, PT.positions_slots(wl, b, 0, k.shape[0]))
    ref = oc.attention(q, wl.block_table, wl.seq_lens, T=T)
    cache = rq.KVCache(mode, bits, hq, hkv, P, wl.num_pages, wl.rot_k, wl.rot_v, max_batch=s.batch,
                       max_query_tokens=T, max_pages_per_seq=wl.block_table.shape[1])
    cache.pages.copy_(torch.from_numpy(oc.pages.reshape(cache.pages.shape)))  # the oracle's own pages
    bt, sl, qd = PT.to_dev(wl.block_table), PT.to_dev(wl.seq_lens), PT.to_dev(q)
    out = cache.extend(qd, bt, sl)
    ver = cache.verify(qd, bt, sl)
    torch.cuda.synchronize()
    assert int(cache.status.item()) == 0
    out, ver = out.cpu().numpy(), ver.cpu().numpy()
    cache.close()
    PT.assert_close(out, ref, "extend attention")
    PT.assert_close(ver, ref, "verify attention")
