"""Parity at the workloads' full sizes, in the launch configuration bench.py times.

For each workload the whole packed cache is built on the GPU, one bench step runs (append of
the step's tokens + attention), and sampled sequences are re-encoded by the CPU oracle from
the same inputs.  Per sampled sequence:
  * codes: the packed bytes match the oracle's, except codes within 1e-6 of a bin boundary
    (counted and bounded);
  * attention over the same cache: the kernels, run on the oracle's own packed pages of the
    sequence, agree with the oracle's fp64 attention within 2e-3 + 1e-3|ref|;
  * end to end, strictly: the bench step's output agrees, within the same tolerance and with no
    exception, with the oracle's attention over the GPU's own packed pages of the sequence;
  * against the oracle's own encoding the output may miss only in kv-head groups whose codes
    hold a near-boundary difference -- there both codes are correct decisions, and one flipped
    code of a dominant token moves the output by more than the tolerance -- which is reported.
Fidelity against attention over the unquantised fp16 cache is reported as cosine similarity.
The extend workload (1,024 query rows per sequence) is checked on sampled rows: row j of an
extend is a decode over the first seq_len - T + j + 1 tokens."""
import numpy as np
import pytest
import torch

import bench
from oracle import oracle as O
from rotation_quantized_kv_rq_gb300 import rq, synth
from tests import parity as PT

pytestmark = pytest.mark.gpu


def _sequence_inputs(spec, b, L, device):
    ks, vs = [], []
    for st in range(0, L, 16384):
        k, v = synth.kv_tokens(spec, b, st, min(16384, L - st), device=device)
        ks.append(k.cpu())
        vs.append(v.cpu())
    return torch.cat(ks).numpy(), torch.cat(vs).numpy()


def _check_sequence(bn, b, out_gpu):
    spec, wl = bn.spec, bn.wl
    L = int(wl.seq_lens[b])
    P = spec.page_size
    npg = (L + P - 1) // P
    k, v = _sequence_inputs(spec, b, L, bn.device)
    oc = O.Cache(spec.mode, spec.bits, spec.num_q_heads, spec.num_kv_heads, P, npg, wl.rot_k, wl.rot_v)
    oc.append(k, v, np.arange(L, dtype=np.int32))
    # packed bytes of the sequence's pages, in order, against the oracle's compact pool
    pages = torch.from_numpy(wl.block_table[b, :npg].astype(np.int64)).to(bn.device)
    gpu = bn.cache.pages.index_select(0, pages).cpu().numpy()        # [npg][Hkv][page_bytes]
    ora = oc.pages.reshape(npg, spec.num_kv_heads, -1)
    # only the bytes of valid tokens are defined: mask the tail of the last page
    vb = 16 * spec.bits
    diff = np.argwhere(gpu != ora)
    in_band = 0
    flipped_heads = set()   # kv heads of this sequence with a near-boundary code or norm difference
    for (pg, h, byte) in diff:
        if byte < P * vb:
            kv, off, norm = 0, int(byte) // vb, False
        elif byte < 2 * P * vb:
            o = int(byte) - P * vb   # inside the V-codes section: find the token owning it
            kv, norm = 1, False
            ub = O.v_unit_bytes(spec.bits)
            off = next(t for t in range(P) for u in range(vb // ub)
                       if O.v_unit_offset(spec.bits, t, u) <= o < O.v_unit_offset(spec.bits, t, u) + ub)
        else:
            kv, rem = divmod(int(byte) - 2 * P * vb, 2 * P)
            off = rem // 2
            norm = True
        t = pg * P + off
        if t >= L:
            continue
        x = (k if kv == 0 else v)[t, h]
        if norm:
            exact = float(np.linalg.norm(x.astype(np.float64)))
            gn = int(gpu[pg, h, 2 * P * vb + kv * 2 * P + 2 * off]) | int(gpu[pg, h, 2 * P * vb + kv * 2 * P + 2 * off + 1]) << 8
            on = int(ora[pg, h, 2 * P * vb + kv * 2 * P + 2 * off]) | int(ora[pg, h, 2 * P * vb + kv * 2 * P + 2 * off + 1]) << 8
            mid = 0.5 * (O.half_to_double(gn) + O.half_to_double(on))
            assert abs(exact - mid) <= 1e-6 * exact, ("norm", b, t, h, kv)
            in_band += 1
            flipped_heads.add(int(h))
            continue
        rot = (wl.rot_k if kv == 0 else wl.rot_v)[h]
        codes, _, margin = O.encode(spec.mode, spec.bits, rot, oc.boundaries, x)
        packed = gpu[pg, h, off * vb:(off + 1) * vb] if kv == 0 else O.v_codes_of(spec.bits, gpu[pg, h], P, off)
        gc = O.unpack(spec.bits, packed)
        bad = np.nonzero(gc != codes)[0]
        assert np.all(margin[bad] < PT.BOUNDARY_BAND), ("code", b, t, h, kv, bad, margin[bad])
        in_band += len(bad)
        if len(bad):
            flipped_heads.add(int(h))
    total_codes = L * spec.num_kv_heads * 2 * 128
    assert in_band <= max(4, total_codes // 200000), (in_band, total_codes)

    q = bn.q.cpu().numpy()
    T = spec.query_tokens
    qb = q[b:b + 1] if T > 1 else q[b:b + 1, None]
    bt1 = np.arange(npg, dtype=np.int32)[None]
    len1 = np.array([L], np.int32)
    if bn.extend:
        # Extend: query row j sees positions 0 .. L - T + j -- a decode over the first L - T + j + 1
        # tokens -- so the oracle is evaluated on sampled rows only, each as that decode.
        rows = sorted({0, T // 2, T - 1})
        ref = np.concatenate([oc.attention(qb[:, j:j + 1], bt1, np.array([L - T + j + 1], np.int32), T=1)
                              for j in rows], axis=1)
    else:
        rows = list(range(T))
        ref = oc.attention(qb, bt1, len1, T=T)
    # the kernels over the oracle's own pages of this sequence: the same dequantised cache
    one = rq.KVCache(spec.mode, spec.bits, spec.num_q_heads, spec.num_kv_heads, P, npg, wl.rot_k, wl.rot_v,
                     max_batch=1, max_query_tokens=T, max_pages_per_seq=npg, device=bn.device)
    one.pages.copy_(torch.from_numpy(oc.pages.reshape(one.pages.shape)))
    qd, btd, lend = PT.to_dev(qb, bn.device), PT.to_dev(bt1, bn.device), PT.to_dev(len1, bn.device)
    if T == 1:
        same = one.decode(qd[:, 0].contiguous(), btd, lend).unsqueeze(1)
    elif bn.extend:
        same = one.extend(qd, btd, lend)
    else:
        same = one.verify(qd, btd, lend)
    same = same.cpu().numpy()[:, rows]
    assert int(one.status.item()) == 0
    one.close()
    err_same = PT.assert_close(same, ref, f"{bn.name} seq {b}, kernels over the oracle's pages")
    got = (out_gpu[b:b + 1] if T > 1 else out_gpu[b:b + 1, None])[:, rows]
    # end to end, strictly: the bench step's output against the oracle's attention over the
    # GPU's own packed pages of this sequence (whatever codes the GPU decided, the attention
    # over them must agree), with no group excused
    og = O.Cache(spec.mode, spec.bits, spec.num_q_heads, spec.num_kv_heads, P, npg, wl.rot_k, wl.rot_v)
    og.pages[:] = gpu.reshape(-1)
    if bn.extend:
        ref_gpu = np.concatenate([og.attention(qb[:, j:j + 1], bt1, np.array([L - T + j + 1], np.int32), T=1)
                                  for j in rows], axis=1)
    else:
        ref_gpu = og.attention(qb, bt1, len1, T=T)
    err_own = PT.assert_close(got, ref_gpu, f"{bn.name} seq {b}, end to end over the GPU's own pages")
    # and against the oracle's own encoding: only kv-head groups holding a near-boundary code
    # may miss (a report of how far the two correct decisions move the output)
    miss = np.abs(got.astype(np.float64) - ref) > PT.ATOL + PT.RTOL * np.abs(ref)   # [1][rows][Hq][d]
    miss_heads = {int(hq) // spec.group for hq in np.nonzero(miss.any(axis=(0, 1, 3)))[0]}
    assert miss_heads <= flipped_heads, (bn.name, b, sorted(miss_heads), sorted(flipped_heads))
    if bn.extend:
        dense = np.concatenate([O.attention_dense(qb[:, j:j + 1], k[None, :L - T + j + 1], v[None, :L - T + j + 1],
                                                  np.array([L - T + j + 1], np.int32), spec.num_q_heads,
                                                  spec.num_kv_heads, T=1) for j in rows], axis=1)
    else:
        dense = O.attention_dense(qb, k[None], v[None], len1, spec.num_q_heads, spec.num_kv_heads, T=T)
    cos = PT.cosine_per_head(got, dense)
    err_e2e = float(np.abs(got.astype(np.float64) - ref).max())
    return err_same, err_own, err_e2e, sorted(miss_heads), in_band, total_codes, float(cos.min()), float(cos.mean())


@pytest.mark.parametrize("name", ["cfg0", "cfg1", "cfg2", "cfg2_32k", "cfg3", "cfg4", "cfg3_prefill", "tq4_32k",
                                  "tq2_32k", "tq3_prefill", "cfg3_extend", "tq3_extend", "tq3_step"])
def test_full_size_workload(name, capsys):
    dev = torch.device("cuda", 0)
    bn = bench.Bench(name, dev)
    bn.step()
    torch.cuda.synchronize(dev)
    assert int(bn.cache.status.item()) == 0
    if bn.prefill_only:
        # the whole 65,536-token prefill: compare every chunk of a few sampled pages
        spec, wl = bn.spec, bn.wl
        k, v = _sequence_inputs(spec, 0, spec.ctx, dev)
        rng = np.random.default_rng(0)
        sample = rng.choice(wl.num_pages, size=64, replace=False)
        oc = O.Cache(spec.mode, spec.bits, spec.num_q_heads, spec.num_kv_heads, spec.page_size, wl.num_pages,
                     wl.rot_k, wl.rot_v)
        pos = np.concatenate([np.arange(p * 16, p * 16 + 16) for p in range(spec.ctx // 16)
                              if wl.block_table[0, p] in set(sample.tolist())])
        mk, mv = oc.append(k[pos], v[pos], synth.slots_for(wl.block_table, 0, pos, 16), with_margins=True)
        gpu = bn.cache.pages.cpu().numpy()
        tokens, margins = [], {}
        for i, t in enumerate(pos):
            s = int(synth.slots_for(wl.block_table, 0, np.array([t]), 16)[0])
            margins[i] = (mk[i], mv[i])
            for h in range(spec.num_kv_heads):
                tokens.append((s // 16, s % 16, h, i))
        compared, in_band = PT.compare_chunks(gpu, oc, tokens, margins, (k[pos], v[pos]))
        assert in_band <= max(4, compared // 200000)
        with capsys.disabled():
            print(f"\n{name}: {compared} codes compared, {in_band} within 1e-6 of a boundary")
        bn.cache.close()
        return
    out = bn.out.cpu().numpy()
    B = bn.spec.batch
    lens = bn.wl.seq_lens
    samples = sorted({0, B - 1, int(np.argmax(lens))})
    for b in samples:
        err_same, err_own, err_e2e, miss, in_band, total, cmin, cmean = _check_sequence(bn, b, out)
        with capsys.disabled():
            print(f"\n{name} seq {b} (ctx {int(lens[b])}): max abs err {err_same:.2e} over the oracle's pages, "
                  f"{err_own:.2e} end to end over the GPU's own pages, {err_e2e:.2e} against the oracle's "
                  f"encoding (kv heads off tolerance: {miss}); near-boundary codes "
                  f"{in_band}/{total}; cosine vs fp16 attention min {cmin:.5f} mean {cmean:.5f}")
    bn.cache.close()
