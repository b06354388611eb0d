"""rq_decode_attention_noalloc, the decode entry point that allocates no device memory.

It serves callers that cannot call cudaMalloc -- a decode loop inside an engine whose memory
pool already holds the device's free memory, or a plugin whose host framework allows no
allocation outside its own allocator.  Its split-K scratch is a fixed 16 MiB array inside the
library, so its results must match the context-based rq_decode_attention on the same inputs,
including on back-to-back calls that reuse the array.

This file is collected last on purpose, so that a run stopping at the first failure has
already run every other test; it also passes when run on its own in a fresh process."""
import numpy as np
import pytest
import torch

from rotation_quantized_kv_rq_gb300 import rq, synth
from tests import parity as PT

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode,bits,hq,hkv,P,lens", [
    (synth.ISO, 4, 64, 8, 16, [3000, 700, 1, 0, 2049]),
    (synth.PLANAR, 3, 32, 8, 64, [5000, 64, 65]),
])
def test_noalloc_matches_context_path_on_two_calls(mode, bits, hq, hkv, P, lens):
    lens = np.asarray(lens, np.int32)
    spec = synth.Spec("noalloc", mode, bits, len(lens), int(lens.max()), hq, hkv, P, seed=11)
    rng = np.random.default_rng(11)
    rot_k = synth.rotation_params(mode, hkv, rng)
    rot_v = synth.rotation_params(mode, hkv, rng)
    bt, num_pages = synth.block_table(spec, lens)
    cache = rq.KVCache(mode, bits, hq, hkv, P, num_pages, rot_k, rot_v, max_batch=len(lens),
                       max_pages_per_seq=bt.shape[1])
    for b, L in enumerate(lens):
        if L == 0:
            continue
        k, v = synth.kv_tokens(spec, b, 0, int(L), device="cuda")
        cache.append(k, v, PT.to_dev(synth.slots_for(bt, b, np.arange(L), P)))
    q = synth.queries(spec, device="cuda")[:, 0].contiguous()
    d_bt, d_lens = PT.to_dev(bt), PT.to_dev(lens)
    ref = cache.decode(q, d_bt, d_lens).clone()

    # Tables live in caller-owned device memory; the codebook is the library's default.
    d_rot_k = PT.to_dev(rot_k)
    d_rot_v = PT.to_dev(rot_v)
    d_cents = PT.to_dev(rq.rq_lloyd_max_codebook(bits, 128))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_np = ref.cpu().numpy().astype(np.float64)
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        rq.rq_decode_attention_noalloc(mode, bits, hq, hkv, P, num_pages, d_rot_k, d_rot_v, d_cents, q, cache.pages,
                                       d_bt, d_lens, out, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        PT.assert_close(out.cpu().numpy(), ref_np, f"no-alloc call {call + 1}")
    cache.close()


def test_noalloc_rejects_batches_beyond_its_scratch():
    """4,096 kv-head rows need more than the 16 MiB scratch holds: a clear capacity error."""
    hq = hkv = 8
    B = 512
    dummy = torch.zeros(1, dtype=torch.float32, device="cuda")
    q = torch.zeros((B, hq, 128), dtype=torch.float16, device="cuda")
    bt = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    lens = torch.ones(B, dtype=torch.int32, device="cuda")
    pages = torch.zeros((1, hkv, 16 * 132), dtype=torch.uint8, device="cuda")
    with pytest.raises(rq.RQError) as e:
        rq.rq_decode_attention_noalloc(synth.PLANAR, 4, hq, hkv, 16, 1, dummy, dummy, dummy, q, pages, bt, lens,
                                       torch.empty_like(q))
    assert e.value.code == rq.RQ_ERR_CAPACITY
