"""Seeded synthetic inputs for the rotation-quantized KV cache workloads.

This module draws random numbers and lays out index tables.  It holds none of the codec's or
attention's arithmetic: rotations are drawn here as parameters (cos/sin of a uniform angle, or
a normalised Gaussian 4-vector), but never applied here.  Both the CUDA path's tests and bench
and the CPU oracle receive the same arrays from here.

Workloads (geometry from the five synthetic decode/verify configurations of this project):

  cfg0  rq4 planar decode, 1 x 1024 ctx, 32 q / 8 kv heads, page 16, identity block table.
  cfg1  rq3 planar decode, 16 x 8192 ctx, 32/8, page 16, permuted pages, per-token K offset
        ~ N(0, 0.5); the step appends 1 token per sequence, then decodes.
  cfg2  rq4 iso decode, 32 sequences with ctx ~ U[1024, 32768], 64/8, page 16, permuted pages.
  cfg2_32k  cfg2 with every ctx = 32768.
  cfg3  rq3 iso chain verify, 8 x 16384 ctx + 6 drafts, 32/8, page 16, permuted pages; the
        step appends the 6 drafts, then verifies.
  cfg3_prefill  quantize-append of 65536 tokens x 8 kv heads (K and V) of one sequence.
  cfg4  rq3 planar decode, 64 x 65536 ctx, 64/8, page 64, permuted pages.
  tq{2,3,4}_32k  TurboQuant (dense random orthogonal rotation) decode at 2, 3 and 4 bits on
        the cfg2_32k geometry and data.
  tq3_prefill  dense-rotation quantize-append of 65536 tokens x 8 kv heads.
  cfg3_extend  extend (chunked prefill): 8 sequences of 15360 cached tokens take 1024 new tokens
        each, appended then attended causally (rq3 iso, 32/8 heads, page 16).
  tq3_extend  cfg3_extend with the dense rotation.
  tq3_step  cfg1 (a decode step of 16 x 8K, 1 new token per sequence) with the dense rotation.

Distributions: Q, V ~ N(0, 1); K ~ N(0, 1) with 4 distinct channels per kv head (drawn from
the seed, fixed for all tokens) multiplied by 10 after sampling; fp16 storage.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

PLANAR, ISO, DENSE = 0, 1, 2
HEAD_DIM = 128


@dataclasses.dataclass(frozen=True)
class Spec:
    name: str
    mode: int
    bits: int
    batch: int
    ctx: int                 # context per sequence after the step (max for ragged)
    num_q_heads: int
    num_kv_heads: int
    page_size: int
    permuted: bool = True
    ragged_min: int = 0      # > 0: ctx ~ U[ragged_min, ctx]
    k_offset_var: float = 0.0
    query_tokens: int = 1    # T: 1 = decode, > 1 = chain verify
    appended: int = 1        # tokens appended by the step (the last ones of each sequence)
    seed: int = 1000

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


SPECS = {
    "cfg0": Spec("cfg0", PLANAR, 4, 1, 1024, 32, 8, 16, permuted=False, appended=0, seed=1000),
    "cfg1": Spec("cfg1", PLANAR, 3, 16, 8192, 32, 8, 16, k_offset_var=0.5, appended=1, seed=1001),
    "cfg2": Spec("cfg2", ISO, 4, 32, 32768, 64, 8, 16, ragged_min=1024, appended=0, seed=1002),
    "cfg2_32k": Spec("cfg2_32k", ISO, 4, 32, 32768, 64, 8, 16, appended=0, seed=1002),
    "cfg3": Spec("cfg3", ISO, 3, 8, 16384 + 6, 32, 8, 16, query_tokens=6, appended=6, seed=1003),
    "cfg4": Spec("cfg4", PLANAR, 3, 64, 65536, 64, 8, 64, appended=0, seed=1004),
    # TurboQuant: the cfg2_32k geometry and seed (same K, V and Q), dense rotation
    "tq4_32k": Spec("tq4_32k", DENSE, 4, 32, 32768, 64, 8, 16, appended=0, seed=1002),
    "tq3_32k": Spec("tq3_32k", DENSE, 3, 32, 32768, 64, 8, 16, appended=0, seed=1002),
    "tq2_32k": Spec("tq2_32k", DENSE, 2, 32, 32768, 64, 8, 16, appended=0, seed=1002),
    # extend: the cfg3 geometry and seed, 1024 new tokens per sequence
    "cfg3_extend": Spec("cfg3_extend", ISO, 3, 8, 16384, 32, 8, 16, query_tokens=1024, appended=1024, seed=1003),
    # TurboQuant on the same geometries: an extend, and a decode step (cfg1's)
    "tq3_extend": Spec("tq3_extend", DENSE, 3, 8, 16384, 32, 8, 16, query_tokens=1024, appended=1024, seed=1003),
    "tq3_step": Spec("tq3_step", DENSE, 3, 16, 8192, 32, 8, 16, k_offset_var=0.5, appended=1, seed=1001),
}
EXTEND_MIN_T = 64  # query tokens from which a step attends with the extend kernel
PREFILL_TOKENS = 65536     # prefill workloads: one sequence, all 8 kv heads, K and V
PREFILL = {"cfg3_prefill": "cfg3", "tq3_prefill": "tq3_32k"}  # workload -> spec it takes its codec from


def prefill_spec(name: str) -> "Spec":
    """The one-sequence, PREFILL_TOKENS-token append workload `name` (see PREFILL)."""
    return dataclasses.replace(SPECS[PREFILL[name]], name=name, batch=1, ctx=PREFILL_TOKENS, ragged_min=0,
                               query_tokens=1, appended=PREFILL_TOKENS)


def scaled(spec: Spec, **kw) -> Spec:
    """The same workload with some fields replaced (e.g. a smaller batch or context)."""
    return dataclasses.replace(spec, **kw)


# ---------------------------------------------------------------------------------------
# Random streams.  One numpy Generator per purpose, spawned from the workload seed.
# ---------------------------------------------------------------------------------------
_STREAMS = ["rot_k", "rot_v", "outliers", "lens", "pages", "torch"]


def _rng(spec_seed: int, purpose: str) -> np.random.Generator:
    ss = np.random.SeedSequence(spec_seed)
    children = ss.spawn(len(_STREAMS))
    return np.random.default_rng(children[_STREAMS.index(purpose)])


def rotation_params(mode: int, num_kv_heads: int, rng: np.random.Generator, head_dim: int = HEAD_DIM):
    """Random per-head rotation parameters, float32.

    planar: [Hkv][head_dim/2][2] = (cos t, sin t), t ~ U[0, 2 pi) per pair per head.
    iso:    [Hkv][head_dim/4][4] = g / |g|, g ~ N(0, I4) per block per head.
    dense:  [Hkv][head_dim][head_dim], a uniformly (Haar) distributed orthogonal matrix per head:
            the Q factor of a Gaussian matrix, its columns' signs fixed by diag(R) > 0.
    """
    if mode == DENSE:
        out = np.empty((num_kv_heads, head_dim, head_dim), np.float32)
        for h in range(num_kv_heads):
            q, r = np.linalg.qr(rng.standard_normal(size=(head_dim, head_dim)))
            out[h] = q * np.sign(np.diag(r))[None, :]
        return out
    if mode == PLANAR:
        theta = rng.uniform(0.0, 2.0 * math.pi, size=(num_kv_heads, head_dim // 2))
        p = np.stack([np.cos(theta), np.sin(theta)], axis=-1)
    else:
        g = rng.standard_normal(size=(num_kv_heads, head_dim // 4, 4))
        p = g / np.linalg.norm(g, axis=-1, keepdims=True)
    return np.ascontiguousarray(p.reshape(num_kv_heads, head_dim).astype(np.float32))


def outlier_channels(spec: Spec) -> np.ndarray:
    """int64 [Hkv][4]: the K channels scaled by 10, distinct within a head."""
    rng = _rng(spec.seed, "outliers")
    return np.stack([rng.choice(HEAD_DIM, size=4, replace=False) for _ in range(spec.num_kv_heads)])


def seq_lens(spec: Spec) -> np.ndarray:
    if spec.ragged_min > 0:
        rng = _rng(spec.seed, "lens")
        return rng.integers(spec.ragged_min, spec.ctx + 1, size=spec.batch).astype(np.int32)
    return np.full(spec.batch, spec.ctx, np.int32)


def block_table(spec: Spec, lens: np.ndarray, extra_pages: int = 0):
    """(block_table int32 [B][max_pages], num_pages).  Pages of all sequences are a seeded
    permutation of 0..num_pages-1 (identity when the spec is not permuted); unused entries are 0."""
    P = spec.page_size
    npg = [(int(l) + P - 1) // P for l in lens]
    max_pages = max(max(npg), 1)
    total = sum(npg) + extra_pages
    ids = np.arange(total, dtype=np.int64)
    if spec.permuted:
        ids = _rng(spec.seed, "pages").permutation(total)
    bt = np.zeros((spec.batch, max_pages), np.int32)
    o = 0
    for b, n in enumerate(npg):
        bt[b, :n] = ids[o:o + n]
        o += n
    return bt, total


def slots_for(bt: np.ndarray, b: int, positions: np.ndarray, page_size: int) -> np.ndarray:
    """Slot ids (page * P + offset) of token positions of sequence b."""
    positions = np.asarray(positions, np.int64)
    return (bt[b, positions // page_size].astype(np.int64) * page_size + positions % page_size).astype(np.int32)


def _torch_gen(spec: Spec, device, salt: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((spec.seed * 1_000_003 + salt) % (2 ** 63))
    return g


def kv_tokens(spec: Spec, b: int, start: int, count: int, device="cpu"):
    """K and V fp16 [count][Hkv][d] for positions start..start+count-1 of sequence b.

    Drawn in fixed chunks of 1024 positions so that any range regenerates the same values on
    the same device type.  K gets the outlier channels (x10) and, when the workload has one,
    a per-token scalar offset ~ N(0, k_offset_var) added to every channel of every kv head."""
    H = spec.num_kv_heads
    CH = 1024
    outs_k, outs_v = [], []
    first, last = start // CH, (start + count - 1) // CH
    out_ch = torch.as_tensor(outlier_channels(spec), device=device)
    for c in range(first, last + 1):
        g = _torch_gen(spec, device, 7919 * (b + 1) + c)
        k = torch.randn((CH, H, HEAD_DIM), generator=g, device=device, dtype=torch.float32)
        v = torch.randn((CH, H, HEAD_DIM), generator=g, device=device, dtype=torch.float32)
        if spec.k_offset_var > 0:
            off = torch.randn((CH, 1, 1), generator=g, device=device, dtype=torch.float32)
            k = k + off * math.sqrt(spec.k_offset_var)
        scale = torch.ones((H, HEAD_DIM), device=device, dtype=torch.float32)
        scale.scatter_(1, out_ch, 10.0)
        k = k * scale
        lo = max(start, c * CH) - c * CH
        hi = min(start + count, (c + 1) * CH) - c * CH
        outs_k.append(k[lo:hi].to(torch.float16))
        outs_v.append(v[lo:hi].to(torch.float16))
    return torch.cat(outs_k), torch.cat(outs_v)


def queries(spec: Spec, device="cpu", batch=None):
    """Q fp16 [B][T][Hq][d]."""
    B = spec.batch if batch is None else batch
    g = _torch_gen(spec, device, 104729)
    q = torch.randn((B, spec.query_tokens, spec.num_q_heads, HEAD_DIM), generator=g, device=device,
                    dtype=torch.float32)
    return q.to(torch.float16)


@dataclasses.dataclass
class Workload:
    spec: Spec
    rot_k: np.ndarray        # float32 [Hkv][d] (dense: [Hkv][d][d])
    rot_v: np.ndarray
    seq_lens: np.ndarray     # int32 [B] (after the step's appends)
    block_table: np.ndarray  # int32 [B][max_pages]
    num_pages: int


def workload(spec: Spec) -> Workload:
    lens = seq_lens(spec)
    bt, total = block_table(spec, lens)
    rk = rotation_params(spec.mode, spec.num_kv_heads, _rng(spec.seed, "rot_k"))
    rv = rotation_params(spec.mode, spec.num_kv_heads, _rng(spec.seed, "rot_v"))
    return Workload(spec, rk, rv, lens, bt, total)
