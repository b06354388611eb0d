"""Benchmark of the rotation-quantized KV cache hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload cfg4] [--impl ours|reference]

A step is one pass of the whole hot path over one batch: the quantize-append of the step's
new tokens, then split-K decode (or chain-verify) attention over the packed cache with its
log-sum-exp combine and inverse rotation done inside the split-K kernel (a dense rotation adds
one launch before it that rotates the queries).  A decode step that appends one token per
sequence (cfg1) runs as one rq_decode_step call: the append is folded into the split-K kernel.
Inputs are synthetic and seeded (rotation_quantized_kv_rq_gb300.synth); the packed cache is
built before timing and stays resident in HBM.

Default workload cfg4: rq3_planar, 64 sequences x 65536 context, 64 q / 8 kv heads, page 64,
permuted block table: the largest configuration (3.36 GB of packed cache, far above the 129 MB
L2; L2 is still flushed, a 512 MB write, before every step outside the per-step CUDA events).
After it, the same process times the 32 x 32768-token rq4 iso decode that the roofline target
is stated at (`target_32k`; `--no-target` skips it).  Any other workload: `--workload NAME`.

Prints one JSON line (rank 0).  `value` = query tokens per second over all ranks (weak
scaling: every rank runs the full workload on its own GPU); `roofline` is the split-K
attention kernel's achieved packed-KV bandwidth against the measured HBM copy peak;
`cpu_baseline` / `--impl reference` time the fp64 CPU oracle on a bounded sample, on all host
cores (a thread per sequence); `cpu_baseline.one_core` is the same on one core.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rotation_quantized_kv_rq_gb300 import rq, synth  # noqa: E402

NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_TFLOPS_SUSTAINED = 1700.0
L2_FLUSH_BYTES = 512 << 20

DESCRIPTIONS = {
    "cfg0": "rq4_planar decode, 1 x 1024 ctx, 32 q / 8 kv heads, head_dim 128, page 16",
    "cfg1": "rq3_planar decode, 16 x 8192 ctx, 32 q / 8 kv heads, head_dim 128, page 16, permuted pages, "
            "append 1 token per sequence + decode",
    "cfg2": "rq4_iso decode, 32 sequences x U[1024, 32768] ctx, 64 q / 8 kv heads, head_dim 128, page 16",
    "cfg2_32k": "rq4_iso decode, 32 x 32768 ctx, 64 q / 8 kv heads, head_dim 128, page 16",
    "cfg3": "rq3_iso chain verify, 8 x 16384 ctx + 6 drafts, 32 q / 8 kv heads, head_dim 128, page 16, "
            "append 6 drafts + verify",
    "cfg3_prefill": "rq3_iso quantize-append of 65536 tokens x 8 kv heads (K and V), page 16",
    "cfg4": "rq3_planar decode, 64 x 65536 ctx, 64 q / 8 kv heads, head_dim 128, page 64",
    "tq4_32k": "tq4 (dense rotation) decode, 32 x 32768 ctx, 64 q / 8 kv heads, head_dim 128, page 16",
    "tq3_32k": "tq3 (dense rotation) decode, 32 x 32768 ctx, 64 q / 8 kv heads, head_dim 128, page 16",
    "tq2_32k": "tq2 (dense rotation) decode, 32 x 32768 ctx, 64 q / 8 kv heads, head_dim 128, page 16",
    "tq3_prefill": "tq3 (dense rotation) quantize-append of 65536 tokens x 8 kv heads (K and V), page 16",
    "cfg3_extend": "rq3_iso extend: 8 x (15360 cached + 1024 new) tokens, 32 q / 8 kv heads, head_dim 128, page 16, "
                   "append the 1024 new tokens + causal extend attention",
    "tq3_extend": "tq3 (dense rotation) extend: 8 x (15360 cached + 1024 new) tokens, 32 q / 8 kv heads, head_dim 128, "
                  "page 16, append the 1024 new tokens + causal extend attention",
    "tq3_step": "tq3 (dense rotation) decode step, 16 x 8192 ctx, 32 q / 8 kv heads, head_dim 128, page 16, "
                "permuted pages, append 1 token per sequence + decode",
}


# ---------------------------------------------------------------------------------------
# distributed plumbing (replicas: no collective on the data path)
# ---------------------------------------------------------------------------------------
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------------
# workload setup
# ---------------------------------------------------------------------------------------
def spec_of(name, batch=None):
    """The workload's Spec; `batch` (profiling a smaller case of the same kernel) keeps its
    first `batch` sequences."""
    s = synth.prefill_spec(name) if name in synth.PREFILL else synth.SPECS[name]
    return synth.scaled(s, batch=batch) if batch else s


class Bench:
    def __init__(self, name, device, batch=None):
        self.name = name
        self.device = device
        self.prefill_only = name in synth.PREFILL
        spec = spec_of(name, batch)
        self.spec = spec
        self.wl = synth.workload(spec)
        s, wl = spec, self.wl
        self.cache = rq.KVCache(s.mode, s.bits, s.num_q_heads, s.num_kv_heads, s.page_size, wl.num_pages, wl.rot_k,
                                wl.rot_v, max_batch=s.batch, max_query_tokens=s.query_tokens,
                                max_pages_per_seq=wl.block_table.shape[1], device=device)
        self.bt = torch.from_numpy(wl.block_table).to(device)
        self.lens = torch.from_numpy(wl.seq_lens).to(device)
        # prefill everything except the step's own tokens
        new_k, new_v, new_slots = [], [], []
        for b in range(s.batch):
            L = int(wl.seq_lens[b])
            keep = L - s.appended
            chunk = 16384
            for st in range(0, keep, chunk):
                cnt = min(chunk, keep - st)
                k, v = synth.kv_tokens(s, b, st, cnt, device=device)
                slots = torch.from_numpy(synth.slots_for(wl.block_table, b, np.arange(st, st + cnt), s.page_size))
                self.cache.append(k, v, slots.to(device))
            if s.appended:
                k, v = synth.kv_tokens(s, b, keep, s.appended, device=device)
                new_k.append(k)
                new_v.append(v)
                new_slots.append(synth.slots_for(wl.block_table, b, np.arange(keep, L), s.page_size))
        if s.appended:
            self.k_new = torch.cat(new_k).contiguous()
            self.v_new = torch.cat(new_v).contiguous()
            self.slots_new = torch.from_numpy(np.concatenate(new_slots)).to(device)
        else:
            self.k_new = self.v_new = self.slots_new = None
        self.q = synth.queries(s, device=device).contiguous()
        if s.query_tokens == 1:
            self.q = self.q[:, 0].contiguous()
        self.out = torch.empty_like(self.q)
        # one token per sequence, then decode: a single rq_decode_step
        self.fused_step = not self.prefill_only and s.appended == 1 and s.query_tokens == 1
        self.extend = not self.prefill_only and s.query_tokens >= synth.EXTEND_MIN_T
        torch.cuda.synchronize(device)
        assert int(self.cache.status.item()) == 0, "range fault while building the cache"

    def step(self):
        s = self.spec
        if self.fused_step:
            self.cache.decode_step(self.q, self.k_new, self.v_new, self.bt, self.lens, out=self.out)
            return
        if self.k_new is not None:
            self.cache.append(self.k_new, self.v_new, self.slots_new)
        if self.prefill_only:
            return
        if s.query_tokens == 1:
            self.cache.decode(self.q, self.bt, self.lens, out=self.out)
        elif self.extend:
            self.cache.extend(self.q, self.bt, self.lens, out=self.out)
        else:
            self.cache.verify(self.q, self.bt, self.lens, out=self.out)

    def launches_per_step(self):
        dense = self.spec.mode == synth.DENSE
        if self.fused_step:  # split-K with the append folded in and the units finished in-kernel; a
            return 2 if dense else 1  # dense rotation: the prologue (queries + tokens), then split-K
        if self.extend:
            return 3 if dense else 2  # append, (dense: the query rotation,) extend attention
        n = 1 if self.k_new is not None else 0
        # split-K (it finishes every unit, R_v^T included); a dense rotation adds the query rotation
        return n if self.prefill_only else n + 1 + (self.spec.mode == synth.DENSE)

    def tokens_per_step(self):
        if self.prefill_only:
            return self.spec.ctx
        return self.spec.batch * self.spec.query_tokens

    def packed_bytes(self):
        s = self.spec
        per = 32 * s.bits + 4
        return int(self.wl.seq_lens.astype(np.int64).sum()) * s.num_kv_heads * per

    def attention_algorithmic_bytes(self):
        """Bytes the split-K kernel must move per launch: the packed cache of every attended
        token-head, the queries, and the block-table entries it reads."""
        s = self.spec
        pages = int(((self.wl.seq_lens + s.page_size - 1) // s.page_size).sum())
        q_bytes = 512 if s.mode == synth.DENSE else 256  # fp32 pre-rotated rows, or fp16 q
        # the step's tokens, when the split-K kernel itself appends them (structured rotations)
        fused = self.append_algorithmic_bytes() if self.fused_step and s.mode != synth.DENSE else 0
        return self.packed_bytes() + s.batch * s.query_tokens * s.num_q_heads * q_bytes + pages * 4 + fused

    def extend_flops(self):
        """Tensor-core FLOPs of the extend kernel per launch: query row j of a sequence of len tokens
        sees len - T + j + 1 keys; per (row, key) 128 multiply-adds for QK^T and 128 for PV."""
        s = self.spec
        T = s.query_tokens
        total = 0
        for L in self.wl.seq_lens.astype(np.int64):
            total += sum(max(0, int(L) - T + j + 1) for j in range(T))
        return float(total) * s.num_q_heads * 4 * 128

    def append_algorithmic_bytes(self):
        n = int(self.slots_new.numel()) if self.slots_new is not None else 0
        per_vec = 256 + 16 * self.spec.bits + 2
        return n * self.spec.num_kv_heads * 2 * per_vec + (0 if self.fused_step else n * 4)


# ---------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------
# NVML clock-event reason bits (nvml.h): the ones a measurement must report
_NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
                 0x80: "hw_power_brake_slowdown"}
CLOCK_Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
           "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
           "clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """Samples the GPU's SM clock, power and clock-event reasons every `period_s` seconds on a
    background thread (NVML through ctypes: it only reads), from before the warm-up to after
    the timed loop.  `mark(t0, t1)` names the timed region; the summary covers the samples
    taken inside it (a region of a few milliseconds still gets samples at 2 ms), with the
    whole run's samples beside them.  Falls back to `nvidia-smi -lms 100` if NVML is missing."""

    def __init__(self, device, period_s=0.002):
        self.device = device
        self.period = period_s
        self.rows = []          # (time, sm_mhz, power_w, reasons bitmask)
        self.window = None
        self.max_mhz = None
        self.source = None
        self._stop = None
        self._thread = None
        self._proc = None

    def _nvml_handle(self):
        import ctypes
        nv = None
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                nv = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if nv is None or nv.nvmlInit_v2() != 0:
            return None, None
        h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(self.device)
        ok = False
        uuid = str(getattr(props, "uuid", "") or "")
        if uuid:
            ok = nv.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(h)) == 0
        if not ok and hasattr(props, "pci_bus_id"):
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
            ok = nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
        if not ok:
            ok = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.device.index or 0), ctypes.byref(h)) == 0
        return (nv, h) if ok else (None, None)

    def _poll(self, nv, h):
        import ctypes
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            t = time.perf_counter()
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:  # NVML_CLOCK_SM
                p = pw.value / 1000.0 if nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 else None
                r = rs.value if get_reasons(h, ctypes.byref(rs)) == 0 else 0
                self.rows.append((t, float(clk.value), p, int(r)))
            self._stop.wait(self.period)

    def __enter__(self):
        import threading
        self._stop = threading.Event()
        try:
            nv, h = self._nvml_handle()
        except Exception:
            nv, h = None, None
        if nv is not None:
            import ctypes
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.source = f"nvml every {self.period * 1e3:g} ms"
            self._thread = threading.Thread(target=self._poll, args=(nv, h), daemon=True)
            self._thread.start()
            return self
        try:  # nvidia-smi fallback
            self._path = os.path.join(tempfile.gettempdir(), f"rq_bench_clocks_{os.getpid()}.csv")
            self._f = open(self._path, "w")
            self._t_start = time.perf_counter()
            self._proc = subprocess.Popen(["nvidia-smi", f"--id={self.device.index or 0}", f"--query-gpu={CLOCK_Q}",
                                           "--format=csv,noheader,nounits", "-lms", "100"],
                                          stdout=self._f, stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi every 100 ms"
        except Exception:
            self._proc = None
        return self

    def __exit__(self, *a):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
            self._f.close()
            names = {5: 0x8, 6: 0x40, 7: 0x20, 8: 0x4}
            with open(self._path) as f:
                lines = [[p.strip() for p in ln.split(",")] for ln in f]
            try:
                os.remove(self._path)
            except OSError:
                pass
            n = max(len(lines), 1)
            for i, parts in enumerate(lines):  # nvidia-smi gives no timestamps: spread them evenly
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    r = sum(bit for col, bit in names.items() if parts[col].lower() == "active")
                    p = float(parts[3]) if parts[3].replace(".", "").isdigit() else None
                    t = self._t_start + (time.perf_counter() - self._t_start) * i / n
                    self.rows.append((t, float(parts[1]), p, r))
                    self.max_mhz = float(parts[2]) if parts[2].replace(".", "").isdigit() else self.max_mhz

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def summary(self):
        if self.source is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"], "samples": 0}

        def summ(rows):
            if not rows:
                return {"sm_mhz": None, "reasons": [], "samples": 0}
            reasons = sorted({name for r in rows for bit, name in _NVML_REASONS.items() if r[3] & bit})
            powers = [r[2] for r in rows if r[2] is not None]
            return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_mhz_min": min(r[1] for r in rows),
                    "reasons": reasons, "samples": len(rows), "power_w_max": max(powers) if powers else None}

        inside = [r for r in self.rows if self.window and self.window[0] <= r[0] <= self.window[1]]
        out = summ(inside)
        out["sm_max_mhz"] = self.max_mhz
        out["source"] = self.source
        out["whole_run"] = summ(self.rows)
        return out


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense fp16/bf16 tensor TFLOP/s sustained over a long loop (the kernel runs inside a step
    loop), measured by cuBLAS bf16 -- fp16 has the same tensor-core rate."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured bf16_tflops_sustained"
    return FALLBACK_TFLOPS_SUSTAINED, "fallback (1.7 PFLOP/s sustained)"


def committed_traffic(kernel_file, workload):
    """DRAM bytes per launch (read + write) from the committed ncu summary
    profiles/traffic_<workload>.txt ("key: value" lines), if it was taken on the current
    kernel source (same sha256); None otherwise."""
    p = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    src = os.path.join(ROOT, "rotation_quantized_kv_rq_gb300", "csrc", kernel_file)
    if not os.path.exists(p):
        return None
    d = {}
    with open(p) as f:
        for ln in f:
            if ":" in ln and not ln.startswith("#"):
                k, v = ln.split(":", 1)
                d[k.strip()] = v.strip()
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if d.get("source_sha256") != sha:
        return None
    try:
        return float(d["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------------------
# the oracle on the host (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------------------
def oracle_step_rate(name, budget_s=10.0, threads=1):
    """Times the CPU oracle doing this workload's step on a sample, on `threads` host threads
    (the oracle's C calls release the GIL, so sequences -- or, for a prefill, 1024-token
    chunks -- run in parallel).  One unit of work is timed alone first; the sample is then as
    many units as fill about `budget_s` seconds on the threads (at most the workload's), their
    packed caches built untimed, and the sample is run repeatedly (steps rewrite the same
    slots) until `budget_s` of wall time has passed.  Returns (tokens/s, description,
    seconds, threads used)."""
    from concurrent.futures import ThreadPoolExecutor
    from oracle import oracle as O
    prefill_only = name in synth.PREFILL
    spec = synth.prefill_spec(name) if prefill_only else synth.SPECS[name]
    wl = synth.workload(spec)
    if prefill_only:
        oc = O.Cache(spec.mode, spec.bits, spec.num_q_heads, spec.num_kv_heads, spec.page_size, wl.num_pages,
                     wl.rot_k, wl.rot_v)
        chunks = []
        for n in range(0, spec.ctx, 1024):
            cnt = min(1024, spec.ctx - n)
            k, v = synth.kv_tokens(spec, 0, n, cnt)
            chunks.append((k.numpy(), v.numpy(),
                           synth.slots_for(wl.block_table, 0, np.arange(n, n + cnt), spec.page_size), cnt))
            if n == 0:  # probe: one chunk alone (after an untimed first call)
                oc.append(*chunks[0][:3])
                t0 = time.perf_counter()
                oc.append(*chunks[0][:3])
                t1 = time.perf_counter() - t0
                want = max(threads, min((spec.ctx + 1023) // 1024, int(budget_s * threads / max(t1, 1e-6))))
            if len(chunks) >= want:
                break
        used = min(threads, len(chunks))
        reps, t0 = 0, time.perf_counter()
        with ThreadPoolExecutor(used) as ex:  # disjoint slots: the chunks write disjoint bytes
            while True:
                list(ex.map(lambda c: oc.append(*c[:3]), chunks))
                reps += 1
                wall = time.perf_counter() - t0
                if wall >= budget_s:
                    break
        n = sum(c[3] for c in chunks)
        return reps * n / wall, (f"quantize-append of the first {n} of {spec.ctx} tokens x {spec.num_kv_heads} kv heads, "
                                 f"{reps} times"), wall, used
    q = synth.queries(spec).numpy()
    P = spec.page_size

    def build(b):  # sequence b's own compact pool, everything but the step's tokens (untimed)
        L = int(wl.seq_lens[b])
        npg = (L + P - 1) // P
        oc = O.Cache(spec.mode, spec.bits, spec.num_q_heads, spec.num_kv_heads, P, npg, wl.rot_k, wl.rot_v)
        keep = L - spec.appended
        for st in range(0, keep, 8192):
            cnt = min(8192, keep - st)
            k, v = synth.kv_tokens(spec, b, st, cnt)
            oc.append(k.numpy(), v.numpy(), np.arange(st, st + cnt, dtype=np.int32))
        new = synth.kv_tokens(spec, b, keep, spec.appended) if spec.appended else None
        return b, L, npg, keep, oc, new

    def step(item):  # the timed work: append of the step's tokens, then attention
        b, L, npg, keep, oc, new = item
        if new is not None:
            oc.append(new[0].numpy(), new[1].numpy(), np.arange(keep, L, dtype=np.int32))
        oc.attention(q[b:b + 1] if spec.query_tokens > 1 else q[b:b + 1, :1], np.arange(npg, dtype=np.int32)[None, :],
                     np.array([L], np.int32), T=spec.query_tokens)

    first = build(0)
    t0 = time.perf_counter()
    step(first)
    t1 = time.perf_counter() - t0
    S = max(1, min(spec.batch, int(budget_s * threads / max(t1, 1e-6))))
    used = min(threads, S)
    with ThreadPoolExecutor(used) as ex:
        items = [first] + list(ex.map(build, range(1, S)))
        rounds, t0 = 0, time.perf_counter()
        while True:
            list(ex.map(step, items))
            rounds += 1
            wall = time.perf_counter() - t0
            if wall >= budget_s:
                break
    return (rounds * S * spec.query_tokens / wall,
            f"{S} of {spec.batch} sequences (full context each), {rounds} steps each", wall, used)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------------------
TARGET_WORKLOAD = "cfg2_32k"  # the long-context decode the roofline target is stated at


def config_of(name, world, batch=None):
    """The `config` object of a workload's JSON line (the same on both arms)."""
    s = spec_of(name, batch)
    wl = synth.workload(s)
    packed = int(wl.seq_lens.astype(np.int64).sum()) * s.num_kv_heads * (32 * s.bits + 4)
    fused = name not in synth.PREFILL and s.appended == 1 and s.query_tokens == 1
    return {"workload": f"{name}: {DESCRIPTIONS[name]}", "batch": s.batch, "ctx": int(s.ctx),
            "query_tokens": s.query_tokens, "bits": s.bits,
            "mode": {synth.PLANAR: "planar", synth.ISO: "iso", synth.DENSE: "dense"}[s.mode],
            "page_size": s.page_size, "fused_decode_step": fused, "packed_kv_bytes": packed,
            "l2": f"flushed before every step ({L2_FLUSH_BYTES >> 20} MB write) outside the per-step events",
            "parallelism": f"replicas x{world}"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    rate, sample, secs, cores = oracle_step_rate(args.workload, budget_s=args.ref_budget, threads=host_cores())
    line = {
        "impl": "reference", "metric": "decode-attn tokens/s", "value": rate, "unit": "tokens/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(args.workload, world),
        "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "the reference arm is the plain fp64 CPU oracle written from the pages (no implementation of "
                "the method exists on the pages); it times the oracle on all host cores, a thread per sequence",
    }
    print(json.dumps(line), flush=True)


def time_steps(bench, K, W, flush, stream):
    """W untimed steps, then K steps each bracketed by CUDA events on the launching stream (the
    attention kernel's own launch by the library's profiling events); L2 is flushed before every
    step, outside the events.  Returns (per-step ms, per-kernel ms, wall seconds of the K steps)."""
    device = stream.device
    for _ in range(W):
        flush.fill_(1.0)
        bench.step()
    torch.cuda.synchronize(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    # torch creates an event's CUDA handle on its first record: record every profiling event
    # once here, so the library can re-record the same handles around its kernel
    for a, b in kev:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for i in range(K):
        flush.fill_(float(i))
        if not bench.prefill_only:
            rq.rq_set_profile_events(bench.cache.ctx, kev[i][0], kev[i][1])
        ev[i][0].record(stream)
        bench.step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    t1 = time.perf_counter()
    if not bench.prefill_only:
        rq.rq_set_profile_events(bench.cache.ctx)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    kern_ms = [a.elapsed_time(b) for a, b in kev] if not bench.prefill_only else step_ms
    return step_ms, kern_ms, (t0, t1)


def fp16_attention_rows(q, k, v, L, T, rows, group):
    """Softmax attention of query rows `rows` (draft indices) of one sequence over its
    UNQUANTISED fp16 cache, in fp32 on the GPU: the fidelity reference.  q [T][Hq][d],
    k / v [L][Hkv][d]; row j sees positions 0 .. L - T + j."""
    kf = k.float().repeat_interleave(group, dim=1).transpose(0, 1)  # [Hq][L][d]
    vf = v.float().repeat_interleave(group, dim=1).transpose(0, 1)
    outs = []
    for j in rows:
        n = L - T + j + 1
        s = torch.einsum("hd,hld->hl", q[j].float(), kf[:, :n]) / math.sqrt(kf.shape[-1])
        outs.append(torch.einsum("hl,hld->hd", torch.softmax(s, dim=-1), vf[:, :n]))
    return torch.stack(outs)  # [rows][Hq][d]


def fidelity(bench, n_seq=3):
    """Cosine similarity per (query row, head) between the bench step's output and attention
    over the unquantised fp16 K/V of a few sampled sequences (first, last, longest)."""
    if bench.prefill_only:
        return None
    s, wl = bench.spec, bench.wl
    T = s.query_tokens
    lens = wl.seq_lens
    seqs = sorted({0, s.batch - 1, int(np.argmax(lens))})[:n_seq]
    rows = sorted({0, T // 2, T - 1}) if T > 6 else list(range(T))
    q = bench.q if T > 1 else bench.q[:, None]
    out = bench.out if T > 1 else bench.out[:, None]
    cos = []
    for b in seqs:
        L = int(lens[b])
        k, v = synth.kv_tokens(s, b, 0, L, device=bench.device)
        ref = fp16_attention_rows(q[b], k, v, L, T, rows, s.group)
        got = out[b, rows].float()
        c = torch.nn.functional.cosine_similarity(got.reshape(-1, got.shape[-1]), ref.reshape(-1, ref.shape[-1]),
                                                  dim=-1)
        cos.append(c)
        del k, v
    c = torch.cat(cos)
    return {"cosine_min": float(c.min()), "cosine_mean": float(c.mean()),
            "sample": f"sequences {seqs}, query rows {rows}, every q head; against softmax attention over the "
                      f"unquantised fp16 K/V (fp32 math on the GPU), outside the timed region"}


def attention_roofline(bench, kern_ms, peak, peak_kind, workload):
    kms = statistics.mean(kern_ms)
    if bench.extend:
        flops = bench.extend_flops()
        tpeak, tkind = measured_tensor_peak()
        achieved = flops / (kms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": tpeak, "unit": "TFLOP/s", "frac": achieved / tpeak,
                "traffic": committed_traffic("rq_extend.cu", workload), "kernel": "extend_kernel",
                "algorithmic_flops_per_launch": flops, "kernel_ms_mean": kms,
                "kernel_ms_median": statistics.median(kern_ms), "peak_source": tkind}
    if bench.prefill_only:
        alg = bench.append_algorithmic_bytes()
        kname = "append_kernel"
    else:
        alg = bench.attention_algorithmic_bytes()
        kname = "attn_splitk_kernel"
    achieved = alg / (kms * 1e-3) / 1e9
    traffic = committed_traffic("rq_attention.cu" if not bench.prefill_only else "rq_append.cu", workload)
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic, "kernel": kname, "algorithmic_bytes_per_launch": alg,
            "kernel_ms_mean": kms, "kernel_ms_median": statistics.median(kern_ms),
            "peak_source": f"{peak_kind} hbm_gbs", "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS}


def run_ours(args, rank, world, local):
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    bench = Bench(args.workload, device, args.batch)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    K = args.steps
    sampler = ClockSampler(device)
    with sampler:
        barrier(world)
        step_ms, kern_ms, (t_wall0, t_wall1) = time_steps(bench, K, args.warmup, flush, stream)
        sampler.mark(t_wall0, t_wall1)
        barrier(world)
    ms = sum(step_ms) / K
    ms = max_over_ranks(ms, world)
    tokens = bench.tokens_per_step()
    value = world * tokens / (ms * 1e-3)
    assert int(bench.cache.status.item()) == 0

    # ---- end to end through the public API: pinned host inputs in, result back to the host.
    # The step's inputs (q, and the new K / V and slots when the step appends) sit in one pinned
    # staging buffer, copied to the device in one transfer; the kernels read views of it.  The
    # result read back is the output rows, or the status word of an append-only step.
    parts = [] if bench.prefill_only else [bench.q]
    if bench.k_new is not None:
        parts += [bench.k_new, bench.v_new] + ([] if bench.fused_step else [bench.slots_new])
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 15) // 16 * 16  # 16-byte aligned views
    h_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(total, dtype=torch.uint8, device=device)
    views = []
    for t, o in zip(parts, offs):
        nb = t.numel() * t.element_size()
        h_in[o:o + nb].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
        views.append(d_in[o:o + nb].view(t.dtype).view(t.shape))
    i0 = 0 if bench.prefill_only else 1
    d_q = None if bench.prefill_only else views[0]
    d_k, d_v = (views[i0], views[i0 + 1]) if bench.k_new is not None else (None, None)
    d_s = views[i0 + 2] if (bench.k_new is not None and not bench.fused_step) else None
    result = bench.cache.status if bench.prefill_only else bench.out
    h_out = torch.empty_like(result, device="cpu").pin_memory()
    h2d = total
    d2h = h_out.numel() * h_out.element_size()
    e2e_times = []
    n_e2e = max(3, min(K, 200))
    for i in range(n_e2e + 2):
        flush.fill_(float(i))
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        d_in.copy_(h_in, non_blocking=True)
        if bench.fused_step:
            bench.cache.decode_step(d_q, d_k, d_v, bench.bt, bench.lens, out=bench.out)
        elif d_k is not None:
            bench.cache.append(d_k, d_v, d_s)
        if not bench.prefill_only and not bench.fused_step:
            if bench.spec.query_tokens == 1:
                bench.cache.decode(d_q, bench.bt, bench.lens, out=bench.out)
            elif bench.extend:
                bench.cache.extend(d_q, bench.bt, bench.lens, out=bench.out)
            else:
                bench.cache.verify(d_q, bench.bt, bench.lens, out=bench.out)
        h_out.copy_(result, non_blocking=True)
        stream.synchronize()
        if i >= 2:
            e2e_times.append(time.perf_counter() - t0)
    e2e_s = max_over_ranks(statistics.median(e2e_times), world)

    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    roof = attention_roofline(bench, kern_ms, peak, peak_kind, args.workload)
    fid = fidelity(bench)
    launches = bench.launches_per_step() * K

    # ---- the long-context decode the roofline target is stated at (32 x 32K rq4 iso), timed
    # the same way in the same process, after the headline workload's own measurement
    target = None
    if not args.no_target and args.workload != TARGET_WORKLOAD and not args.batch:
        bench.cache.close()
        del bench
        torch.cuda.empty_cache()
        tb = Bench(TARGET_WORKLOAD, device)
        tk = max(K, 20)
        with ClockSampler(device) as tsamp:
            t_step, t_kern, (a0, a1) = time_steps(tb, tk, max(args.warmup, 3), flush, stream)
            tsamp.mark(a0, a1)
        assert int(tb.cache.status.item()) == 0
        tr = attention_roofline(tb, t_kern, peak, peak_kind, TARGET_WORKLOAD)
        target = {"workload": f"{TARGET_WORKLOAD}: {DESCRIPTIONS[TARGET_WORKLOAD]}", "steps": tk,
                  "kernel_ms_mean": tr["kernel_ms_mean"], "kernel_ms_median": tr["kernel_ms_median"],
                  "achieved_gbs": tr["achieved"], "frac": tr["frac"], "frac_of_nominal_8tbs": tr["frac_of_nominal_8tbs"],
                  "traffic": tr["traffic"], "algorithmic_bytes_per_launch": tr["algorithmic_bytes_per_launch"],
                  "target_frac_of_nominal_8tbs": 0.70, "clocks": tsamp.summary(),
                  "tokens_per_s": tb.tokens_per_step() / (statistics.mean(t_step) * 1e-3)}
        tb.cache.close()
        del tb

    cpu = None
    if world == 1 and not args.no_cpu_baseline and not args.batch:
        rate, sample, secs, cores = oracle_step_rate(args.workload, budget_s=args.cpu_budget, threads=host_cores())
        rate1, sample1, secs1, _ = oracle_step_rate(args.workload, budget_s=args.cpu_budget / 2, threads=1)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
               "seconds": round(secs, 2),
               "one_core": {"value": rate1, "sample": sample1, "seconds": round(secs1, 2)}}
    s = spec_of(args.workload, args.batch)
    packed = config_of(args.workload, world, args.batch)["packed_kv_bytes"]
    line = {
        "metric": "decode-attn tokens/s", "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": f"u{s.bits} codes, f16 mma, f32 accumulate", "data": "synthetic",
        "config": config_of(args.workload, world, args.batch),
        "packed_kv_gbs": packed / (ms * 1e-3) / 1e9,
        "roofline": roof,
        "target_32k": target,
        "fidelity": fid,
        "cpu_baseline": cpu,
        "e2e": {"value": world * tokens / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3},
        "gpu_launches": launches,
        "clocks": sampler.summary(),
        "wall_s_timed_region": t_wall1 - t_wall0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="cfg4", choices=sorted(DESCRIPTIONS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--ref-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-target", action="store_true",
                    help="skip the 32 x 32K decode sub-record timed after the workload")
    ap.add_argument("--batch", type=int, default=None,
                    help="profiling: the workload's first BATCH sequences only (no baseline or target legs)")
    args = ap.parse_args()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
