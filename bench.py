#!/usr/bin/env python
"""Decode-step benchmark for the paged KV cache library on GB300.

A step is the whole hot path over one batch: copy_blocks (this step's
copy-on-write pairs) -> kv_append (one new K/V row per sequence) ->
paged_attention_decode (split + log-sum-exp combine).  Default workload: the
Llama-3-8B-shaped GQA step (32 query / 8 KV heads, head_dim 128, bf16, block
size 16, batch 256, lognormal context lengths with median 1024 clipped to
[16, 8192], blocks scattered over a pool 1.5x the need), inputs resident in
HBM.  The L2 is flushed (a 512 MB write, then a 256 MB read, so no dirty
lines are left) between timed steps, outside the timed events.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
this machine's host cores instead (the reference arm).  Under torchrun every
rank runs an independent replica of the workload (weak scaling, no collective
on the data path); the timed region is bracketed by barriers and the slowest
rank's time is reported.
"""

from __future__ import annotations

import argparse
import copy
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention: KV HBM GB/s (% of GB300 peak), seq-steps/s"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
# DRAM bytes per launch from ncu captures, keyed by kernel and workload, each
# with the sha256 of the kernel source the counters were taken on
TRAFFIC_DATA = os.path.join(ROOT, "profiles", "dram_traffic.json")
DECODE_SOURCE = os.path.join(ROOT, "paged_kv_cache_68_gb300", "csrc", "decode_kernel.cuh")
PREFILL_SOURCE = os.path.join(ROOT, "paged_kv_cache_68_gb300", "csrc", "prefill_kernel.cuh")

WORKLOAD_TEXT = {
    "llama3_8b_gqa": "Llama-3-8B-shaped GQA decode step: 32 query / 8 KV heads, head_dim 128, bf16, "
                     "block_size 16, batch 256, context ~ clip(round(lognormal(ln 1024, 1.0)), 16, 8192), "
                     "blocks scattered in a pool 1.5x the need, 1 layer, append + attention",
    "opt13b_mha": "OPT-13B-shaped MHA decode step: 40 = 40 heads, head_dim 128, fp16, block_size 16, "
                  "batch 64, context ~ U[128, 2048], pool 1.5x, 1 layer, append + attention",
    "shared_prefix": "shared-prefix parallel sampling: Llama-3-8B GQA shape, bf16, bs 16, 32 prompts x "
                     "2000 tokens, n = 4 samples, 0-256 divergent tokens, CoW copies + append + attention",
    "long_context": "long-context split-KV decode: 32/8 heads, head_dim 128, bf16, batch 8, "
                    "context ~ U[32768, 131072], block_size 16",
    "tiny": "tiny paged decode: 4 sequences with contexts {6, 17, 33, 50} (+1 appended), 4 = 4 heads, "
            "head_dim 64, fp32, block_size 4, 64 blocks placed by a seeded permutation, append + attention",
    "chunked_prefill": "chunked prefill step: Llama-3-8B GQA shape (32/8 heads, head_dim 128, bf16, "
                       "block_size 16), 16 requests x 256-token chunks after cached prefixes of "
                       "U[0, 3840] tokens, blocks scattered in a pool 1.5x the need, 1 layer, "
                       "append of the chunks + causal paged prefill attention",
}
PREFILL_METRIC = "paged chunked-prefill attention: TFLOP/s (% of GB300 bf16 tensor peak), query tokens/s"


# ------------------------------------------------------------------ helpers --

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_TEXT), default="llama3_8b_gqa")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--placement", choices=["random", "identity"], default="random")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (profiling a smaller case)")
    ap.add_argument("--block-size", type=int, default=None,
                    help="block size of the long-context workload (8, 16 or 32)")
    ap.add_argument("--fresh-fork", action="store_true",
                    help="shared-prefix workload: the first decode step after the fork (every "
                         "sample still shares its prompt's partial last block, so with a "
                         "2008-token prompt the step makes 3 copy-on-write copies per prompt)")
    ap.add_argument("--prompt-len", type=int, default=None,
                    help="prompt length of the shared-prefix workload (2000 or 2008)")
    ap.add_argument("--kv-cache", choices=["fp8_e4m3", "int8"], default=None,
                    help="an 8-bit pool (quantising append, dequantising decode) instead of "
                         "the workload's 16-bit one")
    ap.add_argument("--swap-frac", type=float, default=0.0,
                    help="also time kv_swap_blocks out to pinned host memory and back for the "
                         "blocks of this fraction of the sequences")
    ap.add_argument("--cascade", action="store_true",
                    help="shared-prefix workload: decode with the cascade entry point")
    ap.add_argument("--decodes", type=int, default=0,
                    help="chunked-prefill workload: decode requests packed into the batch")
    ap.add_argument("--chunk", type=int, default=None,
                    help="chunked-prefill workload: tokens per chunk (default 256)")
    return ap.parse_args(argv)


def make_workload(name: str, seed: int, device, placement: str = "random", batch=None,
                  block_size=None, prompt_len=None, decodes=0, chunk=None, fresh_fork=False):
    from paged_kv_cache_68_gb300 import workloads as wl
    kw = {} if batch is None else {"batch": batch}
    if name == "llama3_8b_gqa":
        return wl.llama3_8b_gqa(seed, device=device, placement=placement, **kw)
    if name == "opt13b_mha":
        return wl.opt13b_mha(seed, device=device, **kw)
    if name == "shared_prefix":
        if batch is not None:
            kw = {"prompts": batch}
        if prompt_len is not None:
            kw["prompt_len"] = prompt_len
        if fresh_fork:                     # the first step after the fork: no divergent tokens
            import numpy as np
            kw["divergent"] = np.zeros(kw.get("prompts", 32) * 4, np.int64)
        return wl.shared_prefix(seed, device=device, **kw)
    if name == "tiny":
        return wl.tiny(seed, device=device)
    if name == "chunked_prefill":
        if chunk is not None:
            kw["chunk"] = chunk
        return wl.chunked_prefill(seed, decodes=decodes, device=device, **kw)
    if name == "long_context":
        if block_size is not None:
            kw["block_size"] = block_size
        return wl.long_context(seed, device=device, **kw)
    raise ValueError(name)


class L2Flush:
    """Between timed steps: write 512 MB (every line of the 129 MB L2 is
    replaced), then read 256 MB, so that the lines left in L2 are clean.
    Without the read, the step would start with ~129 MB of the flush's dirty
    lines in L2, written back to HBM while the decode streams its K/V -- a
    cost of the flush, not of the step."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(256 << 20, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(key, source):
    """DRAM bytes (read + write) per launch of the kernel under `key` in the
    traffic data file, if its counters were taken on the current source of
    that kernel (else None: the kernel changed since)."""
    try:
        entry = json.load(open(TRAFFIC_DATA))[key]
        sha = hashlib.sha256(open(source, "rb").read()).hexdigest()
    except (OSError, KeyError, ValueError):
        return None
    if entry.get("source_sha256") != sha:
        return None
    return int(entry["dram_bytes_per_launch"])


class ClockSampler:
    """SM clock and throttle reasons sampled while the timed region runs.

    NVML (read-only queries through ctypes) every 2 ms on a background thread;
    ``mark()`` takes one more sample synchronously (call it after the timed
    work is enqueued, while the GPU runs it), so even a region of a few
    milliseconds has samples.  Only samples between ``begin()`` and ``stop()``
    count.  Falls back to ``nvidia-smi -lms 200`` when NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        import ctypes
        import threading
        self.samples, self.t0, self.proc, self.nvml = [], None, None, None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            assert lib.nvmlInit_v2() == 0
            h = ctypes.c_void_p()
            if gpu_id.startswith("GPU-"):
                assert lib.nvmlDeviceGetHandleByUUID(gpu_id.encode(), ctypes.byref(h)) == 0
            else:
                assert lib.nvmlDeviceGetHandleByIndex_v2(int(gpu_id), ctypes.byref(h)) == 0
            reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))   # 1 = NVML_CLOCK_SM
            self.nvml, self.h, self.reasons_fn, self.max_mhz = lib, h, reasons_fn, float(mx.value)
            self.ctypes = ctypes
            self.stop_ev = threading.Event()
            self.lock = threading.Lock()
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()
        except Exception:
            self.nvml = None
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                     "-lms", "200", "-i", gpu_id], stdout=self.file, stderr=subprocess.DEVNULL)
            except OSError:
                self.proc = None

    def _read(self):
        c = self.ctypes
        mhz, rs = c.c_uint(), c.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, c.byref(mhz)) != 0:
            return None
        self.reasons_fn(self.h, c.byref(rs))
        return (time.perf_counter(), float(mhz.value), int(rs.value))

    def _loop(self):
        while not self.stop_ev.is_set():
            r = self._read()
            if r is not None:
                with self.lock:
                    self.samples.append(r)
            time.sleep(0.002)

    def begin(self):
        self.t0 = time.perf_counter()

    def mark(self):
        if self.nvml is not None:
            r = self._read()
            if r is not None:
                with self.lock:
                    self.samples.append(r)

    def stop(self):
        t1 = time.perf_counter()
        if self.nvml is not None:
            self.stop_ev.set()
            self.thread.join(timeout=2)
            t0 = self.t0 if self.t0 is not None else 0.0
            with self.lock:
                inside = [s for s in self.samples if t0 <= s[0] <= t1]
            reasons = set()
            for _, _, bits in inside:
                for bit, name in self.REASONS.items():
                    if bits & bit:
                        reasons.add(name)
            sm = [s[1] for s in inside]
            return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                    "reasons": sorted(reasons), "samples": len(sm), "source": "nvml"}
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [l.strip() for l in self.file.read().splitlines() if l.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi"}


def gpu_uuid(dev) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index or 0)


def dist_setup(n_gpus: int):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend=backend)
    return rank, world, local


def barrier():
    import torch
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def reduce_max_sum(local_ms: float, local_units: float):
    """(max over ranks of local_ms, sum over ranks of local_units)."""
    import torch
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return local_ms, local_units
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def unique_bytes_fields(w, world, dec_ms, q8=None):
    """Shared-prefix steps: decode GB/s against the K/V bytes stored once (the
    prefix counted once per prompt) beside the logical bytes."""
    if "unique_tokens" not in w.info:
        return {}
    row = w.num_kv_heads * w.head_dim * w.elem_bytes * 2 if q8 is None else q8.row_bytes(w)
    ub = int(w.info["unique_tokens"]) * row
    return {"unique_kv_bytes_per_replica": ub,
            "attention_gbs_unique": round(ub * world / (dec_ms * 1e-3) / 1e9, 2),
            "cow_pairs_per_step": int(w.pairs.shape[0])}


def decode_config(args, w, q8, world):
    """The workload description both arms print (the same keys and values)."""
    step_bytes = w.step_bytes() if q8 is None else q8.step_bytes(w)
    kv_bytes = w.kv_bytes() if q8 is None else q8.kv_bytes(w)
    return {"workload": WORKLOAD_TEXT[args.workload]
            + ("" if args.batch is None else f" (batch overridden to {args.batch})")
            + ("" if args.block_size is None else f" (block_size {args.block_size})")
            + ("" if args.prompt_len is None else f" (prompt_len {args.prompt_len})")
            + (" (fresh fork: no divergent tokens yet)" if args.fresh_fork else "")
            + ("" if q8 is None else f", K/V stored as {q8.cache} codes"),
            "seed": args.seed, "placement": args.placement, "global_batch": w.batch * world,
            "kv_cache": q8.cache if q8 is not None else w.dtype,
            "tokens_per_replica": int(w.seq_lens.sum()),
            "kv_bytes_per_replica": kv_bytes, "step_bytes_per_replica": step_bytes,
            "l2": "flushed between timed steps (512 MB write, then 256 MB read: no dirty lines "
                  f"left); K/V read per step {kv_bytes / 1e9:.3f} GB"
                  + (" > 129 MB L2" if kv_bytes > 129e6 else " (smaller than L2: the flush keeps it cold)"),
            "parallelism": f"replicas x{world}"}


def prefill_config(args, w, world, flops):
    return {"workload": WORKLOAD_TEXT[args.workload]
            + ("" if args.batch is None else f" (requests overridden to {args.batch})")
            + ("" if args.chunk is None else f" (chunk {args.chunk})")
            + ("" if not args.decodes else f", + {args.decodes} decode requests"),
            "seed": args.seed, "global_batch": w.batch * world,
            "query_tokens_per_replica": int(w.info["query_tokens"]),
            "context_tokens_per_replica": int(w.seq_lens.sum()),
            "attention_flops_per_replica": flops,
            "l2": "flushed between timed steps (512 MB write, then 256 MB read: no dirty lines left)",
            "parallelism": f"replicas x{world}"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        fields = dict(line.split(":", 1) for line in out.splitlines() if ":" in line)
        name = fields.get("Model name", "").strip()
        vendor = fields.get("Vendor ID", "").strip()
        if name:
            return f"{vendor} {name}".strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


# ----------------------------------------------------------- CPU baseline --

def oracle_sample_step(host_w, seqs, threads, q8=None):
    """One oracle step (copy, append, attention) restricted to `seqs`;
    returns (seconds, algorithmic bytes of that sample).  `q8`: host arrays
    of an 8-bit pool (workloads.Q8Pools) to step instead of the 16-bit one."""
    import numpy as np
    from oracle import c_oracle
    if q8 is not None:
        t0 = time.perf_counter()
        c_oracle.copy_blocks_q8(q8.k_codes, q8.v_codes, q8.k_scales, q8.v_scales, host_w.pairs)
        c_oracle.append_q8(q8.k_codes, q8.v_codes, q8.k_scales, q8.v_scales, host_w.k_new[seqs],
                           host_w.v_new[seqs], host_w.dtype, host_w.slot_mapping[seqs], q8.cache,
                           q8.k_scale, q8.v_scale)
        c_oracle.decode_q8(np.ascontiguousarray(host_w.q[seqs]), host_w.dtype, q8.k_codes,
                           q8.v_codes, q8.k_scales, q8.v_scales, q8.cache,
                           np.ascontiguousarray(host_w.block_tables[seqs]),
                           np.ascontiguousarray(host_w.seq_lens[seqs]), host_w.scale,
                           host_w.num_kv_heads, q8.k_scale, q8.v_scale, num_threads=threads)
        dt = time.perf_counter() - t0
        sub = copy.copy(host_w)
        sub.seq_lens = host_w.seq_lens[seqs]
        sub.q = host_w.q[seqs]
        sub.slot_mapping = host_w.slot_mapping[seqs]
        return dt, q8.step_bytes(sub)
    k, v = host_w.k_pool, host_w.v_pool          # state: appends are idempotent
    t0 = time.perf_counter()
    c_oracle.copy_blocks(k, v, host_w.pairs, host_w.dtype)
    c_oracle.append(k, v, host_w.k_new[seqs], host_w.v_new[seqs], host_w.slot_mapping[seqs],
                    host_w.dtype)
    c_oracle.decode(np.ascontiguousarray(host_w.q[seqs]), k, v, host_w.dtype,
                    np.ascontiguousarray(host_w.block_tables[seqs]),
                    np.ascontiguousarray(host_w.seq_lens[seqs]), host_w.scale,
                    host_w.num_kv_heads, num_threads=threads)
    dt = time.perf_counter() - t0
    L = host_w.seq_lens[seqs].astype(np.int64)
    row = host_w.num_kv_heads * host_w.head_dim * host_w.elem_bytes
    nbytes = int(L.sum()) * row * 2 + len(seqs) * row * 4 + host_w.copy_bytes()
    return dt, nbytes


def q8_on_host(q8):
    """Host numpy copies of an 8-bit pool's arrays (for the oracle)."""
    import dataclasses
    h = lambda a: None if a is None else (a.cpu().numpy() if hasattr(a, "cpu") else a).copy()
    return dataclasses.replace(q8, k_codes=h(q8.k_codes), v_codes=h(q8.v_codes),
                               k_scales=h(q8.k_scales), v_scales=h(q8.v_scales))


def pick_sample(host_w, budget_s, threads, q8=None):
    """Sequences (a prefix of a fixed shuffle) whose oracle step takes about budget_s."""
    import numpy as np
    order = np.random.default_rng(1234).permutation(host_w.batch)
    n = min(host_w.batch, max(1, threads))
    dt, _ = oracle_sample_step(host_w, order[:n], threads, q8)
    if dt < budget_s and n < host_w.batch:
        n = int(min(host_w.batch, max(n, n * budget_s / max(dt, 1e-3))))
    return np.sort(order[:n])


def time_swap(pool, w, frac, flush, K, dev):
    """kv_swap_blocks of every block of a fraction of the sequences: out to a
    pinned host pool, then back into the same blocks (the pool is unchanged),
    each timed with CUDA events after an L2 flush; beside it one contiguous
    pinned-host copy of the same bytes each way (the link's ceiling)."""
    import numpy as np
    import torch
    rng = np.random.default_rng(4321)
    seqs = np.sort(rng.permutation(w.batch)[:max(1, int(round(frac * w.batch)))])
    blocks = [int(w.block_tables[b, j]) for b in seqs
              for j in range(-(-int(w.seq_lens[b]) // w.block_size))]
    n = len(blocks)
    host = pool.host_pool(n)
    pairs = torch.tensor([[g, i] for i, g in enumerate(blocks)], dtype=torch.int32, device=dev)
    nbytes = sum(a[:n].numel() * a.element_size() for a in host if a is not None)
    ref_host = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    ref_dev = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def timed(fn):
        for _ in range(3):
            flush()
            fn()
        ms = 0.0
        for _ in range(K):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ms += e0.elapsed_time(e1)
        return ms / K

    out_ms = timed(lambda: pool.swap_out(host, pairs))
    in_ms = timed(lambda: pool.swap_in(host, pairs))
    d2h_ms = timed(lambda: ref_host.copy_(ref_dev, non_blocking=True))
    h2d_ms = timed(lambda: ref_dev.copy_(ref_host, non_blocking=True))
    assert pool.get_error() == 0, "device error word set during the swap timing"
    gbs = lambda ms: round(nbytes / (ms * 1e-3) / 1e9, 2)
    return {"sequences": int(seqs.shape[0]), "blocks": n, "bytes_per_direction": nbytes,
            "launches_per_direction": 1, "out_ms": round(out_ms, 4), "in_ms": round(in_ms, 4),
            "out_gbs": gbs(out_ms), "in_gbs": gbs(in_ms),
            "contiguous_copy_gbs": {"d2h": gbs(d2h_ms), "h2d": gbs(h2d_ms)},
            "host_memory": "pinned (cudaHostAlloc through torch), addressed by the kernel"}


# --------------------------------------------------------------- our arm --

def run_ours(args):
    import numpy as np
    import torch

    from paged_kv_cache_68_gb300 import pagedkv
    from paged_kv_cache_68_gb300 import workloads as wl

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pagedkv.load()
    w = make_workload(args.workload, args.seed, dev, args.placement, args.batch,
                      args.block_size, args.prompt_len, fresh_fork=args.fresh_fork)
    tv = lambda a: wl.value_to_torch(a, w.dtype, dev)
    k_pool, v_pool = w.k_pool, w.v_pool
    # the step's inputs live back to back in one device buffer (256-byte
    # aligned views), so the end-to-end leg moves them with one copy
    srcs = {"q": tv(w.q), "k_new": tv(w.k_new), "v_new": tv(w.v_new),
            "slots": torch.from_numpy(w.slot_mapping).to(dev),
            "tables": torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(dev),
            "lens": torch.from_numpy(w.seq_lens).to(dev),
            "pairs": torch.from_numpy(np.ascontiguousarray(w.pairs, dtype=np.int32)).to(dev)}
    offs, total = {}, 0
    for n, t in srcs.items():
        offs[n] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    dev_in = torch.empty(max(total, 256), dtype=torch.uint8, device=dev)
    view = {}
    for n, t in srcs.items():
        nb = t.numel() * t.element_size()
        view[n] = dev_in[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)
        view[n].copy_(t)
    q, k_new, v_new = view["q"], view["k_new"], view["v_new"]
    slots, tables, lens, pairs = view["slots"], view["tables"], view["lens"], view["pairs"]
    host_in = dev_in.cpu().pin_memory()
    q8 = None
    if args.kv_cache:
        q8 = wl.q8_pools(w, args.kv_cache, args.seed)
        w.k_pool = w.v_pool = k_pool = v_pool = None              # the 16-bit pools are not used
        torch.cuda.empty_cache()
        pool = pagedkv.KVPool(q8.k_codes, q8.v_codes, cache=q8.cache, dtype=q.dtype,
                              k_scales=q8.k_scales, v_scales=q8.v_scales, k_scale=q8.k_scale,
                              v_scale=q8.v_scale)
    else:
        pool = pagedkv.KVPool(k_pool, v_pool)
    out = torch.empty_like(q)
    cascade = args.cascade and w.groups is not None
    if cascade:
        groups = torch.from_numpy(np.ascontiguousarray(w.groups)).to(dev)
        gcols = [groups[:, i].contiguous() for i in range(3)]
        ws = torch.empty(pagedkv.paged_attention_cascade_workspace_size(
            pool.handle, w.batch, w.num_q_heads, int(groups.shape[0])), dtype=torch.uint8, device=dev)
    else:
        ws = pool.workspace(w.batch, w.num_q_heads)

    def decode():
        if cascade:
            pagedkv.paged_attention_decode_cascade(pool.handle, q, out, tables, lens, w.scale,
                                                   w.num_kv_heads, gcols[0], gcols[1], gcols[2],
                                                   ws, pool.dtype)
        else:
            pool.decode(q, tables, lens, w.scale, out=out, workspace=ws)
    flush = L2Flush(dev)
    n_pairs = int(w.pairs.shape[0])
    # copy (if pairs), append, decode (split, + merge for long contexts; a cascade decode adds
    # the prefix pass)
    dec_launches = pagedkv.paged_attention_decode_launches(pool.handle, w.batch, w.num_q_heads)
    launches_per_step = (1 if n_pairs else 0) + 1 + dec_launches + (1 if cascade else 0)

    def step():
        pool.copy_blocks(pairs)
        pool.append(k_new, v_new, slots)
        decode()

    for _ in range(max(3, args.warmup)):
        flush()
        step()
    torch.cuda.synchronize()
    assert pool.get_error() == 0, "device error word set during warm-up"

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    sampler = ClockSampler(gpu_uuid(dev))
    barrier()
    torch.cuda.synchronize()
    sampler.begin()
    for i in range(K):
        flush()                                   # L2 flush, outside the events
        e = ev[i]
        e[0].record()
        pool.copy_blocks(pairs)
        pool.append(k_new, v_new, slots)
        e[1].record()
        decode()
        e[2].record()
        e[3].record()
    sampler.mark()                                      # the GPU is running the queued steps
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    step_ms = sum(e[0].elapsed_time(e[3]) for e in ev) / K
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    assert pool.get_error() == 0, "device error word set during the timed steps"

    # end to end through the C ABI with host buffers (pinned), copies timed:
    # the step's inputs in one host-to-device copy, the output back
    out_host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in srcs.values())
    d2h = out_host.numel() * out_host.element_size()
    del srcs
    KE = max(1, min(args.e2e_steps, K))
    eve = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(KE)]
    barrier()
    torch.cuda.synchronize()
    for i in range(KE):
        flush()
        eve[i][0].record()
        dev_in.copy_(host_in, non_blocking=True)
        step()
        out_host.copy_(out, non_blocking=True)
        eve[i][1].record()
    torch.cuda.synchronize()
    barrier()
    e2e_ms = sum(e[0].elapsed_time(e[1]) for e in eve) / KE

    swap = None
    if args.swap_frac > 0:
        swap = time_swap(pool, w, args.swap_frac, flush, K, dev)

    step_bytes = w.step_bytes() if q8 is None else q8.step_bytes(w)
    att_bytes = w.attention_bytes() if q8 is None else q8.attention_bytes(w)
    kv_bytes = w.kv_bytes() if q8 is None else q8.kv_bytes(w)
    max_step_ms, total_bytes = reduce_max_sum(step_ms, step_bytes)
    max_e2e_ms, _ = reduce_max_sum(e2e_ms, step_bytes)
    max_dec_ms, _ = reduce_max_sum(dec_ms, att_bytes)
    total_seqs = w.batch * world
    value = total_bytes / (max_step_ms * 1e-3) / 1e9
    peak, peak_kind = measured_hbm_peak()
    # A cascade decode reads each shared block once per group: its algorithmic
    # bytes count the stored (unique) K/V, not the logical per-sequence K/V.
    roof_bytes = att_bytes
    if cascade and "unique_tokens" in w.info:
        row = w.num_kv_heads * w.head_dim * w.elem_bytes * 2 if q8 is None else q8.row_bytes(w)
        roof_bytes = att_bytes - kv_bytes + int(w.info["unique_tokens"]) * row
    achieved = roof_bytes / (dec_ms * 1e-3) / 1e9

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host_w = wl.on_host(w)
        hq8 = None if q8 is None else q8_on_host(q8)
        threads = os.cpu_count() or 1
        seqs = pick_sample(host_w, 10.0, threads, hq8)
        dt, nb, passes = 0.0, 0, 0
        while passes < 3 or dt < 5.0:                   # a few seconds of CPU work at least
            t, b = oracle_sample_step(host_w, seqs, threads, hq8)
            dt, nb, passes = dt + t, nb + b, passes + 1
        # the same on one core (a smaller sample of the same step)
        seqs1 = pick_sample(host_w, 2.0, 1, hq8)
        dt1, nb1, passes1 = 0.0, 0, 0
        while passes1 < 2 or dt1 < 3.0:
            t, b = oracle_sample_step(host_w, seqs1, 1, hq8)
            dt1, nb1, passes1 = dt1 + t, nb1 + b, passes1 + 1
        cpu = {"value": round(nb / dt / 1e9, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
               "cpu_model": cpu_model(),
               "sample": f"{len(seqs)} of {w.batch} sequences of the same step (copy + append + "
                         f"attention, fp64 C oracle, threaded over sequences), {passes} passes, "
                         f"{dt:.1f} s",
               "single_thread": {"value": round(nb1 / dt1 / 1e9, 4), "unit": UNIT, "cores": 1,
                                 "sample": f"{len(seqs1)} of {w.batch} sequences, {passes1} "
                                           f"passes, {dt1:.1f} s"}}

    pool.close()
    if rank != 0:
        return None
    return {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(max_step_ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype if q8 is None else f"{q8.cache} storage, f16 MMA, fp32 softmax",
        "data": "synthetic",
        "config": decode_config(args, w, q8, world),
        "seq_steps_per_s": round(total_seqs / (max_step_ms * 1e-3), 1),
        **unique_bytes_fields(w, world, max_dec_ms, q8),
        "attention_gbs": round(att_bytes * world / (max_dec_ms * 1e-3) / 1e9, 2),
        "roofline": {"bound": "hbm",
                     "kernel": ("paged_decode_prefix + paged_decode_split (+ paged_decode_merge) (the whole cascade decode call)"
                                if cascade else
                                "paged_decode_split (+ paged_decode_merge) (the whole decode call)"),
                     "achieved": round(achieved, 2), "peak": peak, "unit": UNIT,
                     "frac": round(achieved / peak, 4), "peak_kind": f"of {peak_kind}",
                     "traffic": (profiled_traffic("paged_decode_split/llama3_8b_gqa/"
                                                  + ("fp8_e4m3" if q8 is not None else "bf16"),
                                                  DECODE_SOURCE)
                                 if (not cascade and (q8 is None or q8.cache == "fp8_e4m3")
                                     and args.workload == "llama3_8b_gqa"
                                     and args.batch is None and args.seed == 0
                                     and args.placement == "random") else None),
                     "traffic_unit": "bytes per launch (DRAM read + write, ncu)",
                     "algorithmic_bytes": roof_bytes},
        "e2e": {"value": round(total_bytes / (max_e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
                "ms_per_step": round(max_e2e_ms, 5), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "clocks": clocks,
        **({"swap": swap} if swap is not None else {}),
        "gpu_launches": launches_per_step * K,
        "cpu_baseline": cpu,
    }


# ------------------------------------------------------- chunked prefill --

def measured_tensor_peak():
    """Dense bf16 tensor peak: the burst figure (a kernel timed alone)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def oracle_prefill_sample(host_w, reqs, threads):
    """One oracle prefill step (append + attention) restricted to requests
    `reqs`; returns (seconds, algorithmic flops of the sample)."""
    import numpy as np
    from oracle import c_oracle
    cu = host_w.cu_seqlens.astype(np.int64)
    rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in reqs])
    sub_cu = np.concatenate([[0], np.cumsum([cu[b + 1] - cu[b] for b in reqs])]).astype(np.int32)
    k, v = host_w.k_pool, host_w.v_pool          # appends are idempotent
    t0 = time.perf_counter()
    c_oracle.append(k, v, host_w.k_new[rows], host_w.v_new[rows], host_w.slot_mapping[rows],
                    host_w.dtype)
    c_oracle.prefill(np.ascontiguousarray(host_w.q[rows]), k, v, host_w.dtype, sub_cu,
                     np.ascontiguousarray(host_w.block_tables[reqs]),
                     np.ascontiguousarray(host_w.seq_lens[reqs]), host_w.scale,
                     host_w.num_kv_heads, num_threads=threads)
    dt = time.perf_counter() - t0
    sub = copy.copy(host_w)
    sub.cu_seqlens, sub.seq_lens = sub_cu, host_w.seq_lens[reqs]
    return dt, sub.attention_flops()


def pick_prefill_sample(host_w, budget_s, threads):
    """Requests (a prefix of a fixed shuffle) whose oracle step takes about budget_s."""
    import numpy as np
    order = np.random.default_rng(1234).permutation(host_w.batch)
    n = 1
    dt, _ = oracle_prefill_sample(host_w, order[:n], threads)
    if dt < budget_s and n < host_w.batch:
        n = int(min(host_w.batch, max(n, n * budget_s / max(dt, 1e-3))))
    return np.sort(order[:n])


def run_prefill(args):
    """kv_append of the chunks -> paged_attention_prefill, inputs resident in
    HBM; the roofline is the tensor pipe (algorithmic QK and PV flops)."""
    import numpy as np
    import torch

    from paged_kv_cache_68_gb300 import pagedkv
    from paged_kv_cache_68_gb300 import workloads as wl

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pagedkv.load()
    w = make_workload(args.workload, args.seed, dev, batch=args.batch, decodes=args.decodes,
                      chunk=args.chunk)
    tv = lambda a: wl.value_to_torch(a, w.dtype, dev)
    srcs = {"q": tv(w.q), "k_new": tv(w.k_new), "v_new": tv(w.v_new),
            "slots": torch.from_numpy(w.slot_mapping).to(dev),
            "tables": torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(dev),
            "lens": torch.from_numpy(w.seq_lens).to(dev),
            "cu": torch.from_numpy(np.ascontiguousarray(w.cu_seqlens, dtype=np.int32)).to(dev)}
    offs, total = {}, 0
    for n, t in srcs.items():
        offs[n] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    dev_in = torch.empty(total, dtype=torch.uint8, device=dev)
    view = {}
    for n, t in srcs.items():
        nb = t.numel() * t.element_size()
        view[n] = dev_in[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)
        view[n].copy_(t)
    host_in = dev_in.cpu().pin_memory()
    q8 = None
    if args.kv_cache:
        # the same rows as 8-bit codes (the 16-bit pools are not used)
        q8 = wl.q8_pools(w, args.kv_cache, args.seed)
        w.k_pool = w.v_pool = None
        torch.cuda.empty_cache()
        pool = pagedkv.KVPool(q8.k_codes, q8.v_codes, cache=q8.cache, dtype=view["q"].dtype,
                              k_scales=q8.k_scales, v_scales=q8.v_scales, k_scale=q8.k_scale,
                              v_scale=q8.v_scale)
    else:
        pool = pagedkv.KVPool(w.k_pool, w.v_pool)
    out = torch.empty_like(view["q"])
    maxq = int(np.diff(w.cu_seqlens).max())

    def append():
        pool.append(view["k_new"], view["v_new"], view["slots"])

    def prefill():
        pool.prefill(view["q"], view["cu"], maxq, view["tables"], view["lens"], w.scale, out=out)

    flush = L2Flush(dev)
    for _ in range(max(3, args.warmup)):
        flush()
        append()
        prefill()
    torch.cuda.synchronize()
    assert pool.get_error() == 0, "device error word set during warm-up"
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(gpu_uuid(dev))
    barrier()
    torch.cuda.synchronize()
    sampler.begin()
    for i in range(K):
        flush()                                   # L2 flush, outside the events
        e = ev[i]
        e[0].record()
        append()
        e[1].record()
        prefill()
        e[2].record()
    sampler.mark()
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    step_ms = sum(e[0].elapsed_time(e[2]) for e in ev) / K
    pf_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    assert pool.get_error() == 0, "device error word set during the timed steps"

    out_host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    KE = max(1, min(args.e2e_steps, K))
    eve = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(KE)]
    barrier()
    torch.cuda.synchronize()
    for i in range(KE):
        flush()
        eve[i][0].record()
        dev_in.copy_(host_in, non_blocking=True)
        append()
        prefill()
        out_host.copy_(out, non_blocking=True)
        eve[i][1].record()
    torch.cuda.synchronize()
    barrier()
    e2e_ms = sum(e[0].elapsed_time(e[1]) for e in eve) / KE

    flops = w.attention_flops()
    max_step_ms, total_flops = reduce_max_sum(step_ms, flops)
    max_pf_ms, _ = reduce_max_sum(pf_ms, flops)
    max_e2e_ms, _ = reduce_max_sum(e2e_ms, flops)
    qtok = int(w.info["query_tokens"]) * world
    peak, peak_kind = measured_tensor_peak()
    achieved = flops / (pf_ms * 1e-3) / 1e12

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and q8 is None:
        host_w = wl.on_host(w)
        threads = os.cpu_count() or 1
        reqs = pick_prefill_sample(host_w, 10.0, threads)
        dt, fl, passes = 0.0, 0, 0
        while passes < 2 or dt < 5.0:
            t, f = oracle_prefill_sample(host_w, reqs, threads)
            dt, fl, passes = dt + t, fl + f, passes + 1
        cpu = {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
               "kind": "oracle",
               "sample": f"{len(reqs)} of {w.batch} requests of the same step (append + causal "
                         f"prefill attention, fp64 C oracle), {passes} passes, {dt:.1f} s"}
    pool.close()
    if rank != 0:
        return None
    return {
        "metric": PREFILL_METRIC, "value": round(total_flops / (max_step_ms * 1e-3) / 1e12, 2),
        "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(max_step_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype if q8 is None else f"{q8.cache} storage, {w.dtype} MMA, fp32 softmax",
        "data": "synthetic",
        "config": {**prefill_config(args, w, world, flops),
                   "kv_cache": w.dtype if q8 is None else q8.cache},
        "query_tokens_per_s": round(qtok / (max_step_ms * 1e-3), 1),
        "attention_tflops": round(total_flops / (max_pf_ms * 1e-3) / 1e12, 2),
        "roofline": {"bound": "tensor",
                     "kernel": "paged_prefill (tcgen05; the whole prefill call, one kernel)",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"of {peak_kind} (bf16 burst)",
                     "traffic": (profiled_traffic("paged_prefill/chunked_prefill/bf16", PREFILL_SOURCE)
                                 if args.batch is None and args.chunk is None and not args.decodes
                                 and args.seed == 0 and q8 is None else None),
                     "traffic_unit": "bytes per launch (DRAM read + write, ncu)",
                     "algorithmic_flops": flops},
        "e2e": {"value": round(total_flops / (max_e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(max_e2e_ms, 5),
                "h2d_bytes_per_step": int(host_in.numel()),
                "d2h_bytes_per_step": int(out_host.numel() * out_host.element_size())},
        "clocks": clocks,
        "gpu_launches": 2 * K,
        "cpu_baseline": cpu,
    }


def run_prefill_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return None
    import torch

    from oracle import c_oracle
    from paged_kv_cache_68_gb300 import workloads as wl
    c_oracle.build()
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else None
    w = wl.on_host(make_workload(args.workload, args.seed, dev, batch=args.batch,
                                 decodes=args.decodes, chunk=args.chunk))
    threads = os.cpu_count() or 1
    per_step = max(0.05, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    reqs = pick_prefill_sample(w, per_step, threads)
    for _ in range(args.warmup):
        oracle_prefill_sample(w, reqs, threads)
    tot_t, tot_f = 0.0, 0
    for _ in range(args.steps):
        dt, f = oracle_prefill_sample(w, reqs, threads)
        tot_t, tot_f = tot_t + dt, tot_f + f
    value = tot_f / tot_t / 1e12
    sample = (f"{len(reqs)} of {w.batch} requests per step (append + causal prefill attention, "
              f"fp64 C oracle), {args.steps} steps")
    return {
        "impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 6),
        "unit": "TFLOP/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(tot_t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": prefill_config(args, w, int(os.environ.get("WORLD_SIZE", "1")),
                                 w.attention_flops()),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads,
                         "cpu_model": cpu_model(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# -------------------------------------------------------- reference arm --

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import torch

    from oracle import c_oracle
    from paged_kv_cache_68_gb300 import workloads as wl
    c_oracle.build()
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else None
    wd = make_workload(args.workload, args.seed, dev, args.placement, args.batch,
                       args.block_size, args.prompt_len, fresh_fork=args.fresh_fork)
    q8 = None if not args.kv_cache else q8_on_host(wl.q8_pools(wd, args.kv_cache, args.seed))
    w = wl.on_host(wd)
    del wd
    threads = os.cpu_count() or 1
    per_step = max(0.05, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    seqs = pick_sample(w, per_step, threads, q8)
    for _ in range(args.warmup):
        oracle_sample_step(w, seqs, threads, q8)
    tot_t, tot_b = 0.0, 0
    for _ in range(args.steps):
        dt, nb = oracle_sample_step(w, seqs, threads, q8)
        tot_t += dt
        tot_b += nb
    value = tot_b / tot_t / 1e9
    ms = tot_t / args.steps * 1e3
    sample = (f"{len(seqs)} of {w.batch} sequences per step (copy + append + attention, "
              f"fp64 C oracle), {args.steps} steps")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": decode_config(args, w, q8, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "cpu_model": cpu_model(), "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    if args.workload == "chunked_prefill":
        res = run_prefill_reference(args) if args.impl == "reference" else run_prefill(args)
    else:
        res = run_reference(args) if args.impl == "reference" else run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
