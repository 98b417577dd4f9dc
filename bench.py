"""Benchmark of the ring-attention forward pass (one JSON line on stdout).

A step is one ``ra_ring_attention`` call: the whole chunk walk (stats, merges,
normalisation) over one batch of synthetic inputs resident in HBM. Default
workload: bf16, 8 heads, 8192 queries = 8192 keys, head_dim 128, non-causal,
8 contiguous chunks of 1024 walked in ring order by 8 query segments.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--layout contiguous|zigzag|striped] [--impl reference]

N > 1 (under torchrun): every rank runs its own replica of the workload on its
own GPU (the path shards by query segment with no data exchange on one box);
the time is the max over ranks and the value counts every rank's work.
``--impl reference`` times the fp64 CPU oracle instead, on a bounded row
sample of the same workload, on this machine's host cores.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ring_attention fwd TFLOP/s (bf16, causal-adjusted) and % of GB300 tensor peak"
L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2
E2E_STREAMS = 3


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), \
            float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


def _pinned_block(tensors, copy=True):
    """Host tensors shaped like `tensors`, back to back in one pinned buffer
    (holding copies of their values when `copy`)."""
    import torch
    sizes = [t.numel() * t.element_size() for t in tensors]
    buf = torch.empty(sum(sizes), dtype=torch.uint8, pin_memory=True)
    views, at = [], 0
    for t, n in zip(tensors, sizes):
        v = buf[at:at + n].view(t.dtype).view(t.shape)
        if copy:
            v.copy_(t.cpu())
        views.append(v)
        at += n
    return views


def _traffic(kernel_key):
    """DRAM bytes per launch from a committed ncu summary, valid only while the
    kernel's sources are unchanged (their hash is stored next to the counters)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            tab = json.load(f)
        ent = tab[kernel_key]
        srcs = ent["source"] if isinstance(ent["source"], list) else [ent["source"]]
        h = hashlib.sha256()
        for name in srcs:
            with open(os.path.join(ROOT, "blockwise_attention_online_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        return int(ent["bytes_per_launch"]) if h.hexdigest()[:16] == ent["source_sha"] else None
    except Exception:
        return None


_REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class _Nvml:
    """The few NVML reads the clock record needs (read-only; nothing is set)."""

    def __init__(self, cuda_index):
        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        ok = False
        uuid = getattr(torch.cuda.get_device_properties(cuda_index), "uuid", None)
        if uuid is not None:
            for name in (f"GPU-{uuid}", str(uuid)):
                if lib.nvmlDeviceGetHandleByUUID(name.encode(), ctypes.byref(self.h)) == 0:
                    ok = True
                    break
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle for the device")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint()
        lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
        self.max_mhz = float(mx.value)

    def sample(self):
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) != 0:
            return None
        if self.reasons_fn(self.h, ctypes.byref(rs)) != 0:
            rs.value = 0
        return float(mhz.value), int(rs.value)


class ClockSampler:
    """SM clock and clock-event reasons sampled while a timed region runs:
    NVML read every quarter millisecond from a helper thread (so that a region
    of a few milliseconds still gets a dozen samples), else nvidia-smi every
    10 ms."""

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.source = None

    def __enter__(self):
        import threading
        self.samples = []
        self._stop = threading.Event()
        self.proc = None
        try:
            self.nv = _Nvml(self.index)
            self.source = "nvml, 0.25 ms"

            def loop():
                while not self._stop.is_set():
                    s = self.nv.sample()
                    if s is not None:
                        self.samples.append(s)
                    time.sleep(0.00025)

            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
        except Exception:
            self.nv = None
            self.source = "nvidia-smi, 10 ms"
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.index}",
                     "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "10"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception:
                self.proc = None
        return self

    def __exit__(self, *exc):
        if self.nv is not None:
            self._stop.set()
            self.thread.join(timeout=2)
            self.max_mhz = self.nv.max_mhz
            return
        self.max_mhz = None
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            for line in (out or "").splitlines():
                f = [x.strip() for x in line.split(",")]
                try:
                    self.samples.append((float(f[0]), int(f[2], 16)))
                    self.max_mhz = float(f[1])
                except (ValueError, IndexError):
                    continue

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": self.source}
        reasons = set()
        for _, bits in self.samples:
            for b, name in _REASON_BITS.items():
                if bits & b:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(m for m, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(self.samples), "source": self.source}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of ``x`` over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Work of every rank divided by the slowest rank's time."""
    return flops_per_step * steps * world / (max_ms * 1e-3) / 1e12


def build_workload(name, layout, device):
    import torch
    from blockwise_attention_online_gb300 import layouts, workloads
    w = workloads.WORKLOADS[name]
    if layout:
        w = workloads.Workload(**{**w.__dict__, "layout": layout})
    q, k, v = workloads.make_qkv(w, device=device)
    P = w.n_chunks
    rs = layouts.rank_spans(w.layout, w.S, P)
    kc = layouts.shard(k, w.layout, P)
    vc = layouts.shard(v, w.layout, P)
    qs = torch.cat(layouts.shard(q, w.layout, P), dim=2).contiguous()
    del q, k, v
    segs = [(w.S // P, s) for s in rs]
    return w, qs, kc, vc, rs, segs


def _docs(w, mean_len):
    """Packed documents for --docs: seeded boundaries over the workload's
    positions, and the algorithmic FLOPs of one forward with them (exact
    visible pairs: n^2 per document of n positions, n(n+1)/2 when causal)."""
    from blockwise_attention_online_gb300 import workloads
    if not mean_len:
        return None, w.flops()
    b = workloads.packed_documents(w.S, w.seed, mean_len)
    pairs = 0
    for a, z in zip(b[:-1], b[1:]):
        n = z - a
        pairs += n * (n + 1) // 2 if w.causal else n * n
    return b, 4.0 * w.B * w.Hq * w.D * pairs


def run_gpu(args):
    import torch
    import torch.distributed as dist
    from blockwise_attention_online_gb300 import device_status, ring_attention

    world, rank, local = _dist()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    w, qs, kc, vc, rs, segs = build_workload(args.workload, args.layout, dev)
    docs, flops = _docs(w, args.docs)
    out = torch.empty_like(qs)
    m = torch.empty(qs.shape[:3], device=dev, dtype=torch.float32)
    l = torch.empty_like(m)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream()

    def step():
        ring_attention(qs, kc, vc, chunk_spans=rs, q_segments=segs, causal=w.causal,
                       out=out, m=m, l=l, docs=docs)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    device_status()

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # K steps, each after an L2 flush, timed with CUDA events on the stream
    times, clocks = _timed(step, args.steps, 0, flush, stream, dev.index)  # ms per launch
    if world > 1:
        dist.barrier()
    device_status()
    total_ms = sum(times)
    max_ms = max_over_ranks(total_ms, dev)
    value = whole_job_tflops(flops, args.steps, world, max_ms)

    # End to end through the host-buffer entry point: every step copies that
    # step's inputs from pinned host memory to the device, runs the ring pass
    # and copies O, m, l back. Steps rotate over three streams, so that one
    # step's input copies run while another step's kernel runs and a third
    # step's outputs come back (copies in the two directions use separate copy
    # engines; each call has its own device buffers).
    e2e = None
    if not args.no_e2e:
        from blockwise_attention_online_gb300 import ring_attention_host
        # inputs in one pinned buffer (q, the k chunks, the v chunks) and each
        # stream's outputs in another (O, m, l): the library copies each
        # buffer's adjacent tensors with one copy
        hq, *hkv = _pinned_block([qs, *kc, *vc])
        hk, hv = hkv[:len(kc)], hkv[len(kc):]
        ns = args.e2e_streams
        outs = [tuple(_pinned_block([out, m, l], copy=False)) for _ in range(ns)]
        h2d = hq.numel() * hq.element_size() + sum(x.numel() * x.element_size() for x in hk + hv)
        d2h = sum(t.numel() * t.element_size() for t in outs[0])
        n_e2e = max(3, min(args.steps, 100))
        streams = [torch.cuda.Stream(device=dev) for _ in range(ns)]

        def e2e_step(i):
            ho, hm, hl = outs[i % ns]
            ring_attention_host(hq, hk, hv, chunk_spans=rs, q_segments=segs, causal=w.causal,
                                out=ho, m=hm, l=hl, docs=docs, stream=streams[i % ns])

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for i in range(n_e2e):
            e2e_step(i)
        torch.cuda.synchronize()
        el = max_over_ranks(time.perf_counter() - t0, dev)
        e2e = {"value": round(whole_job_tflops(flops, n_e2e, world, el * 1e3), 3),
               "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": n_e2e, "streams": ns,
               "call": "ra_ring_attention_host (pinned host buffers)"}
        device_status()

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return None

    peak_b, peak_s, hbm, src = _peaks()
    mean_ms = total_ms / args.steps
    achieved = flops / (mean_ms * 1e-3) / 1e12
    kernel_key = f"tc_ring_kernel:{w.name}:{w.layout}" + (f":docs{args.docs}" if docs else "")
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_ms / args.steps, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) Q/K/V (bf16), no dataset",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S,
                   "D": w.D, "causal": w.causal, "chunks": w.n_chunks, "layout": w.layout,
                   "ring_order": "segment r visits chunks r, r-1, ...",
                   "flops_per_step": flops,
                   "docs": ({"mean_len": args.docs, "n_docs": len(docs) - 1,
                             "recipe": "workloads.packed_documents(S, seed, mean_len)"}
                            if docs else None),
                   "l2": f"flushed before every step ({L2_FLUSH_BYTES >> 20} MiB write)",
                   "timing": "CUDA events around each step on the launching stream; untimed "
                             "device work queued before the first step, so that its host "
                             "planning does not leave the device idle inside its events",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "pct_of_peak": round(100 * value / world / peak_b, 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak_b,
                     "unit": "TFLOP/s", "frac": round(achieved / peak_b, 4),
                     "traffic": _traffic(kernel_key), "kernel": "tc_ring_kernel<128>",
                     "peak_source": f"{src} bf16 burst (MEASURED_PEAKS.json)" if src == "measured"
                     else "fallback 1.9 PFLOP/s"},
        "clocks": clocks,
        "gpu_launches": args.steps,
        "e2e": e2e,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, docs)
    if not args.no_secondary and world == 1 and args.workload == "bf16_8k" and not docs:
        del qs, kc, vc, out, m, l
        torch.cuda.empty_cache()
        line["secondary"] = secondary_records(dev, flush)
    return line


def _timed(step, steps, warmup, flush, stream, index):
    """Runs ``warmup`` untimed steps, then ``steps`` steps each preceded by an
    L2 flush; returns the CUDA-event time of every step (ms, on ``stream``) and
    the clock record of the timed region."""
    import torch
    for _ in range(warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with ClockSampler(index) as clk:
        # untimed device work queued first, so that the host's preparation of
        # the first step (planning, before its launch) overlaps it instead of
        # leaving the device idle between that step's start event and kernel
        for _ in range(4):
            flush.fill_(0.5)
        for i in range(steps):
            flush.fill_(float(i & 7))
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)], clk.summary()


def _imbalance(w, rs, segs):
    """Per virtual rank (query segment): visible (query, key) pairs and the
    128x128 tile products the kernel schedules; max/mean of each (1.0 is a
    perfect balance)."""
    from blockwise_attention_online_gb300 import segment_work
    lens = [w.S // w.n_chunks] * w.n_chunks
    pairs, tiles = segment_work(w.B, w.Hq, w.Hkv, w.D, segs, lens, rs, w.causal)
    mp, mt = sum(pairs) / len(pairs), sum(tiles) / len(tiles)
    return {"pairs_max_over_mean": round(max(pairs) / mp, 4),
            "tiles_max_over_mean": round(max(tiles) / mt, 4),
            "pairs_per_rank": pairs, "tiles_per_rank": tiles}


def secondary_records(dev, flush, steps_small=5):
    """Further workloads, timed the same way as the headline (L2 flushed per
    step, CUDA events on the launching stream, clocks sampled): the other
    configurations of the forward (with the per-virtual-rank work imbalance of
    each layout), the backward, and the HBM-bound merge kernels."""
    import torch
    from blockwise_attention_online_gb300 import (device_status, merge_lse, merge_stats,
                                                  ring_attention, ring_attention_bwd,
                                                  stats_to_lse)
    peak_b, _, hbm, _ = _peaks()
    stream = torch.cuda.current_stream()
    out = {"forward": [], "backward": [], "hbm_kernels": []}
    # backward of the headline workload, first: like the headline it is timed
    # before the long causal records below heat the GPU to its power cap
    w, qs, kc, vc, rs, segs = build_workload("bf16_8k", None, dev)
    O, m, l = ring_attention(qs, kc, vc, chunk_spans=rs, q_segments=segs, causal=w.causal)
    g = torch.Generator(device=dev).manual_seed(99)
    dout = torch.randn(qs.shape, device=dev, generator=g).to(torch.bfloat16)
    dq = torch.empty(qs.shape, device=dev, dtype=torch.float32)
    dk = [torch.empty(k.shape, device=dev, dtype=torch.float32) for k in kc]
    dv = [torch.empty(v.shape, device=dev, dtype=torch.float32) for v in vc]

    def bstep():
        ring_attention_bwd(qs, kc, vc, O, dout, m, l, chunk_spans=rs, q_segments=segs,
                           causal=w.causal, dq=dq, dk=dk, dv=dv)

    times, clk = _timed(bstep, 20, 3, flush, stream, dev.index)
    device_status()
    ms = sum(times) / len(times)
    tf = 2.5 * w.flops() / (ms * 1e-3) / 1e12
    out["backward"].append({"workload": w.name, "layout": w.layout, "steps": 20, "warmup": 3,
                            "flops_per_step": 2.5 * w.flops(), "ms_per_step": round(ms, 4),
                            "tflops": round(tf, 2), "frac_of_peak": round(tf / peak_b, 4),
                            "clocks": clk})
    del qs, kc, vc, O, m, l, dout, dq, dk, dv
    torch.cuda.empty_cache()
    cases = [("bf16_32k_causal", None, steps_small), ("bf16_128k_gqa_causal", "zigzag", steps_small),
             ("bf16_128k_gqa_causal", "contiguous", steps_small),
             ("bf16_128k_gqa_causal", "striped", steps_small), ("bf16_1m_causal", None, 2)]
    for name, layout, n in cases:
        w, qs, kc, vc, rs, segs = build_workload(name, layout, dev)
        o = torch.empty_like(qs)
        m = torch.empty(qs.shape[:3], device=dev, dtype=torch.float32)
        l = torch.empty_like(m)

        def step():
            ring_attention(qs, kc, vc, chunk_spans=rs, q_segments=segs, causal=w.causal,
                           out=o, m=m, l=l)

        times, clk = _timed(step, n, 3, flush, stream, dev.index)
        device_status()
        ms = sum(times) / len(times)
        tf = w.flops() / (ms * 1e-3) / 1e12
        out["forward"].append({"workload": w.name, "layout": w.layout, "S": w.S, "Hq": w.Hq,
                               "Hkv": w.Hkv, "causal": w.causal, "chunks": w.n_chunks,
                               "steps": n, "warmup": 3, "ms_per_step": round(ms, 4),
                               "tflops": round(tf, 2), "frac_of_peak": round(tf / peak_b, 4),
                               "imbalance": _imbalance(w, rs, segs), "clocks": clk})
        del qs, kc, vc, o, m, l
        torch.cuda.empty_cache()
    out["hbm_kernels"] = hbm_kernel_records(dev, flush, 32 * 32768, 20)
    return out


def hbm_kernel_records(dev, flush, rows, steps, D=128):
    """The HBM-bound kernels, each timed over ``steps`` launches between L2
    flushes: the statistics merge (ra_merge_stats), its log-sum-exp form
    (ra_merge_lse) and ra_stats_to_lse, on ``rows`` rows of head_dim ``D``
    (default: the rows of the 32K causal workload, 32 heads x 32768).
    Algorithmic bytes per row: the merge reads both sides' u, l, m and writes
    the accumulator's, 3 (4D + 8); the lse merge 3 (4D + 4); stats_to_lse
    reads m, l and writes lse, 12."""
    import torch
    from blockwise_attention_online_gb300 import device_status, merge_lse, merge_stats, stats_to_lse
    _, _, hbm, _ = _peaks()
    stream = torch.cuda.current_stream()
    g = torch.Generator(device=dev).manual_seed(7)
    u_a = torch.randn(rows, D, device=dev, generator=g)
    u_b = torch.randn(rows, D, device=dev, generator=g)
    l_a = torch.rand(rows, device=dev, generator=g) + 1
    l_b = torch.rand(rows, device=dev, generator=g) + 1
    m_a = torch.randn(rows, device=dev, generator=g)
    m_b = torch.randn(rows, device=dev, generator=g)
    kern = [("ra_merge_stats", "merge_vec4_kernel",
             lambda: merge_stats(u_a, l_a, m_a, u_b, l_b, m_b), 3 * (4 * D + 8)),
            ("ra_merge_lse", "merge_lse_kernel",
             lambda: merge_lse(u_a, m_a, u_b, m_b), 3 * (4 * D + 4)),
            ("ra_stats_to_lse", "stats_to_lse_kernel",
             lambda: stats_to_lse(m_a, l_a, l_b), 12)]
    recs = []
    for call, kname, fn, bpr in kern:
        times, clk = _timed(fn, steps, 3, flush, stream, dev.index)
        device_status()
        ms = sum(times) / len(times)
        gbs = rows * bpr / (ms * 1e-3) / 1e9
        recs.append({"call": call, "kernel": kname, "rows": rows, "D": D,
                     "bytes_per_row": bpr, "bytes_per_launch": rows * bpr,
                     "ms_per_launch": round(ms, 5), "gbs": round(gbs, 1),
                     "peak_gbs": hbm, "frac_of_peak": round(gbs / hbm, 4),
                     "steps": steps, "warmup": 3, "clocks": clk})
    return recs


def run_gpu_merge(args):
    """--pass merge: only the HBM-bound kernels (one JSON line)."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev, dtype=torch.float32)
    recs = hbm_kernel_records(dev, flush, args.rows, args.steps)
    head = recs[0]
    return {"metric": "ra_merge_stats achieved HBM GB/s", "value": head["gbs"], "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": 3,
            "ms_per_step": head["ms_per_launch"], "higher_is_better": True, "dtype": "f32",
            "data": "synthetic: seeded fp32 statistics", "config": {"workload": "merge",
                                                                    "rows": args.rows, "D": 128},
            "roofline": {"bound": "hbm", "achieved": head["gbs"], "peak": head["peak_gbs"],
                         "unit": "GB/s", "frac": head["frac_of_peak"], "traffic": None,
                         "kernel": head["kernel"]},
            "kernels": recs, "gpu_launches": 3 * args.steps}


def run_gpu_bwd(args):
    """The backward pass of the same workload: one step = ra_ring_attention_bwd
    (two preparation kernels, then one grid of dK/dV and dQ CTAs) on the
    forward's O, m, l and a seeded dO. FLOPs count the standard five products
    of the backward (2.5 x the forward's), causal-adjusted like the forward;
    the design executes seven (S and dP are recomputed by both kinds of CTA)."""
    import torch
    from blockwise_attention_online_gb300 import device_status, ring_attention, ring_attention_bwd

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    w, qs, kc, vc, rs, segs = build_workload(args.workload, args.layout, dev)
    flops = 2.5 * w.flops()
    O, m, l = ring_attention(qs, kc, vc, chunk_spans=rs, q_segments=segs, causal=w.causal)
    g = torch.Generator(device=dev).manual_seed(99)
    dout = torch.randn(qs.shape, device=dev, generator=g).to(torch.bfloat16)
    dq = torch.empty(qs.shape, device=dev, dtype=torch.float32)
    dk = [torch.empty(k.shape, device=dev, dtype=torch.float32) for k in kc]
    dv = [torch.empty(v.shape, device=dev, dtype=torch.float32) for v in vc]
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream()

    def step():
        ring_attention_bwd(qs, kc, vc, O, dout, m, l, chunk_spans=rs, q_segments=segs,
                           causal=w.causal, dq=dq, dk=dk, dv=dv)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    device_status()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    times, clocks = _timed(step, args.steps, 0, flush, stream, dev.index)
    if world > 1:
        dist.barrier()
    device_status()
    total_ms = sum(times)
    max_ms = max_over_ranks(total_ms, dev)
    value = whole_job_tflops(flops, args.steps, world, max_ms)
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return None
    peak_b, _, _, src = _peaks()
    achieved = flops / (total_ms / args.steps * 1e-3) / 1e12
    line = {
        "metric": "ring_attention bwd TFLOP/s (bf16, causal-adjusted, 2.5x the forward's FLOPs)",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) Q/K/V and dO (bf16), no dataset",
        "config": {"workload": w.name, "pass": "backward", "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv,
                   "S": w.S, "D": w.D, "causal": w.causal, "chunks": w.n_chunks,
                   "layout": w.layout, "flops_per_step": flops,
                   "l2": f"flushed before every step ({L2_FLUSH_BYTES >> 20} MiB write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "pct_of_peak": round(100 * value / world / peak_b, 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak_b,
                     "unit": "TFLOP/s", "frac": round(achieved / peak_b, 4), "traffic": None,
                     "kernel": "bwd_kernel<128> (dK/dV and dQ CTAs, one step)",
                     "peak_source": f"{src} bf16 burst (MEASURED_PEAKS.json)"},
        "clocks": clocks,
        "gpu_launches": 3 * args.steps,
        "e2e": None,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline_bwd(w, args.cpu_seconds)
    return line


def cpu_baseline_bwd(w, seconds):
    """The backward oracle timed on a bounded sample: the first query rows of
    head 0 against all keys (their dQ exactly, their share of dK and dV)."""
    import numpy as np
    import oracle
    from blockwise_attention_online_gb300 import workloads
    q, k, v = workloads.make_qkv(w, device="cpu")
    rng = np.random.default_rng(7)
    rows = 64
    done_flops, t0, n = 0.0, time.perf_counter(), 0
    g = w.Hq // w.Hkv
    while time.perf_counter() - t0 < seconds:
        r0 = int(rng.integers(0, max(1, w.S - rows)))
        qs = q[:, :1, r0:r0 + rows].double().numpy()
        ks = k[:, :1].double().numpy()
        vs = v[:, :1].double().numpy()
        do = rng.standard_normal(qs.shape)
        pos_q, pos_k = np.arange(r0, r0 + rows), np.arange(w.S)
        oracle.attention_backward(qs, ks, vs, do, pos_q, pos_k, w.causal, w.D ** -0.5)
        keys = np.minimum(pos_q + 1, w.S).sum() if w.causal else rows * w.S
        done_flops += 10.0 * keys * w.D
        n += 1
    el = time.perf_counter() - t0
    return {"value": round(done_flops / el / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle", "sample": f"{n} blocks of {rows} query rows of head 0 against all "
                                        f"keys (group {g}), {el:.1f} s"}


def _oracle_sample(w, rows_per_head, seed=1234):
    import numpy as np
    from blockwise_attention_online_gb300 import workloads
    q, k, v = workloads.make_qkv(w, device="cpu")
    rng = np.random.default_rng(seed)
    heads = list(range(w.Hq))
    return q.float(), k.float(), v.float(), heads, rng


def _row_flops(w, i, docs=None):
    if docs is None:
        keys = (i + 1) if w.causal else w.S
    else:
        import bisect
        d = bisect.bisect_right(docs, i) - 1
        keys = (i + 1 - docs[d]) if w.causal else (docs[d + 1] - docs[d])
    return 4.0 * keys * w.D


def cpu_baseline(w, seconds, docs=None):
    """The fp64 oracle, as it stands, on a bounded sample of the workload's
    rows, timed on this machine's host cores."""
    import numpy as np
    import oracle
    q, k, v, heads, rng = _oracle_sample(w, 0)
    pos = np.arange(w.S)
    done_flops, rows_done, el = 0.0, 0, 0.0
    t0 = time.perf_counter()
    while el < seconds:
        rows = [(0, int(h), int(rng.integers(0, w.S))) for h in heads]
        oracle.attention_rows(q, k, v, pos, pos, w.causal, w.scale, rows, docs=docs)
        done_flops += sum(_row_flops(w, i, docs) for _, _, i in rows)
        rows_done += len(rows)
        el = time.perf_counter() - t0
    return {"value": round(done_flops / el / 1e12, 6), "unit": "TFLOP/s",
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{rows_done} random query rows (one per head per round) of {w.name}, "
                      f"each exact against all its visible keys, {el:.1f} s"}


def run_reference(args):
    """--impl reference: the fp64 oracle on the host cores, K timed steps, each
    a bounded row sample (one random row per query head) of the workload."""
    import numpy as np
    import oracle
    from blockwise_attention_online_gb300 import workloads
    world, rank, _ = _dist()
    if rank != 0:
        return None
    w = workloads.WORKLOADS[args.workload]
    docs, _ = _docs(w, args.docs)
    q, k, v, heads, rng = _oracle_sample(w, 0)
    pos = np.arange(w.S)

    def one():
        rows = [(0, int(h), int(rng.integers(0, w.S))) for h in heads]
        oracle.attention_rows(q, k, v, pos, pos, w.causal, w.scale, rows, docs=docs)
        return sum(_row_flops(w, i, docs) for _, _, i in rows)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    fl = 0.0
    for _ in range(args.steps):
        fl += one()
    el = time.perf_counter() - t0
    val = fl / el / 1e12
    sample = f"{len(heads)} random query rows per step (one per head) of {w.name}"
    return {"impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic: seeded N(0,1) Q/K/V (bf16 values upcast to f64)",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S,
                       "D": w.D, "causal": w.causal, "chunks": w.n_chunks,
                       "docs": {"mean_len": args.docs, "n_docs": len(docs) - 1} if docs else None},
            "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="bf16_8k")
    ap.add_argument("--layout", default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-streams", type=int, default=E2E_STREAMS,
                    help="streams the end-to-end steps rotate over")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the further records (other workloads, backward, merge kernels)")
    ap.add_argument("--rows", type=int, default=32 * 32768,
                    help="--pass merge: rows of the statistics (head_dim 128)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--docs", type=int, default=0,
                    help="pack the sequence into seeded documents of this mean length "
                         "(forward only; 0 = one document)")
    ap.add_argument("--pass", dest="which", default="fwd", choices=["fwd", "bwd", "merge"],
                    help="time the forward (default), the backward pass or the HBM-bound merge kernels")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        line = run_reference(args)
    elif args.which == "bwd":
        line = run_gpu_bwd(args)
    elif args.which == "merge":
        line = run_gpu_merge(args)
    else:
        line = run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
