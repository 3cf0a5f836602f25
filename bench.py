"""Benchmark of the quantized paged-KV attention path on GB300.

One step = one serving step over a batch: reshape_and_cache of the step's
new tokens (the last query_len tokens of every request) into the fp8 /
int8 paged cache, then attention_with_kv_cache over the whole cache (the
split-KV row-tile kernel, the split merge, and the tensor-core prefill
kernel where the batch has prefills).  The cache holding the earlier
context is written once before timing (state, not per-step input).

Headline workload (the line's `value`): the decode batch -- 64 requests,
query_len 1, kv_len ~ U[1024, 4096], 32 query heads over 8 kv heads,
head_dim 128, block 16, fp8_e4m3 per-tensor scales.  Metric: decode KV GB/s
= the K and V cache bytes the step's attention must read, divided by the
step time.  The same line carries one object per other workload under
"workloads" (the large prefill and the mixed batch in prefill TFLOP/s, the
long-context decode in GB/s), each with its roofline, CPU baseline and
clocks; the mixed batch also reports its prefill and decode parts timed
alone.

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload instead.  Under torchrun each rank
runs an independent replica (replicas only: the path has no exchange).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) per launch of the dominant kernel, from the ncu
# captures summarised in profiles/; valid only while the kernel's sources
# hash as they did when captured.
PROFILED_TRAFFIC = {
    # (workload, kv cache dtype, part of a mixed batch): DRAM bytes read +
    # written by that kernel in one launch, from the ncu capture in `profile`
    # (its "traffic" command; taken while the listed sources hashed to `sha1`).
    (2, "fp8_e4m3", None): {"bytes": 361.342976e6 + 4.596992e6,
                            "profile": "profiles/splitkv_decode_decode_batch.md",
                            "sources": ['kvq_decode.cuh', 'kvq_device.cuh', 'kvq_internal.h'], "sha1": "635463d3cff41345045b05fa4f50b3d17c1b7c78"},
    (5, "fp8_e5m2", None): {"bytes": 269.877760e6 + 4.454912e6,
                            "profile": "profiles/splitkv_decode_long_context.md",
                            "sources": ['kvq_decode.cuh', 'kvq_device.cuh', 'kvq_internal.h'], "sha1": "635463d3cff41345045b05fa4f50b3d17c1b7c78"},
    (4, "int8_per_token_head", "decode"): {"bytes": 484.951296e6 + 5.326592e6,
                                           "profile": "profiles/mixed_batch_int8_per_token_head.md",
                                           "sources": ['kvq_decode.cuh', 'kvq_device.cuh', 'kvq_internal.h'], "sha1": "635463d3cff41345045b05fa4f50b3d17c1b7c78"},
    (4, "int8_per_token_head", "prefill"): {"bytes": 379.163136e6 + 89.351680e6,
                                            "profile": "profiles/mixed_batch_int8_per_token_head.md",
                                            "sources": ['kvq_prefill.cuh', 'kvq_tcgen05.cuh', 'kvq_device.cuh', 'kvq_internal.h'], "sha1": "1960048207eeaf5dafb97e8a77909eb4819e45fe"},
    (3, "fp8_e4m3", None): {"bytes": 37.873152e6 + 0.326400e6,
                            "profile": "profiles/prefill_attention_large_prefill.md",
                            "sources": ['kvq_prefill.cuh', 'kvq_tcgen05.cuh', 'kvq_device.cuh', 'kvq_internal.h'], "sha1": "1960048207eeaf5dafb97e8a77909eb4819e45fe"},
}


def profiled_traffic(workload: int, dtype: str, part=None):
    """The captured DRAM traffic of this workload's dominant kernel (or of
    one part of a mixed batch), or None when there is no capture or the
    kernel changed since."""
    entry = PROFILED_TRAFFIC.get((workload, dtype, part))
    if entry is None:
        return None
    m = hashlib.sha1()
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "int8_kv_cache_reshape_gb300", "csrc")
    for f in entry["sources"]:
        with open(os.path.join(csrc, f), "rb") as fh:
            m.update(fh.read())
    return entry["bytes"] if m.hexdigest() == entry["sha1"] else None


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the GPU is under load."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    """(rank, world, local_rank); initialises a process group under torchrun
    only for the start/stop barriers and the max-over-ranks time."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def kv_bytes_read(wl) -> int:
    """Algorithmic K+V cache bytes the attention reads: every key visible to
    some query of its request, once (the window bounds it)."""
    row = {"auto": 2 * wl.head_dim, "fp8_e4m3": wl.head_dim, "fp8_e5m2": wl.head_dim,
           "int8_per_token_head": wl.head_dim + 4,
           "fp8_per_token_head": wl.head_dim + 4,
           "fp8_e5m2_per_token_head": wl.head_dim + 4}[wl.kv_cache_dtype]
    total = 0
    for Q, L in zip(wl.query_lens, wl.seq_lens):
        if Q == 0:
            continue
        lo = max(0, L - Q - wl.window + 1) if wl.window > 0 else 0
        total += (L - lo) * wl.heads_kv * row * 2
    return total


def attention_flops(wl) -> int:
    """Algorithmic FLOPs: 4 * D per visible (query, key) pair and q head."""
    total = 0
    for Q, L in zip(wl.query_lens, wl.seq_lens):
        for i in range(Q):
            p = L - Q + i
            hi = p + 1 if wl.causal else L
            lo = max(0, p - wl.window + 1) if wl.window > 0 else 0
            total += (hi - lo)
    return total * wl.heads_q * 4 * wl.head_dim


def sub_batch(wl, reqs):
    """The requests `reqs` of a workload as a batch of their own over the same
    caches (their query rows, lengths and table rows)."""
    import torch
    from int8_kv_cache_reshape_gb300 import workloads as W
    qsl = wl.query_start_loc.tolist()
    rows = torch.cat([torch.arange(qsl[r], qsl[r + 1]) for r in reqs]) if reqs else \
        torch.zeros(0, dtype=torch.long)
    ql = [wl.query_lens[r] for r in reqs]
    sub = W.Workload(**{**wl.__dict__})
    sub.query_lens = ql
    sub.seq_lens = [wl.seq_lens[r] for r in reqs]
    sub.q = wl.q[rows].contiguous()
    sub.block_table = wl.block_table[torch.tensor(reqs, dtype=torch.long)].contiguous()
    sub.seq_lens_t = torch.tensor(sub.seq_lens, dtype=torch.int32)
    sub.query_start_loc = torch.zeros(len(reqs) + 1, dtype=torch.int32)
    if reqs:
        sub.query_start_loc[1:] = torch.cumsum(torch.tensor(ql, dtype=torch.int32), 0)
    return sub


def _roofline(decode_metric, kvb, flops, attn_ms, peaks, peaks_src, kernel, traffic=None):
    r = {"bound": "hbm" if decode_metric else "tensor", "kernel": kernel,
         "unit": "GB/s" if decode_metric else "TFLOP/s", "traffic": traffic,
         "peak_source": peaks_src}
    if decode_metric:
        achieved = kvb / (attn_ms * 1e-3) / 1e9
        r.update(achieved=achieved, peak=peaks["hbm_gbs"], frac=achieved / peaks["hbm_gbs"],
                 algorithmic_bytes=kvb)
    else:
        achieved = flops / (attn_ms * 1e-3) / 1e12
        r.update(achieved=achieved, peak=peaks["bf16_tflops"],
                 frac=achieved / peaks["bf16_tflops"], algorithmic_flops=flops)
    return r


def run_workload(args, index, dtype, world, local, with_e2e=True):
    """Time one workload's step; returns (result dict, workload)."""
    import torch
    from int8_kv_cache_reshape_gb300 import workloads as W
    from int8_kv_cache_reshape_gb300 import kvq

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    wl = W.config(index, dtype)
    new = wl.new_token_mask()
    row = kvq.cache_row_bytes(wl.kv_cache_dtype, wl.head_dim)
    shape = (wl.num_blocks, wl.block_size, wl.heads_kv, row)
    kc = torch.empty(shape, dtype=torch.uint8, device=dev)
    vc = torch.empty(shape, dtype=torch.uint8, device=dev)
    key, value = wl.key.to(dev), wl.value.to(dev)
    slots = wl.slot_mapping.to(dev)
    # State: the earlier context's K/V are already in the cache.
    kvq.reshape_and_cache(key, value, kc, vc, slots, wl.kv_cache_dtype, wl.k_scale, wl.v_scale)
    del key, value, slots
    # Per-step inputs: the new tokens' K/V, their slots, q, lengths, table.
    new_idx = torch.nonzero(new).flatten()
    nkey = wl.key[new_idx].contiguous()
    nval = wl.value[new_idx].contiguous()
    nslot = wl.slot_mapping[new_idx].contiguous()
    d_nkey, d_nval, d_nslot = nkey.to(dev), nval.to(dev), nslot.to(dev)
    q = wl.q.to(dev)
    qsl = wl.query_start_loc.to(dev)
    sl = wl.seq_lens_t.to(dev)
    bt = wl.block_table.to(dev)
    out = torch.empty(wl.q.shape, dtype=torch.bfloat16, device=dev)
    sl_host = wl.seq_lens_t.numpy()
    qsl_host = wl.query_start_loc.numpy()
    sched = kvq.get_scheduler_metadata(wl.num_req, wl.heads_q, wl.heads_kv, wl.head_dim,
                                       sl_host, qsl_host, wl.causal, wl.window,
                                       wl.kv_cache_dtype)
    info = sched.info()
    ws = torch.empty(max(1, sched.workspace_bytes), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def l2_flush():
        # Write a buffer larger than L2, then read it back: the inputs are
        # out of L2, and the flush's own dirty lines are written back here
        # rather than inside the timed region.
        flush.zero_()
        flush.max()

    def cache_write():
        kvq.reshape_and_cache(d_nkey, d_nval, kc, vc, d_nslot, wl.kv_cache_dtype, wl.k_scale,
                              wl.v_scale, stream)

    def attention(s=sched, qq=q, qs=qsl, ss=sl, tb=bt, o=out):
        kvq.attention_with_kv_cache(s, qq, kc, vc, qs, ss, tb, wl.sm_scale, wl.causal,
                                    wl.window, wl.soft_cap, wl.k_scale, wl.v_scale, o, ws,
                                    wl.kv_cache_dtype, wl.heads_kv, stream)

    launches_per_step = 1 + info["num_kernel_launches"]
    for _ in range(args.warmup):
        l2_flush()
        cache_write()
        attention()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    # keep the GPU under the same load briefly so the sampler sees it
    t_end = time.perf_counter() + args.clock_window
    while time.perf_counter() < t_end:
        l2_flush()
        cache_write()
        attention()
        torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    _barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        l2_flush()              # L2 flush between steps, outside the timed events
        a, b, c = ev[i]
        a.record(stream)
        cache_write()
        b.record(stream)
        attention()
        c.record(stream)
    torch.cuda.synchronize()
    _barrier(world)
    clk = clocks.stop()
    step_ms = [a.elapsed_time(c) for a, b, c in ev]
    attn_ms = [b.elapsed_time(c) for a, b, c in ev]
    cache_ms = [a.elapsed_time(b) for a, b, c in ev]
    total_ms = _max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    attn_avg = sum(attn_ms) / len(attn_ms)

    kvb = kv_bytes_read(wl)
    flops = attention_flops(wl)
    decode_metric = is_decode_metric(index)
    if decode_metric:
        metric, unit = "decode KV GB/s", "GB/s"
        value = world * kvb / (ms_per_step * 1e-3) / 1e9
    else:
        metric, unit = "prefill TFLOP/s", "TFLOP/s"
        value = world * flops / (ms_per_step * 1e-3) / 1e12

    peaks, peaks_src = _peaks()
    if info["num_prefill_tiles"] and info["num_tiles"]:
        kernel = "tcgen05 prefill + split-KV decode (one attention call)"
    elif info["num_prefill_tiles"]:
        kernel = "tcgen05 prefill attention"
    else:
        kernel = "split-KV decode attention (+ split merge)"
    mixed = bool(info["num_prefill_tiles"] and info["num_tiles"])
    roofline = _roofline(decode_metric, kvb, flops, attn_avg, peaks, peaks_src, kernel,
                         None if mixed else profiled_traffic(index, wl.kv_cache_dtype))

    res = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": f"{wl.kv_cache_dtype} cache, f16 mma / f32 accumulate",
        "data": "synthetic (seeded, torch.Generator cpu, seed 1000 + workload index)",
        "config": {"workload": wl.name, "num_req": wl.num_req, "heads_q": wl.heads_q,
                   "heads_kv": wl.heads_kv, "head_dim": wl.head_dim,
                   "block_size": wl.block_size, "kv_cache_dtype": wl.kv_cache_dtype,
                   "kv_tokens": int(sum(wl.seq_lens)), "query_tokens": wl.num_query_tokens,
                   "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MB write, then read back)",
                   "parallelism": f"replicas x{world}"},
        "kv_bytes_per_step": kvb, "flops_per_step": flops,
        "tokens_per_s": world * wl.num_query_tokens / (ms_per_step * 1e-3),
        "attention_ms": attn_avg, "cache_write_ms": sum(cache_ms) / len(cache_ms),
        "schedule": info,
        "roofline": roofline,
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clk,
    }

    # ---- the mixed batch's two kernels, each timed alone ---------------------
    if info["num_prefill_tiles"] and info["num_tiles"]:
        parts = {}
        ql = wl.query_lens
        for name, reqs in (("prefill", [r for r in range(wl.num_req) if ql[r] * wl.heads_q // wl.heads_kv > 16]),
                           ("decode", [r for r in range(wl.num_req) if ql[r] * wl.heads_q // wl.heads_kv <= 16])):
            sub = sub_batch(wl, reqs)
            s2 = kvq.get_scheduler_metadata(sub.num_req, sub.heads_q, sub.heads_kv, sub.head_dim,
                                            sub.seq_lens_t.numpy(), sub.query_start_loc.numpy(),
                                            sub.causal, sub.window, sub.kv_cache_dtype)
            d_q, d_qsl = sub.q.to(dev), sub.query_start_loc.to(dev)
            d_sl, d_bt = sub.seq_lens_t.to(dev), sub.block_table.to(dev)
            d_out = torch.empty(sub.q.shape, dtype=torch.bfloat16, device=dev)
            for _ in range(args.warmup):
                l2_flush()
                attention(s2, d_q, d_qsl, d_sl, d_bt, d_out)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            torch.cuda.synchronize()
            for a, b in evs:
                l2_flush()
                a.record(stream)
                attention(s2, d_q, d_qsl, d_sl, d_bt, d_out)
                b.record(stream)
            torch.cuda.synchronize()
            ms = sum(a.elapsed_time(b) for a, b in evs) / len(evs)
            pm = name == "decode"
            kvb2, fl2 = kv_bytes_read(sub), attention_flops(sub)
            parts[name] = {
                "requests": len(reqs), "attention_ms": ms,
                "value": (kvb2 / (ms * 1e-3) / 1e9) if pm else (fl2 / (ms * 1e-3) / 1e12),
                "unit": "GB/s" if pm else "TFLOP/s",
                "roofline": _roofline(pm, kvb2, fl2, ms, peaks, peaks_src,
                                      "split-KV decode attention (+ split merge)" if pm
                                      else "tcgen05 prefill attention",
                                      profiled_traffic(index, wl.kv_cache_dtype, name))}
            s2.close()
        res["parts"] = parts

    # ---- the fused decode step (decode batches): plan on the device --------
    fused_ok = all(Q * wl.heads_q // wl.heads_kv <= 16 for Q in wl.query_lens) and wl.causal
    mql = max(wl.query_lens) if wl.query_lens else 1
    if fused_ok:
        step_ws = torch.zeros(kvq.decode_step_workspace_size(
            wl.num_req, wl.heads_q, wl.heads_kv, wl.head_dim, wl.kv_cache_dtype, mql),
            dtype=torch.uint8, device=dev)

        def fused(qq=q, qs=qsl, ss=sl, tb=bt):
            kvq.decode_step(d_nkey, d_nval, d_nslot, kc, vc, qq, qs, ss, tb, mql, wl.sm_scale,
                            wl.window, wl.soft_cap, wl.k_scale, wl.v_scale, out, step_ws,
                            wl.kv_cache_dtype, wl.heads_kv, stream=stream)

        for _ in range(args.warmup):
            l2_flush()
            fused()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        torch.cuda.synchronize()
        for a, b in evs:
            l2_flush()
            a.record(stream)
            fused()
            b.record(stream)
        torch.cuda.synchronize()
        kvq.decode_step_check(step_ws)
        fms = _max_over_ranks(sum(a.elapsed_time(b) for a, b in evs), world) / args.steps
        res["fused_step"] = {
            "call": "kvq_decode_step (cache write + device-built plan + attention in one "
                    "launch, then the merge of its cut tiles)",
            "ms_per_step": fms, "value": world * kvb / (fms * 1e-3) / 1e9, "unit": "GB/s",
            "roofline": _roofline(True, kvb, flops, fms, peaks, peaks_src,
                                  "fused decode step (cache write + split-KV decode)"),
            "gpu_launches_per_step": 2}
        res["gpu_launches"] += args.steps

    # ---- end to end: host buffers through the public API -------------------
    if with_e2e:
        # One pinned staging buffer holds the step's inputs (q, the new K/V
        # rows, their slots, the lengths and the table), each 256-byte
        # aligned, and goes to the device in one copy.
        parts = [wl.q, nkey, nval, nslot, wl.query_start_loc, wl.seq_lens_t, wl.block_table]
        sizes = [t.numel() * t.element_size() for t in parts]
        offs, o = [], 0
        for n in sizes:
            offs.append(o)
            o += (n + 255) // 256 * 256
        h_pack = torch.empty(o, dtype=torch.uint8).pin_memory()
        d_pack = torch.empty(o, dtype=torch.uint8, device=dev)
        for t, off, n in zip(parts, offs, sizes):
            h_pack[off:off + n].copy_(t.contiguous().view(-1).view(torch.uint8))
        dv = [d_pack[off:off + n].view(t.dtype).view(t.shape) for t, off, n in zip(parts, offs, sizes)]
        e_q, e_nkey, e_nval, e_nslot, e_qsl, e_sl, e_bt = dv
        h_out = torch.empty(wl.q.shape, dtype=torch.bfloat16).pin_memory()
        h2d = h_pack.numel()  # the packed buffer the copy moves (tensors + alignment padding)
        d2h = h_out.numel() * h_out.element_size()

        def e2e_two_calls():
            d_pack.copy_(h_pack, non_blocking=True)
            s2 = kvq.get_scheduler_metadata(wl.num_req, wl.heads_q, wl.heads_kv, wl.head_dim,
                                            sl_host, qsl_host, wl.causal, wl.window,
                                            wl.kv_cache_dtype)
            kvq.reshape_and_cache(e_nkey, e_nval, kc, vc, e_nslot, wl.kv_cache_dtype, wl.k_scale,
                                  wl.v_scale, stream)
            kvq.attention_with_kv_cache(s2, e_q, kc, vc, e_qsl, e_sl, e_bt, wl.sm_scale,
                                        wl.causal, wl.window, wl.soft_cap, wl.k_scale,
                                        wl.v_scale, out, ws, wl.kv_cache_dtype, wl.heads_kv,
                                        stream)
            h_out.copy_(out, non_blocking=True)
            stream.synchronize()
            s2.close()

        if fused_ok:
            # a serving loop marshals the step's call once (kvq.Prepared): one
            # C-ABI call copies the packed inputs in, runs the fused step with
            # its output stored straight into the pinned host buffer (or
            # copied back after the step) and waits for the stream
            step_io = kvq.prepare_decode_step_host_io(
                h_pack, d_pack, h_out, 0, e_nkey, e_nval, e_nslot, kc, vc, e_q, e_qsl, e_sl,
                e_bt, mql, wl.sm_scale, wl.window, wl.soft_cap, wl.k_scale, wl.v_scale, None,
                step_ws, wl.kv_cache_dtype, wl.heads_kv, stream=stream)
            step_io_copy = kvq.prepare_decode_step_host_io(
                h_pack, d_pack, h_out, d2h, e_nkey, e_nval, e_nslot, kc, vc, e_q, e_qsl, e_sl,
                e_bt, mql, wl.sm_scale, wl.window, wl.soft_cap, wl.k_scale, wl.v_scale, out,
                step_ws, wl.kv_cache_dtype, wl.heads_kv, stream=stream)
            # the same step captured once (kvq_decode_step_graph_create): a
            # step is one graph launch and its wait
            step_graph = kvq.decode_step_graph(
                h_pack, d_pack, h_out, 0, e_nkey, e_nval, e_nslot, kc, vc, e_q, e_qsl, e_sl,
                e_bt, mql, wl.sm_scale, wl.window, wl.soft_cap, wl.k_scale, wl.v_scale, None,
                step_ws, wl.kv_cache_dtype, wl.heads_kv, stream=stream)

        def e2e_fused():
            step_io()

        def e2e_fused_copy():
            step_io_copy()

        def time_e2e(fn):
            for _ in range(3):
                fn()
            ts = []
            for _ in range(args.steps):
                l2_flush()
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                fn()
                ts.append(time.perf_counter() - t0)
            return _max_over_ranks(sum(ts), world) / args.steps

        def e2e_obj(secs, includes):
            return {"value": world * (kvb if decode_metric else flops) / secs /
                    (1e9 if decode_metric else 1e12),
                    "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": secs * 1e3, "includes": includes}

        two = e2e_obj(time_e2e(e2e_two_calls),
                      "one H2D of the step inputs, host scheduler, reshape_and_cache, "
                      "attention_with_kv_cache, D2H of out")
        if fused_ok:
            res["e2e"] = e2e_obj(time_e2e(step_graph),
                                 "one C-ABI call, kvq_decode_step_graph_launch: the host-buffer "
                                 "step captured once in a CUDA graph, replayed per step -- the "
                                 "fused step (its CTAs read the packed step inputs from pinned "
                                 "host memory and copy them to the device; cache write, plan on "
                                 "the device, attention; merge of the cut tiles) storing out "
                                 "straight into pinned host memory, then stream synchronize")
            res["e2e_host_io"] = e2e_obj(time_e2e(e2e_fused),
                                         "one C-ABI call, kvq_decode_step_host_io: the same step "
                                         "launched by the call (no graph)")
            res["e2e_copy_out"] = e2e_obj(time_e2e(e2e_fused_copy),
                                          "kvq_decode_step_host_io with out in device memory and "
                                          "one D2H copy of it after the step")
            res["e2e_two_calls"] = two
            step_graph.close()
        else:
            res["e2e"] = two
        sched_times = []
        for _ in range(5):
            t1 = time.perf_counter()
            s3 = kvq.get_scheduler_metadata(wl.num_req, wl.heads_q, wl.heads_kv, wl.head_dim,
                                            sl_host, qsl_host, wl.causal, wl.window,
                                            wl.kv_cache_dtype)
            sched_times.append(time.perf_counter() - t1)
            s3.close()
        res["scheduler_host_ms"] = 1e3 * sorted(sched_times)[len(sched_times) // 2]
    sched.close()
    del kc, vc, flush
    torch.cuda.empty_cache()
    return res, wl


def run_gpu(args, rank, world, local):
    return run_workload(args, args.workload, args.kv_cache_dtype, world, local)


class OracleStep:
    """The oracle (as it stands) on a bounded sample of the step: the first
    `nreq` requests -- cache write of their new tokens, then attention of
    their queries over all heads.  Their earlier context is written once in
    setup (untimed)."""

    def __init__(self, wl, nreq: int):
        import numpy as np
        import oracle
        from int8_kv_cache_reshape_gb300 import workloads as W
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        from _harness import ORACLE_DT, cache_shape
        self.oracle, self.W, self.np = oracle, W, np
        self.wl = wl
        self.dt = ORACLE_DT[wl.kv_cache_dtype]
        self.reqs = list(range(min(nreq, wl.num_req)))
        req = wl.token_req.numpy()
        new = wl.new_token_mask().numpy()
        pos = wl.token_pos.numpy()
        L = wl.seq_lens_t.numpy()[req]
        Q = np.array(wl.query_lens)[req]
        in_sample = np.isin(req, self.reqs)
        if wl.window > 0:
            in_sample &= pos >= (L - Q - wl.window + 1)
        self.kc = np.zeros(cache_shape(wl), np.uint8)
        self.vc = np.zeros(cache_shape(wl), np.uint8)
        self.kb, self.vb = W.bf16_bits(wl.key), W.bf16_bits(wl.value)
        self.qb = W.bf16_bits(wl.q)
        slots = wl.slot_mapping.numpy()
        old = np.where(in_sample & ~new, slots, -1)
        oracle.reshape_and_cache(self.kb, self.vb, self.kc, self.vc, old, self.dt, wl.k_scale,
                                 wl.v_scale, wl.block_size)
        self.fresh = np.where(in_sample & new, slots, -1)
        qsl = wl.query_start_loc.numpy()
        self.toks = np.concatenate([np.arange(qsl[r], qsl[r + 1]) for r in self.reqs])
        self.sub = W.Workload(**{**wl.__dict__})
        self.sub.query_lens = [wl.query_lens[r] for r in self.reqs]
        self.sub.seq_lens = [wl.seq_lens[r] for r in self.reqs]
        self.cores = oracle.num_threads()
        self.sample = (f"first {len(self.reqs)} of {wl.num_req} requests: cache write of their "
                       f"new tokens + attention of their {self.sub.num_query_tokens} query "
                       f"tokens over all {wl.heads_q} heads")

    def step(self) -> float:
        wl = self.wl
        t0 = time.perf_counter()
        self.oracle.reshape_and_cache(self.kb, self.vb, self.kc, self.vc, self.fresh, self.dt,
                                      wl.k_scale, wl.v_scale, wl.block_size)
        self.oracle.attention(self.qb, self.kc, self.vc, wl.query_start_loc, wl.seq_lens_t,
                              wl.block_table, wl.heads_kv, wl.block_size, self.dt, wl.sm_scale,
                              wl.causal, wl.window, wl.soft_cap, wl.k_scale, wl.v_scale,
                              tokens=self.toks)
        return time.perf_counter() - t0

    def work(self, decode_metric: bool) -> float:
        return kv_bytes_read(self.sub) if decode_metric else attention_flops(self.sub)


def is_decode_metric(index: int) -> bool:
    return index in (1, 2, 5)


def run_reference(args, rank, world):
    from int8_kv_cache_reshape_gb300 import workloads as W
    if rank != 0:
        return None
    wl = W.config(args.workload, args.kv_cache_dtype)
    decode_metric = is_decode_metric(args.workload)
    ref = OracleStep(wl, args.ref_requests)
    for _ in range(args.warmup):
        ref.step()
    times = [ref.step() for _ in range(args.steps)]
    s = sum(times) / len(times)
    value = ref.work(decode_metric) / s / (1e9 if decode_metric else 1e12)
    unit = "GB/s" if decode_metric else "TFLOP/s"
    return {
        "impl": "reference", "metric": "decode KV GB/s" if decode_metric else "prefill TFLOP/s",
        "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic (seeded)", "config": {"workload": wl.name, "sample": ref.sample},
        "cpu_baseline": {"value": value, "unit": unit, "cores": ref.cores, "kind": "oracle",
                         "sample": ref.sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    ap.add_argument("--workload", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--kv-cache-dtype", default=None)
    ap.add_argument("--clock-window", type=float, default=1.5,
                    help="seconds of untimed load before the timed steps, for clock samples")
    ap.add_argument("--ref-requests", type=int, default=16)
    ap.add_argument("--cpu-requests", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", dest="all_workloads", action="store_false",
                    help="only the headline workload (no per-workload objects)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = _dist()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if rank == 0:
            print(json.dumps(res))
        return
    res, wl = run_gpu(args, rank, world, local)
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl, args.workload, args.cpu_requests)
    if args.all_workloads and args.workload == 2 and args.kv_cache_dtype is None:
        others = []
        for index, dtype in OTHER_WORKLOADS:
            r2, wl2 = run_workload(args, index, dtype, world, local, with_e2e=True)
            entry = {k: r2[k] for k in ("metric", "value", "unit", "ms_per_step", "attention_ms",
                                        "cache_write_ms", "tokens_per_s", "kv_bytes_per_step",
                                        "flops_per_step", "roofline", "e2e", "clocks",
                                        "gpu_launches", "scheduler_host_ms") if k in r2}
            for k in ("fused_step", "e2e_host_io", "e2e_two_calls", "e2e_copy_out"):
                if k in r2:
                    entry[k] = r2[k]
            entry["workload"] = r2["config"]["workload"]
            entry["kv_cache_dtype"] = r2["config"]["kv_cache_dtype"]
            entry["schedule"] = {k: r2["schedule"][k] for k in (
                "num_tiles", "num_pieces", "max_splits", "num_prefill_tiles",
                "num_decode_warps", "workspace_bytes")}
            if "parts" in r2:
                entry["parts"] = r2["parts"]
            if rank == 0 and not args.no_cpu_baseline:
                entry["cpu_baseline"] = cpu_baseline(wl2, index, args.cpu_requests)
            others.append(entry)
            res["gpu_launches"] += r2["gpu_launches"]
        res["workloads"] = others
    if rank == 0:
        print(json.dumps(res))


# The workloads reported beside the headline decode batch (index, dtype).
OTHER_WORKLOADS = [(3, None), (4, "int8_per_token_head"), (4, "fp8_per_token_head"),
                   (4, "fp8_e5m2_per_token_head"), (5, None)]


def cpu_baseline(wl, index, nreq):
    """The oracle on a bounded sample of the workload's step (see OracleStep)."""
    decode_metric = is_decode_metric(index)
    ref = OracleStep(wl, nreq if decode_metric else min(nreq, 1))
    secs = ref.step()
    return {"value": ref.work(decode_metric) / secs / (1e9 if decode_metric else 1e12),
            "unit": "GB/s" if decode_metric else "TFLOP/s", "cores": ref.cores,
            "kind": "oracle", "seconds": secs, "sample": ref.sample}


if __name__ == "__main__":
    main()
