#!/usr/bin/env python3
"""Throughput benchmark of the GB300 attention library.

One step = one pass of the prefill hot path over the batched workload
(B=4, H=16, Nq=Nk=2048, d=128, bf16): attn_fwd non-causal, then attn_fwd
causal, on inputs already resident in HBM.  The headline metric is TFLOPS
with the algorithmic count 4*B*H*Nq*Nk*d per call (halved for the causal
call).  Inputs (100 MB) are smaller than L2, so L2 is flushed (a 256 MB
write) before every timed step, outside the timed events.

Also reported in the same JSON line (timed the same way, not part of
`value`): the long causal prefill (1x32x32768, d=128), FP8 prefill
(2x16x8192, d=128), paged decode (64 requests, H=32, d=128, 64-token
pages), the same decode with 32 query heads over 8 KV heads on the tensor
cores -- both as HBM GB/s of algorithmic bytes -- and causal prefill chunks
over a paged cache (8 requests x 2048 new tokens after 6144 cached, 32 query
heads over 8 KV heads) and a variable-length causal batch (16 packed sequences of 512..4096
tokens, 32 query heads over 8 KV heads) as TFLOPS of exactly counted
visible pairs; and the backward pass of the batched workload (dQ, dK, dV),
as TFLOPS with 2.5x the forward count.

`e2e` is the same step from page-locked host buffers through attn_fwd_host:
Q, K, V are copied in and both calls' O and LSE copied out every step, in
chunks of (b, h) pairs whose copies in both directions overlap the kernels.

`--impl reference` times the float64 CPU oracle (the only reference this
method has) on a bounded row sample of the same workload.

Multi-GPU: one process per GPU (torchrun); every rank runs its own replica of
the step on its own inputs (weak scaling, no data-path collective); the
elapsed time is the max over ranks.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

B, H, N, D = 4, 16, 2048, 128
WORKLOAD = "batched prefill B=4 H=16 Nq=Nk=2048 d=128 bf16, non-causal + causal per step"
METRIC = "attention fwd TFLOPS and % of GB300 tensor peak; paged decode HBM GB/s"


def prefill_flops(b, h, nq, nk, d, causal):
    f = 4.0 * b * h * nq * nk * d
    return f / 2 if causal else f


STEP_FLOPS = prefill_flops(B, H, N, N, D, False) + prefill_flops(B, H, N, N, D, True)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def max_over_ranks(value, device=None):
    """Max of a float over all ranks of the default process group (the
    elapsed time of a weak-scaling replica run is the slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons DURING the
    timed region: NVML through ctypes every ~2 ms from a background thread
    (reading only), plus an nvidia-smi process at 200 ms as a second source."""

    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, torch, device_index):
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self.smi_lines = []
        self._stop = False
        self._nvml = None
        self._handle = None
        self._proc = None
        self._smi_index = str(device_index)
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                bus = None
                try:
                    pr = torch.cuda.get_device_properties(device_index)
                    bus = "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
                except Exception:
                    bus = None
                ok = bus is not None and nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
                if not ok:
                    ok = nv.nvmlDeviceGetHandleByIndex_v2(int(device_index), ctypes.byref(h)) == 0
                if ok:
                    self._nvml, self._handle, self._ct = nv, h, ctypes
                    idx = ctypes.c_uint()
                    if nv.nvmlDeviceGetIndex(h, ctypes.byref(idx)) == 0:
                        self._smi_index = str(idx.value)
                    mx = ctypes.c_uint()
                    if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                        self.max_mhz = float(mx.value)
        except Exception:
            self._nvml = None

    def _poll(self):
        ct, nv, h = self._ct, self._nvml, self._handle
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self._stop:
            if nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(clk)) == 0:
                self.samples.append(float(clk.value))
            if get_reasons(h, ct.byref(rs)) == 0:
                for name, bit in self.REASON_BITS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            time.sleep(0.002)

    def __enter__(self):
        import threading
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", self._smi_index, "--query-gpu=" + self.SMI_FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self._proc = None
        self._thread = None
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *a):
        self._stop = True
        if self._thread is not None:
            self._thread.join(timeout=2)
        if self._proc is not None:
            self._proc.terminate()
            try:
                out, _ = self._proc.communicate(timeout=5)
            except Exception:
                self._proc.kill()
                out = ""
            self.smi_lines = [ln for ln in (out or "").splitlines() if ln.strip()]

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        smi_sm, reasons = [], set(self.reasons)
        mx = self.max_mhz
        for ln in self.smi_lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                smi_sm.append(float(parts[0]))
                mx = max(mx or 0.0, float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        sm = self.samples or smi_sm
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvml" if self.samples else ("nvidia-smi" if smi_sm else "none")}


# ---------------------------------------------------------------- timing helpers

def timed_launches(torch, fn, iters, flush):
    """Run fn() `iters` times, flushing L2 before each; returns per-call ms (CUDA events)."""
    stream = torch.cuda.current_stream()
    times = []
    for _ in range(iters):
        flush()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        e.synchronize()
        times.append(s.elapsed_time(e))
    return times


def traffic_record(kernel_file, key):
    """DRAM bytes per launch from a committed ncu summary, valid only while the
    kernel source is unchanged (sha256 recorded at capture time)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[key]
        with open(os.path.join(ROOT, "attention_attn_fwd_03_gb300", "csrc", kernel_file), "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        if rec.get("source_sha256") != sha:
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import attention_attn_fwd_03_gb300 as attn
    from attention_attn_fwd_03_gb300 import inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    attn.lib()
    peaks = load_peaks()

    flush_buf = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.fill_(1.0)

    # inputs: seeded per rank (each rank is an independent replica)
    q, k, v = (t.to(dev) for t in inputs.dense_qkv(B, H, N, N, D, seed=rank))
    o_nc, l_nc = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=dev)
    o_c, l_c = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=dev)

    def step():
        attn.fwd(q, k, v, causal=False, out=o_nc, lse=l_nc)
        attn.fwd(q, k, v, causal=True, out=o_c, lse=l_c)

    for _ in range(args.warmup):
        flush()
        step()
    attn.device_status()

    # per-launch durations of the dominant kernel (the prefill kernel, both calls)
    nc_ms = timed_launches(torch, lambda: attn.fwd(q, k, v, causal=False, out=o_nc, lse=l_nc), 5, flush)
    c_ms = timed_launches(torch, lambda: attn.fwd(q, k, v, causal=True, out=o_c, lse=l_c), 5, flush)

    # ---- timed region: exactly K steps
    stream = torch.cuda.current_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch, local_rank) as clk:
        for i in range(args.steps):
            flush()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    attn.device_status()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(step_ms)
    if world > 1:
        total_ms = max_over_ranks(total_ms, device=dev)
    ms_per_step = total_ms / args.steps
    value = STEP_FLOPS * world * args.steps / (total_ms * 1e-3) / 1e12

    # ---- end to end through the public API from pinned host buffers: attn_fwd_host
    # pipelines the copies in, the kernels of both mask modes and the copies
    # out over chunks of (b, h) pairs.  For comparison, the same step with
    # serial copies around the device entry point.
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    ho = [torch.empty((B, H, N, D), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    hl = [torch.empty((B, H, N), dtype=torch.float32).pin_memory() for _ in range(2)]
    host_ws = torch.empty(attn.attn_fwd_host_workspace_size(B, H, N, N, D, 2, 0), dtype=torch.uint8, device=dev)

    def e2e_step():
        attn.fwd_host(hq, hk, hv, causal=(False, True), out=ho, lse=hl, workspace=host_ws, synchronize=False)

    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def serial_step():
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        attn.fwd(dq, dk, dv, causal=False, out=o_nc, lse=l_nc)
        attn.fwd(dq, dk, dv, causal=True, out=o_c, lse=l_c)
        ho[0].copy_(o_nc, non_blocking=True)
        ho[1].copy_(o_c, non_blocking=True)
        hl[0].copy_(l_nc, non_blocking=True)
        hl[1].copy_(l_c, non_blocking=True)

    for _ in range(2):
        e2e_step()
        serial_step()
    torch.cuda.synchronize()
    e2e_ms = timed_launches(torch, e2e_step, max(3, min(args.steps, 10)), flush)
    serial_ms = timed_launches(torch, serial_step, max(3, min(args.steps, 10)), flush)
    attn.device_status()
    h2d = 3 * q.numel() * 2
    d2h = 2 * (o_nc.numel() * 2 + l_nc.numel() * 4)
    e2e_val = STEP_FLOPS / (statistics.mean(e2e_ms) * 1e-3) / 1e12

    # ---- dominant kernel roofline (prefill kernel: both calls of the step)
    launch_flops = prefill_flops(B, H, N, N, D, False) + prefill_flops(B, H, N, N, D, True)
    launch_ms = statistics.mean(nc_ms) + statistics.mean(c_ms)
    achieved = launch_flops / (launch_ms * 1e-3) / 1e12
    traffic_nc = traffic_record("prefill.cu", "prefill_bf16_d128_batched_noncausal")
    traffic_c = traffic_record("prefill.cu", "prefill_bf16_d128_batched_causal")
    traffic = (traffic_nc + traffic_c) / 2 if (traffic_nc is not None and traffic_c is not None) else None

    secondary = {}
    if not args.no_secondary:
        secondary = run_secondary(torch, attn, inputs, dev, flush, peaks, rank)

    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), rounded to bf16)",
        "config": {"workload": WORKLOAD, "B": B, "H": H, "Nq": N, "Nk": N, "d": D,
                   "calls_per_step": ["non-causal", "causal"], "flops_per_step": STEP_FLOPS,
                   "l2": "flushed (256 MB write) before every timed step, outside the timed events",
                   "parallelism": "replicas (one independent workload per GPU)"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                     "traffic": traffic, "kernel": "prefill_kernel<128,bf16>",
                     "peak_source": peaks["source"] + " dense bf16 (burst, kernel timed alone)"},
        "e2e": {"value": round(e2e_val, 3), "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(statistics.mean(e2e_ms), 4),
                "api": "attn_fwd_host (chunked copy-in / kernels / copy-out pipeline)",
                "serial_copies_ms_per_step": round(statistics.mean(serial_ms), 4)},
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
        "per_call_ms": {"non_causal": round(statistics.mean(nc_ms), 4), "causal": round(statistics.mean(c_ms), 4)},
        "workloads": secondary,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(sample_seconds=args.cpu_seconds)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_secondary(torch, attn, inputs, dev, flush, peaks, rank):
    out = {}
    reps = 5
    # long causal prefill
    q, k, v = (t.to(dev) for t in inputs.dense_qkv(1, 32, 32768, 32768, 128, seed=rank))
    o, l = torch.empty_like(q), torch.empty((1, 32, 32768), dtype=torch.float32, device=dev)
    attn.fwd(q, k, v, causal=True, out=o, lse=l)
    ms = timed_launches(torch, lambda: attn.fwd(q, k, v, causal=True, out=o, lse=l), reps, flush)
    f = prefill_flops(1, 32, 32768, 32768, 128, True)
    tf = f / (statistics.mean(ms) * 1e-3) / 1e12
    out["long_causal_prefill_1x32x32768_d128"] = {
        "TFLOPS": round(tf, 2), "ms": round(statistics.mean(ms), 4),
        "frac_of_measured_bf16": round(tf / peaks["bf16_tflops"], 4)}
    del q, k, v, o, l
    # FP8 prefill
    q, k, v = inputs.dense_qkv(2, 16, 8192, 8192, 128, seed=rank)
    (q8, dq), (k8, dk), (v8, dv) = (inputs.fp8_quantize(t) for t in (q, k, v))
    q8, k8, v8 = q8.to(dev), k8.to(dev), v8.to(dev)
    o, l = torch.empty((2, 16, 8192, 128), dtype=torch.bfloat16, device=dev), \
        torch.empty((2, 16, 8192), dtype=torch.float32, device=dev)
    attn.fwd_fp8(q8, k8, v8, (dq, dk, dv), out=o, lse=l)
    ms = timed_launches(torch, lambda: attn.fwd_fp8(q8, k8, v8, (dq, dk, dv), out=o, lse=l), reps, flush)
    f = prefill_flops(2, 16, 8192, 8192, 128, False)
    tf = f / (statistics.mean(ms) * 1e-3) / 1e12
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    out["fp8_prefill_2x16x8192_d128"] = {
        "TFLOPS": round(tf, 2), "ms": round(statistics.mean(ms), 4),
        "frac_of_fp8_peak": round(tf / fp8_peak, 4),
        "fp8_peak_note": "measured bf16 burst x 2 (nominal fp8:bf16 dense ratio)"}
    del q, k, v, q8, k8, v8, o, l
    # paged decode
    p = inputs.paged_kv(B=64, H=32, d=128, page_size=64, max_pages=128, num_pages=8192, len_lo=512,
                        len_hi=8192, seed=rank, device=dev)
    o = torch.empty_like(p["q"])
    l = torch.empty((64, 32), dtype=torch.float32, device=dev)
    ws = torch.empty(attn.attn_paged_decode_workspace_size(64, 32, 128, 64, 128), dtype=torch.uint8, device=dev)

    def dec():
        attn.paged_decode(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"], out=o, lse=l,
                          workspace=ws)
    dec()
    ms = timed_launches(torch, dec, reps, flush)
    attn.device_status()
    total_tokens = int(p["seq_lens"].sum().item())
    n_pages = int(((p["seq_lens"].long() + 63) // 64).sum().item())
    alg_bytes = total_tokens * 32 * 128 * 2 * 2 + 2 * (64 * 32 * 128 * 2) + 64 * 32 * 4 + n_pages * 4 + 64 * 4
    gbs = alg_bytes / (statistics.mean(ms) * 1e-3) / 1e9
    out["paged_decode_64req_H32_d128_p64"] = {
        "GBps": round(gbs, 1), "ms": round(statistics.mean(ms), 4), "algorithmic_bytes": alg_bytes,
        "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 4), "frac_of_8TBps": round(gbs / 8000.0, 4),
        "tokens": total_tokens}
    del p, o, l, ws
    torch.cuda.empty_cache()
    # grouped-query paged decode on the tensor cores: 32 query heads over 8 KV heads
    p = inputs.paged_kv(B=64, H=32, d=128, page_size=64, max_pages=128, num_pages=8192, len_lo=512,
                        len_hi=8192, seed=rank, device=dev, H_kv=8)
    o = torch.empty_like(p["q"])
    l = torch.empty((64, 32), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, attn.attn_paged_fwd_workspace_size(64, 64, 1, 32, 8, 128, 64, 128)),
                     dtype=torch.uint8, device=dev)

    def gqa():
        attn.paged_fwd(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"], out=o, lse=l,
                       workspace=ws)
    gqa()
    ms = timed_launches(torch, gqa, reps, flush)
    attn.device_status()
    total_tokens = int(p["seq_lens"].sum().item())
    n_pages = int(((p["seq_lens"].long() + 63) // 64).sum().item())
    alg_bytes = total_tokens * 8 * 128 * 2 * 2 + 2 * (64 * 32 * 128 * 2) + 64 * 32 * 4 + n_pages * 4 + 64 * 4
    gbs = alg_bytes / (statistics.mean(ms) * 1e-3) / 1e9
    out["gqa_paged_decode_64req_H32_Hkv8_d128_p64"] = {
        "GBps": round(gbs, 1), "ms": round(statistics.mean(ms), 4), "algorithmic_bytes": alg_bytes,
        "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 4), "frac_of_8TBps": round(gbs / 8000.0, 4),
        "tokens": total_tokens}
    del p, o, l, ws
    torch.cuda.empty_cache()
    # prefill chunks over a paged cache: 8 requests, 2048 new tokens after a 6144-token prefix, causal
    p = inputs.paged_chunks(B=8, H=32, H_kv=8, d=128, page_size=64, max_pages=128, num_pages=1024,
                            q_lo=2048, q_hi=2048, ctx_lo=6144, ctx_hi=6144, seed=rank, device=dev)
    o = torch.empty_like(p["q"])
    l = torch.empty((p["q"].shape[0], 32), dtype=torch.float32, device=dev)
    wsb = attn.attn_paged_fwd_workspace_size(8, p["q"].shape[0], 2048, 32, 8, 128, 64, 128)
    ws = torch.empty(max(1, wsb), dtype=torch.uint8, device=dev)

    def chunks():
        attn.paged_fwd(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"],
                       cu_seqlens_q=p["cu_seqlens_q"], max_q_len=2048, causal=True, out=o, lse=l, workspace=ws)
    chunks()
    ms = timed_launches(torch, chunks, reps, flush)
    attn.device_status()
    # exact visible (query, key) pairs: query i of a request sees 6144 + i + 1 keys
    pairs = 8 * sum(6144 + i + 1 for i in range(2048))
    f = 4.0 * pairs * 32 * 128
    tf = f / (statistics.mean(ms) * 1e-3) / 1e12
    out["paged_prefill_chunks_8x2048_over_6144_H32_Hkv8_d128_causal"] = {
        "TFLOPS": round(tf, 2), "ms": round(statistics.mean(ms), 4),
        "frac_of_measured_bf16": round(tf / peaks["bf16_tflops"], 4),
        "flops_note": "4 * d * H * visible (query, key) pairs, counted exactly"}
    del p, o, l, ws
    torch.cuda.empty_cache()
    # variable-length batch prefill: 16 packed sequences of 512..4096 tokens, causal self-attention
    p = inputs.varlen_qkv(B=16, H=32, H_kv=8, d=128, q_lo=512, q_hi=4096, seed=rank, device=dev)
    o = torch.empty_like(p["q"])
    l = torch.empty((p["q"].shape[0], 32), dtype=torch.float32, device=dev)
    ws = torch.empty(attn.attn_varlen_fwd_workspace_size(16, p["q"].shape[0], p["max_q_len"], p["max_k_len"], 32, 8,
                                                         128), dtype=torch.uint8, device=dev)

    def varlen():
        attn.varlen_fwd(p["q"], p["k"], p["v"], p["cu_seqlens_q"], p["cu_seqlens_k"], max_q_len=p["max_q_len"],
                        max_k_len=p["max_k_len"], causal=True, out=o, lse=l, workspace=ws)
    varlen()
    ms = timed_launches(torch, varlen, reps, flush)
    attn.device_status()
    lens = (p["cu_seqlens_q"][1:] - p["cu_seqlens_q"][:-1]).long().cpu()
    pairs = int((lens * (lens + 1) // 2).sum())  # query i of a sequence sees i + 1 keys
    f = 4.0 * pairs * 32 * 128
    tf = f / (statistics.mean(ms) * 1e-3) / 1e12
    out["varlen_prefill_16seq_512-4096_H32_Hkv8_d128_causal"] = {
        "TFLOPS": round(tf, 2), "ms": round(statistics.mean(ms), 4), "tokens": int(lens.sum()),
        "frac_of_measured_bf16": round(tf / peaks["bf16_tflops"], 4),
        "flops_note": "4 * d * H * visible (query, key) pairs, counted exactly"}
    del p, o, l, ws
    torch.cuda.empty_cache()
    # backward of the batched prefill (4 x 16 x 2048, d = 128): dQ, dK, dV by recomputation
    q, k, v = (t.to(dev) for t in inputs.dense_qkv(B, H, N, N, D, seed=rank))
    g = torch.Generator(device="cpu").manual_seed(rank + 1)
    do = torch.randn((B, H, N, D), generator=g, dtype=torch.float32).to(torch.bfloat16).to(dev)
    ws = torch.empty(attn.attn_bwd_workspace_size(B, H, N, D), dtype=torch.uint8, device=dev)
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    for causal in (False, True):
        o, l = attn.fwd(q, k, v, causal=causal)

        def bwd():
            attn.bwd(q, k, v, o, l, do, causal=causal, dq=grads[0], dk=grads[1], dv=grads[2], workspace=ws)
        bwd()
        ms = timed_launches(torch, bwd, reps, flush)
        attn.device_status()
        f = 2.5 * prefill_flops(B, H, N, N, D, causal)  # five products of the forward's size
        tf = f / (statistics.mean(ms) * 1e-3) / 1e12
        out["backward_%dx%dx%d_d%d_%s" % (B, H, N, D, "causal" if causal else "non_causal")] = {
            "TFLOPS": round(tf, 2), "ms": round(statistics.mean(ms), 4),
            "frac_of_measured_bf16": round(tf / peaks["bf16_tflops"], 4),
            "flops_note": "2.5 x the forward count (five GEMMs of the forward's size), halved for causal"}
    del q, k, v, do, ws, grads, o, l
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- CPU oracle (reference arm and cpu_baseline)

class OracleSampler:
    """Times the float64 oracle on row samples of the step's workload (inputs
    generated once; the per-row cost calibrated once)."""

    def __init__(self):
        import numpy as np

        import oracle
        from attention_attn_fwd_03_gb300 import inputs

        self.np, self.oracle = np, oracle
        self.q, self.k, self.v = inputs.dense_qkv(B, H, N, N, D, seed=0)
        self.scale = float(np.float32(1.0 / math.sqrt(D)))
        self.threads = oracle.default_threads()
        self.rng = np.random.default_rng(0)
        cal = np.sort(self.rng.choice(B * H * N, size=256, replace=False))
        t0 = time.perf_counter()
        oracle.attention(self.q, self.k, self.v, self.scale, causal=False, rows=cal, nthreads=self.threads)
        self.per_row = max((time.perf_counter() - t0) / 256, 1e-7)

    def run(self, seconds):
        """One timed sample of about `seconds` of CPU work: the same rows, non-causal
        then causal.  Returns (TFLOPS-equivalent, seconds, description)."""
        np = self.np
        n = int(min(B * H * N, max(256, seconds / 1.5 / self.per_row)))
        rows = np.sort(self.rng.choice(B * H * N, size=n, replace=False))
        t0 = time.perf_counter()
        self.oracle.attention(self.q, self.k, self.v, self.scale, causal=False, rows=rows, nthreads=self.threads)
        self.oracle.attention(self.q, self.k, self.v, self.scale, causal=True, rows=rows, nthreads=self.threads)
        secs = time.perf_counter() - t0
        flops = 4.0 * D * N * n + 4.0 * D * float(np.sum(rows % N + 1))
        desc = ("float64 oracle (three-pass softmax per row) on %d of %d rows, non-causal and causal, "
                "of the step's workload; FLOPs = 4*d per visible (row, key) pair" % (n, B * H * N))
        return flops / secs / 1e12, secs, desc


def cpu_baseline(sample_seconds):
    sampler = OracleSampler()
    val, secs, desc = sampler.run(sample_seconds)
    return {"value": round(val, 6), "unit": "TFLOPS", "cores": sampler.threads, "kind": "oracle",
            "sample": desc, "seconds": round(secs, 2)}


def run_reference(args, rank, world):
    if rank != 0:
        return
    sampler = OracleSampler()
    per_step = max(0.2, args.cpu_seconds / max(1, args.steps))
    for _ in range(args.warmup):
        sampler.run(per_step / 2)
    vals, secs, desc = [], [], ""
    for _ in range(args.steps):
        v, s, desc = sampler.run(per_step)
        vals.append(v)
        secs.append(s)
    value = statistics.mean(vals)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.mean(secs), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1), rounded to bf16)",
        "config": {"workload": WORKLOAD, "B": B, "H": H, "Nq": N, "Nk": N, "d": D},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": sampler.threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_profile_case(args):
    """Small fixed workloads for ncu captures: warm-up, then --steps launches of one case."""
    import torch

    import attention_attn_fwd_03_gb300 as attn
    from attention_attn_fwd_03_gb300 import inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    attn.lib()
    case = args.profile_case
    if case == "step":
        q, k, v = (t.to(dev) for t in inputs.dense_qkv(B, H, N, N, D, seed=0))
        fns = [lambda: attn.fwd(q, k, v, causal=False), lambda: attn.fwd(q, k, v, causal=True)]
    elif case == "long_small":
        q, k, v = (t.to(dev) for t in inputs.dense_qkv(1, 4, 32768, 32768, 128, seed=0))
        fns = [lambda: attn.fwd(q, k, v, causal=True)]
    elif case == "fp8":
        q, k, v = inputs.dense_qkv(2, 16, 8192, 8192, 128, seed=0)
        (q8, dq), (k8, dk), (v8, dv) = (inputs.fp8_quantize(t) for t in (q, k, v))
        q8, k8, v8 = q8.to(dev), k8.to(dev), v8.to(dev)
        fns = [lambda: attn.fwd_fp8(q8, k8, v8, (dq, dk, dv))]
    elif case == "decode_small":
        p = inputs.paged_kv(B=8, H=32, d=128, page_size=64, max_pages=128, num_pages=1024, len_lo=512,
                            len_hi=8192, seed=0, device=dev)
        fns = [lambda: attn.paged_decode(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"])]
    elif case == "gqa_decode_small":
        p = inputs.paged_kv(B=16, H=32, d=128, page_size=64, max_pages=128, num_pages=2048, len_lo=512,
                            len_hi=8192, seed=0, device=dev, H_kv=8)
        fns = [lambda: attn.paged_fwd(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"])]
    elif case == "gqa_decode":
        p = inputs.paged_kv(B=64, H=32, d=128, page_size=64, max_pages=128, num_pages=8192, len_lo=512,
                            len_hi=8192, seed=0, device=dev, H_kv=8)
        fns = [lambda: attn.paged_fwd(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"])]
    elif case == "bwd_small":
        q, k, v = (t.to(dev) for t in inputs.dense_qkv(1, 8, 2048, 2048, 128, seed=0))
        do = torch.randn((1, 8, 2048, 128), generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).to(dev)
        o, lse = attn.fwd(q, k, v, causal=True)
        fns = [lambda: attn.bwd(q, k, v, o, lse, do, causal=True)]
    elif case == "chunks_small":
        p = inputs.paged_chunks(B=2, H=32, H_kv=8, d=128, page_size=64, max_pages=128, num_pages=256,
                                q_lo=2048, q_hi=2048, ctx_lo=6144, ctx_hi=6144, seed=0, device=dev)
        fns = [lambda: attn.paged_fwd(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"],
                                      cu_seqlens_q=p["cu_seqlens_q"], max_q_len=2048, causal=True)]
    elif case == "chunks":
        p = inputs.paged_chunks(B=8, H=32, H_kv=8, d=128, page_size=64, max_pages=128, num_pages=1024,
                                q_lo=2048, q_hi=2048, ctx_lo=6144, ctx_hi=6144, seed=0, device=dev)
        fns = [lambda: attn.paged_fwd(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"],
                                      cu_seqlens_q=p["cu_seqlens_q"], max_q_len=2048, causal=True)]
    elif case == "varlen":
        p = inputs.varlen_qkv(B=16, H=32, H_kv=8, d=128, q_lo=512, q_hi=4096, seed=0, device=dev)
        fns = [lambda: attn.varlen_fwd(p["q"], p["k"], p["v"], p["cu_seqlens_q"], p["cu_seqlens_k"],
                                       max_q_len=p["max_q_len"], max_k_len=p["max_k_len"], causal=True)]
    else:
        raise SystemExit("unknown --profile-case %s" % case)
    for _ in range(args.warmup):
        for f in fns:
            f()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.steps):
        for f in fns:
            f()
    e.record()
    e.synchronize()
    attn.device_status()
    print(json.dumps({"profile_case": case, "launches": args.steps * len(fns),
                      "ms_per_iteration": s.elapsed_time(e) / args.steps}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", choices=["step", "long_small", "fp8", "decode_small", "gqa_decode_small",
                                               "gqa_decode", "chunks_small", "chunks", "bwd_small", "varlen"], default=None,
                    help="run one small workload for an ncu capture instead of the benchmark")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    rank, world, local_rank = dist_env()
    if args.profile_case:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
