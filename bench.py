#!/usr/bin/env python3
"""Throughput benchmark of the GB300 attention library.

One step = one pass of the prefill hot path over the long-context causal
workload (B=1, H=32, Nq=Nk=32768, d=128, bf16, causal): one attn_fwd call on
inputs already resident in HBM (805 MB of Q/K/V, larger than the 129 MB L2;
L2 is also flushed with a 256 MB write before every timed step, outside the
timed events).  The headline metric is TFLOPS with the algorithmic count
4*B*H*Nq*Nk*d halved for the causal mask.

The line carries, for that kernel:
  roofline     achieved FLOP/s (CUDA events per launch) against the measured
               dense bf16 burst peak, with the DRAM traffic per launch from the
               committed ncu capture;
  spec_peak    the dense bf16 rate derived on this device: SM count x the
               tensor core's measured FLOP per SM cycle (attn_selftest_mma_rate)
               x SM clock, at the maximum and at the sampled clock;
  e2e          the same step from page-locked host buffers through
               attn_fwd_host (Q, K, V copied in and O, LSE copied out every
               step, overlapped with the kernels);
  cpu_baseline the float64 oracle on the host cores over a stratified row
               sample of the workload (FLOPs counted exactly per visible
               (row, key) pair), extrapolated to the whole workload.

`workloads` holds every other configuration, each with its own roofline and
its own oracle timing: the batched prefill (4x16x2048, non-causal and
causal), FP8 prefill (2x16x8192), paged decode (64 requests, H=32, 64-token
pages) and its grouped-query form (32 query / 8 KV heads), prefill chunks
over a paged cache, a variable-length batch, and the backward pass.

`--impl reference` times the float64 CPU oracle (the only reference this
method has) on bounded row samples of the same workload.

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

# the headline workload: long-context causal prefill
B, H, N, D = 1, 32, 32768, 128
CAUSAL = True
WORKLOAD = "long-context causal prefill B=1 H=32 Nq=Nk=32768 d=128 bf16"
METRIC = "attention fwd TFLOPS and % of GB300 tensor peak; paged decode HBM GB/s"
# the batched prefill workload (reported under workloads)
B2, H2, N2 = 4, 16, 2048
MMA_FLOP = 2 * 128 * 128 * 16  # one 128x128x16 tcgen05.mma


def prefill_flops(b, h, nq, nk, d, causal):
    f = 4.0 * b * h * nq * nk * d
    return f / 2 if causal else f


STEP_FLOPS = prefill_flops(B, H, N, N, D, CAUSAL)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "sm_max_mhz": float(pk.get("sm_max_mhz", 2070.0)), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0,
                "source": "fallback"}


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


# ---------------------------------------------------------------- tensor-core rate and rooflines

def measure_tensor_rate(torch, attn, dev):
    """Dense bf16 FLOP per SM cycle of back-to-back 128x128x16 tcgen05.mma,
    one CTA per SM (attn_selftest_mma_rate).  Returns (SMs, median, min, max)."""
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    cyc = torch.zeros(n_sm, dtype=torch.int64, device=dev)
    n_groups = 4096
    st = attn.attn_selftest_mma_rate(cyc.data_ptr(), n_sm, n_groups, torch.cuda.current_stream(dev).cuda_stream)
    if st != attn.ATTN_OK:
        raise attn.AttnError(st, "attn_selftest_mma_rate")
    attn.device_status()
    rates = [4.0 * n_groups * MMA_FLOP / c for c in cyc.cpu().tolist() if c > 0]
    if not rates:
        raise RuntimeError("tensor-core rate check returned no timings")
    return n_sm, statistics.median(rates), min(rates), max(rates)


class SpecPeak:
    """Dense bf16 peak of this device: SM count x measured FLOP per SM cycle x SM clock."""

    def __init__(self, n_sm, rate, rate_lo, rate_hi, max_mhz):
        self.n_sm, self.rate, self.lo, self.hi, self.max_mhz = n_sm, rate, rate_lo, rate_hi, max_mhz
        self.sampled_mhz = None

    def tflops(self, mhz):
        return self.n_sm * self.rate * mhz * 1e6 / 1e12

    def record(self, achieved_tflops, fp8=False):
        """Fractions of the spec peak for a tensor-bound kernel (FP8: 2x, the nominal fp8:bf16 dense ratio)."""
        mult = 2.0 if fp8 else 1.0
        r = {"frac_of_spec_at_max_clock": round(achieved_tflops / (mult * self.tflops(self.max_mhz)), 4)}
        if self.sampled_mhz:
            r["frac_of_spec_at_sampled_clock"] = round(achieved_tflops / (mult * self.tflops(self.sampled_mhz)), 4)
            r["achieved_flop_per_sm_cycle"] = round(achieved_tflops * 1e12 / (self.n_sm * self.sampled_mhz * 1e6), 1)
        return r

    def summary(self):
        r = {"value": round(self.tflops(self.max_mhz), 1), "unit": "TFLOP/s", "clock_mhz": self.max_mhz,
             "derivation": "SMs (%d, cudaGetDeviceProperties) x %.0f dense bf16 FLOP per SM cycle (measured: "
                           "back-to-back 128x128x16 tcgen05.mma from shared memory into tensor memory, one CTA "
                           "per SM, attn_selftest_mma_rate; per-SM range %.0f..%.0f) x SM clock"
                           % (self.n_sm, self.rate, self.lo, self.hi),
             "flop_per_sm_cycle": round(self.rate, 1), "sms": self.n_sm}
        if self.sampled_mhz:
            r["at_sampled_clock"] = {"value": round(self.tflops(self.sampled_mhz), 1),
                                     "clock_mhz": self.sampled_mhz}
        return r


def tensor_roofline(achieved, peaks, kernel, traffic, fp8=False, sustained=False):
    """`sustained`: the kernel ran back to back for a second or more (power-capped), so the denominator is
    the measured sustained bf16 rate; otherwise the burst rate (a kernel timed alone). Both fractions are
    reported."""
    mult = 2.0 if fp8 else 1.0
    burst = peaks["bf16_tflops"] * mult
    sus = peaks["bf16_tflops_sustained"] * mult
    peak = sus if sustained else burst
    src = peaks["source"] + (" dense bf16 sustained (seconds-long loop, power-capped; the kernel timed the same way)"
                             if sustained else " dense bf16 burst (kernel timed alone)")
    if fp8:
        src += " x 2 (nominal fp8:bf16 dense ratio)"
    return {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "frac_of_burst_peak": round(achieved / burst, 4),
            "frac_of_sustained_peak": round(achieved / sus, 4), "traffic": traffic, "kernel": kernel,
            "peak_source": src}


def hbm_roofline(achieved_gbs, peaks, kernel, traffic):
    return {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved_gbs / peaks["hbm_gbs"], 4), "frac_of_8TBps": round(achieved_gbs / 8000.0, 4),
            "traffic": traffic, "kernel": kernel,
            "peak_source": peaks["source"] + " HBM copy bandwidth (read + write bytes)"}


# ---------------------------------------------------------------- oracle timings (CPU baselines)

def _oracle_threads():
    import oracle
    return oracle.default_threads()


def _baseline(value, unit, secs, sample, extra=None):
    r = {"value": round(value, 6), "unit": unit, "cores": _oracle_threads(), "kind": "oracle", "sample": sample,
         "seconds": round(secs, 2)}
    if extra:
        r.update(extra)
    return r


def causal_row_flops(rows, Nq, Nk, d):
    """Exact FLOPs (4*d per visible (row, key) pair) of flattened BHSD rows under the bottom-right mask."""
    import numpy as np
    i = np.asarray(rows, dtype=np.int64) % Nq
    vis = np.clip(i + 1 + (Nk - Nq), 0, Nk)
    return 4.0 * d * float(vis.sum())


class LongCausalOracle:
    """The float64 oracle on row samples of the headline workload (the long
    causal prefill); its rate calibrated once on a small random sample."""

    def __init__(self, qkv=None):
        import numpy as np

        import oracle
        from attention_attn_fwd_03_gb300 import inputs

        self.np, self.oracle, self.inputs = np, oracle, inputs
        self.q, self.k, self.v = qkv if qkv is not None else inputs.dense_qkv(B, H, N, N, D, seed=0)
        self.scale = float(np.float32(1.0 / math.sqrt(D)))
        self.rng = np.random.default_rng(0)
        cal = np.sort(self.rng.choice(B * H * N, size=64, replace=False))
        t0 = time.perf_counter()
        oracle.attention(self.q, self.k, self.v, self.scale, causal=CAUSAL, rows=cal)
        self.rate = causal_row_flops(cal, N, N, D) / max(time.perf_counter() - t0, 1e-6)

    def _time(self, rows):
        t0 = time.perf_counter()
        self.oracle.attention(self.q, self.k, self.v, self.scale, causal=CAUSAL, rows=rows)
        secs = time.perf_counter() - t0
        return causal_row_flops(rows, N, N, D) / secs / 1e12, secs

    def random_sample(self, seconds):
        """Uniformly drawn rows worth about `seconds` of work: (TFLOPS, seconds, rows)."""
        n = int(min(B * H * N, max(16, seconds * self.rate / (4.0 * D * N / 2))))
        rows = self.np.sort(self.rng.choice(B * H * N, size=n, replace=False))
        tf, secs = self._time(rows)
        return tf, secs, n

    def stratified(self, seconds):
        """The stratified row set (first and last 128 rows, tile-boundary rows,
        random rows) of as many heads as fit in about `seconds`, then random
        rows over all heads for the rest of the time."""
        np = self.np
        per_head = self.inputs.sample_rows(1, N, n_random=0, tile=128, seed=0)
        head_flops = causal_row_flops(per_head, N, N, D)
        n_heads = int(max(1, min(H, 0.5 * seconds * self.rate // head_flops)))
        strata = (np.arange(n_heads, dtype=np.int64)[:, None] * N + per_head[None, :]).ravel()
        left = max(0.0, seconds * self.rate - n_heads * head_flops)
        n_rand = int(min(B * H * N, max(16, left / (4.0 * D * N / 2))))
        rows = np.unique(np.concatenate([strata, self.rng.choice(B * H * N, size=n_rand, replace=False)]))
        tf, secs = self._time(rows)
        full_s = STEP_FLOPS / (tf * 1e12)
        desc = ("float64 oracle (three-pass softmax per row) on %d of %d rows of the workload: the stratified set "
                "(rows 0-127, the last 128 rows, every tile-boundary row) of %d heads plus %d uniformly drawn rows "
                "over all heads; FLOPs = 4*d per visible (row, key) pair; the whole workload extrapolated by its "
                "exact visible-pair count" % (rows.size, B * H * N, n_heads, n_rand))
        return _baseline(tf, "TFLOPS", secs, desc, {"extrapolated": True,
                                                    "extrapolated_full_workload_seconds": round(full_s, 1)})


def oracle_dense(qkv, causal, seconds, descales=None, label="prefill"):
    """The oracle on a dense prefill workload: in full when it fits in about
    `seconds` (rate estimated on a small sample), else on uniformly drawn rows."""
    import numpy as np

    import oracle
    q, k, v = qkv
    BH = q.shape[0] * q.shape[1]
    Nq, Nk, d = q.shape[2], k.shape[2], q.shape[3]
    scale = float(np.float32(1.0 / math.sqrt(d)))
    ds = descales or (1.0, 1.0, 1.0)
    rng = np.random.default_rng(1)

    def rows_flops(rows):
        if causal:
            return causal_row_flops(rows, Nq, Nk, d)
        return 4.0 * d * Nk * len(rows)

    cal = np.sort(rng.choice(BH * Nq, size=min(BH * Nq, 64), replace=False))
    t0 = time.perf_counter()
    oracle.attention(q, k, v, scale, causal=causal, rows=cal, descales=ds)
    rate = rows_flops(cal) / max(time.perf_counter() - t0, 1e-6)
    total = prefill_flops(1, BH, Nq, Nk, d, False) if not causal else causal_row_flops(np.arange(Nq), Nq, Nk, d) * BH
    if total <= 1.5 * seconds * rate:
        rows, what = None, "all %d rows" % (BH * Nq)
        flops = total
    else:
        per_row = total / (BH * Nq)
        n = int(max(64, seconds * rate / per_row))
        rows = np.sort(rng.choice(BH * Nq, size=n, replace=False))
        flops, what = rows_flops(rows), "%d uniformly drawn of %d rows" % (n, BH * Nq)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, scale, causal=causal, rows=rows, descales=ds)
    secs = time.perf_counter() - t0
    desc = ("float64 oracle (three-pass softmax per row) on %s of the %s workload%s; FLOPs = 4*d per visible "
            "(row, key) pair" % (what, label, " (dequantised e4m3 inputs)" if descales else ""))
    return _baseline(flops / secs / 1e12, "TFLOPS", secs, desc)


def _paged_subset(p, reqs, token_major_q=False):
    """CPU copies of requests `reqs` of a paged workload with only their pages,
    renumbered: (q, k_cache, v_cache, block_table, seq_lens, cu_seqlens_q)."""
    import torch
    bt = p["block_table"].cpu()
    sl = p["seq_lens"].cpu()
    page = p["k_cache"].shape[1]
    ids, rows = [], []
    new_bt = torch.full((len(reqs), bt.shape[1]), -1, dtype=torch.int32)
    for i, r in enumerate(reqs):
        n = (int(sl[r]) + page - 1) // page
        new_bt[i, :n] = torch.arange(len(ids), len(ids) + n, dtype=torch.int32)
        ids.extend(int(x) for x in bt[r, :n])
    idx = torch.tensor(ids if ids else [0], dtype=torch.int64, device=p["k_cache"].device)
    kc = p["k_cache"].index_select(0, idx).cpu()
    vc = p["v_cache"].index_select(0, idx).cpu()
    cu = None
    if token_major_q:
        cu_all = p["cu_seqlens_q"].cpu()
        parts, cu_l = [], [0]
        for r in reqs:
            a, e = int(cu_all[r]), int(cu_all[r + 1])
            parts.append(p["q"][a:e].cpu())
            cu_l.append(cu_l[-1] + e - a)
        q = torch.cat(parts)
        cu = torch.tensor(cu_l, dtype=torch.int32)
    else:
        q = p["q"][torch.tensor(reqs, device=p["q"].device)].cpu()
    return q, kc, vc, new_bt, sl[reqs].clone(), cu


def oracle_decode(p, H_kv, n_req, label):
    """The oracle on the first n_req requests of a paged decode workload, as
    GB/s of the same algorithmic bytes the GPU figure counts."""
    import numpy as np

    import oracle
    reqs = list(range(n_req))
    q, kc, vc, bt, sl, _ = _paged_subset(p, reqs)
    H_q, d = q.shape[1], q.shape[2]
    page = kc.shape[1]
    scale = float(np.float32(1.0 / math.sqrt(d)))
    t0 = time.perf_counter()
    if H_kv == H_q:
        oracle.paged_decode(q, kc, vc, bt, sl, scale)
    else:
        oracle.paged_attention(q, kc, vc, bt, sl, scale)
    secs = time.perf_counter() - t0
    nbytes = decode_bytes(sl, H_q, H_kv, d, page)
    desc = ("float64 oracle on %d of the %d requests of the %s workload (all their keys); GB/s of the "
            "algorithmic bytes (K/V of every visible token, q, o, LSE, tables)" % (n_req, p["seq_lens"].numel(),
                                                                                   label))
    return _baseline(nbytes / secs / 1e9, "GB/s", secs, desc)


def decode_bytes(seq_lens, H_q, H_kv, d, page):
    lens = seq_lens.long().cpu()
    B_ = lens.numel()
    tokens = int(lens.sum())
    n_pages = int(((lens + page - 1) // page).sum())
    return tokens * H_kv * d * 2 * 2 + 2 * (B_ * H_q * d * 2) + B_ * H_q * 4 + n_pages * 4 + B_ * 4


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

    # the tensor core's dense bf16 rate per SM cycle (for the spec peak)
    n_sm, rate, rate_lo, rate_hi = measure_tensor_rate(torch, attn, dev)
    spec = SpecPeak(n_sm, rate, rate_lo, rate_hi, peaks["sm_max_mhz"])

    # inputs: seeded per rank (each rank is an independent replica)
    qc, kc, vc = inputs.dense_qkv(B, H, N, N, D, seed=rank)
    q, k, v = qc.to(dev), kc.to(dev), vc.to(dev)
    o, l = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=dev)

    def step():
        attn.fwd(q, k, v, causal=CAUSAL, out=o, lse=l)

    for _ in range(args.warmup):
        flush()
        step()
    attn.device_status()

    # ---- timed region: exactly K steps, one prefill launch each
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
    clocks = clk.summary()
    spec.sampled_mhz = clocks.get("sm_mhz")

    # ---- end to end through the public API from pinned host buffers: attn_fwd_host
    # pipelines the copies in, the kernels and the copies out over chunks of
    # (b, h) pairs.  For comparison, the same step with serial copies around
    # the device entry point.
    hq, hk, hv = (t.pin_memory() for t in (qc, kc, vc))
    ho = torch.empty((B, H, N, D), dtype=torch.bfloat16).pin_memory()
    hl = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    host_ws = torch.empty(attn.attn_fwd_host_workspace_size(B, H, N, N, D, 1, 0), dtype=torch.uint8, device=dev)

    def e2e_step():
        attn.fwd_host(hq, hk, hv, causal=(CAUSAL,), out=[ho], lse=[hl], workspace=host_ws, synchronize=False)

    dq_, dk_, dv_ = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def serial_step():
        dq_.copy_(hq, non_blocking=True)
        dk_.copy_(hk, non_blocking=True)
        dv_.copy_(hv, non_blocking=True)
        attn.fwd(dq_, dk_, dv_, causal=CAUSAL, out=o, lse=l)
        ho.copy_(o, non_blocking=True)
        hl.copy_(l, non_blocking=True)

    for _ in range(2):
        e2e_step()
        serial_step()
    torch.cuda.synchronize()
    e2e_ms = timed_launches(torch, e2e_step, max(3, min(args.steps, 10)), flush)
    serial_ms = timed_launches(torch, serial_step, max(3, min(args.steps, 10)), flush)
    attn.device_status()
    del dq_, dk_, dv_, host_ws
    h2d = 3 * q.numel() * 2
    d2h = o.numel() * 2 + l.numel() * 4
    e2e_val = STEP_FLOPS / (statistics.mean(e2e_ms) * 1e-3) / 1e12

    # ---- dominant kernel roofline: the prefill kernel, one launch per step
    launch_ms = statistics.mean(step_ms)
    achieved = STEP_FLOPS / (launch_ms * 1e-3) / 1e12
    timed_s = sum(step_ms) * 1e-3
    roof = tensor_roofline(achieved, peaks, "prefill_sp_kernel<128,bf16>",
                           traffic_record("prefill_sp.cu", "prefill_sp_bf16_d128_long_causal"),
                           sustained=timed_s >= 1.0)
    roof["timed_region_s"] = round(timed_s, 3)
    roof["algorithmic_bytes"] = 3 * q.numel() * 2 + o.numel() * 2 + l.numel() * 4
    roof.update(spec.record(achieved))

    secondary = {}
    if not args.no_secondary:
        del hq, hk, hv, ho, hl
        secondary = run_secondary(torch, attn, inputs, dev, flush, peaks, spec, rank,
                                  with_oracle=(rank == 0 and world == 1 and not args.no_cpu_baseline),
                                  oracle_seconds=args.cpu_seconds)

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
        "config": {"workload": WORKLOAD, "B": B, "H": H, "Nq": N, "Nk": N, "d": D, "causal": CAUSAL,
                   "flops_per_step": STEP_FLOPS, "flops_convention": "4*B*H*Nq*Nk*d, halved for causal",
                   "l2": "inputs (805 MB) larger than L2; L2 also flushed (256 MB write) before every timed step, "
                         "outside the timed events",
                   "parallelism": "replicas (one independent workload per GPU)"},
        "roofline": roof,
        "spec_peak": spec.summary(),
        "e2e": {"value": round(e2e_val, 3), "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(statistics.mean(e2e_ms), 4),
                "api": "attn_fwd_host (chunked copy-in / kernels / copy-out pipeline, pinned host buffers)",
                "serial_copies_ms_per_step": round(statistics.mean(serial_ms), 4)},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "workloads": secondary,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = LongCausalOracle((qc, kc, vc)).stratified(args.cpu_seconds)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_secondary(torch, attn, inputs, dev, flush, peaks, spec, rank, with_oracle, oracle_seconds):
    """Every other workload: its own timing, roofline and (rank 0, one GPU) oracle timing."""
    out = {}
    reps = 5
    osec = max(2.0, oracle_seconds / 2)

    def prefill_entry(name, ms, flops, kernel, traffic_key, oracle_fn, fp8=False, kernel_file="prefill.cu"):
        tf = flops / (statistics.mean(ms) * 1e-3) / 1e12
        roof = tensor_roofline(tf, peaks, kernel, traffic_record(kernel_file, traffic_key), fp8=fp8)
        roof.update(spec.record(tf, fp8=fp8))
        e = {"value": round(tf, 2), "unit": "TFLOPS", "ms": round(statistics.mean(ms), 4), "flops": flops,
             "roofline": roof}
        if with_oracle and oracle_fn is not None:
            e["cpu_baseline"] = oracle_fn()
        out[name] = e

    # ---- batched prefill, both mask modes (the small batched workload)
    qc, kc, vc = inputs.dense_qkv(B2, H2, N2, N2, D, seed=rank)
    q, k, v = qc.to(dev), kc.to(dev), vc.to(dev)
    o, l = torch.empty_like(q), torch.empty((B2, H2, N2), dtype=torch.float32, device=dev)
    for causal in (False, True):
        attn.fwd(q, k, v, causal=causal, out=o, lse=l)
        ms = timed_launches(torch, lambda: attn.fwd(q, k, v, causal=causal, out=o, lse=l), reps, flush)
        attn.device_status()
        prefill_entry("batched_prefill_4x16x2048_d128_%s" % ("causal" if causal else "non_causal"), ms,
                      prefill_flops(B2, H2, N2, N2, D, causal), "prefill_kernel<128,bf16>",
                      "prefill_bf16_d128_batched_%s" % ("causal" if causal else "noncausal"),
                      lambda: oracle_dense((qc, kc, vc), causal, osec, label="batched prefill"))
    del q, k, v, o, l

    # ---- FP8 prefill
    qc8, kc8, vc8 = inputs.dense_qkv(2, 16, 8192, 8192, 128, seed=rank)
    (q8, dq), (k8, dk), (v8, dv) = (inputs.fp8_quantize(t) for t in (qc8, kc8, vc8))
    del qc8, kc8, vc8
    g8 = [t.to(dev) for t in (q8, k8, v8)]
    o, l = torch.empty((2, 16, 8192, 128), dtype=torch.bfloat16, device=dev), \
        torch.empty((2, 16, 8192), dtype=torch.float32, device=dev)
    attn.fwd_fp8(*g8, (dq, dk, dv), out=o, lse=l)
    ms = timed_launches(torch, lambda: attn.fwd_fp8(*g8, (dq, dk, dv), out=o, lse=l), reps, flush)
    attn.device_status()
    prefill_entry("fp8_prefill_2x16x8192_d128", ms, prefill_flops(2, 16, 8192, 8192, 128, False),
                  "prefill_sp_kernel<128,e4m3>", "prefill_fp8_d128",
                  lambda: oracle_dense((q8, k8, v8), False, osec, descales=(dq, dk, dv), label="FP8 prefill"),
                  fp8=True, kernel_file="prefill_sp.cu")
    del g8, o, l, q8, k8, v8

    # ---- paged decode (multi-head, CUDA cores) and grouped-query decode (tensor cores)
    for H_kv, name, kernel, key in ((32, "paged_decode_64req_H32_d128_p64", "decode_split_kernel<128>",
                                     "decode_paged"),
                                    (8, "gqa_paged_decode_64req_H32_Hkv8_d128_p64", "paged_kernel<128>",
                                     "paged_gqa_decode")):
        p = inputs.paged_kv(B=64, H=32, d=128, page_size=64, max_pages=128, num_pages=8192, len_lo=512,
                            len_hi=8192, seed=rank, device=dev, H_kv=H_kv)
        o = torch.empty_like(p["q"])
        l = torch.empty((64, 32), dtype=torch.float32, device=dev)
        if H_kv == 32:
            ws = torch.empty(attn.attn_paged_decode_workspace_size(64, 32, 128, 128, 64), dtype=torch.uint8,
                             device=dev)

            def fn():
                attn.paged_decode(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"], out=o,
                                  lse=l, workspace=ws)
            kfile = "decode.cu"
        else:
            ws = torch.empty(max(1, attn.attn_paged_fwd_workspace_size(64, 64, 1, 32, 8, 128, 64, 128)),
                             dtype=torch.uint8, device=dev)

            def fn():
                attn.paged_fwd(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"], out=o, lse=l,
                               workspace=ws)
            kfile = "paged.cu"
        fn()
        ms = timed_launches(torch, fn, reps, flush)
        attn.device_status()
        nbytes = decode_bytes(p["seq_lens"], 32, H_kv, 128, 64)
        gbs = nbytes / (statistics.mean(ms) * 1e-3) / 1e9
        e = {"value": round(gbs, 1), "unit": "GB/s", "ms": round(statistics.mean(ms), 4),
             "algorithmic_bytes": nbytes, "tokens": int(p["seq_lens"].sum().item()),
             "roofline": hbm_roofline(gbs, peaks, kernel, traffic_record(kfile, key))}
        if with_oracle:
            e["cpu_baseline"] = oracle_decode(p, H_kv, 16, name)
        out[name] = e
        del p, o, l, ws
        torch.cuda.empty_cache()

    # ---- prefill chunks over a paged cache: 8 requests, 2048 new tokens after a 6144-token prefix, causal
    p = inputs.paged_chunks(B=8, H=32, H_kv=8, d=128, page_size=64, max_pages=128, num_pages=1024,
                            q_lo=2048, q_hi=2048, ctx_lo=6144, ctx_hi=6144, seed=rank, device=dev)
    o = torch.empty_like(p["q"])
    l = torch.empty((p["q"].shape[0], 32), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, attn.attn_paged_fwd_workspace_size(8, p["q"].shape[0], 2048, 32, 8, 128, 64, 128)),
                     dtype=torch.uint8, device=dev)

    def chunks():
        attn.paged_fwd(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"],
                       cu_seqlens_q=p["cu_seqlens_q"], max_q_len=2048, causal=True, out=o, lse=l, workspace=ws)
    chunks()
    ms = timed_launches(torch, chunks, reps, flush)
    attn.device_status()
    pairs = 8 * sum(6144 + i + 1 for i in range(2048))  # query i of a request sees 6144 + i + 1 keys

    def chunks_oracle():
        import numpy as np

        import oracle
        qs, kcs, vcs, bts, sls, cus = _paged_subset(p, [0], token_major_q=True)
        t0 = time.perf_counter()
        oracle.paged_attention(qs, kcs, vcs, bts, sls, float(np.float32(1 / math.sqrt(128))), cu_seqlens_q=cus,
                               causal=True)
        secs = time.perf_counter() - t0
        f = 4.0 * (pairs / 8) * 32 * 128
        return _baseline(f / secs / 1e12, "TFLOPS", secs,
                         "float64 oracle on 1 of the 8 requests (all 2048 new tokens x 32 heads, its 8192 cached "
                         "keys); FLOPs = 4*d per visible (query, key) pair")
    prefill_entry("paged_prefill_chunks_8x2048_over_6144_H32_Hkv8_d128_causal", ms, 4.0 * pairs * 32 * 128,
                  "prefill_kernel<128,bf16,ragged>", "ragged_prefill_chunks", chunks_oracle)
    del p, o, l, ws
    torch.cuda.empty_cache()

    # ---- variable-length batch prefill: 16 packed sequences of 512..4096 tokens, causal self-attention
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

    def varlen_oracle():
        import numpy as np

        import oracle
        cu, cuk = p["cu_seqlens_q"].cpu(), p["cu_seqlens_k"].cpu()
        # the shortest sequences up to about 1/16 of the batch's pairs
        order = sorted(range(16), key=lambda r: int(lens[r]))
        pick, got = [], 0
        for r in order:
            pick.append(r)
            got += int(lens[r]) * (int(lens[r]) + 1) // 2
            if got * 16 >= pairs:
                break
        pick.sort()
        qs = torch.cat([p["q"][int(cu[r]):int(cu[r + 1])].cpu() for r in pick])
        ks = torch.cat([p["k"][int(cuk[r]):int(cuk[r + 1])].cpu() for r in pick])
        vs = torch.cat([p["v"][int(cuk[r]):int(cuk[r + 1])].cpu() for r in pick])
        cs = torch.tensor([0] + list(np.cumsum([int(lens[r]) for r in pick])), dtype=torch.int32)
        t0 = time.perf_counter()
        oracle.varlen_attention(qs, ks, vs, cs, cs, float(np.float32(1 / math.sqrt(128))), causal=True)
        secs = time.perf_counter() - t0
        return _baseline(4.0 * got * 32 * 128 / secs / 1e12, "TFLOPS", secs,
                         "float64 oracle on %d of the 16 sequences (%d tokens x 32 heads); FLOPs = 4*d per "
                         "visible (query, key) pair" % (len(pick), sum(int(lens[r]) for r in pick)))
    prefill_entry("varlen_prefill_16seq_512-4096_H32_Hkv8_d128_causal", ms, 4.0 * pairs * 32 * 128,
                  "prefill_kernel<128,bf16,ragged>", "ragged_prefill_varlen", varlen_oracle)
    out["varlen_prefill_16seq_512-4096_H32_Hkv8_d128_causal"]["tokens"] = int(lens.sum())
    del p, o, l, ws
    torch.cuda.empty_cache()

    # ---- backward of the batched prefill (4 x 16 x 2048, d = 128): dQ, dK, dV by recomputation
    q, k, v = qc.to(dev), kc.to(dev), vc.to(dev)
    g = torch.Generator(device="cpu").manual_seed(rank + 1)
    doc = torch.randn((B2, H2, N2, D), generator=g, dtype=torch.float32).to(torch.bfloat16)
    do = doc.to(dev)
    ws = torch.empty(attn.attn_bwd_workspace_size(B2, H2, N2, D), dtype=torch.uint8, device=dev)
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    for causal in (False, True):
        o, l = attn.fwd(q, k, v, causal=causal)

        def bwd():
            attn.bwd(q, k, v, o, l, do, causal=causal, dq=grads[0], dk=grads[1], dv=grads[2], workspace=ws)
        bwd()
        ms = timed_launches(torch, bwd, reps, flush)
        attn.device_status()

        def bwd_oracle():
            import numpy as np

            import oracle
            sl = (slice(0, 1), slice(0, 2))  # 2 of the 64 (b, h) problems
            t0 = time.perf_counter()
            oracle.attention_bwd(qc[sl], kc[sl], vc[sl], doc[sl], float(np.float32(1 / math.sqrt(D))), causal=causal)
            secs = time.perf_counter() - t0
            f = 2.5 * prefill_flops(1, 2, N2, N2, D, causal)
            return _baseline(f / secs / 1e12, "TFLOPS", secs,
                             "float64 gradient oracle on 2 of the 64 (b, h) problems; FLOPs = 2.5x the forward "
                             "count (five products of the forward's size), halved for causal")
        prefill_entry("backward_4x16x2048_d128_%s" % ("causal" if causal else "non_causal"), ms,
                      2.5 * prefill_flops(B2, H2, N2, N2, D, causal), "bwd_pipe_kernel",
                      "backward_%s" % ("causal" if causal else "noncausal"), bwd_oracle, kernel_file="backward.cu")
    del q, k, v, do, ws, grads, o, l
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    """The float64 oracle, as it stands, on bounded row samples of the headline
    workload; rank 0 only."""
    if rank != 0:
        return
    sampler = LongCausalOracle()
    per_step = max(0.2, args.cpu_seconds / max(1, args.steps))
    for _ in range(args.warmup):
        sampler.random_sample(per_step / 2)
    vals, secs, n = [], [], 0
    for _ in range(args.steps):
        v, s, n = sampler.random_sample(per_step)
        vals.append(v)
        secs.append(s)
    value = statistics.mean(vals)
    desc = ("float64 oracle (three-pass softmax per row) on %d uniformly drawn of the %d rows of the workload per "
            "step; FLOPs = 4*d per visible (row, key) pair" % (n, B * H * N))
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
        "config": {"workload": WORKLOAD, "B": B, "H": H, "Nq": N, "Nk": N, "d": D, "causal": CAUSAL},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": _oracle_threads(), "kind": "oracle",
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
    if case == "step":  # the headline step (long causal prefill), full size
        q, k, v = (t.to(dev) for t in inputs.dense_qkv(B, H, N, N, D, seed=0))
        fns = [lambda: attn.fwd(q, k, v, causal=CAUSAL)]
    elif case == "batched":
        q, k, v = (t.to(dev) for t in inputs.dense_qkv(B2, H2, N2, N2, D, seed=0))
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
    elif case == "decode":  # the benchmark's paged decode workload, full size
        p = inputs.paged_kv(B=64, H=32, d=128, page_size=64, max_pages=128, num_pages=8192, len_lo=512,
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
    elif case == "bwd":  # the benchmark's backward workload (4 x 16 x 2048), non-causal then causal
        q, k, v = (t.to(dev) for t in inputs.dense_qkv(B2, H2, N2, N2, D, seed=0))
        do = torch.randn((B2, H2, N2, D), generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).to(dev)
        fw = [attn.fwd(q, k, v, causal=c) for c in (False, True)]
        fns = [lambda: attn.bwd(q, k, v, fw[0][0], fw[0][1], do, causal=False),
               lambda: attn.bwd(q, k, v, fw[1][0], fw[1][1], do, causal=True)]
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
    ap.add_argument("--profile-case", choices=["step", "batched", "long_small", "fp8", "decode_small", "decode", "gqa_decode_small",
                                               "gqa_decode", "chunks_small", "chunks", "bwd_small", "bwd", "varlen"], default=None,
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
