"""Benchmark of the exact-attention hot path on GB300.

One step = one pass of the forward kernel over the 8k causal prefill workload
(B1 H32 N8192 d128, bf16, seed 2), the headline of the metric (TFLOP/s of
algorithmic work: only unmasked score entries count).  The split-KV decode
over a 32768-token cache (B1 H32 d128, seed 4, automatic chunking) is timed
the same way each step and reported under "decode" (GB/s of K and V read).

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launching stream; the L2 cache is flushed (a 256 MiB write, then a
512 MiB read that writes the flush's dirty lines back) between
steps, outside the events.  Clocks are sampled with nvidia-smi during the
timed region.  `--impl reference` times the float64 CPU oracle instead, on a
bounded sample of the same workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
(N > 1 is launched by torchrun: one independent replica per GPU, weak scaling.)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOP/s vs BF16 TC peak; split-KV decode HBM GB/s vs peak"
PREFILL = "prefill_causal_b1h32_n8192_d128"
DECODE = "decode_b1h32_l32768_d128"
FLUSH_BYTES = 256 << 20
READBACK_BYTES = 512 << 20
# The L2 flush between timed steps: the read writes the fill's dirty lines back before the
# next step, so no step starts with inputs (or pending write-backs) in L2.
L2_NOTE = "flushed between steps outside the timed events (256 MiB write, then 512 MiB read)"


class L2Flush:
    """Evicts the L2 cache between timed steps.

    A write larger than L2 evicts the inputs but leaves L2 full of dirty lines,
    which the next kernel then writes back to HBM: on GB300 that adds ~9 us to
    the 83 us decode step.  A read of a second buffer larger than L2 after the
    write makes those write-backs happen here, outside the timed region; L2
    then holds clean lines of the read buffer only.  The read also keeps the
    GPU busy while the host enqueues the step, so the start event is not
    recorded on an idle GPU ahead of the host's launch."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(FLUSH_BYTES, device=device, dtype=torch.uint8)
        self.r = torch.ones(READBACK_BYTES // 4, device=device, dtype=torch.float32)
        self.acc = torch.empty((), device=device, dtype=torch.float32)

    def __call__(self, value=1):
        self.w.fill_(value)
        self.acc.copy_(self.r.sum())


def prefill_flops(B, H, N, d, causal):
    """Algorithmic FLOPs: 2*d for Q.K and 2*d for W.V per unmasked score."""
    pairs = N * (N + 1) // 2 if causal else N * N
    return 4.0 * d * pairs * B * H


def decode_bytes(H, lens, d):
    """Algorithmic bytes: every cached K and V row of every (b, h) read once."""
    return float(sum(2 * H * n * d * 2 for n in lens))


def spread(ms):
    """Mean, median, extremes and standard deviation of per-step times (ms)."""
    ms = list(ms)
    return {"mean": round(statistics.mean(ms), 4), "median": round(statistics.median(ms), 4),
            "min": round(min(ms), 4), "max": round(max(ms), 4),
            "stdev": round(statistics.stdev(ms), 4) if len(ms) > 1 else 0.0, "n": len(ms)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


KERNEL_SOURCES = {
    "prefill_kernel": ("fa_prefill.cu", "fa_ptx.cuh", "fa_internal.h", "fa_tmap.h"),
    "decode_split_kernel": ("fa_decode.cu", "fa_ptx.cuh", "fa_internal.h"),
    "bwd_main_kernel": ("fa_backward.cu", "fa_ptx.cuh", "fa_internal.h", "fa_tmap.h"),
}


def kernel_sources_hash(kernel):
    """Hash of the source files a kernel is compiled from (stale counters read as null)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_tiled_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if the kernels are unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get(kernel)
    if not ent or ent.get("sources_sha") != kernel_sources_hash(kernel):
        return None
    return ent.get("bytes_per_launch")


# ------------------------------------------------------------------ ranks
def max_over_ranks(values, device, world):
    """Element-wise maximum of per-rank timings (identity on one rank)."""
    if world <= 1:
        return list(values)
    import torch
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def replica_throughput(work_per_rank, ms_slowest, world):
    """Whole-job rate of `world` independent replicas: all ranks' work over the slowest rank's time."""
    return world * work_per_rank / (ms_slowest * 1e-3)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples, 5 ms apart, time-stamped (a 20-step run times ~16 ms).

    The sampler is started before the timed region and only its samples whose
    time stamps fall between mark_start() and mark_end() are summarised."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 5

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=self.file, stderr=subprocess.DEVNULL)
            # do not start timing before the sampler produces rows (bounded wait)
            deadline = time.time() + 10.0
            while time.time() < deadline and os.path.getsize(self.file.name) == 0:
                if self.proc.poll() is not None:
                    break
                time.sleep(0.02)
        except Exception:
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(2.5 * self.PERIOD_MS / 1000.0)  # let the last period's row land
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    @staticmethod
    def _stamp(text):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text, fmt).timestamp()
            except ValueError:
                pass
        return None

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.file.flush()
        with open(self.file.name) as f:
            rows = [[x.strip() for x in r.strip().split(",")] for r in f if r.strip()]
        os.unlink(self.file.name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        parsed = []
        for r in rows:
            if len(r) < 10:
                continue
            try:
                parsed.append((self._stamp(r[0]), float(r[2]), float(r[3]),
                               {n for n, v in zip(names, r[6:10]) if v.lower() == "active"}))
            except ValueError:
                continue
        inside = [x for x in parsed
                  if x[0] is not None and self.t0 is not None and self.t1 is not None
                  and self.t0 - 0.001 <= x[0] <= self.t1 + 0.001]
        use = inside if inside else parsed
        reasons = set().union(*(x[3] for x in use)) if use else set()
        return {"sm_mhz": statistics.median([x[1] for x in use]) if use else None,
                "sm_max_mhz": max(x[2] for x in use) if use else None,
                "reasons": sorted(reasons), "samples": len(inside),
                "samples_window": "inside the timed region" if inside else
                                  "none inside the timed region: all samples of the run"}


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import exact_attention_tiled_gb300 as fa
    from exact_attention_tiled_gb300 import workloads

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = fa.library()
    stream = torch.cuda.current_stream()
    peaks = load_peaks()

    # ---- inputs resident in HBM
    wp = workloads.WORKLOADS[PREFILL]
    Q, K, V = workloads.prefill_inputs(wp.B, wp.H, wp.N, wp.d, wp.seed, device=dev)
    O = torch.empty_like(Q)
    L = torch.empty((wp.B, wp.H, wp.N), device=dev, dtype=torch.float32)
    wd = workloads.WORKLOADS[DECODE]
    q, Kc, Vc = workloads.decode_inputs(wd.B, wd.H, wd.N, wd.d, wd.seed, device=dev)
    seqlens = workloads.decode_seqlens(wd.B, wd.N, wd.seed)
    seq_dev = seqlens.to(dev)
    Od = torch.empty_like(q)
    Ld = torch.empty((wd.B, wd.H), device=dev, dtype=torch.float32)
    ws = torch.empty(fa.fa_decode_workspace_bytes(wd.B, wd.H, wd.N, wd.d, 0, seqlens), device=dev,
                     dtype=torch.uint8)
    chunk, nchunk = fa.fa_decode_plan(wd.B, wd.H, wd.N, wd.d, 0, seqlens)
    flush = L2Flush(dev)

    def prefill():
        fa.fa_forward(Q, K, V, causal=True, out=O, lse=L)

    def decode():
        fa.fa_decode(q, Kc, Vc, seq_dev, num_splits=0, seqlens_host=seqlens, out=Od, lse=Ld,
                     workspace=ws)

    # ---- warm-up: the timed step exactly, flushes included (the first flush of the
    # process is otherwise the first timed step's, and that step runs ~40 % slower)
    for _ in range(args.warmup):
        flush(1)
        prefill()
        flush(2)
        decode()
        torch.cuda.synchronize()
    torch.cuda.synchronize()
    st, site = fa.fa_device_error(clear=True)
    if st != 0:
        raise RuntimeError(f"device error word set during warm-up (site {site:#x})")

    ev = lambda: torch.cuda.Event(enable_timing=True)
    pf_ms, dc_ms = [], []
    launches = 0
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        clk.mark_start()
        t_wall = time.perf_counter()
        for _ in range(args.steps):
            flush(1)
            a, b = ev(), ev()
            a.record(stream)
            prefill()
            b.record(stream)
            launches += 1
            flush(2)
            c, d = ev(), ev()
            c.record(stream)
            decode()
            d.record(stream)
            launches += 2
            torch.cuda.synchronize()
            pf_ms.append(a.elapsed_time(b))
            dc_ms.append(c.elapsed_time(d))
        torch.cuda.synchronize()
        wall = time.perf_counter() - t_wall
        clk.mark_end()
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.summary()
    st, site = fa.fa_device_error(clear=True)
    if st != 0:
        raise RuntimeError(f"device error word set during timing (site {site:#x})")

    # ---- chunk-count sweep of the decode path (same inputs, L2 flushed each time)
    sweep = {}
    for splits in tuple(wd.splits) + (0,):
        ws_s = torch.empty(fa.fa_decode_workspace_bytes(wd.B, wd.H, wd.N, wd.d, splits, seqlens),
                           device=dev, dtype=torch.uint8)
        ts = []
        for i in range(3 + 5):
            flush(4)
            a, b = ev(), ev()
            a.record(stream)
            fa.fa_decode(q, Kc, Vc, seq_dev, num_splits=splits, seqlens_host=seqlens, out=Od, lse=Ld,
                         workspace=ws_s)
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                ts.append(a.elapsed_time(b))
        sweep["auto" if splits == 0 else str(splits)] = round(
            decode_bytes(wd.H, seqlens.tolist(), wd.d) / (statistics.mean(ts) * 1e-3) / 1e9, 1)

    # ---- the other two workload shapes, timed the same way (reported, not the headline)
    def timed(fn, iters=10, warm=3):
        ts = []
        for i in range(warm + iters):
            flush(5)
            a, b = ev(), ev()
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            if i >= warm:
                ts.append(a.elapsed_time(b))
        return statistics.mean(ts)

    others = {}
    w3 = workloads.WORKLOADS["prefill_b8h16_n2048_d64"]
    Q3, K3, V3 = workloads.prefill_inputs(w3.B, w3.H, w3.N, w3.d, w3.seed, w3.amp, device=dev)
    kl3 = workloads.key_lengths(w3.B, w3.N, w3.key_len_seed)
    kl3d = kl3.to(dev)
    for name, kl in (("prefill_b8h16_n2048_d64", None), ("prefill_b8h16_n2048_d64_keypad", kl3d)):
        ms = timed(lambda: fa.fa_forward(Q3, K3, V3, causal=False, key_len=kl))
        fl = prefill_flops(w3.B, w3.H, w3.N, w3.d, False) if kl is None else \
            4.0 * w3.d * w3.N * float(kl3.sum()) * w3.H
        others[name] = {"ms": round(ms, 4), "flops": fl, "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
                        "frac_of_bf16_peak": round(fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)}
    del Q3, K3, V3
    w5 = workloads.WORKLOADS["decode_varlen_b16h32_d128"]
    q5, K5, V5 = workloads.decode_inputs(w5.B, w5.H, w5.N, w5.d, w5.seed, device=dev)
    sl5 = workloads.decode_seqlens(w5.B, w5.N, w5.seed, w5.seqlen_range)
    sl5d = sl5.to(dev)
    ws5 = torch.empty(fa.fa_decode_workspace_bytes(w5.B, w5.H, w5.N, w5.d, 0, sl5), device=dev, dtype=torch.uint8)
    ms = timed(lambda: fa.fa_decode(q5, K5, V5, sl5d, num_splits=0, seqlens_host=sl5, workspace=ws5))
    by5 = decode_bytes(w5.H, sl5.tolist(), w5.d)
    c5, n5 = fa.fa_decode_plan(w5.B, w5.H, w5.N, w5.d, 0, sl5)
    others["decode_varlen_b16h32_d128"] = {"ms": round(ms, 4), "bytes": by5, "gbs": round(by5 / (ms * 1e-3) / 1e9, 1),
                                           "frac_of_hbm_peak": round(by5 / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                                           "chunk_len": c5, "max_chunks": n5}
    del q5, K5, V5
    # paged cache: the decode workload's shape held in scattered blocks of a pool
    for bs in (16, 64):
        qp, Kp, Vp, tbl, slp = workloads.paged_inputs(wd.B, wd.H, bs, wd.d, seqlens, wd.seed, device=dev)
        tbld, slpd = tbl.to(dev), slp.to(dev)
        wsp = torch.empty(fa.fa_decode_workspace_bytes(wd.B, wd.H, tbl.shape[1] * bs, wd.d, 0, slp), device=dev,
                          dtype=torch.uint8)
        ms = timed(lambda: fa.fa_decode_paged(qp, Kp, Vp, tbld, slpd, num_splits=0, seqlens_host=slp,
                                              workspace=wsp))
        byp = decode_bytes(wd.H, slp.tolist(), wd.d)
        others[f"decode_paged_b1h32_l32768_d128_bs{bs}"] = {
            "ms": round(ms, 4), "bytes": byp, "gbs": round(byp / (ms * 1e-3) / 1e9, 1),
            "frac_of_hbm_peak": round(byp / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "block_size": bs, "num_blocks": int(Kp.shape[0])}
        del qp, Kp, Vp
    # FP8 forward of the headline shape: E4M3 Q, K, V (quantised from the same N(0,1) draws),
    # S on the kind::f8f6f4 tensor cores, P V in bf16; includes the E4M3 -> bf16 widening of V
    Q8, K8, V8 = (t.float().to(torch.float8_e4m3fn) for t in (Q, K, V))
    ws8 = torch.empty(fa.fa_forward_fp8_workspace_bytes(wp.B, wp.H, wp.N, wp.d), device=dev, dtype=torch.uint8)
    O8 = torch.empty_like(Q)
    ms = timed(lambda: fa.fa_forward_fp8(Q8, K8, V8, causal=True, out=O8, return_lse=False, workspace=ws8))
    fl = prefill_flops(wp.B, wp.H, wp.N, wp.d, True)
    # roofline: half the FLOPs at the FP8 rate (2x the measured bf16 peak, the nominal ratio), half at bf16
    mixed_peak = 1.0 / (0.5 / (2.0 * peaks["bf16_tflops"]) + 0.5 / peaks["bf16_tflops"])
    others["prefill_fp8_causal_b1h32_n8192_d128"] = {
        "ms": round(ms, 4), "flops": fl, "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
        "frac_of_bf16_peak": round(fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
        "frac_of_mixed_peak": round(fl / (ms * 1e-3) / 1e12 / mixed_peak, 4),
        "mixed_peak_tflops": round(mixed_peak, 1)}
    del Q8, K8, V8, ws8, O8
    # backward (dQ, dK, dV) of the two prefill shapes; algorithmic FLOPs = 5 GEMMs of 2 d per
    # unmasked score = 2.5 x the forward's (CMU 10-423 Lecture 18, 6.1: 10 N^2 d per head)
    for name, (B_, H_, N_, d_, causal_, amp_, seed_) in (
            ("backward_causal_b1h32_n8192_d128", (wp.B, wp.H, wp.N, wp.d, True, 1.0, wp.seed)),
            ("backward_b8h16_n2048_d64", (w3.B, w3.H, w3.N, w3.d, False, w3.amp, w3.seed))):
        Qb, Kb, Vb = workloads.prefill_inputs(B_, H_, N_, d_, seed_, amp_, device=dev)
        gb = torch.Generator(device=dev)
        gb.manual_seed(seed_ + 1000)
        dOb = torch.randn(Qb.shape, generator=gb, device=dev, dtype=torch.float32).to(torch.bfloat16)
        Ob, Lb = fa.fa_forward(Qb, Kb, Vb, causal=causal_)
        dQb, dKb, dVb = torch.empty_like(Qb), torch.empty_like(Qb), torch.empty_like(Qb)
        wsb = torch.empty(fa.fa_backward_workspace_bytes(B_, H_, N_, d_), device=dev, dtype=torch.uint8)
        ms = timed(lambda: fa.fa_backward(Qb, Kb, Vb, Ob, dOb, Lb, causal=causal_, dQ=dQb, dK=dKb, dV=dVb,
                                          workspace=wsb))
        fl = 2.5 * prefill_flops(B_, H_, N_, d_, causal_)
        others[name] = {"ms": round(ms, 4), "flops": fl, "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
                        "frac_of_bf16_peak": round(fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)}
        if d_ == 64:
            # fa_backward_atomic_dq: dQ accumulated by the dK/dV CTAs with TMA reductions
            # (d = 64 only); not bitwise reproducible in dQ
            wsa = torch.empty(fa.library().fa_backward_atomic_dq_workspace_bytes(B_, H_, N_, d_), device=dev,
                              dtype=torch.uint8)
            ms = timed(lambda: fa.fa_backward(Qb, Kb, Vb, Ob, dOb, Lb, causal=causal_, dQ=dQb, dK=dKb, dV=dVb,
                                              workspace=wsa, atomic_dq=True))
            others[name + "_atomic_dq"] = {
                "ms": round(ms, 4), "flops": fl, "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
                "frac_of_bf16_peak": round(fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)}
            del wsa
        del Qb, Kb, Vb, dOb, Ob, Lb, dQb, dKb, dVb
    st, site = fa.fa_device_error(clear=True)
    if st != 0:
        raise RuntimeError(f"device error word set by the other workloads (site {site:#x})")

    # ---- end to end through the public call with host buffers: fa_forward_host copies
    # the pinned Q, K, V in, runs the forward and copies O, L back inside the call
    Qh, Kh, Vh = (t.cpu().pin_memory() for t in (Q, K, V))
    Oh = torch.empty(O.shape, dtype=O.dtype).pin_memory()
    Lh = torch.empty(L.shape, dtype=L.dtype).pin_memory()
    wsh = torch.empty(fa.fa_forward_host_workspace_bytes(wp.B, wp.H, wp.N, wp.d), device=dev, dtype=torch.uint8)
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush(3)
        a, b = ev(), ev()
        a.record(stream)
        fa.fa_forward_host(Qh, Kh, Vh, causal=True, out=Oh, lse=Lh, workspace=wsh, stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            e2e_ms.append(a.elapsed_time(b))
    if not (torch.equal(Oh.view(torch.int16), O.cpu().view(torch.int16)) and torch.equal(Lh, L.cpu())):
        raise RuntimeError("fa_forward_host differs from fa_forward on the timed workload")
    h2d = 3 * Q.numel() * Q.element_size()
    d2h = O.numel() * O.element_size() + L.numel() * L.element_size()

    flops = prefill_flops(wp.B, wp.H, wp.N, wp.d, wp.causal)
    dbytes = decode_bytes(wd.H, seqlens.tolist(), wd.d)
    pf, dc, ee = max_over_ranks([statistics.mean(pf_ms), statistics.mean(dc_ms), statistics.mean(e2e_ms)],
                                dev, world)

    tflops = replica_throughput(flops, pf, world) / 1e12
    gbs = replica_throughput(dbytes, dc, world) / 1e9
    e2e_tflops = replica_throughput(flops, ee, world) / 1e12
    per_gpu_tflops = flops / (pf * 1e-3) / 1e12
    per_gpu_gbs = dbytes / (dc * 1e-3) / 1e9
    src = peaks["source"]
    result = {
        "metric": METRIC,
        "value": round(tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(pf, 4),
        "step_ms": spread(pf_ms),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": PREFILL, "B": wp.B, "H": wp.H, "N": wp.N, "d": wp.d, "causal": True,
                   "seed": wp.seed, "flops_per_step": flops, "parallelism": "replicas",
                   "l2": L2_NOTE},
        "roofline": {"bound": "tensor", "achieved": round(per_gpu_tflops, 2),
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(per_gpu_tflops / peaks["bf16_tflops"], 4),
                     "frac_of_sustained": round(per_gpu_tflops / peaks["bf16_tflops_sustained"], 4),
                     "frac_of_2250_nominal": round(per_gpu_tflops / 2250.0, 4),
                     "peak_source": f"bf16 burst, of {src}",
                     "traffic": recorded_traffic("prefill_kernel"),
                     "kernel": "prefill_kernel<128>"},
        "e2e": {"value": round(e2e_tflops, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(ee, 4), "step_ms": spread(e2e_ms),
                "path": "fa_forward_host: pinned host buffers, copies inside the call, pipelined by head groups"},
        "decode": {"workload": DECODE, "value": round(gbs, 1), "unit": "GB/s",
                   "ms_per_step": round(dc, 4), "step_ms": spread(dc_ms), "bytes_per_step": dbytes,
                   "num_splits": "auto",
                   "chunk_len": chunk, "chunks_per_seq": nchunk, "gbs_by_num_splits": sweep,
                   "roofline": {"bound": "hbm", "achieved": round(per_gpu_gbs, 1),
                                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": round(per_gpu_gbs / peaks["hbm_gbs"], 4),
                                "frac_of_8tbs_nominal": round(per_gpu_gbs / 8000.0, 4),
                                "peak_source": f"HBM copy, of {src}",
                                "traffic": recorded_traffic("decode_split_kernel"),
                                "kernel": "decode_split_kernel<128> + decode_merge_kernel<128>"}},
        "other_workloads": others,
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 3),
    }
    return result


# ------------------------------------------------------------------ oracle
def oracle_sample(seconds_target, seed=0):
    """Time the float64 oracle on sampled rows of the prefill workload.

    Returns (TFLOP/s of algorithmic work, threads, description)."""
    import numpy as np
    import oracle
    from exact_attention_tiled_gb300 import workloads

    wp = workloads.WORKLOADS[PREFILL]
    Q, K, V = workloads.prefill_inputs(wp.B, wp.H, wp.N, wp.d, wp.seed)
    threads = oracle.max_threads()
    total = wp.B * wp.H * wp.N
    rng = np.random.default_rng(seed)

    def run(nrows):
        rows = np.sort(rng.choice(total, size=nrows, replace=False))
        i = rows % wp.N
        work = float(np.sum(4.0 * wp.d * (i + 1)))
        t0 = time.perf_counter()
        oracle.sdpa_rows(Q, K, V, rows, causal=True, nthreads=threads)
        return work, time.perf_counter() - t0

    w, t = run(max(64, threads * 8))
    rate = w / max(t, 1e-6)
    nrows = int(min(total, max(64, seconds_target * rate / (4.0 * wp.d * wp.N / 2))))
    w, t = run(nrows)
    return w / t / 1e12, threads, f"{nrows} random query rows of {PREFILL} ({w:.3e} FLOP in {t:.1f} s)"


def host_cpu():
    """Model name of the host CPU and the cores this process may run on."""
    model = None
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                key, val = key.strip(), val.strip()
                if key and val and key not in fields:
                    fields[key] = val
    except OSError:
        pass
    for key in ("model name", "Model", "Hardware"):
        if key in fields:
            model = fields[key]
            break
    if model is None and "CPU implementer" in fields:
        model = f"implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    import platform
    try:
        affinity = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        affinity = os.cpu_count() or 1
    return {"cpu_model": model or platform.processor() or platform.machine(),
            "machine": platform.machine(), "affinity_cores": affinity}


def oracle_decode_rate(q, Kc, Vc, seqlens, threads):
    """GB/s of cached K and V the float64 oracle attends per second (no split)."""
    import oracle
    H, d = int(q.shape[1]), int(q.shape[2])
    nbytes = decode_bytes(H, [int(n) for n in seqlens], d)
    t0 = time.perf_counter()
    oracle.decode(q, Kc, Vc, seqlens, nthreads=threads)
    return nbytes / max(time.perf_counter() - t0, 1e-9) / 1e9


def oracle_extras(threads):
    """The oracle on the whole decode workload (all threads and one thread) and
    on the tiny prefill case (one thread), beside the sampled prefill rate."""
    import oracle
    from exact_attention_tiled_gb300 import workloads

    out = host_cpu()
    w = workloads.make(DECODE)
    out["decode"] = {
        "workload": DECODE, "unit": "GB/s",
        "value": oracle_decode_rate(w["q"], w["Kc"], w["Vc"], w["seqlens"], threads), "cores": threads,
        "value_1_thread": oracle_decode_rate(w["q"], w["Kc"], w["Vc"], w["seqlens"], 1),
    }
    del w
    t = workloads.make("tiny_n256_d64")
    wt = workloads.WORKLOADS["tiny_n256_d64"]
    flops = prefill_flops(wt.B, wt.H, wt.N, wt.d, wt.causal)
    tiny = {"workload": "tiny_n256_d64", "unit": "ms"}
    for key, n in (("ms", threads), ("ms_1_thread", 1)):
        t0 = time.perf_counter()
        oracle.sdpa_forward(t["Q"], t["K"], t["V"], causal=wt.causal, nthreads=n)
        tiny[key] = (time.perf_counter() - t0) * 1e3
    tiny["tflops_1_thread"] = flops / (tiny["ms_1_thread"] * 1e-3) / 1e12
    out["tiny"] = tiny
    return out


# Key order of the printed line: the contract's keys first, the per-workload detail last.
LINE_ORDER = ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks",
              "cpu_baseline", "step_ms", "wall_s_timed_region", "decode", "other_workloads")


def rounded(x, digits=4):
    """Floats in nested dicts to `digits` significant digits (integers and strings unchanged)."""
    if isinstance(x, float):
        return float(f"{x:.{digits}g}")
    if isinstance(x, dict):
        return {k: rounded(v, digits) for k, v in x.items()}
    return x


def ordered_line(res):
    out = {k: res[k] for k in LINE_ORDER if k in res}
    out.update({k: v for k, v in res.items() if k not in out})
    if "cpu_baseline" in out:
        out["cpu_baseline"] = rounded(out["cpu_baseline"])
    return out


def run_reference(args):
    per_step = max(1.0, 150.0 / max(1, args.steps + args.warmup))
    vals = []
    desc = ""
    threads = 0
    for i in range(args.warmup + args.steps):
        v, threads, desc = oracle_sample(per_step, seed=i)
        if i >= args.warmup:
            vals.append(v)
    val = statistics.mean(vals)
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": val,
        "unit": "TFLOP/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": None,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": PREFILL, "B": 1, "H": 32, "N": 8192, "d": 128, "causal": True, "seed": 2},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step: {desc}", **oracle_extras(threads)},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def record_traffic(report, kernel, units_note):
    """Store DRAM bytes per launch of `kernel` from an ncu report into profiles/dram_traffic.json."""
    out = subprocess.run(["ncu", "-i", report, "--page", "raw", "--csv"], capture_output=True, text=True,
                         check=True).stdout
    import csv
    rows = list(csv.reader(out.splitlines()))
    hdr, data = rows[0], rows[2:]
    name_i = hdr.index("Kernel Name")
    rd, wr = hdr.index("dram__bytes_read.sum"), hdr.index("dram__bytes_write.sum")
    units = rows[1]
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    vals = [float(r[rd].replace(",", "")) * scale[units[rd]] + float(r[wr].replace(",", "")) * scale[units[wr]]
            for r in data if kernel in r[name_i]]
    if not vals:
        raise SystemExit(f"no launch of {kernel} in {report}")
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    rec = {}
    if os.path.exists(path):
        with open(path) as f:
            rec = json.load(f)
    rec[kernel] = {"bytes_per_launch": statistics.mean(vals), "launches": len(vals),
                   "sources_sha": kernel_sources_hash(kernel), "note": units_note}
    with open(path, "w") as f:
        json.dump(rec, f, indent=1, sort_keys=True)
    print(json.dumps(rec[kernel]))


def run_profile_case(args):
    """Warm-up launches plus `steps` launches of one kernel, nothing else (for ncu)."""
    import torch
    import exact_attention_tiled_gb300 as fa
    from exact_attention_tiled_gb300 import workloads
    dev = torch.device("cuda", 0)
    if args.profile == "prefill":
        wp = workloads.WORKLOADS[PREFILL]
        Q, K, V = workloads.prefill_inputs(wp.B, wp.H, wp.N, wp.d, wp.seed, device=dev)
        run = lambda: fa.fa_forward(Q, K, V, causal=True)
    elif args.profile == "prefill_fp8":
        wp = workloads.WORKLOADS[PREFILL]
        Q, K, V = workloads.prefill_inputs(wp.B, wp.H, wp.N, wp.d, wp.seed, device=dev)
        Q8, K8, V8 = (t.float().to(torch.float8_e4m3fn) for t in (Q, K, V))
        ws8 = torch.empty(fa.fa_forward_fp8_workspace_bytes(wp.B, wp.H, wp.N, wp.d), device=dev, dtype=torch.uint8)
        run = lambda: fa.fa_forward_fp8(Q8, K8, V8, causal=True, workspace=ws8)
    elif args.profile == "prefill64":
        # the batched d64 shape (B8 H16 N2048, x0.5): 192 MiB of inputs, more than L2
        w3 = workloads.WORKLOADS["prefill_b8h16_n2048_d64"]
        Q, K, V = workloads.prefill_inputs(w3.B, w3.H, w3.N, w3.d, w3.seed, w3.amp, device=dev)
        run = lambda: fa.fa_forward(Q, K, V, causal=False)
    elif args.profile in ("backward", "backward_atomic"):
        # the batched d64 shape (B8 H16 N2048): ~0.3 GB on the device (plus the fp32 dQ
        # of the dQ-accumulating variant)
        w3 = workloads.WORKLOADS["prefill_b8h16_n2048_d64"]
        Q, K, V = workloads.prefill_inputs(w3.B, w3.H, w3.N, w3.d, w3.seed, w3.amp, device=dev)
        gb = torch.Generator(device=dev)
        gb.manual_seed(w3.seed + 1000)
        dO = torch.randn(Q.shape, generator=gb, device=dev, dtype=torch.float32).to(torch.bfloat16)
        O, L = fa.fa_forward(Q, K, V)
        atomic = args.profile == "backward_atomic"
        run = lambda: fa.fa_backward(Q, K, V, O, dO, L, atomic_dq=atomic)
    elif args.profile == "backward128":
        # the causal d128 backward on half the heads of the headline shape (B1 H16 N8192):
        # 168 MB of inputs (more than L2), ~0.4 GB on the device with the gradients
        wp = workloads.WORKLOADS[PREFILL]
        Q, K, V = workloads.prefill_inputs(wp.B, wp.H // 2, wp.N, wp.d, wp.seed, device=dev)
        gb = torch.Generator(device=dev)
        gb.manual_seed(wp.seed + 1000)
        dO = torch.randn(Q.shape, generator=gb, device=dev, dtype=torch.float32).to(torch.bfloat16)
        O, L = fa.fa_forward(Q, K, V, causal=True)
        run = lambda: fa.fa_backward(Q, K, V, O, dO, L, causal=True)
    else:
        wd = workloads.WORKLOADS[DECODE]
        q, Kc, Vc = workloads.decode_inputs(wd.B, wd.H, wd.N, wd.d, wd.seed, device=dev)
        seqlens = workloads.decode_seqlens(wd.B, wd.N, wd.seed)
        sd = seqlens.to(dev)
        run = lambda: fa.fa_decode(q, Kc, Vc, sd, num_splits=0, seqlens_host=seqlens)
    for _ in range(args.warmup + args.steps):
        run()
    torch.cuda.synchronize()
    st, site = fa.fa_device_error(clear=True)
    print(json.dumps({"profile_case": args.profile, "launches": args.warmup + args.steps,
                      "device_error": st}))
    if st != 0:
        sys.exit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--profile", choices=["prefill", "prefill64", "prefill_fp8", "decode", "backward", "backward_atomic",
                                          "backward128"],
                    default=None,
                    help="only launch one kernel warmup+steps times (for ncu captures)")
    ap.add_argument("--record-traffic", nargs=3, metavar=("REPORT", "KERNEL", "NOTE"), default=None,
                    help="write DRAM bytes per launch of KERNEL from an ncu report to profiles/")
    args = ap.parse_args()
    if args.record_traffic:
        record_traffic(*args.record_traffic)
        return
    if args.profile:
        run_profile_case(args)
        return
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(ordered_line(run_reference(args))), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        # the oracle baseline on the host cores belongs to the single-GPU line only
        if world == 1:
            v, threads, desc = oracle_sample(args.cpu_seconds)
            res["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                   "sample": desc, **oracle_extras(threads)}
        print(json.dumps(ordered_line(res)), flush=True)
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
