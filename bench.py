"""Benchmark of the Mamba-3 scan library on B300.

One step = one full pass of the scan over one batch of synthetic input:
for the prefill workloads a single ``m3_scan_prefill`` call over every
token (writing y and the final state), for the decode workloads the whole
1024-step decode loop.  Default workload: the SISO prefill shaped like a
1.5B-scale layer (batch 8, L 4096, 32 heads, P 64, N 128, bf16 inputs).

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead
(the only reference this project has: the pages ship no code).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "Mamba-3 scan tokens/s (prefill) & decode steps/s; % of HBM/tensor roofline"
L2_BYTES = 126 * 1024 ** 2
PKG = "state_space_sequence_06_b300"


def peaks():
    """HBM GB/s and dense bf16 TFLOP/s (burst: the kernels are timed alone)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6400.0, 1800.0, "fallback"


def workload_bytes(wl) -> dict:
    """Algorithmic bytes of one pass: every input read once, y written once,
    the f32 state read (when it carries in) and written once."""
    isz = 2 if wl.dtype == "bf16" else 4
    ysz = 2 if wl.y_bf16 else 4
    H, P, N, R = wl.nheads, wl.headdim, wl.dstate, wl.rank
    G = wl.groups
    # per token and head: x, dt, and lam / theta unless they are the special
    # values (not read at all then); B and C once per group of heads
    per_in = R * P + 1 + (0 if wl.euler else 1) + (0 if wl.real else N // 2) + 2 * R * N * G / H
    if wl.kind == "decode":
        units = wl.batch * H
        per_step_in = int(round(units * per_in * isz))
        carry = units * (R * N + R * P) * isz * 2  # read old, write new
        state = units * N * P * 4 * 2
        y = units * R * P * ysz
        return dict(per_unit_of_work=per_step_in + carry + state + y, unit="step",
                    inputs=per_step_in, state=state, carry=carry, y=y)
    tokens = wl.seqlen * (wl.batch if wl.kind == "prefill" else 1)
    th = tokens * H
    per_th_in = per_in * isz
    nseq = wl.nseq if wl.kind == "varlen" else wl.batch
    state = nseq * H * N * P * 4 * 2  # h0 read + h_final write
    carry = nseq * H * (R * N + R * P) * isz * 2
    total = int(round(th * (per_th_in + R * P * ysz))) + state + carry
    return dict(per_unit_of_work=total, unit="pass", inputs=int(round(th * per_th_in)), y=th * R * P * ysz,
                state=state, carry=carry, per_token_head=per_th_in + R * P * ysz)


def contraction_flops(wl) -> dict:
    """Tensor-core work of one chunked prefill pass.

    ``algorithmic``: the chunked form's contractions per token and head,
    2QR^2 N (scores C B^T) + 2QR^2 P (intra output S' X) + 2RNP (inter
    output C^H G') + 2RNP (chunk state B^T W X), for the chunk Q the kernel
    runs (the quadratic form of the Mamba-2 duality the chunked scan uses).
    ``issued``: what the kernel actually issues on the tensor cores: every
    product of a rotated operand, of S' and of W X is a hi/lo pair of f16
    operands taking three (or two) MMAs; the real-state variant's B and C
    are exact in f16 and take one."""
    if wl.kind == "decode" or wl.dtype != "bf16":
        return {}
    Q, R, N, P = wl.chunk, wl.rank, wl.dstate, wl.headdim
    tokens = wl.seqlen * (wl.batch if wl.kind == "prefill" else 1)
    th = tokens * wl.nheads
    per_th = 2 * Q * R * R * N + 2 * Q * R * R * P + 4 * R * N * P
    rot = 1 if wl.real else 3  # products with a rotated B or C operand
    # per chunk of MR = QR rows: MMA 1 (MR x MR x N), 2 (MR x P x MR, S' hi/lo),
    # 3 (MR x P x N, C hi/lo; one product without rotation), 4 (N x P x MR)
    MR = Q * R
    issued_chunk = (2 * MR * MR * N * rot + 2 * MR * P * MR * 2 + 2 * MR * P * N * (1 if wl.real else 2)
                    + 2 * N * P * MR * (2 if wl.real else 3))
    return {"algorithmic": th * per_th, "issued": th * issued_chunk // Q, "per_token_head": per_th}


# the sources each kernel is compiled from (its launcher included)
KERNEL_SOURCES = {
    "prefill": ["csrc/chunked.cuh", "csrc/recurrent.cuh", "csrc/umma.cuh", "csrc/common.cuh", "csrc/m3scan.cu",
                "include/m3scan.h"],
    "decode_step": ["csrc/decode.cuh", "csrc/umma.cuh", "csrc/common.cuh", "csrc/m3scan.cu", "include/m3scan.h"],
}


def _code_only(src: str) -> str:
    """C/C++/CUDA source without comments, blank lines or trailing spaces:
    an edit to a comment leaves the compiled kernel, so the hash, alone."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(ln.rstrip() for ln in src.splitlines() if ln.strip())


def kernel_source_hash(kind):
    """Hash of the code a kernel is built from (comments excluded): a
    committed DRAM-traffic figure counts only while it matches."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        path = os.path.join(ROOT, rel if rel.startswith("include") else os.path.join(PKG, rel))
        with open(path) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_for(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        e = d.get(kernel_key)
        if e and e.get("source_sha") == kernel_source_hash(kernel_key.split(":")[0]):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """SM clocks and throttle reasons sampled every few ms during a timed
    region, read from the driver's NVML library through ctypes (reading
    only; no setting is touched)."""

    NVML_CLOCK_SM = 1
    REASONS = {
        "sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
        "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80,
    }

    def __init__(self, cuda_index: int, period_s: float = 0.005):
        self.idx, self.period = cuda_index, period_s
        self.samples, self.max_mhz, self.err = [], None, None

    def _open(self):
        import ctypes

        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(self.idx)
        bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0".encode()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
            raise RuntimeError("no NVML handle for " + bus.decode())
        self.lib, self.h, self.ct = lib, h, ctypes
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
            self.max_mhz = mx.value
        self.get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")

    def __enter__(self):
        import threading
        try:
            self._open()
        except Exception as e:  # pragma: no cover - depends on the box
            self.err = repr(e)[:120]
            return self
        self.stop = threading.Event()
        ct, lib, h = self.ct, self.lib, self.h
        sm, rs = ct.c_uint(), ct.c_ulonglong()

        def sample():
            if lib.nvmlDeviceGetClockInfo(h, self.NVML_CLOCK_SM, ct.byref(sm)) == 0 and \
                    self.get_reasons(h, ct.byref(rs)) == 0:
                self.samples.append((sm.value, rs.value))

        # the first queries of a process are slow: take them here, before the
        # caller's timed region starts, and keep only the later samples
        sample()
        self.samples.clear()
        self._sample = sample

        started = threading.Event()

        def run():
            while not self.stop.is_set():
                sample()
                started.set()
                self.stop.wait(self.period)

        # the caller's timed region starts once the thread runs its loop (its
        # start-up then takes no host time from the first launch)
        self.th = threading.Thread(target=run, daemon=True)
        self.th.start()
        started.wait(0.5)
        return self

    def restart(self):
        """Drop the samples taken so far (those before a timed region) and
        take one at its start."""
        if self.err is None:
            self.samples.clear()
            self._sample()

    def __exit__(self, *a):
        if self.err is None:
            self.stop.set()
            self.th.join(timeout=2)

    def summary(self):
        if self.err is not None or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [self.err or "no samples"]}
        sm = [x for x, _ in self.samples]
        reasons = sorted({n for _, r in self.samples for n, bit in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(sm), "sm_mhz_min": min(sm)}


# ------------------------------------------------------------------ oracle arm


def oracle_rate(wl, seconds=15.0):
    """Time the CPU oracle, as it stands, on a bounded sample of the workload
    (whole units, all their tokens), on all host cores.  Returns the rate in
    the workload's unit and a description of the sample."""
    import oracle

    cores = os.cpu_count() or 1
    if wl.kind == "decode":
        steps = 64
        d = synth.decode_inputs(wl, steps=steps)
        units = list(range(min(wl.batch * wl.nheads, cores * 4)))
        kw = dict(batch=wl.batch, H=wl.nheads, P=wl.headdim, N=wl.dstate, R=wl.rank, dtype=wl.dtype,
                  steps=steps, units=units, nthreads=cores)
        t0 = time.perf_counter()
        reps = 0
        while True:
            oracle.decode(d, **kw)
            reps += 1
            el = time.perf_counter() - t0
            if el > seconds or reps >= 50:
                break
        unit_steps_per_s = reps * len(units) * steps / el
        rate = unit_steps_per_s / (wl.batch * wl.nheads)  # whole-batch decode steps/s
        return rate, cores, f"{len(units)} of {wl.batch * wl.nheads} units x {steps} steps, {reps} reps, {el:.1f} s"
    inp = synth.prefill_inputs(wl)
    cu = wl.cu_seqlens if wl.kind == "varlen" else None
    nseq = wl.nseq if cu is not None else wl.batch
    U = nseq * wl.nheads
    kw = dict(batch=wl.batch, L=wl.seqlen, H=wl.nheads, P=wl.headdim, N=wl.dstate, R=wl.rank,
              dtype=wl.dtype, cu_seqlens=cu, nthreads=cores)
    units = list(range(min(U, cores)))
    t0 = time.perf_counter()
    done_tok_heads = 0
    reps = 0
    while True:
        _, _, _, _, spans = oracle.prefill(inp, units=units, **kw)
        done_tok_heads += sum(s[2] for s in spans)
        reps += 1
        el = time.perf_counter() - t0
        if el > seconds or reps >= 100:
            break
    rate = done_tok_heads / el / wl.nheads  # tokens/s (a token = one position across all heads)
    return rate, cores, f"{len(units)} of {U} units (all tokens), {reps} reps, {el:.1f} s"


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    metric_unit = "steps/s" if wl.kind == "decode" else "tokens/s"
    times = []
    rate = cores = sample = None
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        rate, cores, sample = oracle_rate(wl, seconds=max(2.0, 60.0 / max(1, args.warmup + args.steps)))
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": metric_unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl),
        "cpu_baseline": {"value": rate, "unit": metric_unit, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": rate, "unit": metric_unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "the pages ship no code; the reference arm is the CPU oracle (complex double, sequential per unit)",
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(torch, dist, world, value, device):
    """The largest of every rank's `value` (the job's time is its slowest
    rank's); timing only, no data of the scan crosses ranks."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank_step, steps, world, total_ms):
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return units_per_rank_step * steps * world / (total_ms / 1e3)


# A GPU that idled for a few seconds (the parity check and the oracle run
# on the host before a line is timed) runs its first tens of milliseconds
# about 5 % slower than in steady state (measured: 0.460 against 0.437 ms a
# headline pass, with the SM clock already at its maximum).  So the warm-up
# is the W passes asked for and then more, untimed, until the device has
# been busy for WARM_UP_MIN_S.
WARM_UP_MIN_S = 0.3


def warm_up(step, w, torch):
    """W untimed passes, then more until WARM_UP_MIN_S seconds have gone by
    (at most 10,000 passes)."""
    t0 = time.perf_counter()
    for _ in range(w):
        step()
    torch.cuda.synchronize()
    n = w
    while time.perf_counter() - t0 < WARM_UP_MIN_S and n < 10000:
        step()
        n += 1
        if n % 8 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()


def config_of(wl):
    c = {"workload": wl.name, "kind": wl.kind, "batch": wl.batch, "seq_len": wl.seqlen, "heads": wl.nheads,
         "headdim": wl.headdim, "dstate": wl.dstate, "mimo_rank": wl.rank, "in_dtype": wl.dtype,
         "global_batch": (wl.nseq if wl.kind == "varlen" else wl.batch) * wl.shards}
    if wl.kind != "decode":
        c["chunk"] = wl.chunk
    if wl.kind == "varlen":
        c["nseq"] = wl.nseq
    if wl.ngroups:
        c["ngroups"] = wl.ngroups
    if wl.prologue:
        c["prologue"] = "fused: dt = softplus(dt + dt_bias), B and C rows RMS-normalised"
    c["y_dtype"] = "bf16" if wl.y_bf16 else "f32"
    c["warm_up"] = f"the W passes, then untimed passes until the device has been busy {WARM_UP_MIN_S} s"
    if wl.real or wl.euler:
        c["special_case"] = "Mamba-2: " + ", ".join(
            ([("theta = 0 (real state)")] if wl.real else []) + (["lam = 1 (first order)"] if wl.euler else []))
    return c


# ------------------------------------------------------------------ GPU arm


def prologue_kw(wl, m3, t):
    """Prologue arguments of a scan call: raw-input workloads have the kernel
    apply softplus(dt + dt_bias) and the RMS norm of B and C rows."""
    if not wl.prologue:
        return {}
    return dict(prologue=m3.M3_PRO_DT_SOFTPLUS | m3.M3_PRO_BC_NORM, dt_bias=t["dt_bias"])


def dev_tensor(torch, a):
    if a is None:  # lam = 1 / theta = 0
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.cuda()


def measure(wl, args, m3, torch, dist, world, local, stream, headline):
    """Time `args.steps` passes of `wl` after `args.warmup` untimed ones.
    Returns the JSON fields for it (the headline also gets e2e, the CPU
    oracle baseline and a sampled parity check)."""
    algo = {"auto": m3.M3_ALGO_AUTO, "recurrent": m3.M3_ALGO_RECURRENT, "chunked": m3.M3_ALGO_CHUNKED}[args.algo]
    hbm_peak, _, peak_src = peaks()
    dims_dtype = m3.M3_BF16 if wl.dtype == "bf16" else m3.M3_F32
    H, P, N, R = wl.nheads, wl.headdim, wl.dstate, wl.rank
    byt = workload_bytes(wl)
    ev_pairs = []
    cu = None

    if wl.kind == "decode":
        d = synth.decode_inputs(wl)
        T = wl.seqlen
        t = {k: dev_tensor(torch, d[k]) for k in ("x", "B", "C", "dt", "lam", "theta", "A", "D")}
        st = m3.m3_state_alloc(m3.make_dims(wl.batch, H, P, N, R, dims_dtype))
        hv, pB, px = st.views()
        h0, pB0, px0 = dev_tensor(torch, d["h0"]), dev_tensor(torch, d["prev_B"]), dev_tensor(torch, d["prev_x"])
        y = torch.empty((wl.batch, H, R, P), dtype=torch.bfloat16 if wl.y_bf16 else torch.float32, device="cuda")
        del d

        per_tok = {k: ([None] * T if t[k] is None else [t[k][i] for i in range(T)])
                   for k in ("x", "B", "C", "dt", "lam", "theta")}

        def reset():
            hv.copy_(h0)  # every pass starts from the same initial state and carry
            pB.copy_(pB0)
            px.copy_(px0)

        def launch(i):
            m3.m3_decode_step(per_tok["x"][i], per_tok["B"][i], per_tok["C"][i], per_tok["dt"][i],
                              per_tok["lam"][i], per_tok["theta"][i], t["A"], t["D"], y, st)

        # The T-token pass is captured once as a CUDA graph of the library's
        # own decode kernels (one launch per token): replaying it removes the
        # host's per-call cost, which is not the kernel's, from the pass time.
        reset()
        for i in range(T):  # eager pass first: lazy module loading and kernel attributes happen here
            launch(i)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(T):
                launch(i)
        torch.cuda.synchronize()

        def step():
            reset()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            ev_pairs.append((e0, e1))

        def per_launch_median_ms():
            """Median device time of one decode kernel: events around every
            launch of one eager pass (after the timed region)."""
            reset()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(T)]
            torch.cuda.synchronize()
            for i in range(T):
                evs[i][0].record(stream)
                launch(i)
                evs[i][1].record(stream)
            torch.cuda.synchronize()
            return statistics.median(a.elapsed_time(b) for a, b in evs)

        launches_per_step, units_per_step, unit_name = T, T, "steps/s"
        kernel_key = f"decode_step:{wl.name}"
        path_dtype = "f32"
    else:
        inp = synth.prefill_inputs(wl)
        t = {k: dev_tensor(torch, inp[k]) for k in ("x", "B", "C", "dt", "lam", "theta", "A", "D")}
        t["dt_bias"] = dev_tensor(torch, inp.get("dt_bias"))
        pkw = prologue_kw(wl, m3, t)
        nseq = wl.batch
        if wl.kind == "varlen":
            cu = torch.from_numpy(wl.cu_seqlens).cuda()
            nseq = wl.nseq
        st = m3.m3_state_alloc(m3.make_dims(nseq, H, P, N, R, dims_dtype))
        y = torch.empty(t["x"].shape, dtype=torch.bfloat16 if wl.y_bf16 else torch.float32, device="cuda")

        def step():
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            m3.m3_scan_prefill(t["x"], t["B"], t["C"], t["dt"], t["lam"], t["theta"], t["A"], t["D"], y,
                               state=st, cu_seqlens=cu, algo=algo, chunk=wl.chunk, **pkw)
            e1.record(stream)
            ev_pairs.append((e0, e1))

        per_launch_median_ms = None
        launches_per_step = 1
        units_per_step = wl.seqlen * (wl.batch if wl.kind == "prefill" else 1)  # tokens
        unit_name = "tokens/s"
        kernel_key = f"prefill:{wl.name}:{args.algo}"
        # which prefill kernel runs: the chunked one multiplies f16 operand
        # pairs on the tensor cores (f32 accumulation); the recurrent one is f32
        path_dtype = "f32"
        if wl.dtype == "bf16" and algo != m3.M3_ALGO_RECURRENT:
            try:
                m3.m3_scan_prefill(t["x"], t["B"], t["C"], t["dt"], t["lam"], t["theta"], t["A"], t["D"], y,
                                   state=st, cu_seqlens=cu, algo=m3.M3_ALGO_CHUNKED, chunk=wl.chunk, **pkw)
                path_dtype = "f16x2 (hi/lo f16 operands, f32 accumulate)"
            except m3.M3Error as e:
                if e.status != m3.M3_ERR_UNSUPPORTED:
                    raise
        torch.cuda.synchronize()

    parity = None
    if headline and wl.kind != "decode":
        try:
            parity = sampled_parity(wl, m3, t, y, st, cu, algo)
        except Exception as e:  # reported, never hides a number
            parity = {"error": repr(e)[:200]}

    # the sampler starts before the warm-up, so that the device does not idle
    # between the warm-up and the timed region; its samples are those of the
    # timed region
    with ClockSampler(local) as clk:
        warm_up(step, args.warmup, torch)
        ev_pairs.clear()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        clk.restart()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            step()
        g1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    total_ms = max_over_ranks(torch, dist, world, g0.elapsed_time(g1), "cuda")
    kern_ms = [a.elapsed_time(b) for a, b in ev_pairs]
    status = m3.m3_device_status()
    # the dominant kernel's roofline: algorithmic bytes of one launch over its
    # average duration (events on the launching stream)
    per_launch_ms = statistics.mean(kern_ms) / launches_per_step
    bytes_per_launch = byt["per_unit_of_work"]  # one prefill pass, or one decode step
    achieved = bytes_per_launch / (per_launch_ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved / hbm_peak, "traffic": traffic_for(kernel_key),
            "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else peak_src,
            "algorithmic_bytes_per_launch": bytes_per_launch,
            "kernel_ms_per_launch": per_launch_ms}
    if per_launch_median_ms is not None:
        # decode: the pass time / T above includes the gaps between launches
        # (none to speak of in a graph); this is the kernel alone
        roof["kernel_ms_per_launch_median_eager"] = per_launch_median_ms()
    fl = contraction_flops(wl) if path_dtype.startswith("f16x2") else {}
    if fl:
        _, tc_peak, tc_src = peaks()
        sec = per_launch_ms / 1e3
        ideal_s = bytes_per_launch / (hbm_peak * 1e9)  # the pass at the HBM roofline
        roof["tensor"] = {
            "achieved": fl["algorithmic"] / sec / 1e12, "peak": tc_peak, "unit": "TFLOP/s",
            "frac": fl["algorithmic"] / sec / 1e12 / tc_peak,
            "flops_per_launch": fl["algorithmic"], "flops_per_token_head": fl["per_token_head"],
            "issued_mma_flops_per_launch": fl["issued"],
            "issued_frac": fl["issued"] / sec / 1e12 / tc_peak,
            "ceiling_frac_at_hbm_roofline": fl["algorithmic"] / ideal_s / 1e12 / tc_peak,
            "peak_source": tc_src + " (MEASURED_PEAKS.json bf16_tflops, dense bf16 burst)"
            if tc_src == "measured" else tc_src}
    out = {
        "value": job_rate(units_per_step, args.steps, world, total_ms), "unit": unit_name,
        "ms_per_step": total_ms / args.steps, "dtype": path_dtype,
        "roofline": roof,
        "gpu_launches": launches_per_step * args.steps, "device_status": status,
        "clocks": clk.summary(), "parity": parity, "config": config_of(wl),
    }
    if headline and not args.no_e2e:
        out["e2e"] = measure_e2e(wl, m3, torch, t, y, st, cu, algo, args, world)
    st.free()
    del t, y
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="siso_b8_l4096")
    ap.add_argument("--algo", default="auto", choices=["auto", "recurrent", "chunked"])
    ap.add_argument("--quick", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--decode-steps", type=int, default=0,
                    help="decode workloads: tokens per pass (default: the workload's 1024); "
                         "smaller passes keep profiler captures small")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    wls = synth.workloads()
    if args.decode_steps > 0:
        for k, w in list(wls.items()):
            if w.kind == "decode":
                wls[k] = synth.scaled(w, seqlen=args.decode_steps)
    if args.impl == "reference":
        return run_reference(args, wls[args.workload])

    import torch
    import torch.distributed as dist

    import state_space_sequence_06_b300 as m3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    stream = torch.cuda.current_stream()
    # weak scaling: each rank runs its own shard (a distinct group of
    # sequences) of a global batch world times the workload's
    wls = {k: synth.shard(w, rank, world) for k, w in wls.items()}
    wl = wls[args.workload]
    if wl.backward:  # a line of its own, run only by name
        return run_backward(wl, args, m3, torch, dist, world, rank, local, stream)

    head = measure(wl, args, m3, torch, dist, world, local, stream, headline=True)
    others = []
    if not args.quick:
        for name in ("mimo4_b8_l4096", "long_l16384", "varlen_16", "siso_n64_b8_l4096", "mamba2_b8_l4096",
                     "siso_g1_b8_l4096", "mimo4_g1_b8_l4096", "siso_ybf16_b8_l4096", "siso_prologue_b8_l4096",
                     "decode_siso_b256", "decode_mimo4_b256",
                     "decode_siso_n64_b256", "decode_mamba2_b256", "decode_siso_g1_b256", "tiny_f32"):
            if name == args.workload:
                continue
            sargs = argparse.Namespace(**vars(args))
            if wls[name].kind == "decode":
                sargs.steps = 5  # one step = the whole 1024-token decode loop
            r = measure(wls[name], sargs, m3, torch, dist, world, local, stream, headline=False)
            others.append({"workload": name, "value": r["value"], "unit": r["unit"], "ms_per_step": r["ms_per_step"],
                           "dtype": r["dtype"], "roofline_frac": r["roofline"]["frac"],
                           "achieved_gbs": r["roofline"]["achieved"],
                           "kernel_ms_per_launch": r["roofline"]["kernel_ms_per_launch"],
                           "kernel_ms_per_launch_median_eager":
                               r["roofline"].get("kernel_ms_per_launch_median_eager"),
                           "tensor_frac": (r["roofline"].get("tensor") or {}).get("frac"),
                           "gpu_launches": r["gpu_launches"], "device_status": r["device_status"],
                           "clocks": r["clocks"]})

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            r_, cores, sample = oracle_rate(wl, seconds=15.0)
            cpu = {"value": r_, "unit": head["unit"], "cores": cores, "kind": "oracle", "sample": sample}
        except Exception as e:
            cpu = {"error": repr(e)[:200]}

    if rank == 0:
        print(json.dumps(contract_line(head, cpu, others, args, world)), flush=True)
    if world > 1:
        dist.destroy_process_group()


def contract_line(head, cpu, others, args, world):
    """The one JSON line of a run: the headline measurement `head` (from
    measure()), the CPU oracle baseline and the other workloads' lines."""
    return {
        "metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": head["dtype"],
        "data": "synthetic (seeded generator; shapes of the pages' 1.5B-scale workloads)",
        "config": dict(head["config"], algo=args.algo,
                       l2=("inputs larger than L2 (%.2f GB per pass vs 126 MB L2)"
                           % (head["roofline"]["algorithmic_bytes_per_launch"] / 1e9)),
                       parallelism=f"replicas over independent units x{world}"),
        "roofline": head["roofline"], "cpu_baseline": cpu, "e2e": head.get("e2e"),
        "gpu_launches": head["gpu_launches"], "device_status": head["device_status"],
        "clocks": head["clocks"], "parity": head["parity"], "workloads": others,
    }


def backward_flops(wl) -> int:
    """Contraction FLOPs of one chunked backward pass: per chunk of MR = QR
    rows, the chunk sums Z = Bt^T (f x) and U = Ct^T (e^Lam dy) (2 N MR P
    each), and the gradient contractions: S and dM (2 MR^2 N, 2 MR^2 P), the
    inter output Ct Gs (2 MR P N), dX = M^T dY + Bt dG (2 MR^2 P + 2 MR N P),
    dCt = dS Bt + dY Gs^T and dBt = dS^T Ct + X dG^T (2 (2 MR^2 N + 2 MR N P))."""
    Q, R, N, P = 64 // wl.rank, wl.rank, wl.dstate, wl.headdim
    MR = Q * R
    per_chunk = (2 * (2 * N * MR * P) + 2 * MR * MR * N + 2 * MR * MR * P + 2 * MR * P * N
                 + 2 * MR * MR * P + 2 * MR * N * P + 2 * (2 * MR * MR * N + 2 * MR * N * P))
    nch = -(-wl.seqlen // Q)
    return per_chunk * nch * wl.batch * wl.nheads


def fp32_peak_tflops():
    """FP32 FMA peak of a B300 from its unit counts and clock: 148 SMs x 128
    FP32 lanes x 2 FLOP per FMA x the maximum SM clock (2032 MHz)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f)["sm_max_mhz"])
    except Exception:
        mhz = 2032.0
    return 148 * 128 * 2 * mhz * 1e6 / 1e12


def run_backward(wl, args, m3, torch, dist, world, rank, local, stream):
    """Time m3_scan_prefill_backward on a prefill workload with a seeded
    dL/dy and dL/dh_final; one pass = every gradient of the batch (the
    chunked kernels where the shape has them: --algo auto or chunked; the
    token-serial kernel: --algo recurrent).  Roofline: the contraction
    FLOPs of the chunked form against the FP32 FMA peak (the dominant
    kernel, the chunk gradients, is f32 SIMT: bound "alu"; the chunk sums
    run on the tensor cores for ranks 1 and 2).  Unit 0's gradients are checked against the
    oracle's adjoint."""
    import oracle

    H, P, N, R, L, b = wl.nheads, wl.headdim, wl.dstate, wl.rank, wl.seqlen, wl.batch
    algo = {"auto": m3.M3_ALGO_AUTO, "recurrent": m3.M3_ALGO_RECURRENT, "chunked": m3.M3_ALGO_CHUNKED}[args.algo]
    inp = synth.prefill_inputs(wl)
    rng = np.random.default_rng(0)
    dy = rng.normal(size=(b, L, H, R, P)).astype(np.float32)
    dhf = rng.normal(size=(b, H, N // 2, P, 2)).astype(np.float32)
    t = {k: dev_tensor(torch, inp[k]) for k in ("x", "B", "C", "dt", "lam", "theta", "A", "D", "h0", "prev_B",
                                                "prev_x")}
    dy_d, dhf_d = dev_tensor(torch, dy), dev_tensor(torch, dhf)

    def once():
        return m3.m3_scan_prefill_backward(t["x"], t["B"], t["C"], t["dt"], t["lam"], t["theta"], t["A"], t["D"],
                                           dy_d, h0=t["h0"], prev_B=t["prev_B"], prev_x=t["prev_x"],
                                           dh_final=dhf_d, algo=algo)

    box = {}

    def warm():
        box["out"] = once()

    steps = args.steps if algo != m3.M3_ALGO_RECURRENT else min(args.steps, 3)
    with ClockSampler(local) as clk:  # (started before the warm-up, as in measure())
        warm_up(warm, args.warmup, torch)
        out = box["out"]
        clk.restart()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            out = once()
        e1.record(stream)
        torch.cuda.synchronize()
    total_ms = max_over_ranks(torch, dist, world, e0.elapsed_time(e1), "cuda")
    status = m3.m3_device_status()
    # parity of unit 0 (sequence 0, head 0) against the adjoint oracle
    w = lambda k: oracle._widen(inp[k], wl.dtype)  # noqa: E731
    g = 0  # head 0 reads group 0
    _, _, ref = oracle.unit_backward(w("x")[0, :, 0], w("B")[0, :, g], w("C")[0, :, g], w("dt")[0, :, 0],
                                     w("lam")[0, :, 0], w("theta")[0, :, 0], float(inp["A"][0]),
                                     float(inp["D"][0]), inp["h0"][0, 0, ..., 0] + 1j * inp["h0"][0, 0, ..., 1],
                                     w("prev_B")[0, 0], w("prev_x")[0, 0], dy[0, :, 0].astype(np.float64),
                                     dhf[0, 0, ..., 0] + 1j * dhf[0, 0, ..., 1])
    err = {}
    for gk, rk in (("dx", "x"), ("dB", "B"), ("dC", "C"), ("ddt", "dt"), ("dlam", "lam"), ("dtheta", "theta")):
        got = out[gk][0, :, 0].double().cpu().numpy()
        err[gk] = float(np.max(np.abs(got - ref[rk])) / max(np.sqrt(np.mean(ref[rk] ** 2)), 1e-30))
    isz = 2 if wl.dtype == "bf16" else 4
    th = b * L * H
    in_bytes = th * (R * P + 2 * R * N + 2 + N // 2) * isz + th * R * P * 4
    out_bytes = th * (R * P + 2 * R * N + 2 + N // 2) * 4
    byt = in_bytes + out_bytes
    per_ms = total_ms / steps
    hbm_peak, _, peak_src = peaks()
    flops = backward_flops(wl)
    alu_peak = fp32_peak_tflops()
    achieved = flops / (per_ms / 1e3) / 1e12
    if rank == 0:
        kernel = ("token-serial" if algo == m3.M3_ALGO_RECURRENT
                  else "chunked (f32 SIMT gradients; tcgen05 chunk sums for ranks 1 and 2)")
        print(json.dumps({
            "metric": "Mamba-3 scan backward tokens/s", "value": b * L * world / (per_ms / 1e3), "unit": "tokens/s",
            "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": per_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(config_of(wl), **{"pass": "backward (all gradients, f32)", "kernel": kernel}),
            "roofline": {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
                         "frac": achieved / alu_peak, "traffic": None,
                         "peak_source": "derived: 148 SMs x 128 FP32 lanes x 2 FLOP x max SM clock",
                         "flops_per_launch": flops, "kernel_ms_per_launch": per_ms,
                         "hbm": {"algorithmic_bytes_per_launch": byt, "achieved_gbs": byt / (per_ms / 1e3) / 1e9,
                                 "peak": hbm_peak, "frac": byt / (per_ms / 1e3) / 1e9 / hbm_peak,
                                 "peak_source": peak_src}},
            "gpu_launches": steps * (1 if algo == m3.M3_ALGO_RECURRENT else 5), "device_status": status,
            "clocks": clk.summary(), "parity": {"unit": 0, "max_err_over_rms": err}}), flush=True)


def sampled_parity(wl, m3, t, y, st, cu, algo):
    """Two units of the timed configuration against the oracle, max |err|
    over them divided by the rms of the whole output tensor."""
    import torch

    import oracle

    inp = synth.prefill_inputs(wl)
    cu_np = wl.cu_seqlens if wl.kind == "varlen" else None
    nseq = wl.nseq if cu_np is not None else wl.batch
    U = nseq * wl.nheads
    hv, pB, px = st.views()
    hv.zero_()
    pB.zero_()
    px.zero_()
    m3.m3_scan_prefill(t["x"], t["B"], t["C"], t["dt"], t["lam"], t["theta"], t["A"], t["D"], y, state=st,
                       cu_seqlens=cu, algo=algo, chunk=wl.chunk, **prologue_kw(wl, m3, t))
    torch.cuda.synchronize()
    rms = float(torch.sqrt((y.double() ** 2).mean()).item())
    units = [0, U - 1]
    dtype = wl.dtype
    if wl.prologue:
        inp = oracle.apply_prologue(inp, wl.dtype, dt_softplus=True, bc_norm=True, dt_bias=inp["dt_bias"])
        dtype = "f64"
    yo, ho, _, _, spans = oracle.prefill(inp, batch=wl.batch, L=wl.seqlen, H=wl.nheads, P=wl.headdim,
                                         N=wl.dstate, R=wl.rank, dtype=dtype, cu_seqlens=cu_np, units=units)
    err = 0.0
    for u, (b, t0, n, hd, _) in zip(units, spans):
        g = y[b, t0:t0 + n, hd].double().cpu().numpy()
        err = max(err, float(np.max(np.abs(g - yo[u]))))
    hv.zero_()
    pB.zero_()
    px.zero_()
    return {"units": units, "max_err_over_rms_y": err / rms}


def measure_e2e(wl, m3, torch, t, y, st, cu, algo, args, world):
    """The same metric through the public API from pinned host buffers: each
    step copies its inputs host -> device, runs the scan and copies y back.

    Steps are pipelined over two sets of device buffers and three streams:
    the upload of step i + 1 (copy stream) and the download of step i - 1
    (a second copy stream, the other direction of the link) overlap the scan
    of step i, ordered by events: a set's inputs are overwritten only after
    the scan that read them, its y only after the download that read it."""
    if wl.kind == "decode":
        return measure_e2e_decode(wl, m3, torch, t, st, args, world)
    keys = tuple(k for k in ("x", "B", "C", "dt", "lam", "theta") if t[k] is not None)
    host = {k: torch.empty(t[k].shape, dtype=t[k].dtype, pin_memory=True) for k in keys}
    for k in keys:
        host[k].copy_(t[k])
    sets = [{k: t[k] for k in keys}, {k: torch.empty_like(t[k]) for k in keys}]
    ys = [y, torch.empty_like(y)]
    yh = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for _ in range(2)]
    torch.cuda.synchronize()
    h2d = sum(host[k].numel() * host[k].element_size() for k in keys)
    d2h = y.numel() * y.element_size()
    units = wl.seqlen * (wl.batch if wl.kind == "prefill" else 1)
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    scanned = [None, None]   # set j's last scan done (its inputs read, its y written)
    fetched = [None, None]   # set j's last download done (its y read)

    def one(i):
        j = i % 2
        with torch.cuda.stream(up):
            if scanned[j] is not None:
                up.wait_event(scanned[j])
            for k in keys:
                sets[j][k].copy_(host[k], non_blocking=True)
            loaded = ev()
            loaded.record(up)
        comp.wait_event(loaded)
        if fetched[j] is not None:
            comp.wait_event(fetched[j])
        d = sets[j]
        m3.m3_scan_prefill(d["x"], d["B"], d["C"], d["dt"], d.get("lam"), d.get("theta"), t["A"], t["D"], ys[j],
                           state=st, cu_seqlens=cu, algo=algo, chunk=wl.chunk, stream=comp,
                           **prologue_kw(wl, m3, t))
        scanned[j] = ev()
        scanned[j].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(scanned[j])
            yh[j].copy_(ys[j], non_blocking=True)
            fetched[j] = ev()
            fetched[j].record(down)

    steps = max(3, min(args.steps, 10))
    for i in range(2):
        one(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    return {"value": units * steps * world / el, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "pipeline": "two buffer sets; upload of step i+1 and download of step i-1 overlap the scan of step i"}


def measure_e2e_decode(wl, m3, torch, t, st, args, world):
    """Decode end to end: each pass copies the inputs of its T tokens from
    pinned host memory, runs T decode steps (each writing its own slice of
    a [T][b][H][R][P] output) and copies every step's y back."""
    keys = tuple(k for k in ("x", "B", "C", "dt", "lam", "theta") if t[k] is not None)
    host = {k: torch.empty(t[k].shape, dtype=t[k].dtype, pin_memory=True) for k in keys}
    for k in keys:
        host[k].copy_(t[k])
    T = t["x"].shape[0]
    y_all = torch.empty(t["x"].shape, dtype=torch.bfloat16 if wl.y_bf16 else torch.float32, device="cuda")
    yh = torch.empty(y_all.shape, dtype=y_all.dtype, pin_memory=True)
    torch.cuda.synchronize()
    h2d = sum(host[k].numel() * host[k].element_size() for k in keys)
    d2h = y_all.numel() * y_all.element_size()

    def one():
        for k in keys:
            t[k].copy_(host[k], non_blocking=True)
        lam, th = t["lam"], t["theta"]
        for i in range(T):
            m3.m3_decode_step(t["x"][i], t["B"][i], t["C"][i], t["dt"][i], None if lam is None else lam[i],
                              None if th is None else th[i], t["A"], t["D"], y_all[i], st)
        yh.copy_(y_all, non_blocking=True)

    steps = max(2, min(args.steps, 3))
    one()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    return {"value": T * steps * world / el, "unit": "steps/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h}


if __name__ == "__main__":
    main()
