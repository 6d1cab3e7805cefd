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
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "Mamba-3 scan tokens/s (prefill) & decode steps/s; % of HBM/tensor roofline"
L2_BYTES = 126 * 1024 ** 2


def peaks():
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
    H, P, N, R = wl.nheads, wl.headdim, wl.dstate, wl.rank
    if wl.kind == "decode":
        units = wl.batch * H
        per_step_in = units * (R * P + 2 * R * N + 2 + N // 2) * isz
        carry = units * (R * N + R * P) * isz * 2  # read old, write new
        state = units * N * P * 4 * 2
        y = units * R * P * 4
        return dict(per_unit_of_work=per_step_in + carry + state + y, unit="step",
                    inputs=per_step_in, state=state, carry=carry, y=y)
    tokens = wl.seqlen * (wl.batch if wl.kind == "prefill" else 1)
    th = tokens * H
    per_th_in = (R * P + 2 * R * N + 2 + N // 2) * isz
    nseq = wl.nseq if wl.kind == "varlen" else wl.batch
    state = nseq * H * N * P * 4 * 2  # h0 read + h_final write
    carry = nseq * H * (R * N + R * P) * isz * 2
    total = th * (per_th_in + R * P * 4) + state + carry
    return dict(per_unit_of_work=total, unit="pass", inputs=th * per_th_in, y=th * R * P * 4,
                state=state, carry=carry, per_token_head=per_th_in + R * P * 4)


def kernel_source_hash():
    h = hashlib.sha256()
    for d in ("state_space_sequence_06_b300/csrc", "include"):
        for fn in sorted(os.listdir(os.path.join(ROOT, d))):
            with open(os.path.join(ROOT, d, fn), "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        e = d.get(kernel_key)
        if e and e.get("source_sha") == kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during timing."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


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


def config_of(wl):
    c = {"workload": wl.name, "kind": wl.kind, "batch": wl.batch, "seq_len": wl.seqlen, "heads": wl.nheads,
         "headdim": wl.headdim, "dstate": wl.dstate, "rank": wl.rank, "in_dtype": wl.dtype}
    if wl.kind != "decode":
        c["chunk"] = wl.chunk
    if wl.kind == "varlen":
        c["nseq"] = wl.nseq
    return c


# ------------------------------------------------------------------ GPU arm


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="siso_b8_l4096")
    ap.add_argument("--algo", default="auto", choices=["auto", "recurrent", "chunked"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    wl = synth.workloads()[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)

    import torch
    import torch.distributed as dist

    import state_space_sequence_06_b300 as m3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    algo = {"auto": m3.M3_ALGO_AUTO, "recurrent": m3.M3_ALGO_RECURRENT, "chunked": m3.M3_ALGO_CHUNKED}[args.algo]
    hbm_peak, tc_peak, peak_src = peaks()
    stream = torch.cuda.current_stream()

    def dev(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.bfloat16)
        return t.cuda()

    dims_dtype = m3.M3_BF16 if wl.dtype == "bf16" else m3.M3_F32
    H, P, N, R = wl.nheads, wl.headdim, wl.dstate, wl.rank
    byt = workload_bytes(wl)
    ev_pairs = []

    if wl.kind == "decode":
        d = synth.decode_inputs(wl)
        T = wl.seqlen
        t = {k: dev(d[k]) for k in ("x", "B", "C", "dt", "lam", "theta", "A", "D")}
        A, D = t["A"], t["D"]
        st = m3.m3_state_alloc(m3.make_dims(wl.batch, H, P, N, R, dims_dtype))
        hv, pB, px = st.views()
        h0 = dev(d["h0"])
        pB0, px0 = dev(d["prev_B"]), dev(d["prev_x"])
        y = torch.empty((wl.batch, H, R, P), dtype=torch.float32, device="cuda")

        def step():
            hv.copy_(h0)  # every pass starts from the same initial state
            pB.copy_(pB0)
            px.copy_(px0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(T):
                m3.m3_decode_step(t["x"][i], t["B"][i], t["C"][i], t["dt"][i], t["lam"][i], t["theta"][i],
                                  A, D, y, st)
            e1.record(stream)
            ev_pairs.append((e0, e1))

        launches_per_step = T
        units_per_step = T  # decode steps
        unit_name = "steps/s"
        kernel_key = f"decode_step:{wl.name}"
        bytes_per_launch = byt["per_unit_of_work"]
        h2d = sum(d[k].nbytes for k in ("x", "B", "C", "dt", "lam", "theta"))
        d2h = T * y.numel() * 4
    else:
        inp = synth.prefill_inputs(wl)
        t = {k: dev(inp[k]) for k in ("x", "B", "C", "dt", "lam", "theta", "A", "D")}
        cu = None
        nseq = wl.batch
        if wl.kind == "varlen":
            cu = torch.from_numpy(wl.cu_seqlens).cuda()
            nseq = wl.nseq
        st = m3.m3_state_alloc(m3.make_dims(nseq, H, P, N, R, dims_dtype))
        y = torch.empty(t["x"].shape, dtype=torch.float32, device="cuda")

        def step():
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            m3.m3_scan_prefill(t["x"], t["B"], t["C"], t["dt"], t["lam"], t["theta"], t["A"], t["D"], y,
                               state=st, cu_seqlens=cu, algo=algo, chunk=wl.chunk)
            e1.record(stream)
            ev_pairs.append((e0, e1))

        launches_per_step = 1
        units_per_step = wl.seqlen * (wl.batch if wl.kind == "prefill" else 1)  # tokens
        unit_name = "tokens/s"
        kernel_key = f"prefill:{wl.name}:{args.algo}"
        bytes_per_launch = byt["per_unit_of_work"]
        h2d = sum(inp[k].nbytes for k in ("x", "B", "C", "dt", "lam", "theta"))
        d2h = y.numel() * 4

    # which prefill kernel runs: the chunked one multiplies bf16 operands on
    # the tensor cores (f32 accumulation); the recurrent one is f32 throughout
    path_dtype = "f32"
    if wl.kind != "decode" and wl.dtype == "bf16" and algo != m3.M3_ALGO_RECURRENT:
        try:
            m3.m3_scan_prefill(t["x"], t["B"], t["C"], t["dt"], t["lam"], t["theta"], t["A"], t["D"], y,
                               state=st, cu_seqlens=cu, algo=m3.M3_ALGO_CHUNKED, chunk=wl.chunk)
            path_dtype = "bf16"
        except m3.M3Error as e:
            if e.status != m3.M3_ERR_UNSUPPORTED:
                raise
    torch.cuda.synchronize()

    # quick sampled parity check of the timed configuration (oracle on 2 units)
    parity = None
    try:
        parity = sampled_parity(wl, m3, t, y, st, step if wl.kind == "decode" else None)
    except Exception as e:  # reported, never hides a number
        parity = {"error": repr(e)[:200]}

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ev_pairs.clear()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
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
    total_ms = g0.elapsed_time(g1)
    if world > 1:
        tt = torch.tensor([total_ms], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt.item())
    kern_ms = [a.elapsed_time(b) for a, b in ev_pairs]
    ms_per_step = total_ms / args.steps
    value = units_per_step * args.steps * world / (total_ms / 1e3)
    status = m3.m3_device_status()

    # end to end through the public API with host buffers: H2D of the step's
    # inputs from pinned memory, the scan, D2H of y, all inside the timed region
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(wl, m3, torch, t, y, st, algo, args, world, stream)

    per_launch_ms = statistics.mean(kern_ms) / launches_per_step
    achieved = bytes_per_launch / launches_per_step / (per_launch_ms / 1e3) / 1e9 if wl.kind != "decode" else \
        bytes_per_launch / (per_launch_ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
            "traffic": traffic_for(kernel_key), "peak_source": peak_src,
            "algorithmic_bytes_per_launch": bytes_per_launch / (1 if wl.kind != "decode" else 1),
            "kernel_ms_per_launch": per_launch_ms}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            r_, cores, sample = oracle_rate(wl, seconds=15.0)
            cpu = {"value": r_, "unit": unit_name, "cores": cores, "kind": "oracle", "sample": sample}
        except Exception as e:
            cpu = {"error": repr(e)[:200]}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": unit_name, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": path_dtype,
            "data": "synthetic (seeded generator; shapes of the pages' 1.5B-scale workloads)",
            "config": dict(config_of(wl), algo=args.algo,
                           l2="inputs larger than L2 (%.2f GB per pass vs 126 MB L2)" % (bytes_per_launch / 1e9)
                           if wl.kind != "decode" else "state larger than L2 (%.0f MB)" % (byt["state"] / 2 / 1e6),
                           parallelism=f"replicas over independent units x{world}"),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps, "device_status": status,
            "clocks": clk.summary(), "parity": parity,
        }
        print(json.dumps(line), flush=True)
    st.free()
    if world > 1:
        dist.destroy_process_group()


def sampled_parity(wl, m3, t, y, st, decode_step_fn):
    """Compare two units of the timed configuration with the oracle."""
    import torch

    import oracle

    if wl.kind == "decode":
        return None  # covered by tests/test_gpu_decode.py at full size
    inp = synth.prefill_inputs(wl) if wl.kind != "decode" else None
    cu = wl.cu_seqlens if wl.kind == "varlen" else None
    nseq = wl.nseq if cu is not None else wl.batch
    U = nseq * wl.nheads
    hv, pB, px = st.views()
    hv.zero_()
    pB.zero_()
    px.zero_()
    m3.m3_scan_prefill(t["x"], t["B"], t["C"], t["dt"], t["lam"], t["theta"], t["A"], t["D"], y, state=st,
                       cu_seqlens=None if cu is None else torch.from_numpy(cu).cuda(), chunk=wl.chunk)
    torch.cuda.synchronize()
    units = [0, U - 1]
    yo, ho, _, _, spans = oracle.prefill(inp, batch=wl.batch, L=wl.seqlen, H=wl.nheads, P=wl.headdim,
                                         N=wl.dstate, R=wl.rank, dtype=wl.dtype, cu_seqlens=cu, units=units)
    errs = []
    for u, (b, t0, n, hd, _) in zip(units, spans):
        g = y[b, t0:t0 + n, hd].double().cpu().numpy()
        r = yo[u]
        errs.append(float(np.max(np.abs(g - r)) / np.sqrt(np.mean(r ** 2))))
    hv.zero_()
    pB.zero_()
    px.zero_()
    return {"units": units, "max_err_over_rms_y": max(errs)}


def measure_e2e(wl, m3, torch, t, y, st, algo, args, world, stream):
    """Same metric through the public API from host buffers."""
    keys = ("x", "B", "C", "dt", "lam", "theta")
    host = {k: torch.empty(t[k].shape, dtype=t[k].dtype, pin_memory=True) for k in keys}
    for k in keys:
        host[k].copy_(t[k])
    yh = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
    torch.cuda.synchronize()
    h2d = sum(host[k].numel() * host[k].element_size() for k in keys)
    if wl.kind == "decode":
        T = wl.seqlen
        d2h = T * y.numel() * 4
        yall = torch.empty((T,) + tuple(y.shape), dtype=y.dtype, pin_memory=True)

        def one():
            for k in keys:
                t[k].copy_(host[k], non_blocking=True)
            for i in range(T):
                m3.m3_decode_step(t["x"][i], t["B"][i], t["C"][i], t["dt"][i], t["lam"][i], t["theta"][i],
                                  t["A"], t["D"], y, st)
                yall[i].copy_(y, non_blocking=True)
        units = T
    else:
        d2h = y.numel() * 4
        cu = torch.from_numpy(wl.cu_seqlens).cuda() if wl.kind == "varlen" else None

        def one():
            for k in keys:
                t[k].copy_(host[k], non_blocking=True)
            m3.m3_scan_prefill(t["x"], t["B"], t["C"], t["dt"], t["lam"], t["theta"], t["A"], t["D"], y,
                               state=st, cu_seqlens=cu, algo=algo, chunk=wl.chunk)
            yh.copy_(y, non_blocking=True)
        units = wl.seqlen * (wl.batch if wl.kind == "prefill" else 1)
    steps = max(3, min(args.steps, 10))
    for _ in range(2):
        one()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    return {"value": units * steps * world / el, "unit": "steps/s" if wl.kind == "decode" else "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


if __name__ == "__main__":
    main()
