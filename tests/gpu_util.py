"""Helpers shared by the GPU parity tests: move generator arrays to the
device, run the library through its C ABI binding, and measure errors the
way the tolerance is stated (max |err| / rms(reference))."""
from __future__ import annotations

import numpy as np
import torch

import state_space_sequence_06_b300 as m3

TOL = {"f32": 1e-4, "bf16": 1e-2}


def dev(a: np.ndarray | None, dtype: str | None = None) -> torch.Tensor | None:
    """numpy -> CUDA tensor; uint16 arrays are bf16 bit patterns; None stays
    None (an input the library treats as its special value)."""
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.cuda()


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    return float(np.max(np.abs(got - ref)) / max(rms, 1e-30))


def assert_close(got, ref, tol, what):
    e = rel_err(got, ref)
    assert e <= tol, f"{what}: max|err|/rms = {e:.3e} > {tol:.1e}"
    return e


def prefill_gpu(inp: dict, wl, *, state=None, cu=None, algo=m3.M3_ALGO_AUTO, chunk=0, y_dtype=torch.float32,
                prologue=0):
    """Run m3_scan_prefill on device copies of ``inp``; returns y (torch)."""
    t = {k: dev(v) for k, v in inp.items() if k in ("x", "B", "C", "dt", "lam", "theta", "A", "D")}
    b, L, H, R, P = inp["x"].shape
    y = torch.empty((b, L, H, R, P), dtype=y_dtype, device="cuda")
    cu_t = None if cu is None else torch.from_numpy(np.asarray(cu, np.int32)).cuda()
    m3.m3_scan_prefill(t["x"], t["B"], t["C"], t["dt"], t["lam"], t["theta"], t["A"], t["D"], y,
                       state=state, cu_seqlens=cu_t, algo=algo, chunk=chunk, prologue=prologue,
                       dt_bias=dev(inp.get("dt_bias")) if prologue else None)
    return y


def state_for(wl_dims, h0=None, prev_B=None, prev_x=None):
    """Allocate a library state and load an initial h / carry into it."""
    st = m3.m3_state_alloc(m3.make_dims(*wl_dims))
    h, pB, px = st.views()
    if h0 is not None:
        h.copy_(dev(np.asarray(h0, np.float32)))
    if prev_B is not None:
        pB.copy_(dev(prev_B))
    if prev_x is not None:
        px.copy_(dev(prev_x))
    return st


def widen(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return widen(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.detach().cpu().numpy().astype(np.float64)
