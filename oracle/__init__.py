"""CPU oracle of the Mamba-3 SSM state scan (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never loads it and
shares no code with it.

``m3_oracle.c`` walks the recurrence token by token in complex double (see
its header for the equations and the readings taken where the pages are
silent).  ``backward.py`` is the exact gradient of that forward pass, and
``apply_prologue`` the fused prologue (softplus of dt, RMS norm of B and C).  This wrapper only builds the table of units (which (sequence,
head) pairs to walk, and where their tokens live) and converts arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "m3_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libm3oracle.so")

DTYPE_CODE = {"f32": 0, "bf16": 1, "f64": 2}


class _Unit(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "ntok", "x0", "xs", "b0", "bs", "s0", "ss", "q0", "qs", "y0", "ys", "head")]


def compile_lib(src: str, out: str) -> str:
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_lib(_SRC, _LIB_PATH)
    return _LIB_PATH


def load(path: str | None = None):
    """Load the oracle library (``path`` lets tests load a modified copy)."""
    if path is None:
        path = build()
    lib = ctypes.CDLL(path)
    lib.m3_oracle_run.argtypes = [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
    ] + [ctypes.c_void_p] * 12 + [ctypes.c_int]
    lib.m3_oracle_run.restype = ctypes.c_int
    return lib


_default = None


def _lib():
    global _default
    if _default is None:
        _default = load()
    return _default


def _c(a, dtype=None):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def run_units(units, R, P, N, dtype, x, B, C, dt, lam, theta, A, D, h, prev_B, prev_x, ytot,
              nthreads=None, lib=None):
    """Low-level call: ``units`` is a list of dicts with the _Unit fields."""
    lib = lib or _lib()
    tab = (_Unit * max(1, len(units)))()
    for i, u in enumerate(units):
        for k, v in u.items():
            setattr(tab[i], k, int(v))
    h = np.ascontiguousarray(h, dtype=np.float64)
    prev_B = np.ascontiguousarray(prev_B, dtype=np.float64)
    prev_x = np.ascontiguousarray(prev_x, dtype=np.float64)
    y = np.zeros(ytot, dtype=np.float64)
    keep = []
    ptrs = []
    for a in (x, B, C, dt, lam, theta):
        a, p = _c(a)
        keep.append(a)
        ptrs.append(p)
    A_, pA = _c(A, np.float64)
    D_, pD = _c(D, np.float64)
    nthreads = nthreads or os.cpu_count() or 1
    rc = lib.m3_oracle_run(
        ctypes.addressof(tab), len(units), R, P, N, DTYPE_CODE[dtype], *ptrs, pA, pD,
        h.ctypes.data, prev_B.ctypes.data, prev_x.ctypes.data, y.ctypes.data, nthreads,
    )
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return y, h, prev_B, prev_x


def prefill(inp: dict, *, batch, L, H, P, N, R, dtype, cu_seqlens=None, units=None,
            h0=None, prev_B=None, prev_x=None, nthreads=None, lib=None):
    """Run the oracle over a prefill workload (or a subset of its units).

    ``inp`` holds x [b][L][H][R][P], B/C [b][L][G][R][N] (G groups of
    consecutive heads share B and C; G = H: one per head), dt/lam [b][L][H],
    theta [b][L][H][N/2], A/D [H].  Units are ``s*H + h`` where s is the
    batch row, or the sequence index when ``cu_seqlens`` is given (then
    b == 1).  ``h0``/``prev_B``/``prev_x`` are per-sequence initial states
    ([S][H][N/2][P][2], [S][H][R][N], [S][H][R][P]); zero when omitted.

    Returns ``(y, h, prev_B, prev_x, spans)``: ``y`` in the full layout
    [b][L][H][R][P] when every unit is walked, else a dict unit -> [T][R][P];
    ``h`` etc. per walked unit in ``units`` order.
    """
    nseq = batch if cu_seqlens is None else len(cu_seqlens) - 1
    all_units = list(range(nseq * H))
    sel = all_units if units is None else list(units)
    K = N // 2
    G = np.shape(inp["B"])[2]
    tab, spans, yoff = [], [], 0
    for u in sel:
        s, hd = divmod(u, H)
        if cu_seqlens is None:
            b, t_beg, ntok = s, 0, L
        else:
            b, t_beg, ntok = 0, int(cu_seqlens[s]), int(cu_seqlens[s + 1] - cu_seqlens[s])
        tok0 = b * L + t_beg
        tab.append(dict(
            ntok=ntok,
            x0=(tok0 * H + hd) * R * P, xs=H * R * P,
            b0=(tok0 * G + hd // (H // G)) * R * N, bs=G * R * N,
            s0=tok0 * H + hd, ss=H,
            q0=(tok0 * H + hd) * K, qs=H * K,
            y0=yoff, ys=R * P, head=hd,
        ))
        spans.append((b, t_beg, ntok, hd, yoff))
        yoff += ntok * R * P

    def per_unit(a, shape):
        if a is None:
            return np.zeros((len(sel),) + shape)
        a = _widen(a, dtype).reshape((nseq * H,) + shape)
        return a[sel]

    h = np.zeros((len(sel), K, P, 2)) if h0 is None else \
        np.asarray(h0, np.float64).reshape((nseq * H, K, P, 2))[sel]
    pB = per_unit(prev_B, (R, N))
    px = per_unit(prev_x, (R, P))
    lam, theta = _lam_theta(inp, K)
    yflat, h, pB, px = run_units(tab, R, P, N, dtype, inp["x"], inp["B"], inp["C"], inp["dt"],
                                 lam, theta, inp["A"], inp["D"], h, pB, px, yoff,
                                 nthreads=nthreads, lib=lib)
    if units is None:
        y = np.zeros((batch, L, H, R, P))
        for (b, t_beg, ntok, hd, off) in spans:
            y[b, t_beg:t_beg + ntok, hd] = yflat[off:off + ntok * R * P].reshape(ntok, R, P)
    else:
        y = {u: yflat[off:off + ntok * R * P].reshape(ntok, R, P)
             for u, (b, t_beg, ntok, hd, off) in zip(sel, spans)}
    return y, h.reshape((len(sel), K, P, 2)), pB, px, spans


def decode(inp: dict, *, batch, H, P, N, R, dtype, steps, units=None, nthreads=None, lib=None):
    """Run ``steps`` single-token decode steps from the initial state in ``inp``.

    ``inp`` holds per-step tensors x [T][b][H][R][P], B/C [T][b][G][R][N],
    dt/lam [T][b][H], theta [T][b][H][N/2] plus h0, prev_B, prev_x.  Units
    are ``b*H + h``.  Returns ``(y, h, prev_B, prev_x)`` with y
    [T][b][H][R][P] when every unit is walked, else a dict unit -> [T][R][P].
    """
    K = N // 2
    G = np.shape(inp["B"])[2]  # B/C [T][b][G][R][N]
    sel = list(range(batch * H)) if units is None else list(units)
    tab = []
    for i, u in enumerate(sel):
        b, hd = divmod(u, H)
        tab.append(dict(
            ntok=steps,
            x0=u * R * P, xs=batch * H * R * P,
            b0=(b * G + hd // (H // G)) * R * N, bs=batch * G * R * N,
            s0=u, ss=batch * H,
            q0=u * K, qs=batch * H * K,
            y0=i * steps * R * P, ys=R * P, head=hd,
        ))
    h = np.asarray(inp["h0"], np.float64).reshape(batch * H, K, P, 2)[sel]
    pB = _widen(inp["prev_B"], dtype).reshape(batch * H, R, N)[sel]
    px = _widen(inp["prev_x"], dtype).reshape(batch * H, R, P)[sel]
    lam, theta = _lam_theta(inp, K)
    yflat, h, pB, px = run_units(tab, R, P, N, dtype, inp["x"], inp["B"], inp["C"], inp["dt"],
                                 lam, theta, inp["A"], inp["D"], h, pB, px,
                                 len(sel) * steps * R * P, nthreads=nthreads, lib=lib)
    yu = yflat.reshape(len(sel), steps, R, P)
    if units is None:
        y = yu.reshape(batch, H, steps, R, P).transpose(2, 0, 1, 3, 4).copy()
    else:
        y = {u: yu[i] for i, u in enumerate(sel)}
    return y, h.reshape(len(sel), K, P, 2), pB, px


BC_NORM_EPS = 1e-6


def softplus(z):
    """log(1 + e^z) in double, written as max(z, 0) + log1p(e^-|z|): no
    overflow for large z, no cancellation for very negative z."""
    z = np.asarray(z, np.float64)
    return np.maximum(z, 0.0) + np.log1p(np.exp(-np.abs(z)))


def rms_normalize(a, eps=BC_NORM_EPS):
    """Each row (last axis) divided by its root mean square,
    a / sqrt(mean(a^2) + eps): the BC/QK norm ("Mamba-3: an inference-first
    LLM", section "Implementation and kernel optimisation")."""
    a = np.asarray(a, np.float64)
    return a / np.sqrt(np.mean(a * a, axis=-1, keepdims=True) + eps)


def apply_prologue(inp: dict, dtype: str, *, dt_softplus=False, bc_norm=False, dt_bias=None) -> dict:
    """The inputs as the scan sees them after the fused prologue, in double
    (run the oracle on the result with dtype "f64").  dt becomes
    softplus(dt + dt_bias[h]) (heads on dt's last axis, in prefill and
    decode layouts); every row over N of B, C and the carried prev_B is
    RMS-normalised.  The other inputs are widened unchanged; lam and theta
    given as None stay None, h0, A and D are kept as they are."""
    out = {}
    for k, v in inp.items():
        out[k] = v if (v is None or k in ("A", "D", "h0", "dt_bias")) else _widen(v, dtype)
    if dt_softplus:
        bias = 0.0 if dt_bias is None else np.asarray(dt_bias, np.float64)
        out["dt"] = softplus(out["dt"] + bias)
    if bc_norm:
        for k in ("B", "C", "prev_B"):
            if out.get(k) is not None:
                out[k] = rms_normalize(out[k])
    return out


def _lam_theta(inp, K):
    """lam and theta of ``inp``; None stands for lam = 1 and theta = 0 (the
    first-order, real-state special case), written out as arrays."""
    lam, theta = inp.get("lam"), inp.get("theta")
    dt = np.asarray(inp["dt"])  # the C oracle reads every input in dt's storage type
    if lam is None:
        lam = np.full(dt.shape, 0x3F80, np.uint16) if dt.dtype == np.uint16 else np.ones(dt.shape, dt.dtype)
    if theta is None:
        theta = np.zeros(dt.shape + (K,), dt.dtype)
    return lam, theta


def _widen(a, dtype):
    a = np.asarray(a)
    if dtype == "bf16" and a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


# the backward pass (gradients of the forward above), for training parity cases
from .backward import prefill_backward, unit_backward  # noqa: E402,F401
