"""Mamba-3 SSM state scan on B300 (sm_103a): Python binding of libm3scan.

The compute runs in the CUDA library ``libm3scan.so`` built from
``csrc/`` (see ``build.py``); its C ABI is ``include/m3scan.h``.  This
module only marshals arguments: torch tensors in, raw device pointers and
sizes out, one ctypes call per entry point, same names as the C ABI.
There is no CPU fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libm3scan.so")

M3_OK, M3_ERR_INVALID_ARG, M3_ERR_UNSUPPORTED, M3_ERR_CUDA, M3_ERR_TIMEOUT, M3_ERR_ALLOC, M3_ERR_SCRATCH = range(7)
M3_F32, M3_BF16 = 0, 1
M3_ALGO_AUTO, M3_ALGO_RECURRENT, M3_ALGO_CHUNKED = 0, 1, 2
M3_PRO_DT_SOFTPLUS, M3_PRO_BC_NORM = 1, 2
# include/m3scan_testing.h
(M3_TEST_KERNEL_NONE, M3_TEST_KERNEL_CHUNKED, M3_TEST_KERNEL_CHUNKED_BALANCED, M3_TEST_KERNEL_RECURRENT,
 M3_TEST_KERNEL_CHUNKED_SPLIT) = range(5)
M3_TEST_FAULT_NONE, M3_TEST_FAULT_SKIP_HANDOVER_RELEASE = 0, 1

SYMBOLS = ("m3_state_alloc", "m3_state_free", "m3_state_view", "m3_scan_prefill",
           "m3_decode_step", "m3_device_status", "m3_status_string", "m3_scan_prefill_backward")


class M3Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {m3_status_string(status)} (status {status})")


class m3_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("nheads", ctypes.c_int32), ("headdim", ctypes.c_int32),
                ("dstate", ctypes.c_int32), ("rank", ctypes.c_int32), ("in_dtype", ctypes.c_int32)]


class m3_state_ptrs(ctypes.Structure):
    _fields_ = [("dims", m3_dims), ("h", ctypes.c_void_p), ("prev_B", ctypes.c_void_p),
                ("prev_x", ctypes.c_void_p)]


class m3_prefill_args(ctypes.Structure):
    _fields_ = [("dims", m3_dims), ("seqlen", ctypes.c_int64), ("chunk", ctypes.c_int32),
                ("algo", ctypes.c_int32)] + \
        [(n, ctypes.c_void_p) for n in ("x", "B", "C", "dt", "lam", "theta", "A", "D", "cu_seqlens")] + \
        [("nseq", ctypes.c_int32), ("y", ctypes.c_void_p), ("ngroups", ctypes.c_int32),
         ("y_dtype", ctypes.c_int32), ("prologue", ctypes.c_int32), ("dt_bias", ctypes.c_void_p)]


class m3_decode_args(ctypes.Structure):
    _fields_ = [("dims", m3_dims)] + \
        [(n, ctypes.c_void_p) for n in ("x", "B", "C", "dt", "lam", "theta", "A", "D", "y")] + \
        [("ngroups", ctypes.c_int32), ("y_dtype", ctypes.c_int32), ("prologue", ctypes.c_int32),
         ("dt_bias", ctypes.c_void_p)]


class m3_backward_args(ctypes.Structure):
    _fields_ = [("dims", m3_dims), ("seqlen", ctypes.c_int64)] + \
        [(n, ctypes.c_void_p) for n in ("x", "B", "C", "dt", "lam", "theta", "A", "D", "h0", "prev_B", "prev_x",
                                        "dy", "dh_final", "dx", "dB", "dC", "ddt", "dlam", "dtheta", "dA", "dD",
                                        "dh0", "dprev_B", "dprev_x")] + \
        [("ngroups", ctypes.c_int32), ("algo", ctypes.c_int32), ("chunk", ctypes.c_int32),
         ("prologue", ctypes.c_int32), ("dt_bias", ctypes.c_void_p), ("ddt_bias", ctypes.c_void_p)]


class m3_launch_info(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("grid", ctypes.c_int32), ("scratch_bytes", ctypes.c_int64)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libm3scan.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libm3scan.so is not built ({path}); run state_space_sequence_06_b300/build.py")
    lib = ctypes.CDLL(path)
    vp = ctypes.c_void_p
    lib.m3_state_alloc.argtypes = [ctypes.POINTER(m3_dims), ctypes.POINTER(vp), vp]
    lib.m3_state_free.argtypes = [vp]
    lib.m3_state_view.argtypes = [vp, ctypes.POINTER(m3_state_ptrs)]
    lib.m3_scan_prefill.argtypes = [ctypes.POINTER(m3_prefill_args), vp, vp]
    lib.m3_scan_prefill_noalloc.argtypes = [ctypes.POINTER(m3_prefill_args), vp, vp]
    lib.m3_decode_step.argtypes = [ctypes.POINTER(m3_decode_args), vp, vp]
    lib.m3_scan_prefill_backward.argtypes = [ctypes.POINTER(m3_backward_args), vp]
    lib.m3_device_status.argtypes = [vp]
    lib.m3_test_set_fault.argtypes = [ctypes.c_int32, ctypes.c_int64]
    lib.m3_test_last_launch.argtypes = [ctypes.POINTER(m3_launch_info)]
    for f in ("m3_state_alloc", "m3_state_free", "m3_state_view", "m3_scan_prefill",
              "m3_scan_prefill_noalloc", "m3_decode_step", "m3_device_status", "m3_scan_prefill_backward",
              "m3_test_set_fault", "m3_test_last_launch"):
        getattr(lib, f).restype = ctypes.c_int
    lib.m3_status_string.argtypes = [ctypes.c_int]
    lib.m3_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def m3_status_string(status: int) -> str:
    return load_library().m3_status_string(int(status)).decode()


def _check(rc: int, what: str):
    if rc != M3_OK:
        raise M3Error(rc, what)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t):
    if t is None:
        return None
    if not (t.is_cuda and t.is_contiguous()):
        raise ValueError("tensors must be contiguous CUDA tensors")
    return t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return M3_BF16
    if t.dtype == torch.float32:
        return M3_F32
    raise ValueError(f"unsupported input dtype {t.dtype}")


class _DeviceArray:
    """Zero-copy view of library-owned device memory (CUDA array interface)."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 3, "strides": None}


class State:
    """A library-allocated m3_state; ``h``, ``prev_B`` and ``prev_x`` are
    zero-copy torch views of its device buffers."""

    def __init__(self, handle, dims: m3_dims):
        self.handle = handle
        self.dims = dims

    @property
    def _as_parameter_(self):
        return self.handle

    def views(self):
        p = m3_state_view(self)
        d = p.dims
        K = d.dstate // 2
        ts = "<f4" if d.in_dtype == M3_F32 else "<u2"
        h = torch.as_tensor(_DeviceArray(p.h, (d.batch, d.nheads, K, d.headdim, 2), "<f4"), device="cuda")
        pB = torch.as_tensor(_DeviceArray(p.prev_B, (d.batch, d.nheads, d.rank, d.dstate), ts), device="cuda")
        px = torch.as_tensor(_DeviceArray(p.prev_x, (d.batch, d.nheads, d.rank, d.headdim), ts), device="cuda")
        if d.in_dtype == M3_BF16:
            pB, px = pB.view(torch.bfloat16), px.view(torch.bfloat16)
        return h, pB, px

    def free(self):
        if self.handle:
            m3_state_free(self)
            self.handle = None


def make_dims(batch, nheads, headdim, dstate, rank, in_dtype) -> m3_dims:
    return m3_dims(batch, nheads, headdim, dstate, rank, in_dtype)


def m3_state_alloc(dims: m3_dims, stream=None) -> State:
    h = ctypes.c_void_p()
    _check(load_library().m3_state_alloc(ctypes.byref(dims), ctypes.byref(h), _stream(stream)),
           "m3_state_alloc")
    return State(h.value, dims)


def m3_state_free(state: State):
    _check(load_library().m3_state_free(state.handle), "m3_state_free")


def m3_state_view(state: State) -> m3_state_ptrs:
    out = m3_state_ptrs()
    _check(load_library().m3_state_view(state.handle, ctypes.byref(out)), "m3_state_view")
    return out


def m3_scan_prefill(x, B, C, dt, lam, theta, A, D, y, *, state: State | None = None,
                    cu_seqlens=None, chunk: int = 0, algo: int = M3_ALGO_AUTO, prologue: int = 0,
                    dt_bias=None, stream=None, _entry="m3_scan_prefill"):
    """Prefill.  x [b][L][H][R][P], B/C [b][L][G][R][N] (G groups of heads;
    G = H: one per head), dt/lam [b][L][H], theta [b][L][H][N/2] (all bf16
    or all f32; lam None: lam = 1, theta None: theta = 0), A/D [H] f32,
    y [b][L][H][R][P] f32 or bf16 (written; bf16 is the f32 result rounded
    to nearest even).  ``cu_seqlens`` (int32 CUDA tensor) packs sequences
    in a batch of one row.  ``prologue`` (M3_PRO_* flags) makes the kernel
    apply softplus(dt + dt_bias) and/or the RMS norm of B and C rows."""
    b, L, H, R, P = x.shape
    N = B.shape[-1]
    a = m3_prefill_args()
    a.dims = m3_dims(b, H, P, N, R, _dtype_code(x))
    a.ngroups = B.shape[2]  # B and C [b][L][G][R][N]: G = H is one per head
    a.y_dtype = _dtype_code(y)
    a.prologue, a.dt_bias = prologue, _ptr(dt_bias)
    a.seqlen, a.chunk, a.algo = L, chunk, algo
    a.x, a.B, a.C, a.dt, a.lam, a.theta = (_ptr(t) for t in (x, B, C, dt, lam, theta))
    a.A, a.D, a.y = _ptr(A), _ptr(D), _ptr(y)
    if cu_seqlens is not None:
        a.cu_seqlens = _ptr(cu_seqlens)
        a.nseq = cu_seqlens.numel() - 1
    _check(getattr(load_library(), _entry)(ctypes.byref(a), state.handle if state else None, _stream(stream)),
           _entry)


def m3_scan_prefill_noalloc(x, B, C, dt, lam, theta, A, D, y, *, state: State | None = None,
                            cu_seqlens=None, chunk: int = 0, algo: int = M3_ALGO_AUTO, prologue: int = 0,
                            dt_bias=None, stream=None):
    """m3_scan_prefill without device-memory allocation in the call: its
    scratch is a fixed buffer in the library (calls that overlap in time
    race on it; M3_ERR_SCRATCH when a request needs more)."""
    m3_scan_prefill(x, B, C, dt, lam, theta, A, D, y, state=state, cu_seqlens=cu_seqlens, chunk=chunk,
                    algo=algo, prologue=prologue, dt_bias=dt_bias, stream=stream,
                    _entry="m3_scan_prefill_noalloc")


def m3_decode_step(x, B, C, dt, lam, theta, A, D, y, state: State, stream=None, prologue: int = 0,
                   dt_bias=None):
    """One decode step.  x [b][H][R][P], B/C [b][G][R][N] (G groups of heads;
    G = H: one per head), dt/lam [b][H], theta [b][H][N/2] (lam / theta
    None: 1 / 0), A/D [H] f32, y [b][H][R][P] f32 or bf16 (written)."""
    b, H, R, P = x.shape
    N = B.shape[-1]
    a = m3_decode_args()
    a.dims = m3_dims(b, H, P, N, R, _dtype_code(x))
    a.ngroups = B.shape[1]
    a.y_dtype = _dtype_code(y)
    a.prologue, a.dt_bias = prologue, _ptr(dt_bias)
    a.x, a.B, a.C, a.dt, a.lam, a.theta = (_ptr(t) for t in (x, B, C, dt, lam, theta))
    a.A, a.D, a.y = _ptr(A), _ptr(D), _ptr(y)
    _check(load_library().m3_decode_step(ctypes.byref(a), state.handle, _stream(stream)),
           "m3_decode_step")


def m3_scan_prefill_backward(x, B, C, dt, lam, theta, A, D, dy, *, h0=None, prev_B=None, prev_x=None,
                             dh_final=None, algo: int = M3_ALGO_AUTO, chunk: int = 0, prologue: int = 0,
                             dt_bias=None, stream=None) -> dict:
    """Gradients of a loss with respect to every prefill input, given dy =
    dL/dy [b][L][H][R][P] f32 (and dh_final = dL/dh_final [b][H][N/2][P][2]).
    Inputs as for m3_scan_prefill (fixed-length batch); h0 [b][H][N/2][P][2]
    f32, prev_B / prev_x the carry.  ``algo``: AUTO (the chunked kernel
    where the shape has it), RECURRENT (token-serial) or CHUNKED.  With
    ``prologue`` flags the inputs are raw and the gradients are with respect
    to them (``ddt_bias`` too).  Returns f32 CUDA tensors dx, dB, dC, ddt,
    dlam, dtheta, dA, dD, dh0, dprev_B, dprev_x (and ddt_bias) in the
    inputs' layouts (allocated here; the kernels are the library's)."""
    b, L, H, R, P = x.shape
    N = B.shape[-1]
    f32 = dict(dtype=torch.float32, device=x.device)
    out = dict(dx=torch.empty(x.shape, **f32), dB=torch.empty(B.shape, **f32), dC=torch.empty(C.shape, **f32),
               ddt=torch.empty(dt.shape, **f32), dlam=torch.empty(dt.shape, **f32),
               dtheta=torch.empty(dt.shape + (N // 2,), **f32), dA=torch.empty(H, **f32),
               dD=torch.empty(H, **f32), dh0=torch.empty((b, H, N // 2, P, 2), **f32),
               dprev_B=torch.empty((b, H, R, N), **f32), dprev_x=torch.empty((b, H, R, P), **f32))
    if prologue & M3_PRO_DT_SOFTPLUS:
        out["ddt_bias"] = torch.empty(H, **f32)
    a = m3_backward_args()
    a.dims = m3_dims(b, H, P, N, R, _dtype_code(x))
    a.seqlen, a.ngroups = L, B.shape[2]
    a.algo, a.chunk, a.prologue, a.dt_bias = algo, chunk, prologue, _ptr(dt_bias)
    for name, t in (("x", x), ("B", B), ("C", C), ("dt", dt), ("lam", lam), ("theta", theta), ("A", A),
                    ("D", D), ("h0", h0), ("prev_B", prev_B), ("prev_x", prev_x), ("dy", dy),
                    ("dh_final", dh_final)):
        setattr(a, name, _ptr(t))
    for name, t in out.items():
        setattr(a, name, _ptr(t))
    _check(load_library().m3_scan_prefill_backward(ctypes.byref(a), _stream(stream)), "m3_scan_prefill_backward")
    return out


def m3_device_status(stream=None) -> int:
    return load_library().m3_device_status(_stream(stream))


def m3_test_set_fault(fault: int, wait_limit_ns: int = 0):
    """Test hook: plant a fault (M3_TEST_FAULT_*) in the following prefill
    launches and set their bounded-wait limit (0: the default)."""
    _check(load_library().m3_test_set_fault(int(fault), int(wait_limit_ns)), "m3_test_set_fault")


def m3_test_last_launch() -> m3_launch_info:
    """Test hook: the kernel, grid and handover scratch of the last prefill."""
    out = m3_launch_info()
    _check(load_library().m3_test_last_launch(ctypes.byref(out)), "m3_test_last_launch")
    return out
