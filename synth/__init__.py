"""Seeded synthetic inputs for the Mamba-3 scan workloads.

The workloads stand in for the pages' H100 measurements on a 1.5B model
("Together AI announces Mamba-3", inference-speed table): the shapes are
those of a 1.5B-scale Mamba-3 layer, the values are drawn from fixed
distributions, and nothing comes from a dataset or a checkpoint.

This module holds none of the scan's arithmetic.  It only draws tensors
(through ``m3_synth.c``) and returns them as numpy arrays; bf16 tensors are
returned as ``uint16`` bit patterns.  Both the CPU oracle and the GPU path
consume these arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "m3_synth.c")
_LIB_PATH = os.path.join(_HERE, "libm3synth.so")

# tensor stream ids (part of the generator's definition: changing one changes the data)
S_X, S_B, S_C, S_DT, S_A, S_THETA, S_LAM, S_D, S_H0, S_PREVB, S_PREVX, S_LENS, S_DTBIAS = range(1, 14)

# distribution kinds, as in m3_synth.c
K_NORMAL, K_NORMAL_RMS, K_SOFTPLUS, K_NEG_EXP, K_UNIFORM, K_SIGMOID = range(6)
OUT_F32, OUT_BF16, OUT_F64 = 0, 1, 2

RMS_EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile the generator into ``synth/libm3synth.so`` (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def _get_lib():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.synth_fill.argtypes = [
            ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_double,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
        ]
        lib.synth_fill.restype = ctypes.c_int
        lib.synth_lengths.argtypes = [
            ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_void_p,
        ]
        lib.synth_lengths.restype = ctypes.c_int
        _lib = lib
    return _lib


def fill(shape, stream, kind, p0=0.0, p1=1.0, dtype="f32", seed=0, offset=0, row_len=0):
    """Draw a tensor of ``shape`` (elements ``offset..`` of stream ``stream``)."""
    out_code = {"f32": OUT_F32, "bf16": OUT_BF16, "f64": OUT_F64}[dtype]
    np_dtype = {"f32": np.float32, "bf16": np.uint16, "f64": np.float64}[dtype]
    out = np.empty(shape, dtype=np_dtype)
    rc = _get_lib().synth_fill(
        seed, stream, kind, float(p0), float(p1), int(offset), int(out.size), int(row_len),
        out_code, out.ctypes.data,
    )
    if rc != 0:
        raise ValueError("synth_fill rejected its arguments")
    return out


def lengths(count, lo, hi, seed=0, stream=S_LENS):
    out = np.empty(count, dtype=np.int32)
    if _get_lib().synth_lengths(seed, stream, lo, hi, count, out.ctypes.data) != 0:
        raise ValueError("synth_lengths rejected its arguments")
    return out


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64 exactly."""
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_to_f64(a) if dtype == "bf16" else a.astype(np.float64)


@dataclass
class Workload:
    """One synthetic workload: shapes, dtype and the distribution recipe."""

    name: str
    kind: str  # "prefill" | "varlen" | "decode"
    batch: int
    seqlen: int  # tokens per sequence (prefill); steps (decode); total tokens (varlen)
    nheads: int
    headdim: int
    dstate: int
    rank: int = 1
    dtype: str = "bf16"
    chunk: int = 64
    dt_shift: float = -4.0
    h0_std: float = 0.0  # 0: zero initial state
    carry: bool = False  # draw an initial previous-token (B, x) carry
    nseq: int = 0  # varlen: number of sequences
    len_lo: int = 0
    len_hi: int = 0
    seed: int = 0
    real: bool = False   # theta = 0: a real state (given as None)
    euler: bool = False  # lam = 1: first-order exponential Euler (given as None)
    ngroups: int = 0  # B/C groups shared by nheads/ngroups consecutive heads; 0: one per head
    y_bf16: bool = False  # output y in bf16 (else f32)
    # raw inputs for the fused prologue: dt the pre-activation N(dt_shift, 1)
    # with a per-head bias N(0, 0.5), B and C (and the carried B) N(0, 2^2)
    # without row normalisation
    prologue: bool = False
    backward: bool = False  # a training-pass workload: the backward of this prefill (timed by name only)
    cu_seqlens: np.ndarray | None = field(default=None, repr=False)
    # shard of a global problem: this shard's `batch` sequences (varlen:
    # `nseq` sequences) are number shard_index*batch.. of a global batch of
    # shards*batch
    shard_index: int = 0
    shards: int = 1
    tok_offset: int = 0  # varlen: first global token of this shard

    @property
    def groups(self) -> int:
        return self.ngroups or self.nheads

    @property
    def units(self) -> int:
        return (self.nseq if self.kind == "varlen" else self.batch) * self.nheads


# The five workloads (config 3 has two variants, config 4 two parts).
def workloads() -> dict:
    w = {
        "tiny_f32": Workload("tiny_f32", "prefill", 1, 64, 2, 16, 16, 1, "f32", chunk=64),
        "siso_b8_l4096": Workload("siso_b8_l4096", "prefill", 8, 4096, 32, 64, 128, 1, "bf16", chunk=64),
        "mimo4_b8_l4096": Workload("mimo4_b8_l4096", "prefill", 8, 4096, 32, 64, 64, 4, "bf16", chunk=16),
        "decode_siso_b256": Workload(
            "decode_siso_b256", "decode", 256, 1024, 32, 64, 128, 1, "bf16", h0_std=0.1, carry=True
        ),
        "decode_mimo4_b256": Workload(
            "decode_mimo4_b256", "decode", 256, 1024, 32, 64, 64, 4, "bf16", h0_std=0.1, carry=True
        ),
        "long_l16384": Workload("long_l16384", "prefill", 1, 16384, 32, 64, 128, 1, "bf16", chunk=64, dt_shift=-3.0),
        # Mamba-3 with half the state (N 64: 32 complex pairs), the size at which the pages report
        # Mamba-2's N 128 perplexity
        "siso_n64_b8_l4096": Workload("siso_n64_b8_l4096", "prefill", 8, 4096, 32, 64, 64, 1, "bf16", chunk=64),
        "decode_siso_n64_b256": Workload(
            "decode_siso_n64_b256", "decode", 256, 1024, 32, 64, 64, 1, "bf16", h0_std=0.1, carry=True),
        # the Mamba-2 special case on the same shapes: real state (theta = 0), first order (lam = 1)
        "mamba2_b8_l4096": Workload("mamba2_b8_l4096", "prefill", 8, 4096, 32, 64, 128, 1, "bf16", chunk=64,
                                    real=True, euler=True),
        "decode_mamba2_b256": Workload(
            "decode_mamba2_b256", "decode", 256, 1024, 32, 64, 128, 1, "bf16", h0_std=0.1, carry=True,
            real=True, euler=True),
        # B and C shared by all heads (one group), as a mixer layer usually projects them
        "siso_g1_b8_l4096": Workload("siso_g1_b8_l4096", "prefill", 8, 4096, 32, 64, 128, 1, "bf16", chunk=64,
                                     ngroups=1),
        "mimo4_g1_b8_l4096": Workload("mimo4_g1_b8_l4096", "prefill", 8, 4096, 32, 64, 64, 4, "bf16", chunk=16,
                                      ngroups=1),
        "decode_siso_g1_b256": Workload(
            "decode_siso_g1_b256", "decode", 256, 1024, 32, 64, 128, 1, "bf16", h0_std=0.1, carry=True,
            ngroups=1),
        # the same SISO prefill with y written in bf16
        "siso_ybf16_b8_l4096": Workload("siso_ybf16_b8_l4096", "prefill", 8, 4096, 32, 64, 128, 1, "bf16",
                                        chunk=64, y_bf16=True),
        # the same SISO prefill from raw inputs: dt before softplus, B and C before the RMS norm
        "siso_prologue_b8_l4096": Workload("siso_prologue_b8_l4096", "prefill", 8, 4096, 32, 64, 128, 1, "bf16",
                                           chunk=64, prologue=True),
        # the backward pass of a prefill: batch 2, L 1024, and the SISO layer shape of the prefill line
        "backward_siso_b2_l1024": Workload("backward_siso_b2_l1024", "prefill", 2, 1024, 32, 64, 128, 1, "bf16",
                                           h0_std=0.1, carry=True, backward=True),
        "backward_siso_b8_l4096": Workload("backward_siso_b8_l4096", "prefill", 8, 4096, 32, 64, 128, 1, "bf16",
                                           h0_std=0.1, carry=True, backward=True),
        "backward_mimo4_b8_l4096": Workload("backward_mimo4_b8_l4096", "prefill", 8, 4096, 32, 64, 64, 4, "bf16",
                                            chunk=16, h0_std=0.1, carry=True, backward=True),
        "varlen_16": Workload(
            "varlen_16", "varlen", 1, 0, 32, 64, 128, 1, "bf16", chunk=64, dt_shift=-3.0,
            nseq=16, len_lo=256, len_hi=8192,
        ),
    }
    v = w["varlen_16"]
    lens = lengths(v.nseq, v.len_lo, v.len_hi, seed=v.seed)
    v.cu_seqlens = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    v.seqlen = int(v.cu_seqlens[-1])
    return w


def shard(wl: Workload, rank: int, world: int) -> Workload:
    """Rank `rank`'s part of the global problem made of `world` copies of
    `wl`'s batch: the global batch is world*batch sequences (varlen:
    world*nseq packed sequences, lengths drawn for all of them), and this
    rank holds a contiguous group of them.  Per-head weights (A, D) are the
    same on every rank.  Concatenating the shards' tensors over ranks gives
    exactly the global problem's tensors."""
    if not (0 <= rank < world):
        raise ValueError("rank out of range")
    out = scaled(wl, shard_index=rank, shards=world)
    if wl.kind == "varlen":
        lens = lengths(wl.nseq * world, wl.len_lo, wl.len_hi, seed=wl.seed)
        glob = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        mine = lens[rank * wl.nseq:(rank + 1) * wl.nseq]
        out.cu_seqlens = np.concatenate([[0], np.cumsum(mine)]).astype(np.int32)
        out.seqlen = int(out.cu_seqlens[-1])
        out.tok_offset = int(glob[rank * wl.nseq])
    return out


def scaled(wl: Workload, **kw) -> Workload:
    """A copy of ``wl`` with some fields replaced (smaller parity-test sizes)."""
    d = dict(wl.__dict__)
    d.update(kw)
    return Workload(**d)


def varlen_cu_seqlens(lens) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lens, dtype=np.int64))]).astype(np.int32)


def prefill_inputs(wl: Workload) -> dict:
    """All tensors of a prefill workload.

    Layouts (token-major, heads inside):  x [b][L][H][R][P], B and C
    [b][L][G][R][N] (G = ngroups, else H), dt and lam [b][L][H], theta
    [b][L][H][N/2]; A and D [H] float32.  For a varlen workload b = 1 and
    L = total tokens.
    """
    b, L, H, P, N, R = wl.batch, wl.seqlen, wl.nheads, wl.headdim, wl.dstate, wl.rank
    G = wl.groups
    dt_ = wl.dtype
    s = wl.seed
    # first token (over b*L) and first unit of this shard in the global problem
    t0 = wl.tok_offset if wl.kind == "varlen" else wl.shard_index * b * L
    u0 = wl.shard_index * (wl.nseq if wl.kind == "varlen" else b) * H

    def tok(shape, stream, kind, p0, p1, row_len=0):
        per_tok = int(np.prod(shape[2:]))
        return fill(shape, stream, kind, p0, p1, dt_, s, offset=t0 * per_tok, row_len=row_len)

    def unit(shape, stream, kind, p0, p1, dtype, row_len=0):
        per_unit = int(np.prod(shape[2:]))
        return fill(shape, stream, kind, p0, p1, dtype, s, offset=u0 * per_unit, row_len=row_len)

    d = {
        "x": tok((b, L, H, R, P), S_X, K_NORMAL, 0.0, 1.0),
        "B": tok((b, L, G, R, N), S_B, K_NORMAL, 0.0, 2.0) if wl.prologue else
        tok((b, L, G, R, N), S_B, K_NORMAL_RMS, RMS_EPS, 0.0, row_len=N),
        "C": tok((b, L, G, R, N), S_C, K_NORMAL, 0.0, 2.0) if wl.prologue else
        tok((b, L, G, R, N), S_C, K_NORMAL_RMS, RMS_EPS, 0.0, row_len=N),
        "dt": tok((b, L, H), S_DT, K_NORMAL, wl.dt_shift, 1.0) if wl.prologue else
        tok((b, L, H), S_DT, K_SOFTPLUS, wl.dt_shift, 0.0),
        "lam": tok((b, L, H), S_LAM, K_SIGMOID, 0.0, 0.0),
        "theta": tok((b, L, H, N // 2), S_THETA, K_UNIFORM, 0.0, np.pi),
        "A": fill((H,), S_A, K_NEG_EXP, 0.0, 0.5, "f32", s),
        "D": fill((H,), S_D, K_NORMAL, 0.0, 1.0, "f32", s),
    }
    if wl.real:
        d["theta"] = None
    if wl.euler:
        d["lam"] = None
    if wl.prologue:
        d["dt_bias"] = fill((H,), S_DTBIAS, K_NORMAL, 0.0, 0.5, "f32", s)
    nseq = wl.nseq if wl.kind == "varlen" else b
    if wl.h0_std > 0:
        d["h0"] = unit((nseq, H, N // 2, P, 2), S_H0, K_NORMAL, 0.0, wl.h0_std, "f32")
    if wl.carry:
        d["prev_B"] = unit((nseq, H, R, N), S_PREVB, K_NORMAL, 0.0, 2.0, dt_) if wl.prologue else \
            unit((nseq, H, R, N), S_PREVB, K_NORMAL_RMS, RMS_EPS, 0.0, dt_, row_len=N)
        d["prev_x"] = unit((nseq, H, R, P), S_PREVX, K_NORMAL, 0.0, 1.0, dt_)
    return d


def decode_inputs(wl: Workload, steps: int | None = None, first_step: int = 0) -> dict:
    """Per-step decode inputs for steps first_step .. first_step+steps.

    Layouts: x [T][b][H][R][P], B and C [T][b][G][R][N], dt and lam
    [T][b][H], theta [T][b][H][N/2]; initial state h0 [b][H][N/2][P][2]
    float32 and the previous-token carry prev_B [b][H][R][N], prev_x
    [b][H][R][P].  Step t is element range t*size.. of each stream, so any
    window of steps is drawn identically.
    """
    T = wl.seqlen if steps is None else steps
    b, H, P, N, R = wl.batch, wl.nheads, wl.headdim, wl.dstate, wl.rank
    G = wl.groups
    dt_ = wl.dtype
    s = wl.seed

    def step_fill(inner, stream, kind, p0, p1, row_len=0):
        n = int(np.prod(inner))  # this shard's elements per step
        if wl.shards == 1:
            return fill((T,) + inner, stream, kind, p0, p1, dt_, s, offset=first_step * n, row_len=row_len)
        # step t of the global problem is elements t*n*world.. of the stream; this shard's slice is
        # at rank*n inside it
        out = np.empty((T,) + inner, dtype=np.uint16 if dt_ == "bf16" else np.float32)
        for t in range(T):
            out[t] = fill(inner, stream, kind, p0, p1, dt_, s,
                          offset=((first_step + t) * wl.shards + wl.shard_index) * n, row_len=row_len)
        return out

    u0 = wl.shard_index * b * H  # first unit of this shard

    def unit(shape, stream, kind, p0, p1, dtype, row_len=0):
        per_unit = int(np.prod(shape[2:]))
        return fill(shape, stream, kind, p0, p1, dtype, s, offset=u0 * per_unit, row_len=row_len)

    d = {
        "x": step_fill((b, H, R, P), S_X, K_NORMAL, 0.0, 1.0),
        "B": step_fill((b, G, R, N), S_B, K_NORMAL, 0.0, 2.0) if wl.prologue else
        step_fill((b, G, R, N), S_B, K_NORMAL_RMS, RMS_EPS, 0.0, row_len=N),
        "C": step_fill((b, G, R, N), S_C, K_NORMAL, 0.0, 2.0) if wl.prologue else
        step_fill((b, G, R, N), S_C, K_NORMAL_RMS, RMS_EPS, 0.0, row_len=N),
        "dt": step_fill((b, H), S_DT, K_NORMAL, wl.dt_shift, 1.0) if wl.prologue else
        step_fill((b, H), S_DT, K_SOFTPLUS, wl.dt_shift, 0.0),
        "lam": step_fill((b, H), S_LAM, K_SIGMOID, 0.0, 0.0),
        "theta": step_fill((b, H, N // 2), S_THETA, K_UNIFORM, 0.0, np.pi),
        "A": fill((H,), S_A, K_NEG_EXP, 0.0, 0.5, "f32", s),
        "D": fill((H,), S_D, K_NORMAL, 0.0, 1.0, "f32", s),
    }
    if wl.real:
        d["theta"] = None
    if wl.euler:
        d["lam"] = None
    if wl.prologue:
        d["dt_bias"] = fill((H,), S_DTBIAS, K_NORMAL, 0.0, 0.5, "f32", s)
    if wl.h0_std > 0:
        d["h0"] = unit((b, H, N // 2, P, 2), S_H0, K_NORMAL, 0.0, wl.h0_std, "f32")
    else:
        d["h0"] = np.zeros((b, H, N // 2, P, 2), np.float32)
    if wl.carry:
        d["prev_B"] = unit((b, H, R, N), S_PREVB, K_NORMAL, 0.0, 2.0, dt_) if wl.prologue else \
            unit((b, H, R, N), S_PREVB, K_NORMAL_RMS, RMS_EPS, 0.0, dt_, row_len=N)
        d["prev_x"] = unit((b, H, R, P), S_PREVX, K_NORMAL, 0.0, 1.0, dt_)
    else:
        z = np.uint16 if dt_ == "bf16" else np.float32
        d["prev_B"] = np.zeros((b, H, R, N), z)
        d["prev_x"] = np.zeros((b, H, R, P), z)
    return d
