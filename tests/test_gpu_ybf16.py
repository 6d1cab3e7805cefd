"""y written in bf16 (y_dtype = M3_BF16) through every kernel.

Each kernel computes y in f32 exactly as for an f32 output and rounds it
once, to nearest even, at the store.  So the bf16 output must equal the
f32 output of the same call rounded on the host, bit for bit, and the
state and carry must not change at all.  Against the oracle the bound is
the f32 bound plus one bf16 rounding, 2^-8 of |y| (bf16 keeps 8
significant bits).
"""
import numpy as np
import pytest
import torch

import oracle
import state_space_sequence_06_b300 as m3
import synth
from gpu_util import TOL, dev, prefill_gpu, state_for, to_np
from test_gpu_prefill import dims_of, oracle_kw

pytestmark = pytest.mark.gpu

ROUND = 2.0 ** -8


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy()


def _both(wl, algo=m3.M3_ALGO_AUTO, cu=None):
    """Run the prefill twice on the same inputs and initial state, y in f32
    then in bf16; returns the inputs, both outputs and both final states."""
    inp = synth.prefill_inputs(wl)
    out = []
    for yd in (torch.float32, torch.bfloat16):
        st = state_for(dims_of(wl, batch=wl.nseq if wl.kind == "varlen" else None), inp.get("h0"),
                       inp.get("prev_B"), inp.get("prev_x"))
        y = prefill_gpu(inp, wl, state=st, algo=algo, cu=cu, y_dtype=yd)
        assert m3.m3_device_status() == m3.M3_OK
        h, pB, px = (v.clone() for v in st.views())
        st.free()
        out.append((y, h, pB, px))
    return inp, out


def _check(wl, inp, out, cu=None, what=""):
    (y32, h32, pB32, px32), (y16, h16, pB16, px16) = out
    assert y16.dtype == torch.bfloat16
    assert np.array_equal(_bits(y16), _bits(y32.to(torch.bfloat16))), f"{what}: bf16 y is not the f32 y rounded"
    assert torch.equal(h16, h32) and torch.equal(pB16, pB32) and torch.equal(px16, px32), f"{what}: state"
    yo, _, _, _, _ = oracle.prefill(inp, **oracle_kw(wl), cu_seqlens=cu, h0=inp.get("h0"),
                                    prev_B=inp.get("prev_B"), prev_x=inp.get("prev_x"))
    rms = np.sqrt(np.mean(yo ** 2))
    err = np.max(np.abs(to_np(y16).reshape(yo.shape) - yo) - ROUND * np.abs(yo)) / rms
    assert err <= TOL[wl.dtype], f"{what}: max(|err| - 2^-8 |y|)/rms = {err:.3e}"


SHAPES = {
    "siso_n128": dict(dstate=128, rank=1, chunk=64),
    "mimo4": dict(dstate=64, rank=4, chunk=16),
    "mamba2": dict(dstate=128, rank=1, chunk=64, real=True, euler=True),
    "odd_shape": dict(dstate=48, rank=2, chunk=64, headdim=32),
}


@pytest.mark.parametrize("algo", [m3.M3_ALGO_AUTO, m3.M3_ALGO_RECURRENT])
@pytest.mark.parametrize("shape", list(SHAPES))
def test_prefill_y_bf16(shape, algo):
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=2, seqlen=201, nheads=4, h0_std=0.3, carry=True,
                      **SHAPES[shape])
    inp, out = _both(wl, algo)
    _check(wl, inp, out, what=f"{shape} algo {algo}")


def test_prefill_y_bf16_balanced_schedule():
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=5, seqlen=600, nheads=32, h0_std=0.3, carry=True,
                      dt_shift=-3.0)
    inp, out = _both(wl)
    _check(wl, inp, out, what="balanced")


def test_prefill_y_bf16_f32_inputs():
    wl = synth.scaled(synth.workloads()["tiny_f32"], seqlen=77, nheads=3, h0_std=0.3, carry=True)
    inp, out = _both(wl)
    _check(wl, inp, out, what="f32 inputs")


def test_prefill_y_bf16_varlen():
    wl = synth.scaled(synth.workloads()["varlen_16"], nseq=4, len_lo=10, len_hi=300, nheads=4)
    lens = synth.lengths(wl.nseq, wl.len_lo, wl.len_hi, seed=wl.seed)
    wl.cu_seqlens = synth.varlen_cu_seqlens(lens)
    wl.seqlen = int(wl.cu_seqlens[-1])
    inp, out = _both(wl, cu=wl.cu_seqlens)
    _check(wl, inp, out, cu=wl.cu_seqlens, what="varlen")


def test_full_size_y_bf16():
    """The bf16-output SISO line (batch 8, L 4096, 32 heads) in its launch
    configuration: bf16 y equals the f32 y rounded, everywhere."""
    wl = synth.workloads()["siso_ybf16_b8_l4096"]
    inp = synth.prefill_inputs(wl)
    y32 = prefill_gpu(inp, wl)
    y16 = prefill_gpu(inp, wl, y_dtype=torch.bfloat16)
    assert m3.m3_device_status() == m3.M3_OK
    assert np.array_equal(_bits(y16), _bits(y32.to(torch.bfloat16)))


@pytest.mark.parametrize("N,R,P", [(128, 1, 64), (64, 4, 64), (24, 3, 8)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_y_bf16(N, R, P, dtype):
    """Two states from the same start, stepped on the same tokens, one with
    y in f32 and one in bf16: every step's bf16 y is the f32 y rounded and
    the states stay identical."""
    wl = synth.Workload("t", "decode", 3, 0, 4, P, N, R, dtype, h0_std=0.1, carry=True)
    d = synth.decode_inputs(wl, steps=9)
    b, H = wl.batch, wl.nheads
    dims = (b, H, P, N, R, m3.M3_BF16 if dtype == "bf16" else m3.M3_F32)
    sts = [state_for(dims, d["h0"], d["prev_B"], d["prev_x"]) for _ in range(2)]
    t = {k: dev(d[k]) for k in ("x", "B", "C", "dt", "lam", "theta", "A", "D")}
    ys = [torch.empty((b, H, R, P), dtype=yd, device="cuda") for yd in (torch.float32, torch.bfloat16)]
    for i in range(9):
        for st, y in zip(sts, ys):
            m3.m3_decode_step(t["x"][i], t["B"][i], t["C"][i], t["dt"][i], t["lam"][i], t["theta"][i], t["A"],
                              t["D"], y, st)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(ys[1]), _bits(ys[0].to(torch.bfloat16))), f"step {i}"
    assert m3.m3_device_status() == m3.M3_OK
    for a, b_ in zip(sts[0].views(), sts[1].views()):
        assert torch.equal(a, b_)
    for st in sts:
        st.free()


def test_bad_y_dtype_is_rejected():
    """An unknown y_dtype code is M3_ERR_INVALID_ARG at the C ABI, before
    any launch; the binding refuses other torch dtypes itself."""
    import ctypes

    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=1, seqlen=64, nheads=2)
    inp = synth.prefill_inputs(wl)
    with pytest.raises(ValueError):
        prefill_gpu(inp, wl, y_dtype=torch.float16)
    t = {k: dev(inp[k]) for k in ("x", "B", "C", "dt", "lam", "theta", "A", "D")}
    y = torch.empty(t["x"].shape, dtype=torch.float32, device="cuda")
    a = m3.m3_prefill_args()
    a.dims = m3.make_dims(1, 2, 64, 128, 1, m3.M3_BF16)
    a.seqlen = 64
    a.x, a.B, a.C, a.dt, a.lam, a.theta = (t[k].data_ptr() for k in ("x", "B", "C", "dt", "lam", "theta"))
    a.A, a.D, a.y = t["A"].data_ptr(), t["D"].data_ptr(), y.data_ptr()
    a.y_dtype = 7
    rc = m3.load_library().m3_scan_prefill(ctypes.byref(a), None, torch.cuda.current_stream().cuda_stream)
    assert rc == m3.M3_ERR_INVALID_ARG
    a.y_dtype = m3.M3_F32
    rc = m3.load_library().m3_scan_prefill(ctypes.byref(a), None, torch.cuda.current_stream().cuda_stream)
    assert rc == m3.M3_OK
    torch.cuda.synchronize()
