"""The fused prologue through every kernel: dt through softplus with a
per-head bias, and the RMS norm of B and C rows (and of the carried B),
against the oracle run on the inputs its own prologue produced.  The
inputs are raw (dt the pre-activation, B and C rows of RMS about 2), so
a kernel that skipped either step would miss by far more than the bound.
The carry must still hold the raw last B and x."""
import numpy as np
import pytest
import torch

import oracle
import state_space_sequence_06_b300 as m3
import synth
from gpu_util import TOL, assert_close, dev, prefill_gpu, state_for, to_np, widen
from test_gpu_prefill import dims_of

pytestmark = pytest.mark.gpu

SP, NORM = m3.M3_PRO_DT_SOFTPLUS, m3.M3_PRO_BC_NORM
MODES = {"softplus": SP, "norm": NORM, "both": SP | NORM}
SHAPES = {
    "siso_n128": dict(dstate=128, rank=1, chunk=64),
    "siso_n64": dict(dstate=64, rank=1, chunk=64),
    "mimo4": dict(dstate=64, rank=4, chunk=16),
    "mimo2_n128": dict(dstate=128, rank=2, chunk=32),
    "mamba2": dict(dstate=128, rank=1, chunk=64, real=True, euler=True),
    "odd_shape": dict(dstate=48, rank=2, chunk=64, headdim=32),
}


def _oracle_prefill(inp, wl, mode, cu=None):
    p = oracle.apply_prologue(inp, wl.dtype, dt_softplus=bool(mode & SP), bc_norm=bool(mode & NORM),
                              dt_bias=inp.get("dt_bias"))
    return oracle.prefill(p, batch=wl.batch, L=wl.seqlen, H=wl.nheads, P=wl.headdim, N=wl.dstate, R=wl.rank,
                          dtype="f64", cu_seqlens=cu, h0=p.get("h0"), prev_B=p.get("prev_B"), prev_x=p.get("prev_x"))


def _last_raw(inp, wl):
    """The raw carry a fixed-length prefill must leave: each unit's last B
    (its group's row) and x."""
    b, L, H, G = wl.batch, wl.seqlen, wl.nheads, wl.groups
    lastB = inp["B"][:, L - 1][:, np.arange(H) // (H // G)]  # [b][H][R][N]
    return lastB, inp["x"][:, L - 1]


def _inputs(wl, mode):
    """Raw inputs; without the softplus step dt must already be a step size
    (positive), so it is the plain workload's dt (the same draws through
    the generator's softplus)."""
    inp = synth.prefill_inputs(wl)
    if not mode & SP:
        inp["dt"] = synth.prefill_inputs(synth.scaled(wl, prologue=False))["dt"]
    return inp


def _run(wl, mode, algo=m3.M3_ALGO_AUTO, what=""):
    inp = _inputs(wl, mode)
    st = state_for(dims_of(wl), inp.get("h0"), inp.get("prev_B"), inp.get("prev_x"))
    y = prefill_gpu(inp, wl, state=st, algo=algo, prologue=mode)
    assert m3.m3_device_status() == m3.M3_OK
    yo, ho, _, _, _ = _oracle_prefill(inp, wl, mode)
    tol = TOL[wl.dtype]
    assert_close(y.cpu().numpy(), yo, tol, f"{what} y")
    h, pB, px = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, tol, f"{what} h_final")
    lastB, lastx = _last_raw(inp, wl)
    assert np.array_equal(to_np(pB).reshape(lastB.shape), widen(lastB)), f"{what} carry B (raw)"
    assert np.array_equal(to_np(px).reshape(lastx.shape), widen(lastx)), f"{what} carry x (raw)"
    st.free()


@pytest.mark.parametrize("algo", [m3.M3_ALGO_AUTO, m3.M3_ALGO_RECURRENT])
@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("shape", list(SHAPES))
def test_prefill_prologue(shape, mode, algo):
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=2, seqlen=201, nheads=4, h0_std=0.3, carry=True,
                      prologue=True, ngroups=2, **SHAPES[shape])
    _run(wl, MODES[mode], algo, f"{shape} {mode} algo {algo}")


@pytest.mark.parametrize("shape", ["siso_n128", "mimo4"])
def test_balanced_schedule_prologue(shape):
    """Units cut between CTAs: the second part starts from a handed-over raw
    carry, normalised and through softplus like any other."""
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=5, seqlen=600, nheads=32, h0_std=0.3, carry=True,
                      prologue=True, **SHAPES[shape])
    _run(wl, SP | NORM, what=f"balanced {shape}")


def test_prologue_f32_inputs():
    wl = synth.scaled(synth.workloads()["tiny_f32"], seqlen=77, nheads=3, h0_std=0.3, carry=True, prologue=True)
    _run(wl, SP | NORM, what="f32")


def test_prologue_varlen():
    wl = synth.scaled(synth.workloads()["varlen_16"], nseq=5, len_lo=10, len_hi=300, nheads=4, prologue=True)
    lens = synth.lengths(wl.nseq, wl.len_lo, wl.len_hi, seed=wl.seed)
    wl.cu_seqlens = synth.varlen_cu_seqlens(lens)
    wl.seqlen = int(wl.cu_seqlens[-1])
    inp = synth.prefill_inputs(wl)
    y = prefill_gpu(inp, wl, cu=wl.cu_seqlens, prologue=SP | NORM)
    yo, _, _, _, _ = _oracle_prefill(inp, wl, SP | NORM, cu=wl.cu_seqlens)
    assert_close(y.cpu().numpy(), yo, TOL["bf16"], "varlen y")


def test_real_state_with_norm_is_token_serial():
    """The real-state chunked variant has no BC norm: CHUNKED reports it,
    AUTO runs the token-serial kernel."""
    wl = synth.scaled(synth.workloads()["mamba2_b8_l4096"], batch=1, seqlen=130, nheads=2, prologue=True)
    inp = synth.prefill_inputs(wl)
    with pytest.raises(m3.M3Error) as e:
        prefill_gpu(inp, wl, algo=m3.M3_ALGO_CHUNKED, prologue=NORM)
    assert e.value.status == m3.M3_ERR_UNSUPPORTED
    y = prefill_gpu(inp, wl, algo=m3.M3_ALGO_CHUNKED, prologue=SP)  # softplus alone is fine there
    yo, _, _, _, _ = _oracle_prefill(inp, wl, SP)
    assert_close(y.cpu().numpy(), yo, TOL["bf16"], "real-state softplus y")


def test_unknown_prologue_bits_are_rejected():
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=1, seqlen=64, nheads=2, prologue=True)
    with pytest.raises(m3.M3Error) as e:
        prefill_gpu(synth.prefill_inputs(wl), wl, prologue=8)
    assert e.value.status == m3.M3_ERR_INVALID_ARG


def test_full_size_prologue_every_output():
    """The prologue SISO line (batch 8, L 4096, 32 heads, raw dt, B and C)
    in its launch configuration: every output and final state."""
    wl = synth.workloads()["siso_prologue_b8_l4096"]
    inp = synth.prefill_inputs(wl)
    st = state_for(dims_of(wl))
    y = prefill_gpu(inp, wl, state=st, prologue=SP | NORM)
    assert m3.m3_device_status() == m3.M3_OK
    yo, ho, _, _, _ = _oracle_prefill(inp, wl, SP | NORM)
    assert_close(y.cpu().numpy(), yo, TOL["bf16"], "prologue y")
    h, _, _ = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, TOL["bf16"], "prologue h_final")
    st.free()


@pytest.mark.parametrize("N,R,P,G", [(128, 1, 64, 2), (64, 4, 64, 1), (24, 3, 8, 4)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_prologue(N, R, P, G, dtype):
    """Decode steps with both prologue steps from a raw carry: every step's
    y, the final state, and the raw carry of the last step."""
    T = 11
    wl = synth.Workload("t", "decode", 3, 0, 4, P, N, R, dtype, h0_std=0.1, carry=True, prologue=True, ngroups=G)
    d = synth.decode_inputs(wl, steps=T)
    b, H = wl.batch, wl.nheads
    st = state_for((b, H, P, N, R, m3.M3_BF16 if dtype == "bf16" else m3.M3_F32), d["h0"], d["prev_B"], d["prev_x"])
    t = {k: dev(d[k]) for k in ("x", "B", "C", "dt", "lam", "theta", "A", "D", "dt_bias")}
    y = torch.empty((b, H, R, P), dtype=torch.float32, device="cuda")
    ys = []
    for i in range(T):
        m3.m3_decode_step(t["x"][i], t["B"][i], t["C"][i], t["dt"][i], t["lam"][i], t["theta"][i], t["A"], t["D"],
                          y, st, prologue=SP | NORM, dt_bias=t["dt_bias"])
        ys.append(y.cpu().numpy().copy())
    assert m3.m3_device_status() == m3.M3_OK
    p = oracle.apply_prologue(d, dtype, dt_softplus=True, bc_norm=True, dt_bias=d["dt_bias"])
    yo, ho, _, _ = oracle.decode(p, batch=b, H=H, P=P, N=N, R=R, dtype="f64", steps=T)
    tol = TOL[dtype]
    assert_close(np.stack(ys), yo, tol, "decode y")
    h, pB, px = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, tol, "decode h_final")
    lastB = d["B"][T - 1][:, np.arange(H) // (H // G)]
    assert np.array_equal(to_np(pB).reshape(lastB.shape), widen(lastB))
    assert np.array_equal(to_np(px).reshape(d["x"][T - 1].shape), widen(d["x"][T - 1]))
    st.free()
