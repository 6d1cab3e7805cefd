"""The backward pass (m3_scan_prefill_backward) against the oracle's exact
adjoint: every gradient (x, B, C, dt, lam, theta, A, D, the initial state
and the carry) for a random dL/dy and dL/dh_final, with an initial state
and carry, grouped B/C, SISO and MIMO, f32 and bf16 inputs and the
theta = 0 / lam = 1 special case.  The arithmetic is f32 on inputs both
sides read identically, so the bound is the same max|err| / rms(reference)
as the forward's."""
import numpy as np
import pytest
import torch

import oracle
import state_space_sequence_06_b300 as m3
import synth
from gpu_util import TOL, assert_close, dev

pytestmark = pytest.mark.gpu

CASES = {
    "siso_f32_grouped": dict(batch=2, seqlen=37, nheads=4, headdim=8, dstate=16, rank=1, dtype="f32", ngroups=2),
    "mimo2_f32": dict(batch=2, seqlen=29, nheads=3, headdim=4, dstate=8, rank=2, dtype="f32"),
    "siso_bf16_one_group": dict(batch=1, seqlen=50, nheads=4, headdim=16, dstate=32, rank=1, dtype="bf16",
                                ngroups=1),
    "mamba2_mode_f32": dict(batch=2, seqlen=33, nheads=2, headdim=8, dstate=16, rank=1, dtype="f32", real=True,
                            euler=True),
}
PAIRS = [("dx", "x"), ("dB", "B"), ("dC", "C"), ("ddt", "dt"), ("dlam", "lam"), ("dtheta", "theta"),
         ("dA", "A"), ("dD", "D"), ("dh0", "h0"), ("dprev_B", "prev_B"), ("dprev_x", "prev_x")]


@pytest.mark.parametrize("case", list(CASES))
def test_backward_matches_the_adjoint_oracle(case):
    wl = synth.Workload("t", "prefill", h0_std=0.3, carry=True, **CASES[case])
    inp = synth.prefill_inputs(wl)
    b, L, H, P, N, R = wl.batch, wl.seqlen, wl.nheads, wl.headdim, wl.dstate, wl.rank
    rng = np.random.default_rng(len(case))
    dy = rng.normal(size=(b, L, H, R, P)).astype(np.float32)
    dhf = rng.normal(size=(b, H, N // 2, P, 2)).astype(np.float32)
    t = {k: dev(inp[k]) for k in ("x", "B", "C", "dt", "lam", "theta", "A", "D", "h0", "prev_B", "prev_x")}
    out = m3.m3_scan_prefill_backward(t["x"], t["B"], t["C"], t["dt"], t["lam"], t["theta"], t["A"], t["D"],
                                      dev(dy), h0=t["h0"], prev_B=t["prev_B"], prev_x=t["prev_x"],
                                      dh_final=dev(dhf))
    torch.cuda.synchronize()
    _, _, ref = oracle.prefill_backward(inp, dy, batch=b, L=L, H=H, P=P, N=N, R=R, dtype=wl.dtype,
                                        h0=inp["h0"], prev_B=inp["prev_B"], prev_x=inp["prev_x"], dh_final=dhf)
    for gk, rk in PAIRS:
        got = out[gk].cpu().numpy().astype(np.float64).reshape(np.shape(ref[rk]))
        assert_close(got, ref[rk], TOL[wl.dtype], f"{case} {gk}")


def test_backward_rejects_bad_arguments():
    wl = synth.Workload("t", "prefill", 1, 8, 4, 8, 16, 1, "f32", ngroups=3)
    inp = synth.prefill_inputs(synth.scaled(wl, ngroups=0))
    t = {k: dev(inp[k]) for k in ("x", "B", "C", "dt", "lam", "theta", "A", "D")}
    dy = torch.zeros(t["x"].shape, dtype=torch.float32, device="cuda")
    bad_B = torch.zeros((1, 8, 3, 1, 16), dtype=torch.float32, device="cuda")  # 3 groups do not divide 4 heads
    with pytest.raises(m3.M3Error) as e:
        m3.m3_scan_prefill_backward(t["x"], bad_B, bad_B, t["dt"], t["lam"], t["theta"], t["A"], t["D"], dy)
    assert e.value.status == m3.M3_ERR_INVALID_ARG


# ---- the chunked kernel (every chunk of every unit in parallel, f32)

CHUNKED = {
    "siso_n128_ragged": dict(batch=2, seqlen=200, nheads=3, headdim=64, dstate=128, rank=1, dtype="bf16"),
    "siso_n64_grouped_f32": dict(batch=1, seqlen=150, nheads=4, headdim=64, dstate=64, rank=1, dtype="f32",
                                 ngroups=2),
    "mimo4": dict(batch=2, seqlen=100, nheads=2, headdim=64, dstate=64, rank=4, dtype="bf16"),
    "mimo2_n128_one_group": dict(batch=1, seqlen=77, nheads=2, headdim=64, dstate=128, rank=2, dtype="bf16",
                                 ngroups=1),
    "mamba2_mode": dict(batch=1, seqlen=130, nheads=2, headdim=64, dstate=128, rank=1, dtype="bf16", real=True,
                        euler=True),
    "strong_decay": dict(batch=1, seqlen=160, nheads=2, headdim=64, dstate=128, rank=1, dtype="bf16", dt_shift=1.5),
    "one_token": dict(batch=2, seqlen=1, nheads=2, headdim=64, dstate=64, rank=4, dtype="bf16"),
}
# f32 arithmetic on both sides of the same rounded inputs
CHUNKED_TOL = 1e-3


def _backward_case(cfg, seed, state=True, **kw):
    wl = synth.Workload("t", "prefill", h0_std=0.3 if state else 0.0, carry=state, **cfg)
    inp = synth.prefill_inputs(wl)
    b, L, H, P, N, R = wl.batch, wl.seqlen, wl.nheads, wl.headdim, wl.dstate, wl.rank
    rng = np.random.default_rng(seed)
    dy = rng.normal(size=(b, L, H, R, P)).astype(np.float32)
    dhf = rng.normal(size=(b, H, N // 2, P, 2)).astype(np.float32)
    keys = ("x", "B", "C", "dt", "lam", "theta", "A", "D") + (("h0", "prev_B", "prev_x") if state else ())
    t = {k: dev(inp[k]) for k in keys}
    for k in ("h0", "prev_B", "prev_x"):
        t.setdefault(k, None)
    return wl, inp, t, dy, dhf


def _run(t, dy, dhf, **kw):
    out = m3.m3_scan_prefill_backward(t["x"], t["B"], t["C"], t["dt"], t["lam"], t["theta"], t["A"], t["D"],
                                      dev(dy), h0=t["h0"], prev_B=t["prev_B"], prev_x=t["prev_x"],
                                      dh_final=dev(dhf), **kw)
    torch.cuda.synchronize()
    return out


def _oracle(wl, inp, dy, dhf, state=True, **kw):
    return oracle.prefill_backward(inp, dy, batch=wl.batch, L=wl.seqlen, H=wl.nheads, P=wl.headdim, N=wl.dstate,
                                   R=wl.rank, dtype=wl.dtype, h0=inp["h0"] if state else None,
                                   prev_B=inp["prev_B"] if state else None,
                                   prev_x=inp["prev_x"] if state else None, dh_final=dhf, **kw)[2]


@pytest.mark.parametrize("case", list(CHUNKED))
def test_chunked_backward_matches_the_adjoint_oracle(case):
    wl, inp, t, dy, dhf = _backward_case(CHUNKED[case], len(case))
    out = _run(t, dy, dhf, algo=m3.M3_ALGO_CHUNKED)
    ref = _oracle(wl, inp, dy, dhf)
    for gk, rk in PAIRS:
        got = out[gk].cpu().numpy().astype(np.float64).reshape(np.shape(ref[rk]))
        assert_close(got, ref[rk], CHUNKED_TOL, f"{case} {gk}")


@pytest.mark.parametrize("shape", [dict(dstate=128, rank=1), dict(dstate=64, rank=4)], ids=["siso_n128", "mimo4"])
def test_chunked_backward_long_sequence_every_gradient(shape):
    """N 128 / P 64 SISO and N 64 MIMO rank 4 over 1024 tokens (16 and 64
    chunks chained through the state and adjoint), every gradient."""
    cfg = dict(batch=1, seqlen=1024, nheads=2, headdim=64, dtype="bf16", dt_shift=-3.0, **shape)
    wl, inp, t, dy, dhf = _backward_case(cfg, 3)
    out = _run(t, dy, dhf, algo=m3.M3_ALGO_CHUNKED)
    ref = _oracle(wl, inp, dy, dhf)
    for gk, rk in PAIRS:
        got = out[gk].cpu().numpy().astype(np.float64).reshape(np.shape(ref[rk]))
        assert_close(got, ref[rk], CHUNKED_TOL, f"long {gk}")


def test_chunked_and_token_serial_kernels_agree_and_chunked_is_deterministic():
    cfg = dict(batch=2, seqlen=300, nheads=4, headdim=64, dstate=128, rank=1, dtype="bf16", ngroups=2)
    wl, inp, t, dy, dhf = _backward_case(cfg, 5)
    a = _run(t, dy, dhf, algo=m3.M3_ALGO_CHUNKED)
    a2 = _run(t, dy, dhf, algo=m3.M3_ALGO_CHUNKED)
    s = _run(t, dy, dhf, algo=m3.M3_ALGO_RECURRENT)
    for gk, _ in PAIRS:
        assert torch.equal(a[gk], a2[gk]), f"{gk} differs between two identical calls"
        assert_close(a[gk].cpu().numpy(), s[gk].cpu().numpy().astype(np.float64), CHUNKED_TOL, f"chunked vs serial {gk}")


@pytest.mark.parametrize("algo", [m3.M3_ALGO_CHUNKED, m3.M3_ALGO_RECURRENT], ids=["chunked", "serial"])
def test_backward_through_the_fused_prologue(algo):
    """Raw inputs with the prologue flags (softplus of dt + dt_bias, RMS norm
    of B, C and the carried B): gradients with respect to the raw inputs and
    dt_bias against the oracle's chained adjoint."""
    cfg = dict(batch=1, seqlen=130, nheads=4, headdim=64, dstate=128, rank=1, dtype="bf16", ngroups=2,
               prologue=True)
    wl, inp, t, dy, dhf = _backward_case(cfg, 7)
    bias = dev(inp["dt_bias"])
    pro = m3.M3_PRO_DT_SOFTPLUS | m3.M3_PRO_BC_NORM
    out = _run(t, dy, dhf, algo=algo, prologue=pro, dt_bias=bias)
    ref = _oracle(wl, inp, dy, dhf, dt_softplus=True, bc_norm=True, dt_bias=inp["dt_bias"])
    for gk, rk in PAIRS + [("ddt_bias", "dt_bias")]:
        got = out[gk].cpu().numpy().astype(np.float64).reshape(np.shape(ref[rk]))
        assert_close(got, ref[rk], CHUNKED_TOL, f"prologue {gk}")


def test_chunked_backward_refuses_shapes_it_has_no_kernel_for():
    cfg = dict(batch=1, seqlen=20, nheads=2, headdim=32, dstate=16, rank=1, dtype="f32")
    wl, inp, t, dy, dhf = _backward_case(cfg, 1)
    with pytest.raises(m3.M3Error) as e:
        _run(t, dy, dhf, algo=m3.M3_ALGO_CHUNKED)
    assert e.value.status == m3.M3_ERR_UNSUPPORTED
    out = _run(t, dy, dhf)  # AUTO: the token-serial kernel
    ref = _oracle(wl, inp, dy, dhf)
    assert_close(out["dx"].cpu().numpy(), ref["x"], TOL["f32"], "auto dx")
