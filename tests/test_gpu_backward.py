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
