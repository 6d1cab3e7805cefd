"""The split schedule of the chunked prefill (few (sequence, head) units on
many SMs: each unit cut into segments; a state-only pass gives every
segment's own final state, a small kernel chains them, and the full pass
runs every segment from its exact initial state) against the oracle: y,
the final state and the carry, with and without an initial state, for
SISO, MIMO, grouped B/C, the real-state variant, strong decay, the fused
prologue and bf16 y.  The library's test hook confirms the schedule."""
import numpy as np
import pytest
import torch

import oracle
import state_space_sequence_06_b300 as m3
import synth
from gpu_util import TOL, assert_close, dev, prefill_gpu, state_for, to_np

pytestmark = pytest.mark.gpu

CASES = {
    "siso": dict(batch=1, seqlen=1000, nheads=2, dstate=128, rank=1, chunk=64),
    "siso_n64_one_group": dict(batch=2, seqlen=777, nheads=2, dstate=64, rank=1, chunk=64, ngroups=1),
    "mimo4": dict(batch=1, seqlen=1000, nheads=2, dstate=64, rank=4, chunk=16),
    "mimo2_n128": dict(batch=1, seqlen=640, nheads=3, dstate=128, rank=2, chunk=32),
    "mamba2_mode": dict(batch=1, seqlen=900, nheads=2, dstate=128, rank=1, chunk=64, real=True, euler=True),
    "strong_decay": dict(batch=1, seqlen=700, nheads=2, dstate=128, rank=1, chunk=64, dt_shift=1.5),
    "long_dt": dict(batch=1, seqlen=3000, nheads=1, dstate=128, rank=1, chunk=64, dt_shift=-3.0),
}


def _check(wl, inp, state, prologue=0, y_dtype=torch.float32):
    dims = (wl.batch, wl.nheads, wl.headdim, wl.dstate, wl.rank, m3.M3_BF16)
    st = state_for(dims, inp["h0"], inp["prev_B"], inp["prev_x"]) if state else state_for(dims)
    y = prefill_gpu(inp, wl, state=st, chunk=wl.chunk, prologue=prologue, y_dtype=y_dtype)
    info = m3.m3_test_last_launch()
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    assert info.kernel == m3.M3_TEST_KERNEL_CHUNKED_SPLIT, info.kernel
    src, dtype = inp, wl.dtype
    if prologue:
        src = oracle.apply_prologue(inp, wl.dtype, dt_softplus=True, bc_norm=True, dt_bias=inp["dt_bias"])
        dtype = "f64"
    kw = dict(h0=inp["h0"], prev_B=src["prev_B"], prev_x=src["prev_x"]) if state else {}
    yo, ho, pBo, pxo, _ = oracle.prefill(src, batch=wl.batch, L=wl.seqlen, H=wl.nheads, P=wl.headdim, N=wl.dstate,
                                         R=wl.rank, dtype=dtype, **kw)
    if y_dtype == torch.bfloat16:  # the f32 bound plus one bf16 rounding of each output
        gy = to_np(y)
        bound = TOL["bf16"] * np.sqrt(np.mean(yo ** 2)) + 2.0 ** -8 * np.abs(yo)
        assert (np.abs(gy - yo) <= bound).all(), float(np.max(np.abs(gy - yo) - bound))
    else:
        assert_close(to_np(y), yo, TOL["bf16"], "y")
    h, pB, px = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, TOL["bf16"], "h_final")
    # the carry is the last token's raw B and x
    last = {k: inp[k][:, -1] for k in ("B", "x")}
    G = inp["B"].shape[2]
    want_B = np.repeat(last["B"], wl.nheads // G, axis=1)
    assert np.array_equal(to_np(pB).reshape(want_B.shape), synth.to_f64(want_B, "bf16"))
    assert np.array_equal(to_np(px).reshape(last["x"].shape), synth.to_f64(last["x"], "bf16"))
    st.free()


@pytest.mark.parametrize("state", [True, False], ids=["state", "fresh"])
@pytest.mark.parametrize("case", list(CASES))
def test_split_schedule_matches_the_oracle(case, state):
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], h0_std=0.3 if state else 0.0, carry=state,
                      **CASES[case])
    _check(wl, synth.prefill_inputs(wl), state)


def test_split_schedule_with_the_fused_prologue_and_bf16_y():
    wl = synth.scaled(synth.workloads()["siso_prologue_b8_l4096"], batch=1, seqlen=1100, nheads=2, h0_std=0.3,
                      carry=True, ngroups=1)
    _check(wl, synth.prefill_inputs(wl), True, prologue=m3.M3_PRO_DT_SOFTPLUS | m3.M3_PRO_BC_NORM,
           y_dtype=torch.bfloat16)
