"""A bounded device wait that runs out: the library reports M3_ERR_TIMEOUT
and the device stays usable.

The failure is planted on the host side of a handover, through the
library's test hook (include/m3scan_testing.h): in a balanced-schedule
prefill, the CTAs that write handover slots leave them unpublished, so
each CTA that reads one waits for a flag that nothing sets.  The waits are
limited to 20 ms for this call; each then gives up, makes every role of
its CTA leave (the MMA threads first wait for their issued products, so
the TMEM is freed only when nothing writes it), and records M3_ERR_TIMEOUT
in the library's status word.  Nothing traps, no address is invalid and no
loop is endless.  A normal call afterwards on the same device must match
the oracle."""
import numpy as np
import pytest
import torch

import oracle
import state_space_sequence_06_b300 as m3
import synth
from gpu_util import TOL, assert_close, dev

pytestmark = pytest.mark.gpu

WAIT_NS = 20_000_000


def _inputs():
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    # more (sequence, head) units than SMs, two chunks each: the balanced schedule
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=nsm // 32 + 2, seqlen=128, nheads=32)
    inp = synth.prefill_inputs(wl)
    t = {k: dev(inp[k]) for k in ("x", "B", "C", "dt", "lam", "theta", "A", "D")}
    return wl, inp, t


def _call(t, y):
    m3.m3_scan_prefill(t["x"], t["B"], t["C"], t["dt"], t["lam"], t["theta"], t["A"], t["D"], y)


def test_handover_wait_runs_out_then_the_library_recovers():
    wl, inp, t = _inputs()
    y = torch.full(tuple(inp["x"].shape), float("nan"), dtype=torch.float32, device="cuda")
    assert m3.m3_device_status() == m3.M3_OK  # nothing pending from earlier tests
    m3.m3_test_set_fault(m3.M3_TEST_FAULT_SKIP_HANDOVER_RELEASE, WAIT_NS)
    try:
        _call(t, y)
        info = m3.m3_test_last_launch()
        status = m3.m3_device_status()  # synchronises the stream
    finally:
        m3.m3_test_set_fault(m3.M3_TEST_FAULT_NONE, 0)
    assert info.kernel == m3.M3_TEST_KERNEL_CHUNKED_BALANCED, "the shape must take the balanced schedule"
    assert status == m3.M3_ERR_TIMEOUT
    assert m3.m3_device_status() == m3.M3_OK  # read and cleared
    # the units whose handover never came are incomplete; the units no CTA cut completed
    yc = y.cpu().numpy()
    assert np.isnan(yc).any() and np.isfinite(yc).mean() > 0.3

    # the same device, a normal call: every output against the oracle
    y2 = torch.empty(tuple(inp["x"].shape), dtype=torch.float32, device="cuda")
    _call(t, y2)
    assert m3.m3_test_last_launch().kernel == m3.M3_TEST_KERNEL_CHUNKED_BALANCED
    assert m3.m3_device_status() == m3.M3_OK
    yo, _, _, _, _ = oracle.prefill(inp, batch=wl.batch, L=wl.seqlen, H=wl.nheads, P=wl.headdim, N=wl.dstate,
                                    R=wl.rank, dtype=wl.dtype)
    assert_close(y2.cpu().numpy(), yo, TOL["bf16"], "y after the timeout")
