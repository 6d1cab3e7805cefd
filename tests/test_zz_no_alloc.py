"""m3_scan_prefill_noalloc (fixed scratch in the library, no allocation in
the call) against m3_scan_prefill: the same outputs, final state and carry,
bit for bit, over two chained calls in a row, on a batch that has more
(sequence, head) units than the GPU has SMs (the schedule that uses
scratch, checked through the library's test hook).  The noalloc call maps
no device memory (the free memory the driver reports does not change).
Self-contained: it passes alone and after the other tests."""
import numpy as np
import pytest
import torch

import state_space_sequence_06_b300 as m3
import synth
from gpu_util import dev, state_for, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [dict(dstate=128, rank=1, chunk=64), dict(dstate=64, rank=4, chunk=16)],
                         ids=["siso", "mimo4"])
def test_noalloc_matches_prefill_over_two_calls(shape):
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    batch = nsm // 32 + 2  # 32 heads: more units than SMs
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=batch, seqlen=700, nheads=32, h0_std=0.3,
                      carry=True, dt_shift=-3.0, **shape)
    inp = synth.prefill_inputs(wl)
    dims = (wl.batch, wl.nheads, wl.headdim, wl.dstate, wl.rank, m3.M3_BF16)
    t = {k: dev(inp[k]) for k in ("x", "B", "C", "dt", "lam", "theta", "A", "D")}
    results = []
    for fn in (m3.m3_scan_prefill, m3.m3_scan_prefill_noalloc):
        st = state_for(dims, inp["h0"], inp["prev_B"], inp["prev_x"])
        ybuf = [torch.empty(tuple(inp["x"].shape), dtype=torch.float32, device="cuda") for _ in range(2)]
        torch.cuda.synchronize()
        ys = []
        for i in range(2):  # the second call continues from the first's state and carry
            free0 = torch.cuda.mem_get_info()[0]
            fn(t["x"], t["B"], t["C"], t["dt"], t["lam"], t["theta"], t["A"], t["D"], ybuf[i], state=st)
            info = m3.m3_test_last_launch()
            torch.cuda.synchronize()
            # the shape really takes the schedule that uses scratch
            assert info.kernel == m3.M3_TEST_KERNEL_CHUNKED_BALANCED and info.scratch_bytes > 0
            if fn is m3.m3_scan_prefill_noalloc and i == 1:
                # no device memory was mapped by the call (the first call on a
                # device may load the library's module, so the second is checked)
                assert torch.cuda.mem_get_info()[0] == free0
            ys.append(ybuf[i].cpu().numpy())
        assert m3.m3_device_status() == m3.M3_OK
        h, pB, px = st.views()
        results.append((ys, to_np(h), to_np(pB), to_np(px)))
        st.free()
    (ya, ha, pBa, pxa), (yb, hb, pBb, pxb) = results
    for i in range(2):
        assert np.array_equal(ya[i], yb[i]), f"y of call {i + 1}"
    assert np.array_equal(ha, hb) and np.array_equal(pBa, pBb) and np.array_equal(pxa, pxb)
    assert np.isfinite(ya[1]).all() and np.abs(ya[1]).max() > 0
