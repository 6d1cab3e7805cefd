"""The Mamba-2 special case through the same entry points: theta = 0 (a
real state, passed as NULL) and lam = 1 (first-order exponential Euler,
passed as NULL), each alone and together, for the chunked kernel (its
real-state variant), the token-serial kernel and the decode step, against
the oracle fed theta = 0 and lam = 1."""
import numpy as np
import pytest

import oracle
import state_space_sequence_06_b300 as m3
import synth
from gpu_util import TOL, assert_close, prefill_gpu, state_for, to_np
from test_gpu_decode import check, run_decode
from test_gpu_prefill import dims_of, oracle_kw

pytestmark = pytest.mark.gpu

MODES = {"real+euler": dict(real=True, euler=True), "real": dict(real=True), "euler": dict(euler=True)}
SHAPES = {
    "siso_n128": dict(batch=2, seqlen=333, nheads=3, headdim=64, dstate=128, rank=1, chunk=64),
    "siso_n64": dict(batch=2, seqlen=200, nheads=2, headdim=64, dstate=64, rank=1, chunk=64),
    "mimo4": dict(batch=2, seqlen=201, nheads=3, headdim=64, dstate=64, rank=4, chunk=16),
    "odd_shape": dict(batch=2, seqlen=45, nheads=2, headdim=32, dstate=48, rank=2, chunk=64),
}


@pytest.mark.parametrize("algo", [m3.M3_ALGO_AUTO, m3.M3_ALGO_RECURRENT])
@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("mode", list(MODES))
def test_prefill_special_cases(mode, shape, algo):
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], h0_std=0.3, carry=True, **SHAPES[shape],
                      **MODES[mode])
    inp = synth.prefill_inputs(wl)
    st = state_for(dims_of(wl), inp["h0"], inp["prev_B"], inp["prev_x"])
    y = prefill_gpu(inp, wl, state=st, algo=algo)
    yo, ho, pBo, pxo, _ = oracle.prefill(inp, **oracle_kw(wl), h0=inp["h0"], prev_B=inp["prev_B"],
                                         prev_x=inp["prev_x"])
    assert_close(y.cpu().numpy(), yo, TOL["bf16"], f"{mode} {shape} y")
    h, pB, px = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, TOL["bf16"], f"{mode} {shape} h_final")
    assert np.array_equal(to_np(pB).reshape(pBo.shape), pBo)
    assert np.array_equal(to_np(px).reshape(pxo.shape), pxo)
    st.free()


def test_real_state_chunked_variant_is_selected():
    """theta = NULL with a supported shape runs the chunked kernel (the
    explicit CHUNKED request succeeds); an unsupported one reports so."""
    wl = synth.scaled(synth.workloads()["mamba2_b8_l4096"], batch=1, seqlen=130, nheads=2)
    inp = synth.prefill_inputs(wl)
    y = prefill_gpu(inp, wl, algo=m3.M3_ALGO_CHUNKED)
    yo, _, _, _, _ = oracle.prefill(inp, **oracle_kw(wl))
    assert_close(y.cpu().numpy(), yo, TOL["bf16"], "chunked real-state y")
    wl2 = synth.scaled(wl, headdim=32)
    with pytest.raises(m3.M3Error) as e:
        prefill_gpu(synth.prefill_inputs(wl2), wl2, algo=m3.M3_ALGO_CHUNKED)
    assert e.value.status == m3.M3_ERR_UNSUPPORTED


def test_full_size_mamba2_every_output():
    """The benchmark's Mamba-2 line (batch 8, L 4096, 32 heads, N 128, real
    state, lam = 1) in its launch configuration: every output and final
    state against the oracle."""
    wl = synth.workloads()["mamba2_b8_l4096"]
    inp = synth.prefill_inputs(wl)
    st = state_for(dims_of(wl))
    y = prefill_gpu(inp, wl, state=st)
    assert m3.m3_device_status() == m3.M3_OK
    yo, ho, _, _, _ = oracle.prefill(inp, **oracle_kw(wl))
    assert_close(y.cpu().numpy(), yo, TOL["bf16"], "mamba2 y")
    h, _, _ = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, TOL["bf16"], "mamba2 h_final")
    st.free()


@pytest.mark.parametrize("N,R,P", [(128, 1, 64), (64, 4, 64), (24, 3, 8)])
@pytest.mark.parametrize("mode", list(MODES))
def test_decode_special_cases(mode, N, R, P):
    wl = synth.Workload("t", "decode", 3, 0, 4, P, N, R, "bf16", h0_std=0.1, carry=True, **MODES[mode])
    gpu, ref = run_decode(wl, 29)
    check(gpu, ref, "bf16", f"decode {mode} N{N} R{R} P{P}")
