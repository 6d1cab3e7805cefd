"""B and C shared by groups of heads, through every kernel: the chunked
tensor-core prefill (SISO, MIMO, the real-state variant, on one CTA per
unit and on the balanced schedule that cuts units between CTAs), the
token-serial prefill and the decode step, against the oracle run on the
same grouped inputs."""
import numpy as np
import pytest

import oracle
import state_space_sequence_06_b300 as m3
import synth
from gpu_util import TOL, assert_close, prefill_gpu, state_for, to_np
from test_gpu_decode import check, run_decode
from test_gpu_prefill import dims_of, oracle_kw

pytestmark = pytest.mark.gpu

SHAPES = {
    "siso_n128": dict(dstate=128, rank=1, chunk=64),
    "mimo4": dict(dstate=64, rank=4, chunk=16),
    "mamba2": dict(dstate=128, rank=1, chunk=64, real=True, euler=True),
    "odd_shape": dict(dstate=48, rank=2, chunk=64, headdim=32),
}


def _run(wl, algo=m3.M3_ALGO_AUTO, what=""):
    inp = synth.prefill_inputs(wl)
    assert inp["B"].shape[2] == wl.groups
    st = state_for(dims_of(wl), inp.get("h0"), inp.get("prev_B"), inp.get("prev_x"))
    y = prefill_gpu(inp, wl, state=st, algo=algo)
    assert m3.m3_device_status() == m3.M3_OK
    yo, ho, pBo, pxo, _ = oracle.prefill(inp, **oracle_kw(wl), h0=inp.get("h0"), prev_B=inp.get("prev_B"),
                                         prev_x=inp.get("prev_x"))
    tol = TOL[wl.dtype]
    assert_close(y.cpu().numpy(), yo, tol, f"{what} y")
    h, pB, px = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, tol, f"{what} h_final")
    assert np.array_equal(to_np(pB).reshape(pBo.shape), pBo), f"{what} carry B"
    assert np.array_equal(to_np(px).reshape(pxo.shape), pxo), f"{what} carry x"
    st.free()


@pytest.mark.parametrize("algo", [m3.M3_ALGO_AUTO, m3.M3_ALGO_RECURRENT])
@pytest.mark.parametrize("G", [1, 2])
@pytest.mark.parametrize("shape", list(SHAPES))
def test_prefill_grouped_small(shape, G, algo):
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=2, seqlen=201, nheads=4, h0_std=0.3, carry=True,
                      ngroups=G, **SHAPES[shape])
    _run(wl, algo, f"{shape} G{G}")


@pytest.mark.parametrize("G", [1, 4])
@pytest.mark.parametrize("shape", ["siso_n128", "mimo4", "mamba2"])
def test_balanced_schedule_grouped(shape, G):
    """More units than SMs (5 x 32 heads, L 600): units cut between CTAs,
    each part reading its group's B/C."""
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=5, seqlen=600, nheads=32, h0_std=0.3,
                      carry=True, dt_shift=-3.0, ngroups=G, **SHAPES[shape])
    _run(wl, what=f"balanced {shape} G{G}")


def test_prefill_grouped_f32():
    wl = synth.scaled(synth.workloads()["tiny_f32"], seqlen=77, nheads=4, h0_std=0.3, carry=True, ngroups=2)
    _run(wl, what="f32 G2")


def test_grouped_varlen():
    wl = synth.scaled(synth.workloads()["varlen_16"], nseq=5, len_lo=10, len_hi=300, nheads=4, ngroups=2)
    lens = synth.lengths(wl.nseq, wl.len_lo, wl.len_hi, seed=wl.seed)
    wl.cu_seqlens = synth.varlen_cu_seqlens(lens)
    wl.seqlen = int(wl.cu_seqlens[-1])
    inp = synth.prefill_inputs(wl)
    y = prefill_gpu(inp, wl, cu=wl.cu_seqlens)
    yo, _, _, _, _ = oracle.prefill(inp, **oracle_kw(wl), cu_seqlens=wl.cu_seqlens)
    assert_close(y.cpu().numpy(), yo, TOL["bf16"], "varlen G2 y")


def test_groups_must_divide_heads():
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=1, seqlen=64, nheads=4, ngroups=3)
    with pytest.raises(m3.M3Error) as e:
        prefill_gpu(synth.prefill_inputs(wl), wl)
    assert e.value.status == m3.M3_ERR_INVALID_ARG


def test_full_size_grouped_every_output():
    """The grouped SISO benchmark line (batch 8, L 4096, 32 heads sharing
    one B/C) in its launch configuration: every output and final state."""
    wl = synth.workloads()["siso_g1_b8_l4096"]
    inp = synth.prefill_inputs(wl)
    st = state_for(dims_of(wl))
    y = prefill_gpu(inp, wl, state=st)
    assert m3.m3_device_status() == m3.M3_OK
    yo, ho, _, _, _ = oracle.prefill(inp, **oracle_kw(wl))
    assert_close(y.cpu().numpy(), yo, TOL["bf16"], "siso G1 y")
    h, _, _ = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, TOL["bf16"], "siso G1 h_final")
    st.free()


@pytest.mark.parametrize("N,R,P,G", [(128, 1, 64, 1), (64, 4, 64, 2), (24, 3, 8, 1)])
def test_decode_grouped(N, R, P, G):
    wl = synth.Workload("t", "decode", 3, 0, 4, P, N, R, "bf16", h0_std=0.1, carry=True, ngroups=G)
    gpu, ref = run_decode(wl, 29)
    check(gpu, ref, "bf16", f"decode G{G} N{N} R{R} P{P}")


def test_decode_full_size_grouped_sampled():
    wl = synth.workloads()["decode_siso_g1_b256"]
    rng = np.random.default_rng(1)
    units = sorted(set([0, wl.batch * wl.nheads - 1] + list(rng.choice(wl.batch * wl.nheads, 10, replace=False))))
    gpu, ref = run_decode(wl, wl.seqlen, units=units, window=128)
    check(gpu, ref, wl.dtype, wl.name)
