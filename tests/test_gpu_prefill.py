"""GPU parity of m3_scan_prefill against the oracle (element by element),
for every prefill kernel, at small sizes with ragged chunks, with initial
states and carries, packed variable-length batches, and at full size on
sampled units."""
import numpy as np
import pytest
import torch

import oracle
import state_space_sequence_06_b300 as m3
import synth
from gpu_util import TOL, assert_close, dev, prefill_gpu, state_for, to_np

pytestmark = pytest.mark.gpu

ALGOS = [m3.M3_ALGO_RECURRENT, m3.M3_ALGO_AUTO]


def dims_of(wl, batch=None):
    return (batch or wl.batch, wl.nheads, wl.headdim, wl.dstate, wl.rank,
            m3.M3_BF16 if wl.dtype == "bf16" else m3.M3_F32)


def oracle_kw(wl, L=None):
    return dict(batch=wl.batch, L=L if L is not None else wl.seqlen, H=wl.nheads, P=wl.headdim,
                N=wl.dstate, R=wl.rank, dtype=wl.dtype)


def test_tiny_f32_config():
    """The tiny all-f32 workload (batch 1, L 64, 2 heads, P 16, N 16) at 1e-4."""
    wl = synth.workloads()["tiny_f32"]
    inp = synth.prefill_inputs(wl)
    st = state_for(dims_of(wl))
    y = prefill_gpu(inp, wl, state=st)
    yo, ho, pBo, pxo, _ = oracle.prefill(inp, **oracle_kw(wl))
    assert_close(y.cpu().numpy(), yo, TOL["f32"], "tiny y")
    h, pB, px = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, TOL["f32"], "tiny h_final")
    assert np.array_equal(to_np(pB).reshape(pBo.shape), pBo)
    assert np.array_equal(to_np(px).reshape(pxo.shape), pxo)
    st.free()


SMALL = {
    "siso": dict(batch=2, seqlen=333, nheads=3, headdim=64, dstate=128, rank=1, chunk=64),
    "mimo4": dict(batch=2, seqlen=201, nheads=3, headdim=64, dstate=64, rank=4, chunk=16),
    "siso_long_dt": dict(batch=1, seqlen=517, nheads=2, headdim=64, dstate=128, rank=1, chunk=64, dt_shift=-3.0),
    "odd_shape": dict(batch=2, seqlen=45, nheads=2, headdim=32, dstate=48, rank=2, chunk=64),
    # large dt: chunks whose summed log-decay falls below -60, where the
    # chunked kernel takes its per-element decay path (see the coverage test)
    "siso_strong_decay": dict(batch=1, seqlen=300, nheads=4, headdim=64, dstate=128, rank=1, chunk=64, dt_shift=1.5),
    "mimo4_strong_decay": dict(batch=1, seqlen=150, nheads=4, headdim=64, dstate=64, rank=4, chunk=16, dt_shift=4.0),
}


@pytest.mark.parametrize("case", ["siso_strong_decay", "mimo4_strong_decay"])
def test_strong_decay_cases_cover_both_decay_paths(case):
    """The strong-decay cases really contain chunks on both sides of the
    -60 log-decay threshold (chunk sums of dt * A in f32)."""
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], **SMALL[case])
    inp = synth.prefill_inputs(wl)
    dt = synth.to_f64(inp["dt"], wl.dtype).astype(np.float32)[0]  # [L][H]
    A = inp["A"].astype(np.float32)
    sums = []
    for c0 in range(0, wl.seqlen, wl.chunk):
        sums.append((dt[c0:c0 + wl.chunk] * A[None, :]).sum(0))
    sums = np.concatenate(sums)
    assert (sums <= -60).any() and (sums > -60).any(), sums


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("case", list(SMALL))
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_small_with_state(case, dtype, algo):
    """Ragged lengths, a random initial state and carry; y, h_final and the
    carry against the oracle."""
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], dtype=dtype, h0_std=0.3, carry=True, **SMALL[case])
    inp = synth.prefill_inputs(wl)
    st = state_for(dims_of(wl), inp["h0"], inp["prev_B"], inp["prev_x"])
    y = prefill_gpu(inp, wl, state=st, algo=algo)
    yo, ho, pBo, pxo, _ = oracle.prefill(inp, **oracle_kw(wl), h0=inp["h0"], prev_B=inp["prev_B"],
                                         prev_x=inp["prev_x"])
    tol = TOL[dtype]
    assert_close(y.cpu().numpy(), yo, tol, f"{case} y")
    h, pB, px = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, tol, f"{case} h_final")
    assert np.array_equal(to_np(pB).reshape(pBo.shape), pBo)
    assert np.array_equal(to_np(px).reshape(pxo.shape), pxo)
    st.free()


@pytest.mark.parametrize("algo", ALGOS)
def test_stateless_and_split(algo):
    """No state: zero start.  Split: prefill(L) = prefill(L1) + prefill(L-L1)
    through the state, on the GPU."""
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=2, seqlen=300, nheads=2)
    inp = synth.prefill_inputs(wl)
    y_full = prefill_gpu(inp, wl, algo=algo).cpu().numpy()
    yo, _, _, _, _ = oracle.prefill(inp, **oracle_kw(wl))
    assert_close(y_full, yo, TOL["bf16"], "stateless y")
    st = state_for(dims_of(wl))
    L1 = 131
    head = {k: (v[:, :L1] if v.ndim >= 3 else v) for k, v in inp.items()}
    tail = {k: (np.ascontiguousarray(v[:, L1:]) if v.ndim >= 3 else v) for k, v in inp.items()}
    ya = prefill_gpu(head, wl, state=st, algo=algo).cpu().numpy()
    yb = prefill_gpu(tail, wl, state=st, algo=algo).cpu().numpy()
    assert_close(np.concatenate([ya, yb], 1), yo, TOL["bf16"], "split y")
    st.free()


@pytest.mark.parametrize("algo", ALGOS)
def test_prefill_then_decode(algo):
    """GPU prefill of L-k tokens then k GPU decode steps equals the oracle's
    prefill of all L tokens."""
    wl = synth.scaled(synth.workloads()["mimo4_b8_l4096"], batch=2, seqlen=100, nheads=2)
    inp = synth.prefill_inputs(wl)
    L, k = wl.seqlen, 7
    st = state_for(dims_of(wl))
    head = {n: (v[:, :L - k] if v.ndim >= 3 else v) for n, v in inp.items()}
    ya = prefill_gpu(head, wl, state=st, algo=algo).cpu().numpy()
    b, H, R, P = wl.batch, wl.nheads, wl.rank, wl.headdim
    y = torch.empty((b, H, R, P), dtype=torch.float32, device="cuda")
    A, D = dev(inp["A"]), dev(inp["D"])
    yd = []
    for t in range(L - k, L):
        tt = {n: dev(np.ascontiguousarray(inp[n][:, t])) for n in ("x", "B", "C", "dt", "lam", "theta")}
        m3.m3_decode_step(tt["x"], tt["B"], tt["C"], tt["dt"], tt["lam"], tt["theta"], A, D, y, st)
        yd.append(y.cpu().numpy())
    yo, ho, _, _, _ = oracle.prefill(inp, **oracle_kw(wl))
    got = np.concatenate([ya, np.stack(yd, 1)], 1)
    assert_close(got, yo, TOL["bf16"], "prefill+decode y")
    h, _, _ = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, TOL["bf16"], "prefill+decode h")
    st.free()


@pytest.mark.parametrize("algo", ALGOS)
def test_varlen_small(algo):
    """Packed batch with an empty sequence, a one-token sequence and ragged
    ones; per-sequence initial states; state and carry restart at each
    boundary."""
    lens = [37, 1, 0, 130, 64, 65]
    cu = synth.varlen_cu_seqlens(lens)
    wl = synth.scaled(synth.workloads()["varlen_16"], seqlen=int(cu[-1]), nheads=3, nseq=len(lens),
                      cu_seqlens=cu, h0_std=0.2, carry=True)
    wl_state = synth.scaled(wl, batch=len(lens))
    inp = synth.prefill_inputs(wl)
    init = synth.prefill_inputs(wl_state)  # per-sequence h0 and carry
    st = state_for(dims_of(wl, batch=len(lens)), init["h0"], init["prev_B"], init["prev_x"])
    y = prefill_gpu(inp, wl, state=st, cu=cu, algo=algo).cpu().numpy()
    yo, ho, pBo, pxo, _ = oracle.prefill(inp, **oracle_kw(wl), cu_seqlens=cu, h0=init["h0"],
                                         prev_B=init["prev_B"], prev_x=init["prev_x"])
    assert_close(y, yo, TOL["bf16"], "varlen y")
    h, pB, px = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, TOL["bf16"], "varlen h")
    assert np.array_equal(to_np(pB).reshape(pBo.shape), pBo)
    assert np.array_equal(to_np(px).reshape(pxo.shape), pxo)
    st.free()


def test_varlen_more_units_than_sms_longest_first():
    """More (sequence, head) units than SMs in a packed batch: the chunked
    launch runs the longest sequences' units first (an order computed on
    the device, ties and empty sequences included); every output, final
    state and carry against the oracle."""
    lens = [130, 0, 64, 257, 1, 130, 65, 200, 33, 0, 129, 64]
    cu = synth.varlen_cu_seqlens(lens)
    wl = synth.scaled(synth.workloads()["varlen_16"], seqlen=int(cu[-1]), nheads=16, nseq=len(lens),
                      cu_seqlens=cu, h0_std=0.2, carry=True)
    wl_state = synth.scaled(wl, batch=len(lens))
    inp = synth.prefill_inputs(wl)
    init = synth.prefill_inputs(wl_state)
    st = state_for(dims_of(wl, batch=len(lens)), init["h0"], init["prev_B"], init["prev_x"])
    y = prefill_gpu(inp, wl, state=st, cu=cu, algo=0)
    info = m3.m3_test_last_launch()
    y = y.cpu().numpy()
    assert info.kernel == m3.M3_TEST_KERNEL_CHUNKED and info.grid == 16 * len(lens)
    assert info.scratch_bytes == 4 * len(lens)  # the sequence order
    yo, ho, pBo, pxo, _ = oracle.prefill(inp, **oracle_kw(wl), cu_seqlens=cu, h0=init["h0"],
                                         prev_B=init["prev_B"], prev_x=init["prev_x"])
    assert_close(y, yo, TOL["bf16"], "varlen y")
    h, pB, px = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, TOL["bf16"], "varlen h")
    assert np.array_equal(to_np(pB).reshape(pBo.shape), pBo)
    assert np.array_equal(to_np(px).reshape(pxo.shape), pxo)
    st.free()


def test_empty_sequence_is_noop():
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=1, seqlen=0, nheads=1)
    x = torch.empty((1, 0, 1, 1, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((1, 0, 1, 1, 128), dtype=torch.bfloat16, device="cuda")
    s = torch.empty((1, 0, 1), dtype=torch.bfloat16, device="cuda")
    th = torch.empty((1, 0, 1, 64), dtype=torch.bfloat16, device="cuda")
    A = torch.full((1,), -1.0, device="cuda")
    y = torch.empty((1, 0, 1, 1, 64), device="cuda")
    st = state_for(dims_of(wl))
    h, _, _ = st.views()
    h.fill_(0.5)
    # empty tensors have no storage: pass aligned placeholders through the raw ABI
    buf = torch.empty(64, dtype=torch.float32, device="cuda")
    a = m3.m3_prefill_args()
    a.dims = m3.make_dims(1, 1, 64, 128, 1, m3.M3_BF16)
    a.seqlen = 0
    for f in ("x", "B", "C", "dt", "lam", "theta", "A", "D", "y"):
        setattr(a, f, buf.data_ptr())
    import ctypes
    assert m3.load_library().m3_scan_prefill(ctypes.byref(a), st.handle, None) == m3.M3_OK
    torch.cuda.synchronize()
    assert torch.all(h == 0.5)
    st.free()
    del x, B, s, th, A, y


def test_invalid_arguments_return_status():
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=2, seqlen=8, nheads=2)
    inp = synth.prefill_inputs(wl)
    st = state_for(dims_of(wl, batch=3))  # wrong batch for this call
    with pytest.raises(m3.M3Error) as e:
        prefill_gpu(inp, wl, state=st)
    assert e.value.status == m3.M3_ERR_INVALID_ARG
    st.free()
    wl32 = synth.scaled(wl, dtype="f32")
    with pytest.raises(m3.M3Error) as e:
        prefill_gpu(synth.prefill_inputs(wl32), wl32, algo=m3.M3_ALGO_CHUNKED)
    assert e.value.status == m3.M3_ERR_UNSUPPORTED


FULL = ["siso_b8_l4096", "mimo4_b8_l4096", "long_l16384", "varlen_16"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_output(name):
    """Full-size workloads in the benchmark's launch configuration, every
    output and every final state against the oracle (which finishes these
    in seconds on the host cores): max |err| / rms over the whole tensor."""
    wl = synth.workloads()[name]
    inp = synth.prefill_inputs(wl)
    cu = wl.cu_seqlens if wl.kind == "varlen" else None
    nseq = wl.nseq if cu is not None else wl.batch
    st = state_for(dims_of(wl, batch=nseq))
    y = prefill_gpu(inp, wl, state=st, cu=cu)
    assert m3.m3_device_status() == m3.M3_OK
    yo, ho, _, _, _ = oracle.prefill(inp, **oracle_kw(wl), cu_seqlens=cu)
    assert_close(y.cpu().numpy(), yo, TOL[wl.dtype], f"{name} y")
    h, _, _ = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, TOL[wl.dtype], f"{name} h_final")
    st.free()


@pytest.mark.parametrize("shape", [dict(dstate=128, rank=1, chunk=64), dict(dstate=64, rank=4, chunk=16),
                                   dict(dstate=128, rank=1, chunk=64, real=True, euler=True),
                                   dict(dstate=64, rank=1, chunk=64)],
                         ids=["siso", "mimo4", "mamba2", "siso_n64"])
def test_balanced_schedule_with_state(shape):
    """More units than SMs (5 x 32 heads, L 600 with a ragged last chunk):
    the chunked kernel cuts units between CTAs and hands state and carry
    over; with an initial state and carry, every output, the final state
    and the carry against the oracle."""
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=5, seqlen=600, nheads=32, h0_std=0.3,
                      carry=True, dt_shift=-3.0, **shape)
    inp = synth.prefill_inputs(wl)
    st = state_for(dims_of(wl), inp["h0"], inp["prev_B"], inp["prev_x"])
    y = prefill_gpu(inp, wl, state=st)
    assert m3.m3_device_status() == m3.M3_OK
    yo, ho, pBo, pxo, _ = oracle.prefill(inp, **oracle_kw(wl), h0=inp["h0"], prev_B=inp["prev_B"],
                                         prev_x=inp["prev_x"])
    assert_close(y.cpu().numpy(), yo, TOL["bf16"], "balanced y")
    h, pB, px = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, TOL["bf16"], "balanced h_final")
    assert np.array_equal(to_np(pB).reshape(pBo.shape), pBo)
    assert np.array_equal(to_np(px).reshape(pxo.shape), pxo)
    st.free()


CHUNKED_SHAPES = [(128, 1, 64), (64, 1, 64), (64, 4, 16), (64, 2, 32), (128, 2, 32)]


@pytest.mark.parametrize("N,R,Q", CHUNKED_SHAPES)
@pytest.mark.parametrize("L", [1, 31, 64, 65, 200])
def test_chunked_shapes_ragged(N, R, Q, L):
    """Every chunked-kernel variant against the oracle, explicitly selected,
    at lengths that end inside, at and just past a chunk boundary, with an
    initial state and a carry."""
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=2, seqlen=L, nheads=3, dstate=N, rank=R,
                      chunk=Q, h0_std=0.3, carry=True, dt_shift=-3.0)
    inp = synth.prefill_inputs(wl)
    st = state_for(dims_of(wl), inp["h0"], inp["prev_B"], inp["prev_x"])
    y = prefill_gpu(inp, wl, state=st, algo=m3.M3_ALGO_CHUNKED, chunk=Q)
    assert m3.m3_device_status() == m3.M3_OK
    yo, ho, pBo, pxo, _ = oracle.prefill(inp, **oracle_kw(wl), h0=inp["h0"], prev_B=inp["prev_B"],
                                         prev_x=inp["prev_x"])
    assert_close(y.cpu().numpy(), yo, TOL["bf16"], f"chunked N{N} R{R} Q{Q} L{L} y")
    h, pB, px = st.views()
    assert_close(to_np(h).reshape(ho.shape), ho, TOL["bf16"], f"chunked N{N} R{R} Q{Q} L{L} h")
    assert np.array_equal(to_np(pB).reshape(pBo.shape), pBo)
    assert np.array_equal(to_np(px).reshape(pxo.shape), pxo)
    st.free()


def test_chunked_matches_recurrent_closely():
    """The two GPU kernels agree far inside the tolerance on a mid-size case
    (the recurrent kernel is f32 throughout)."""
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=2, seqlen=700, nheads=4)
    inp = synth.prefill_inputs(wl)
    ya = prefill_gpu(inp, wl, algo=m3.M3_ALGO_CHUNKED).cpu().numpy()
    yb = prefill_gpu(inp, wl, algo=m3.M3_ALGO_RECURRENT).cpu().numpy()
    yo, _, _, _, _ = oracle.prefill(inp, **oracle_kw(wl))
    ea = assert_close(ya, yo, TOL["bf16"], "chunked")
    eb = assert_close(yb, yo, 1e-5, "recurrent")
    assert eb < ea
