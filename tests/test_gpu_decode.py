"""GPU parity of m3_decode_step against the oracle (element by element)."""
import numpy as np
import pytest
import torch

import oracle
import state_space_sequence_06_b300 as m3
import synth
from gpu_util import TOL, dev, state_for, to_np

pytestmark = pytest.mark.gpu


def run_decode(wl, steps, units=None, window=None):
    """Run `steps` decode steps on the GPU for every unit of wl; return
    (y per step [T][b][H][R][P] for the sampled units or all, final h, carry)
    and the oracle's results for the same units."""
    b, H, P, N, R = wl.batch, wl.nheads, wl.headdim, wl.dstate, wl.rank
    init = synth.decode_inputs(wl, steps=1)  # h0 / carry do not depend on the window
    st = state_for((b, H, P, N, R, m3.M3_BF16 if wl.dtype == "bf16" else m3.M3_F32),
                   init["h0"], init["prev_B"], init["prev_x"])
    window = window or steps
    ys = []
    sel = list(range(b * H)) if units is None else list(units)
    y = torch.empty((b, H, R, P), dtype=torch.float32, device="cuda")
    sumsq = torch.zeros((), dtype=torch.float64, device="cuda")  # over every unit and step
    allin = {}
    for s0 in range(0, steps, window):
        n = min(window, steps - s0)
        d = synth.decode_inputs(wl, steps=n, first_step=s0)
        t = {k: dev(d[k]) for k in ("x", "B", "C", "dt", "lam", "theta")}
        A, D = dev(d["A"]), dev(d["D"])
        for i in range(n):
            lam_i = None if t["lam"] is None else t["lam"][i]
            th_i = None if t["theta"] is None else t["theta"][i]
            m3.m3_decode_step(t["x"][i], t["B"][i], t["C"][i], t["dt"][i], lam_i, th_i, A, D, y, st)
            sumsq += (y.double() ** 2).sum()
            ys.append(y.reshape(b * H, R, P)[sel].cpu().numpy())
        for k in ("x", "B", "C", "dt", "lam", "theta"):
            if d[k] is None:  # lam = 1 / theta = 0: the oracle takes None the same way
                continue
            a = d[k]
            if k in ("B", "C") and a.shape[2] != H:  # grouped: the oracle below takes one head per row
                a = np.repeat(a, H // a.shape[2], axis=2)
            v = a.reshape((n, b * H) + a.shape[3:])[:, sel] if k not in ("dt", "lam") else \
                a.reshape(n, b * H)[:, sel]
            allin.setdefault(k, []).append(v)
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    h, pB, px = st.views()
    gpu = dict(y=np.stack(ys), y_rms=float(torch.sqrt(sumsq / (steps * y.numel())).item()),
               h_rms=float(torch.sqrt((h.double() ** 2).mean()).item()),
               h=to_np(h).reshape(b * H, N // 2, P, 2)[sel],
               pB=to_np(pB).reshape(b * H, R, N)[sel], px=to_np(px).reshape(b * H, R, P)[sel])
    st.free()
    # oracle over the sampled units only: pack them as a batch of len(sel) rows with one head each
    heads = np.array([u % H for u in sel])
    sub = {k: np.concatenate(v, 0) for k, v in allin.items()}
    T = steps
    sub = dict(x=sub["x"].reshape(T, len(sel), 1, R, P), B=sub["B"].reshape(T, len(sel), 1, R, N),
               C=sub["C"].reshape(T, len(sel), 1, R, N), dt=sub["dt"].reshape(T, len(sel), 1),
               lam=sub["lam"].reshape(T, len(sel), 1) if "lam" in sub else None,
               theta=sub["theta"].reshape(T, len(sel), 1, N // 2) if "theta" in sub else None)
    yo, ho, pBo, pxo = [], [], [], []
    for i, u in enumerate(sel):
        one = {k: (None if v is None else np.ascontiguousarray(v[:, i:i + 1])) for k, v in sub.items()}
        one["A"] = init["A"][heads[i]:heads[i] + 1]
        one["D"] = init["D"][heads[i]:heads[i] + 1]
        one["h0"] = init["h0"].reshape(b * H, N // 2, P, 2)[u:u + 1]
        one["prev_B"] = init["prev_B"].reshape(b * H, R, N)[u:u + 1]
        one["prev_x"] = init["prev_x"].reshape(b * H, R, P)[u:u + 1]
        y_, h_, pB_, px_ = oracle.decode(one, batch=1, H=1, P=P, N=N, R=R, dtype=wl.dtype, steps=T)
        yo.append(y_[:, 0, 0])
        ho.append(h_[0])
        pBo.append(pB_[0])
        pxo.append(px_[0])
    ref = dict(y=np.stack(yo, 1), h=np.stack(ho), pB=np.stack(pBo), px=np.stack(pxo))
    return gpu, ref


def check(gpu, ref, dtype, what):
    """max |err| over the checked units / rms over every unit (the GPU's
    own outputs stand in for the reference rms: they differ by ~1e-6)."""
    tol = TOL[dtype]
    ey = np.max(np.abs(gpu["y"] - ref["y"])) / gpu["y_rms"]
    eh = np.max(np.abs(gpu["h"] - ref["h"])) / gpu["h_rms"]
    assert ey <= tol, f"{what} y: max|err|/rms = {ey:.3e} > {tol:.1e}"
    assert eh <= tol, f"{what} h_final: max|err|/rms = {eh:.3e} > {tol:.1e}"
    assert np.array_equal(gpu["pB"], ref["pB"]), f"{what} carry B"
    assert np.array_equal(gpu["px"], ref["px"]), f"{what} carry x"


@pytest.mark.parametrize("N,R,P", [(128, 1, 64), (64, 4, 64), (16, 2, 32), (24, 3, 8), (256, 1, 16)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_small(N, R, P, dtype):
    wl = synth.Workload("t", "decode", 3, 0, 4, P, N, R, dtype, h0_std=0.1, carry=True)
    gpu, ref = run_decode(wl, 37)
    check(gpu, ref, dtype, f"decode N{N} R{R} P{P} {dtype}")


def test_decode_zero_state_no_carry():
    wl = synth.Workload("t", "decode", 2, 0, 2, 64, 128, 1, "bf16")
    gpu, ref = run_decode(wl, 9)
    check(gpu, ref, "bf16", "decode from zero state")


@pytest.mark.parametrize("name", ["decode_siso_b256", "decode_mimo4_b256"])
def test_decode_full_size_sampled(name):
    """The full workload (batch 256, 32 heads, 1024 steps) in the launch
    configuration the benchmark times; the oracle checks sampled units at
    every step."""
    wl = synth.workloads()[name]
    rng = np.random.default_rng(0)
    units = sorted(set([0, wl.batch * wl.nheads - 1] + list(rng.choice(wl.batch * wl.nheads, 10, replace=False))))
    gpu, ref = run_decode(wl, wl.seqlen, units=units, window=128)
    check(gpu, ref, wl.dtype, name)


@pytest.mark.parametrize("name", ["decode_siso_b256", "decode_mimo4_b256"])
def test_decode_full_size_every_unit(name):
    """Every unit of the full workload (batch 256, 32 heads: 8192 units) for
    256 steps, in the benchmark's launch configuration: every output of
    every step and the whole final state against the oracle, the carry bit
    for bit.  (The sampled test above walks all 1024 steps.)"""
    wl = synth.workloads()[name]
    steps = 256
    b, H, P, N, R = wl.batch, wl.nheads, wl.headdim, wl.dstate, wl.rank
    d = synth.decode_inputs(wl, steps=steps)
    st = state_for((b, H, P, N, R, m3.M3_BF16), d["h0"], d["prev_B"], d["prev_x"])
    t = {k: dev(d[k]) for k in ("x", "B", "C", "dt", "lam", "theta", "A", "D")}
    ys = torch.empty((steps, b, H, R, P), dtype=torch.float32, device="cuda")
    for i in range(steps):
        m3.m3_decode_step(t["x"][i], t["B"][i], t["C"][i], t["dt"][i], t["lam"][i], t["theta"][i], t["A"], t["D"],
                          ys[i], st)
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    h, pB, px = st.views()
    gh, gpB, gpx = to_np(h), to_np(pB), to_np(px)
    gy = ys.cpu().numpy().astype(np.float64)
    st.free()
    yo, ho, pBo, pxo = oracle.decode(d, batch=b, H=H, P=P, N=N, R=R, dtype=wl.dtype, steps=steps)
    tol = TOL[wl.dtype]
    ey = np.max(np.abs(gy - yo)) / np.sqrt(np.mean(yo ** 2))
    eh = np.max(np.abs(gh.reshape(ho.shape) - ho)) / np.sqrt(np.mean(ho ** 2))
    assert ey <= tol, f"{name} y over every unit: {ey:.3e}"
    assert eh <= tol, f"{name} h_final over every unit: {eh:.3e}"
    assert np.array_equal(gpB.reshape(pBo.shape), pBo) and np.array_equal(gpx.reshape(pxo.shape), pxo)
