"""Pins of the oracle's fused prologue (softplus of dt, RMS norm of B and C
rows) against things other than itself: closed forms and identities of
softplus, the input generator's own softplus (another formula, written
separately), the defining property of the norm, and invariances of the
whole scan that hold only when the norm acts on each row over N."""
import numpy as np
import pytest

import oracle
import synth


def test_softplus_closed_forms():
    assert oracle.softplus(0.0) == pytest.approx(np.log(2.0), rel=1e-15)
    z = np.linspace(-30, 30, 601)
    # softplus(z) - softplus(-z) = z and softplus(z) > max(z, 0)
    assert np.allclose(oracle.softplus(z) - oracle.softplus(-z), z, rtol=0, atol=1e-13)
    assert np.all(oracle.softplus(z) > np.maximum(z, 0))
    # tails: e^z for very negative z, z + e^-z for large z
    assert oracle.softplus(-700.0) == pytest.approx(np.exp(-700.0), rel=1e-12)
    assert oracle.softplus(40.0) == pytest.approx(40.0 + np.exp(-40.0), rel=1e-15)
    assert np.isfinite(oracle.softplus(1e4))


def test_softplus_matches_the_generators_formula():
    """The generator draws dt as log1p(exp(z)) of z = N(0,1) + shift; the
    same draws taken raw (N(shift, 1)) go through the oracle's softplus."""
    n = 4096
    for shift in (-4.0, 0.0, 3.0):
        raw = synth.fill((n,), synth.S_DT, synth.K_NORMAL, shift, 1.0, "f64")
        gen = synth.fill((n,), synth.S_DT, synth.K_SOFTPLUS, shift, 0.0, "f64")
        assert np.allclose(oracle.softplus(raw), gen, rtol=1e-14, atol=0)


def test_bias_enters_before_softplus():
    """dt_bias is added to the pre-activation: raw draws N(0, 1) with a
    per-head bias equal to the generator's shift give the generator's own
    softplus(N(0, 1) + shift), head by head."""
    shifts = np.array([-4.0, -1.0, 2.0])
    raw = synth.fill((2, 50, 3), synth.S_DT, synth.K_NORMAL, 0.0, 1.0, "f64")
    out = oracle.apply_prologue({"dt": raw}, "f64", dt_softplus=True, dt_bias=shifts)["dt"]
    for h, sh in enumerate(shifts):
        gen = synth.fill((2, 50, 3), synth.S_DT, synth.K_SOFTPLUS, sh, 0.0, "f64")
        assert np.allclose(out[..., h], gen[..., h], rtol=1e-14, atol=0)


def test_rms_normalize_definition():
    rng = np.random.default_rng(0)
    a = rng.normal(0, 3, (5, 7, 64)) * rng.uniform(0.1, 10, (5, 7, 1))
    n = oracle.rms_normalize(a)
    ms = np.mean(a * a, axis=-1, keepdims=True)
    # each row keeps its direction and ends with mean square ms / (ms + eps)
    assert np.allclose(np.mean(n * n, axis=-1, keepdims=True), ms / (ms + oracle.BC_NORM_EPS), rtol=1e-13)
    assert np.allclose(n * np.sqrt(ms + oracle.BC_NORM_EPS), a, rtol=1e-13)
    assert np.array_equal(oracle.rms_normalize(np.zeros(8)), np.zeros(8))


def _scan(inp, wl, **pro):
    kw = dict(batch=wl.batch, L=wl.seqlen, H=wl.nheads, P=wl.headdim, N=wl.dstate, R=wl.rank, nthreads=1)
    p = oracle.apply_prologue(inp, wl.dtype, dt_bias=inp.get("dt_bias"), **pro)
    return oracle.prefill(p, **kw, dtype="f64", h0=p.get("h0"), prev_B=p.get("prev_B"), prev_x=p.get("prev_x"))


@pytest.mark.parametrize("R", [1, 2])
def test_norm_undoes_a_positive_scale_of_each_row(R):
    """Scaling every row of B and C (and the carried B) by its own positive
    factor c changes nothing after the norm but the epsilon's share,
    eps / (2 c^2 mean(v^2)), at most about 2e-6 here (rows of 16 values of
    N(0, 2^2), c >= 0.5): the norm acts per (token, group, rank) row over N."""
    wl = synth.Workload("t", "prefill", 2, 23, 4, 8, 16, R, "f32", h0_std=0.2, carry=True, prologue=True,
                        ngroups=2)
    inp = synth.prefill_inputs(wl)
    rng = np.random.default_rng(1)
    scaled = dict(inp)
    for k in ("B", "C", "prev_B"):
        scaled[k] = inp[k].astype(np.float64) * rng.uniform(0.5, 4.0, inp[k].shape[:-1] + (1,))
    y1, h1, _, _, _ = _scan(inp, wl, bc_norm=True, dt_softplus=True)
    y2, h2, _, _, _ = _scan(scaled, wl, bc_norm=True, dt_softplus=True)
    assert np.allclose(y1, y2, rtol=1e-5, atol=1e-5 * np.sqrt(np.mean(y1 ** 2)))
    assert np.allclose(h1, h2, rtol=1e-5, atol=1e-5 * np.sqrt(np.mean(h1 ** 2)))
    # and the norm does matter: without it the scaled inputs give another result
    y3, _, _, _, _ = _scan(scaled, wl, dt_softplus=True)
    assert not np.allclose(y1, y3, rtol=1e-2)


def test_a_normalisation_over_the_wrong_axis_is_caught():
    """Normalising over the rank axis instead of N gives another result
    (so the invariance above pins the axis)."""
    wl = synth.Workload("t", "prefill", 1, 17, 2, 8, 16, 2, "f32", prologue=True)
    inp = synth.prefill_inputs(wl)
    y1, _, _, _, _ = _scan(inp, wl, bc_norm=True)
    wrong = dict(inp)
    for k in ("B", "C"):
        a = inp[k].astype(np.float64)
        wrong[k] = a / np.sqrt(np.mean(a * a, axis=-2, keepdims=True) + 1e-6)
    y2, _, _, _, _ = _scan(wrong, wl)
    assert not np.allclose(y1, y2, rtol=1e-3)


def test_prologue_on_already_normalised_inputs_is_the_plain_scan():
    """The plain workloads' B and C rows are drawn already RMS-normalised and
    their dt already through softplus: the norm leaves them (to 1e-6), and
    softplus of the generator's raw draws rebuilds their dt."""
    wl = synth.Workload("t", "prefill", 1, 40, 2, 8, 16, 1, "f32")
    inp = synth.prefill_inputs(wl)
    kw = dict(batch=1, L=40, H=2, P=8, N=16, R=1, nthreads=1)
    y_plain, _, _, _, _ = oracle.prefill(inp, **kw, dtype="f32")
    raw = dict(inp, dt=synth.fill((1, 40, 2), synth.S_DT, synth.K_NORMAL, wl.dt_shift, 1.0, "f32"))
    p = oracle.apply_prologue(raw, "f32", dt_softplus=True, bc_norm=True)
    y_pro, _, _, _, _ = oracle.prefill(p, **kw, dtype="f64")
    assert np.allclose(y_pro, y_plain, rtol=0, atol=1e-5 * np.sqrt(np.mean(y_plain ** 2)))


def test_decode_prologue_continues_prefill_prologue():
    """Prefill with the prologue, then decode steps with the prologue (the
    carry holds the raw last B, normalised again when used), equals one
    prologue prefill over all tokens."""
    H, P, N, R, L, T = 2, 8, 16, 2, 20, 4
    wl = synth.Workload("t", "prefill", 1, L + T, H, P, N, R, "f32", prologue=True, ngroups=1)
    inp = synth.prefill_inputs(wl)
    kw = dict(batch=1, H=H, P=P, N=N, R=R, nthreads=1)
    full = oracle.apply_prologue(inp, "f32", dt_softplus=True, bc_norm=True, dt_bias=inp["dt_bias"])
    y_all, _, _, _, _ = oracle.prefill(full, L=L + T, dtype="f64", **kw)
    _, h, _, px, _ = oracle.prefill({k: (v if k in ("A", "D", "dt_bias") else v[:, :L]) for k, v in full.items()},
                                    L=L, dtype="f64", **kw)
    raw_last_B = np.repeat(inp["B"][:, L - 1], H, axis=1).reshape(H, R, N)  # group 0 for both heads
    dec = {k: np.ascontiguousarray(np.swapaxes(inp[k][:, L:], 0, 1)) for k in ("x", "B", "C", "dt", "lam", "theta")}
    dec.update(A=inp["A"], D=inp["D"], h0=h, prev_B=raw_last_B, prev_x=px)
    p = oracle.apply_prologue(dec, "f32", dt_softplus=True, bc_norm=True, dt_bias=inp["dt_bias"])
    y_dec, _, _, _ = oracle.decode(p, steps=T, dtype="f64", **kw)
    assert np.allclose(y_dec[:, 0], y_all[0, L:], rtol=1e-9, atol=1e-9)
