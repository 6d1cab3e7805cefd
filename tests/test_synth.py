"""The seeded input generator: deterministic, windowed draws agree with full
draws, distributions and bf16 rounding are what the recipe says."""
import numpy as np
import torch

import synth


def test_deterministic_and_windowed():
    a = synth.fill((1000,), synth.S_X, synth.K_NORMAL, 0.0, 1.0, "f32", seed=3)
    b = synth.fill((1000,), synth.S_X, synth.K_NORMAL, 0.0, 1.0, "f32", seed=3)
    assert np.array_equal(a, b)
    w = synth.fill((100,), synth.S_X, synth.K_NORMAL, 0.0, 1.0, "f32", seed=3, offset=400)
    assert np.array_equal(w, a[400:500])
    c = synth.fill((1000,), synth.S_X, synth.K_NORMAL, 0.0, 1.0, "f32", seed=4)
    assert not np.array_equal(a, c)


def test_distributions():
    n = 200_000
    z = synth.fill((n,), synth.S_X, synth.K_NORMAL, 0.0, 1.0, "f64")
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    u = synth.fill((n,), synth.S_THETA, synth.K_UNIFORM, 0.0, np.pi, "f64")
    assert u.min() >= 0 and u.max() < np.pi and abs(u.mean() - np.pi / 2) < 0.01
    dt = synth.fill((n,), synth.S_DT, synth.K_SOFTPLUS, -4.0, 0.0, "f64")
    zz = np.log(np.expm1(dt)) + 4.0  # invert softplus(z - 4)
    assert abs(zz.mean()) < 0.01 and abs(zz.std() - 1) < 0.01
    a = synth.fill((n,), synth.S_A, synth.K_NEG_EXP, 0.0, 0.5, "f64")
    assert (a < 0).all() and abs(np.log(-a).std() - 0.5) < 0.01
    lam = synth.fill((n,), synth.S_LAM, synth.K_SIGMOID, 0.0, 0.0, "f64")
    assert (lam > 0).all() and (lam < 1).all() and abs(lam.mean() - 0.5) < 0.01
    B = synth.fill((1000, 128), synth.S_B, synth.K_NORMAL_RMS, synth.RMS_EPS, 0.0, "f64", row_len=128)
    rms = np.sqrt((B ** 2).mean(axis=1))
    assert np.allclose(rms, 1.0, atol=1e-5)


def test_bf16_rounding_matches_torch():
    f = synth.fill((50_000,), synth.S_X, synth.K_NORMAL, 0.0, 3.0, "f32", seed=9)
    h = synth.fill((50_000,), synth.S_X, synth.K_NORMAL, 0.0, 3.0, "bf16", seed=9)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(h, ref)


def test_lengths_and_workloads():
    w = synth.workloads()
    v = w["varlen_16"]
    lens = np.diff(v.cu_seqlens)
    assert len(lens) == 16 and lens.min() >= 256 and lens.max() <= 8192
    assert v.seqlen == int(v.cu_seqlens[-1])
    assert w["siso_b8_l4096"].units == 256 and w["mimo4_b8_l4096"].rank == 4
