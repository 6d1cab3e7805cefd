"""The oracle's stand-ins for the special values: lam = None means lam = 1
and theta = None means theta = 0, for bf16 and f32 inputs, in prefill and
decode (the C oracle reads every input in dt's storage type, so the
stand-ins must be stored the same way)."""
import numpy as np
import pytest

import oracle
import synth


def _explicit(inp, dtype):
    d = dict(inp)
    dt = np.asarray(inp["dt"])
    d["lam"] = np.full(dt.shape, 0x3F80, np.uint16) if dtype == "bf16" else np.ones(dt.shape, np.float32)
    K = inp["B"].shape[-1] // 2
    d["theta"] = np.zeros(dt.shape + (K,), dt.dtype)
    return d


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prefill_none_equals_explicit(dtype):
    wl = synth.scaled(synth.workloads()["siso_b8_l4096"], batch=1, seqlen=37, nheads=2, dstate=16,
                      dtype=dtype, h0_std=0.3, carry=True)
    inp = synth.prefill_inputs(wl)
    kw = dict(batch=1, L=37, H=2, P=64, N=16, R=1, dtype=dtype, h0=inp["h0"], prev_B=inp["prev_B"],
              prev_x=inp["prev_x"], nthreads=1)
    none = dict(inp, lam=None, theta=None)
    ya, ha = oracle.prefill(none, **kw)[:2]
    yb, hb = oracle.prefill(_explicit(inp, dtype), **kw)[:2]
    assert np.array_equal(ya, yb) and np.array_equal(ha, hb)
    # and they are not the general case's values (the stand-ins matter)
    yc = oracle.prefill(inp, **kw)[0]
    assert not np.allclose(ya, yc)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_none_equals_explicit(dtype):
    wl = synth.Workload("t", "decode", 2, 0, 2, 8, 16, 2, dtype, h0_std=0.1, carry=True)
    inp = synth.decode_inputs(wl, steps=5)
    kw = dict(batch=2, H=2, P=8, N=16, R=2, dtype=dtype, steps=5, nthreads=1)
    ya, ha = oracle.decode(dict(inp, lam=None, theta=None), **kw)[:2]
    yb, hb = oracle.decode(_explicit(inp, dtype), **kw)[:2]
    assert np.array_equal(ya, yb) and np.array_equal(ha, hb)
