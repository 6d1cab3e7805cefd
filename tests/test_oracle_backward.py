"""Pins of the backward oracle: its forward replica equals the (pinned) C
oracle, and every gradient matches central finite differences of the C
oracle's own forward pass in double (loss = sum(dy * y) + sum(dh * h_final))
along a random direction per input, for SISO and MIMO, grouped B/C, with an
initial state and carry.  A slip in any adjoint term (a missing conjugate,
a weight taken from the wrong token, a dropped carry term) moves one of
these directional derivatives by far more than the tolerance."""
import numpy as np
import pytest

import oracle

KEYS = ("x", "B", "C", "dt", "lam", "theta", "A", "D", "h0", "prev_B", "prev_x")


def _case(R, G, seed=0):
    rng = np.random.default_rng(seed)
    b, L, H, P, N = 2, 9, 4, 3, 6
    K = N // 2
    inp = dict(x=rng.normal(size=(b, L, H, R, P)), B=rng.normal(size=(b, L, G, R, N)),
               C=rng.normal(size=(b, L, G, R, N)), dt=rng.uniform(0.05, 0.6, (b, L, H)),
               lam=rng.uniform(0.1, 0.9, (b, L, H)), theta=rng.uniform(0, np.pi, (b, L, H, K)),
               A=-rng.uniform(0.2, 2.0, H), D=rng.normal(size=H))
    st = dict(h0=rng.normal(size=(b, H, K, P, 2)) * 0.5, prev_B=rng.normal(size=(b, H, R, N)),
              prev_x=rng.normal(size=(b, H, R, P)))
    dims = dict(batch=b, L=L, H=H, P=P, N=N, R=R)
    dy = rng.normal(size=(b, L, H, R, P))
    dh = rng.normal(size=(b, H, K, P, 2))
    return inp, st, dims, dy, dh


def _loss(inp, st, dims, dy, dh):
    y, h, _, _, _ = oracle.prefill(inp, **dims, dtype="f64", nthreads=1, **st)
    return float(np.sum(dy * y) + np.sum(dh * h.reshape(dh.shape)))


@pytest.mark.parametrize("R,G", [(1, 4), (2, 2), (1, 1)])
def test_forward_replica_is_the_oracle(R, G):
    inp, st, dims, dy, dh = _case(R, G)
    y, hf, _ = oracle.prefill_backward(inp, dy, **dims, dtype="f64", dh_final=dh, **st)
    yo, ho, _, _, _ = oracle.prefill(inp, **dims, dtype="f64", nthreads=1, **st)
    assert np.allclose(y, yo, rtol=1e-12, atol=1e-12)
    assert np.allclose(hf.reshape(ho.shape), ho, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("R,G", [(1, 4), (2, 2), (1, 1)])
def test_gradients_match_finite_differences(R, G):
    inp, st, dims, dy, dh = _case(R, G)
    _, _, grads = oracle.prefill_backward(inp, dy, **dims, dtype="f64", dh_final=dh, **st)
    rng = np.random.default_rng(7)
    eps = 1e-6
    for key in KEYS:
        src = st if key in st else inp
        v = rng.normal(size=np.shape(src[key]))
        plus = {k: (w + eps * v if k == key else w) for k, w in src.items()}
        minus = {k: (w - eps * v if k == key else w) for k, w in src.items()}
        if key in st:
            fd = (_loss(inp, plus, dims, dy, dh) - _loss(inp, minus, dims, dy, dh)) / (2 * eps)
        else:
            fd = (_loss(plus, st, dims, dy, dh) - _loss(minus, st, dims, dy, dh)) / (2 * eps)
        an = float(np.sum(grads[key] * v))
        assert abs(an - fd) <= 1e-6 * max(1.0, abs(fd)), f"{key}: adjoint {an:.9g} vs finite difference {fd:.9g}"


def test_special_values_lam_one_theta_zero():
    """lam and theta given as None (first order, real state): the gradient
    still matches finite differences in dt, B and x."""
    inp, st, dims, dy, dh = _case(1, 4, seed=3)
    inp = dict(inp, lam=None, theta=None)
    _, _, grads = oracle.prefill_backward(inp, dy, **dims, dtype="f64", dh_final=dh, **st)
    rng = np.random.default_rng(11)
    eps = 1e-6
    for key in ("dt", "B", "x", "A"):
        v = rng.normal(size=np.shape(inp[key]))
        fd = (_loss(dict(inp, **{key: inp[key] + eps * v}), st, dims, dy, dh)
              - _loss(dict(inp, **{key: inp[key] - eps * v}), st, dims, dy, dh)) / (2 * eps)
        assert abs(float(np.sum(grads[key] * v)) - fd) <= 1e-6 * max(1.0, abs(fd)), key


BACKWARD_MUTANTS = [
    ("no_conjugate_on_a", "Gs = np.conj(a[t])[:, None] * Gh", "Gs = a[t][:, None] * Gh"),
    ("beta_from_current_token", "Gu[t - 1] += bet[t] * Gs", "Gu[t - 1] += bet[t - 1] * Gs"),
    ("carry_gradient_dropped", "Gu_m1 = bet[0] * Gs", "Gu_m1 = 0 * Gs"),
    ("lam_sign", 'g["lam"][t] = -dt[t] * dbet + dt[t] * dgam', 'g["lam"][t] = dt[t] * dbet + dt[t] * dgam'),
    ("theta_from_real_part", 'g["theta"][t] = dt[t] * Gz.imag', 'g["theta"][t] = dt[t] * Gz.real'),
]


@pytest.mark.parametrize("name,find,repl", BACKWARD_MUTANTS, ids=[m[0] for m in BACKWARD_MUTANTS])
def test_backward_mutant_is_caught(monkeypatch, name, find, repl):
    """Plant one slip in a copy of the adjoint and check that the finite
    differences catch it."""
    import importlib.util
    import os

    src = open(os.path.join(os.path.dirname(oracle.__file__), "backward.py")).read()
    assert find in src, f"mutation site for {name} not found"
    spec = importlib.util.spec_from_loader("oracle._backward_mutant", loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    exec(compile(src.replace(find, repl, 1), f"<{name}>", "exec"), mod.__dict__)
    monkeypatch.setattr(oracle, "prefill_backward", mod.prefill_backward)
    with pytest.raises(AssertionError):
        for R, G in [(1, 4), (2, 2)]:
            test_gradients_match_finite_differences(R, G)


def _loss_prologue(inp, st, dims, dy, dh, bias):
    post = oracle.apply_prologue(dict(inp, prev_B=st["prev_B"]), "f64", dt_softplus=True, bc_norm=True, dt_bias=bias)
    st2 = dict(st, prev_B=post.pop("prev_B"))
    y, h, _, _, _ = oracle.prefill(post, **dims, dtype="f64", nthreads=1, **st2)
    return float(np.sum(dy * y) + np.sum(dh * h.reshape(dh.shape)))


@pytest.mark.parametrize("R,G", [(1, 4), (2, 2)])
def test_prologue_gradients_match_finite_differences(R, G):
    """With the fused prologue (softplus of dt + dt_bias, RMS norm of B, C
    and the carried B rows) the gradients are with respect to the raw
    inputs: central finite differences of the prologue-then-scan forward
    oracle along a random direction per raw input, dt_bias included."""
    inp, st, dims, dy, dh = _case(R, G, seed=5)
    inp = dict(inp, dt=inp["dt"] * 8 - 3)  # pre-activations on both sides of 0
    bias = np.random.default_rng(9).normal(size=dims["H"]) * 0.5
    _, _, g = oracle.prefill_backward(inp, dy, **dims, dtype="f64", dh_final=dh, dt_softplus=True, bc_norm=True,
                                      dt_bias=bias, **st)
    rng = np.random.default_rng(13)
    eps = 1e-6
    for key in ("dt", "B", "C", "prev_B", "x", "dt_bias"):
        if key == "dt_bias":
            v = rng.normal(size=bias.shape)
            fd = (_loss_prologue(inp, st, dims, dy, dh, bias + eps * v)
                  - _loss_prologue(inp, st, dims, dy, dh, bias - eps * v)) / (2 * eps)
        else:
            src = st if key in st else inp
            v = rng.normal(size=np.shape(src[key]))
            pl = {k: (w + eps * v if k == key else w) for k, w in src.items()}
            mi = {k: (w - eps * v if k == key else w) for k, w in src.items()}
            if key in st:
                fd = (_loss_prologue(inp, pl, dims, dy, dh, bias) - _loss_prologue(inp, mi, dims, dy, dh, bias)) / (2 * eps)
            else:
                fd = (_loss_prologue(pl, st, dims, dy, dh, bias) - _loss_prologue(mi, st, dims, dy, dh, bias)) / (2 * eps)
        an = float(np.sum(g[key] * v))
        assert abs(an - fd) <= 1e-6 * max(1.0, abs(fd)), f"{key}: adjoint {an:.9g} vs finite difference {fd:.9g}"


def test_rms_norm_backward_slips_are_caught():
    """The norm's Jacobian pin is sharp: the full chain dv = s (dn - n
    mean(dn n)) matches the finite difference of B, and dropping its
    projection term (dv = s dn) misses it by far more than the bound."""
    from oracle import backward as ob

    inp, st, dims, dy, dh = _case(1, 4, seed=5)
    bias = np.zeros(dims["H"])
    post = oracle.apply_prologue(dict(inp, prev_B=st["prev_B"]), "f64", dt_softplus=True, bc_norm=True, dt_bias=bias)
    post_grads = ob._prefill_backward(post, dy, **dims, dtype="f64", h0=st["h0"], prev_B=post["prev_B"],
                                      prev_x=st["prev_x"], dh_final=dh)[2]
    v = np.random.default_rng(1).normal(size=inp["B"].shape)
    eps = 1e-6
    fd = (_loss_prologue(dict(inp, B=inp["B"] + eps * v), st, dims, dy, dh, bias)
          - _loss_prologue(dict(inp, B=inp["B"] - eps * v), st, dims, dy, dh, bias)) / (2 * eps)
    right = float(np.sum(ob._rms_norm_backward(inp["B"], post_grads["B"], oracle.BC_NORM_EPS) * v))
    assert abs(right - fd) <= 1e-6 * max(1.0, abs(fd))
    s = 1.0 / np.sqrt(np.mean(inp["B"] ** 2, axis=-1, keepdims=True) + oracle.BC_NORM_EPS)
    wrong = float(np.sum(s * post_grads["B"] * v))
    assert abs(wrong - fd) > 1e-4 * max(1.0, abs(fd))
