"""Pins for the CPU oracle: checks that tie it to something other than itself.

Each ``pin_*`` function takes an oracle library handle (the default build, or
a copy with a planted mistake) and raises AssertionError when the oracle
disagrees with what the method and the mathematics fix.  Sources of truth:

* closed forms of the recurrence (zero input, constant input);
* ``scipy.signal.lfilter``: with constant dt, lam and theta the recurrence
  of every state entry is a first-order IIR filter driven by u_t;
* a brute-force unrolled sum (the quadratic, attention-like form) on L <= 16;
* the parity example of "Together AI announces Mamba-3" (section 2,
  complex-valued states: the rotation lets the state track whether the
  number of 1s read so far is even or odd), as a stored fixture;
* structural identities: rank-R superposition of SISO runs, permutation
  invariance of the real state when theta = 0, independence from the carry
  when lam = 1 (first-order exponential-Euler, the Mamba-2 rule in the
  discretisation table of the same page), split and carry equalities.
"""
from __future__ import annotations

import os

import numpy as np
import scipy.signal

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def run1(lib, x, B, C, dt, lam, theta, A, D, h0=None, pB=None, px=None):
    """One unit (batch 1, one head), f64 inputs: x [L][R][P], B/C [L][R][N],
    dt/lam [L], theta [L][N/2].  Returns y [L][R][P], h [N/2][P] complex,
    carry (B [R][N], x [R][P])."""
    L, R, P = x.shape
    N = B.shape[2]
    inp = dict(x=x.reshape(1, L, 1, R, P), B=B.reshape(1, L, 1, R, N), C=C.reshape(1, L, 1, R, N),
               dt=np.asarray(dt, float).reshape(1, L, 1), lam=np.asarray(lam, float).reshape(1, L, 1),
               theta=theta.reshape(1, L, 1, N // 2), A=np.array([A], float), D=np.array([D], float))
    h0c = None if h0 is None else np.stack([h0.real, h0.imag], -1).reshape(1, 1, N // 2, P, 2)
    y, h, cB, cx, _ = oracle.prefill(
        inp, batch=1, L=L, H=1, P=P, N=N, R=R, dtype="f64", h0=h0c,
        prev_B=None if pB is None else pB.reshape(1, 1, R, N),
        prev_x=None if px is None else px.reshape(1, 1, R, P), nthreads=1, lib=lib)
    return y[0, :, 0], h[0, ..., 0] + 1j * h[0, ..., 1], cB[0], cx[0]


def cplx(v):
    """Real vector [..., N] -> complex [..., N/2] with (2k, 2k+1) = (re, im)."""
    return v[..., 0::2] + 1j * v[..., 1::2]


def _rand(rng, L, R, P, N, dt_shift=-1.0):
    x = rng.standard_normal((L, R, P))
    B = rng.standard_normal((L, R, N))
    C = rng.standard_normal((L, R, N))
    dt = np.log1p(np.exp(rng.standard_normal(L) + dt_shift))
    lam = 1 / (1 + np.exp(-rng.standard_normal(L)))
    theta = rng.uniform(0, np.pi, (L, N // 2))
    return x, B, C, dt, lam, theta


def close(a, b, tol=1e-10, what=""):
    a, b = np.asarray(a), np.asarray(b)
    err = np.max(np.abs(a - b)) / max(1e-300, np.max(np.abs(b)))
    assert err <= tol, f"{what}: relative max error {err:.3e} > {tol}"


# --------------------------------------------------------------------------


def pin_zero_input_closed_form(lib):
    """B = 0 so u = 0: h_t = h0 * exp(sum_{s<=t} dt_s (A + i theta_s)) and
    y_t = Re(conj(Chat_t) h_t) + D x_t, written in real components."""
    rng = np.random.default_rng(1)
    L, R, P, N = 20, 2, 3, 8
    x, B, C, dt, lam, theta = _rand(rng, L, R, P, N)
    B[:] = 0
    A, D = -0.7, 0.37
    h0 = rng.standard_normal((N // 2, P)) + 1j * rng.standard_normal((N // 2, P))
    y, h, _, _ = run1(lib, x, B, C, dt, lam, theta, A, D, h0=h0)
    expo = np.cumsum(dt[:, None] * (A + 1j * theta), axis=0)  # [L][N/2]
    ht = h0[None] * np.exp(expo)[:, :, None]  # [L][N/2][P]
    # Re(conj(c) h) = c_re h_re + c_im h_im, c_re = C[2k], c_im = C[2k+1]
    yref = (np.einsum("trk,tkp->trp", C[:, :, 0::2], ht.real)
            + np.einsum("trk,tkp->trp", C[:, :, 1::2], ht.imag) + D * x)
    close(y, yref, what="zero-input y")
    close(h, ht[-1], what="zero-input h_final")


def pin_lfilter_constant_params(lib):
    """Constant dt, lam, theta: every entry h[k][p] is the IIR filter
    h_t = a h_{t-1} + b u_{t-1} + g u_t, i.e. lfilter([g, b], [1, -a]) of
    u, with the initial condition (h_{-1} = h0, u_{-1} = carry) set by
    lfiltic.  Rank R = 3 so u sums three outer products."""
    rng = np.random.default_rng(2)
    L, R, P, N = 33, 3, 4, 6
    x, B, C, _, _, _ = _rand(rng, L, R, P, N)
    dt0, lam0, A, D = 0.31, 0.27, -0.9, -0.4
    th = rng.uniform(0, np.pi, N // 2)
    h0 = rng.standard_normal((N // 2, P)) + 1j * rng.standard_normal((N // 2, P))
    pB, px = rng.standard_normal((R, N)), rng.standard_normal((R, P))
    y, h, cB, cx = run1(lib, x, B, C, np.full(L, dt0), np.full(L, lam0), np.tile(th, (L, 1)), A, D,
                        h0=h0, pB=pB, px=px)
    u = np.einsum("trk,trp->tkp", cplx(B), x)
    u_prev = np.einsum("rk,rp->kp", cplx(pB), px)
    hs = np.zeros((L, N // 2, P), complex)
    for k in range(N // 2):
        a = np.exp(dt0 * (A + 1j * th[k]))
        bco = [lam0 * dt0, (1 - lam0) * dt0 * a]
        aco = [1.0, -a]
        for p in range(P):
            zi = scipy.signal.lfiltic(bco, aco, y=[h0[k, p]], x=[u_prev[k, p]])
            hs[:, k, p], _ = scipy.signal.lfilter(bco, aco, u[:, k, p], zi=zi)
    yref = np.einsum("trk,tkp->trp", np.conj(cplx(C)), hs).real + D * x
    close(h, hs[-1], what="lfilter h_final")
    close(y, yref, what="lfilter y")
    close(cB, B[-1], 0, "carry B")
    close(cx, x[-1], 0, "carry x")


def pin_constant_input_closed_form(lib):
    """Constant B, x, dt, lam, theta from a zero state without a carry:
    h_t = a^t g u + (b + g) u (1 - a^t)/(1 - a), b = (1-lam) dt a, g = lam dt."""
    rng = np.random.default_rng(3)
    L, R, P, N = 200, 1, 2, 4
    B1 = rng.standard_normal((R, N))
    x1 = rng.standard_normal((R, P))
    C1 = rng.standard_normal((R, N))
    dt0, lam0, A = 0.2, 0.6, -0.5
    th = np.array([0.3, 2.0])
    y, h, _, _ = run1(lib, np.tile(x1, (L, 1, 1)), np.tile(B1, (L, 1, 1)), np.tile(C1, (L, 1, 1)),
                      np.full(L, dt0), np.full(L, lam0), np.tile(th, (L, 1)), A, 0.0)
    a = np.exp(dt0 * (A + 1j * th))[:, None]
    g, b = lam0 * dt0, (1 - lam0) * dt0 * a
    u = np.einsum("rk,rp->kp", cplx(B1), x1)
    t = np.arange(L)[:, None, None]
    ht = a[None] ** t * g * u + (b + g) * u * (1 - a[None] ** t) / (1 - a)
    close(h, ht[-1], what="constant-input h")
    yref = np.einsum("rk,tkp->trp", np.conj(cplx(C1)), ht).real
    close(y, yref, what="constant-input y")


def pin_lambda_one_is_exponential_euler(lib):
    """lam = 1 gives b = 0 and g = dt: the first-order exponential-Euler rule
    h_t = a_t h_{t-1} + dt_t u_t.  So the carry cannot matter, and with
    constant dt, theta the state is lfilter([dt], [1, -a]) of u."""
    rng = np.random.default_rng(4)
    L, R, P, N = 25, 2, 3, 4
    x, B, C, dt, _, theta = _rand(rng, L, R, P, N)
    lam = np.ones(L)
    pB, px = rng.standard_normal((R, N)), rng.standard_normal((R, P))
    y1, h1, _, _ = run1(lib, x, B, C, dt, lam, theta, -0.6, 0.2, pB=pB, px=px)
    y0, h0, _, _ = run1(lib, x, B, C, dt, lam, theta, -0.6, 0.2)
    close(y1, y0, 1e-13, "lam=1 carry independence y")
    close(h1, h0, 1e-13, "lam=1 carry independence h")
    dt0, th = 0.4, theta[0]
    _, h2, _, _ = run1(lib, x, B, C, np.full(L, dt0), lam, np.tile(th, (L, 1)), -0.6, 0.2)
    u = np.einsum("trk,trp->tkp", cplx(B), x)
    for k in range(N // 2):
        a = np.exp(dt0 * (-0.6 + 1j * th[k]))
        ref = scipy.signal.lfilter([dt0], [1.0, -a], u[:, k, :], axis=0)
        close(h2[k], ref[-1], what="lam=1 Euler filter")


def brute_force(x, B, C, dt, lam, theta, A, D, h0, pB, px):
    """Unrolled sum, token by token, pure Python (tiny sizes only):
    h_t = Pi(0,t) (h0 + (1-lam_0) dt_0 u_{-1})
          + sum_{j<=t} Pi(j+1,t) w_tj u_j,  w_tt = lam_t dt_t,
            w_tj = lam_j dt_j + (1-lam_{j+1}) dt_{j+1}  (j < t),
    Pi(j,t) = prod_{s=j..t} exp(dt_s (A + i theta_s))."""
    L, R, P = x.shape
    K = B.shape[2] // 2
    Bh, Ch = cplx(B), cplx(C)
    ubar = [[sum(complex(cplx(pB)[r, k]) * px[r, p] for r in range(R)) for p in range(P)] for k in range(K)]
    u = [[[sum(complex(Bh[j, r, k]) * x[j, r, p] for r in range(R)) for p in range(P)]
          for k in range(K)] for j in range(L)]

    def Pi(j, t, k):
        acc = 1.0 + 0j
        for s in range(j, t + 1):
            acc *= np.exp(dt[s] * (A + 1j * theta[s, k]))
        return acc

    y = np.zeros((L, R, P))
    hs = np.zeros((L, K, P), complex)
    for t in range(L):
        for k in range(K):
            for p in range(P):
                v = Pi(0, t, k) * (h0[k, p] + (1 - lam[0]) * dt[0] * ubar[k][p])
                for j in range(t + 1):
                    w = lam[j] * dt[j] + ((1 - lam[j + 1]) * dt[j + 1] if j < t else 0.0)
                    v += Pi(j + 1, t, k) * w * u[j][k][p]
                hs[t, k, p] = v
        for r in range(R):
            for p in range(P):
                y[t, r, p] = sum((np.conj(Ch[t, r, k]) * hs[t, k, p]).real for k in range(K)) + D * x[t, r, p]
    return y, hs[-1]


def pin_brute_force_unrolled(lib):
    rng = np.random.default_rng(5)
    for (L, R, P, N) in [(1, 1, 2, 2), (7, 2, 2, 4), (16, 3, 2, 4)]:
        x, B, C, dt, lam, theta = _rand(rng, L, R, P, N)
        h0 = rng.standard_normal((N // 2, P)) + 1j * rng.standard_normal((N // 2, P))
        pB, px = rng.standard_normal((R, N)), rng.standard_normal((R, P))
        y, h, _, _ = run1(lib, x, B, C, dt, lam, theta, -0.8, 0.5, h0=h0, pB=pB, px=px)
        yref, href = brute_force(x, B, C, dt, lam, theta, -0.8, 0.5, h0, pB, px)
        close(y, yref, what=f"brute force y L={L}")
        close(h, href, what=f"brute force h L={L}")


def load_parity_fixture():
    bits, signs = None, None
    with open(os.path.join(GOLDEN, "parity_example.txt")) as f:
        for line in f:
            line = line.strip()
            if line.startswith("bits:"):
                bits = [int(c) for c in line.split(":", 1)[1].strip()]
            elif line.startswith("signs:"):
                signs = [1 if c == "+" else -1 for c in line.split(":", 1)[1].strip()]
    return np.array(bits), np.array(signs)


def pin_parity_example(lib):
    """A = 0, dt = 1, theta_t = pi * bit_t, x = 0, h0 = 1: each 1-bit turns
    the state by pi, so Re(h_t) = +1 or -1 with the parity of the bits read
    so far (fixture signs), whatever lam is.  Read through y with C = (1, 0)."""
    bits, signs = load_parity_fixture()
    L, R, P, N = len(bits), 1, 2, 4
    rng = np.random.default_rng(6)
    x = np.zeros((L, R, P))
    B = rng.standard_normal((L, R, N))
    C = np.zeros((L, R, N))
    C[:, :, 0::2] = 1.0
    theta = np.pi * np.tile(bits[:, None], (1, N // 2)).astype(float)
    y, h, _, _ = run1(lib, x, B, C, np.ones(L), rng.uniform(0, 1, L), theta, 0.0, 0.0,
                      h0=np.ones((N // 2, P), complex))
    got = np.sign(y[:, 0, 0])
    assert np.array_equal(got, signs), "parity signs differ from the fixture"
    close(y[:, 0, :], (N // 2) * signs[:, None] * np.ones((1, P)), 1e-12, "parity magnitude")


def pin_theta_zero_real_state(lib):
    """theta = 0: the N/2 complex pairs are N independent real states, so
    permuting the real components of B and C together leaves y unchanged
    (it does not when theta != 0 and the permutation crosses pairs)."""
    rng = np.random.default_rng(7)
    L, R, P, N = 30, 2, 3, 8
    x, B, C, dt, lam, _ = _rand(rng, L, R, P, N)
    perm = np.array([3, 6, 0, 5, 1, 7, 2, 4])
    th0 = np.zeros((L, N // 2))
    y1, _, _, _ = run1(lib, x, B, C, dt, lam, th0, -0.5, 0.1)
    y2, _, _, _ = run1(lib, x, B[:, :, perm], C[:, :, perm], dt, lam, th0, -0.5, 0.1)
    close(y1, y2, 1e-12, "theta=0 permutation invariance")
    th = rng.uniform(0.5, 2.5, (L, N // 2))
    y3, _, _, _ = run1(lib, x, B, C, dt, lam, th, -0.5, 0.1)
    y4, _, _, _ = run1(lib, x, B[:, :, perm], C[:, :, perm], dt, lam, th, -0.5, 0.1)
    assert np.max(np.abs(y3 - y4)) > 1e-3, "rotation should break the permutation invariance"


def pin_mimo_superposition(lib):
    """Rank R: the state is the sum of the R rank-1 (SISO) states driven by
    (B_r, x_r); output rank r' reads it with C_r' and adds D x_r'."""
    rng = np.random.default_rng(8)
    L, R, P, N = 24, 4, 3, 6
    x, B, C, dt, lam, theta = _rand(rng, L, R, P, N)
    pB, px = rng.standard_normal((R, N)), rng.standard_normal((R, P))
    A, D = -0.45, 0.8
    y, h, _, _ = run1(lib, x, B, C, dt, lam, theta, A, D, pB=pB, px=px)
    hsum = 0
    for r in range(R):
        _, hr, _, _ = run1(lib, x[:, r:r + 1], B[:, r:r + 1], C[:, :1], dt, lam, theta, A, 0.0,
                           pB=pB[r:r + 1], px=px[:, :][r:r + 1])
        hsum = hsum + hr
    close(h, hsum, what="superposition h")
    for r2 in range(R):
        yr = D * x[:, r2]
        for r in range(R):
            y_, _, _, _ = run1(lib, x[:, r:r + 1], B[:, r:r + 1], C[:, r2:r2 + 1], dt, lam, theta,
                               A, 0.0, pB=pB[r:r + 1], px=px[r:r + 1])
            yr = yr + y_[:, 0]
        close(y[:, r2], yr, what=f"superposition y rank {r2}")
    y1, h1, _, _ = run1(lib, x[:, :1], B[:, :1], C[:, :1], dt, lam, theta, A, D)
    assert y1.shape == (L, 1, P) and h1.shape == (N // 2, P)


def pin_split_and_carry(lib):
    """prefill(L) = prefill(L1) then prefill(L - L1) from the returned state
    and carry; the carry returned is the last token's (B, x)."""
    rng = np.random.default_rng(9)
    L, R, P, N = 40, 2, 3, 6
    x, B, C, dt, lam, theta = _rand(rng, L, R, P, N)
    y, h, cB, cx = run1(lib, x, B, C, dt, lam, theta, -0.3, 0.6)
    for L1 in (1, 17, 39):
        ya, ha, pBa, pxa = run1(lib, x[:L1], B[:L1], C[:L1], dt[:L1], lam[:L1], theta[:L1], -0.3, 0.6)
        yb, hb, cBb, cxb = run1(lib, x[L1:], B[L1:], C[L1:], dt[L1:], lam[L1:], theta[L1:], -0.3, 0.6,
                                h0=ha, pB=pBa, px=pxa)
        close(np.concatenate([ya, yb]), y, 1e-12, f"split y at {L1}")
        close(hb, h, 1e-12, f"split h at {L1}")
        close(cBb, cB, 0, "split carry B")
        close(cxb, cx, 0, "split carry x")


ALL_PINS = [
    pin_zero_input_closed_form,
    pin_lfilter_constant_params,
    pin_constant_input_closed_form,
    pin_lambda_one_is_exponential_euler,
    pin_brute_force_unrolled,
    pin_parity_example,
    pin_theta_zero_real_state,
    pin_mimo_superposition,
    pin_split_and_carry,
]


def _multi(rng, b, L, H, R, P, N):
    return dict(
        x=rng.standard_normal((b, L, H, R, P)), B=rng.standard_normal((b, L, H, R, N)),
        C=rng.standard_normal((b, L, H, R, N)),
        dt=np.log1p(np.exp(rng.standard_normal((b, L, H)) - 1)),
        lam=1 / (1 + np.exp(-rng.standard_normal((b, L, H)))),
        theta=rng.uniform(0, np.pi, (b, L, H, N // 2)),
        A=-np.exp(0.5 * rng.standard_normal(H)), D=rng.standard_normal(H))


def pin_prefill_then_decode(lib):
    """prefill(L) = prefill(L - k) then k single-token decode steps, with the
    decode inputs in step-major layout [T][b][H]..."""
    rng = np.random.default_rng(10)
    b, L, H, R, P, N, k = 2, 21, 3, 2, 3, 4, 6
    d = _multi(rng, b, L, H, R, P, N)
    kw = dict(H=H, P=P, N=N, R=R, dtype="f64", lib=lib, nthreads=2)
    y, h, cB, cx, _ = oracle.prefill(d, batch=b, L=L, **kw)
    head = {n: (v[:, :L - k] if v.ndim >= 3 else v) for n, v in d.items()}
    ya, ha, pBa, pxa, _ = oracle.prefill(head, batch=b, L=L - k, **kw)
    step = {n: (np.ascontiguousarray(np.moveaxis(v[:, L - k:], 1, 0)) if v.ndim >= 3 else v)
            for n, v in d.items()}
    step.update(h0=ha, prev_B=pBa, prev_x=pxa)
    yd, hd, cBd, cxd = oracle.decode(step, batch=b, steps=k, **kw)
    close(np.concatenate([ya, np.moveaxis(yd, 0, 1)], axis=1), y, 1e-12, "prefill+decode y")
    close(hd, h, 1e-12, "prefill+decode h")
    close(cBd, cB, 0, "prefill+decode carry B")
    close(cxd, cx, 0, "prefill+decode carry x")


def pin_varlen_equals_separate(lib):
    """A packed batch with cu_seqlens equals separate calls per sequence:
    the state and the carry start from zero at every sequence boundary."""
    rng = np.random.default_rng(11)
    lens = [5, 1, 9, 4]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, H, R, P, N = int(cu[-1]), 2, 2, 3, 4
    d = _multi(rng, 1, T, H, R, P, N)
    kw = dict(H=H, P=P, N=N, R=R, dtype="f64", lib=lib, nthreads=2)
    y, h, cB, cx, _ = oracle.prefill(d, batch=1, L=T, cu_seqlens=cu, **kw)
    for s, n in enumerate(lens):
        sub = {k: (v[:, cu[s]:cu[s + 1]] if v.ndim >= 3 else v) for k, v in d.items()}
        ys, hs, cBs, cxs, _ = oracle.prefill(sub, batch=1, L=n, **kw)
        close(y[:, cu[s]:cu[s + 1]], ys, 1e-13, f"varlen y seq {s}")
        close(h[s * H:(s + 1) * H], hs, 1e-13, f"varlen h seq {s}")
        close(cB[s * H:(s + 1) * H], cBs, 0, f"varlen carry seq {s}")


ALL_PINS += [pin_prefill_then_decode, pin_varlen_equals_separate]
