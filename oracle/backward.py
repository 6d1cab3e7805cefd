"""Backward pass of the scan for training (test infrastructure, like the
rest of this package): the exact gradient of the oracle's forward pass.

The pages train the models but describe no backward kernel ("Together AI
announces Mamba-3", sections 1-3 give the forward recurrence); this is the
adjoint of that recurrence, written out step by step in complex double, per
(sequence, head) unit and token by token, for small parity cases.

Forward, per unit (pairs k, columns p, ranks r):
    a_t = exp(dt_t (A + i theta_t)),  beta'_t = (1 - lam_t) dt_t,  gamma_t = lam_t dt_t
    u_t = sum_r Bhat_t[r] x_t[r]^T
    s_t = h_{t-1} + beta'_t u_{t-1}          (h_{-1} = h0, u_{-1} from the carry)
    h_t = a_t s_t + gamma_t u_t
    y_t[r] = Re(conj(Chat_t[r]) h_t) + D x_t[r]
Gradients of a real loss with respect to a complex quantity z are kept as
G_z = dL/dRe z + i dL/dIm z; then for w = c z, G_z = conj(c) G_w, and for
a = exp(z), G_z = conj(a) G_a.  Going backwards through the tokens:
    G_h(t) = sum_r dy_t[r] Chat_t[r] + G_s(t+1)      (G_s(T) = dL/dh_final)
    G_s(t) = conj(a_t) G_h(t)
    G_a(t) = sum_p G_h(t) conj(s_t),  G_z(t) = conj(a_t) G_a(t)
    G_u(t) = gamma_t G_h(t) + beta'_{t+1} G_s(t+1)
    dgamma_t = Re sum G_h(t) conj(u_t),  dbeta'_t = Re sum G_s(t) conj(u_{t-1})
and the chain to the inputs: dt through Re G_z A + Im G_z theta and the two
weights, lam through the two weights, theta_k through dt Im G_z, A through
dt Re G_z, B from G_u x, x from Re(G_u conj(Bhat)) plus D dy, C from dy h,
D from dy x, the carry from G_u(-1) and h0 from G_s(0).
"""
from __future__ import annotations

import numpy as np


def _pairs(v):
    """[..., N] real with (re, im) interleaved -> [..., N/2] complex."""
    return v[..., 0::2] + 1j * v[..., 1::2]


def _unpairs(z):
    """[..., K] complex -> [..., 2K] real, (re, im) interleaved."""
    out = np.empty(z.shape[:-1] + (2 * z.shape[-1],))
    out[..., 0::2] = z.real
    out[..., 1::2] = z.imag
    return out


def unit_backward(x, B, C, dt, lam, theta, A, D, h0, prev_B, prev_x, dy, dh_final=None):
    """One unit, all arrays float64: x [T][R][P], B/C [T][R][N], dt/lam [T],
    theta [T][N/2], A/D scalars, h0 [N/2][P] complex, prev_B [R][N],
    prev_x [R][P], dy [T][R][P], dh_final [N/2][P] complex or None.
    Returns (y, h_final, grads) with grads a dict of the same shapes."""
    T = len(dt)
    Bc, Cc = _pairs(B), _pairs(C)                    # [T][R][K]
    a = np.exp(dt[:, None] * (A + 1j * theta))       # [T][K]
    bet, gam = (1.0 - lam) * dt, lam * dt
    u = np.einsum("trk,trp->tkp", Bc, x)             # [T][K][P]
    u_m1 = np.einsum("rk,rp->kp", _pairs(prev_B), prev_x)
    s = np.empty_like(u)
    hs = np.empty_like(u)
    h = np.asarray(h0, complex)
    for t in range(T):
        s[t] = h + bet[t] * (u[t - 1] if t else u_m1)
        h = a[t][:, None] * s[t] + gam[t] * u[t]
        hs[t] = h
    y = np.einsum("trk,tkp->trp", np.conj(Cc), hs).real + D * x

    g = {k: np.zeros_like(v) for k, v in (("x", x), ("B", B), ("C", C), ("dt", dt), ("lam", lam),
                                          ("theta", theta), ("prev_B", prev_B), ("prev_x", prev_x))}
    dA = 0.0
    dD = float(np.sum(dy * x))
    gx = D * dy
    Gs_next = np.zeros_like(h) if dh_final is None else np.asarray(dh_final, complex)
    Gu = np.zeros_like(u)
    for t in range(T - 1, -1, -1):
        Gh = np.einsum("rp,rk->kp", dy[t], Cc[t]) + Gs_next
        Gs = np.conj(a[t])[:, None] * Gh
        Ga = np.sum(Gh * np.conj(s[t]), axis=1)      # [K]
        Gz = np.conj(a[t]) * Ga
        Gu[t] += gam[t] * Gh
        dgam = np.sum(Gh * np.conj(u[t])).real
        u_prev = u[t - 1] if t else u_m1
        dbet = np.sum(Gs * np.conj(u_prev)).real
        if t:
            Gu[t - 1] += bet[t] * Gs
        else:
            Gu_m1 = bet[0] * Gs
        g["dt"][t] = np.sum(Gz.real) * A + np.sum(Gz.imag * theta[t]) + (1.0 - lam[t]) * dbet + lam[t] * dgam
        g["lam"][t] = -dt[t] * dbet + dt[t] * dgam
        g["theta"][t] = dt[t] * Gz.imag
        dA += dt[t] * np.sum(Gz.real)
        g["C"][t] = _unpairs(np.einsum("rp,kp->rk", dy[t], hs[t]))
        Gs_next = Gs
    dh0 = Gs_next
    # u_t = sum_r Bhat_t[r] x_t[r]^T
    g["B"] = _unpairs(np.einsum("tkp,trp->trk", Gu, x))
    g["x"] = gx + np.einsum("tkp,trk->trp", Gu, np.conj(Bc)).real
    g["prev_B"] = _unpairs(np.einsum("kp,rp->rk", Gu_m1, prev_x))
    g["prev_x"] = np.einsum("kp,rk->rp", Gu_m1, np.conj(_pairs(prev_B))).real
    g["A"], g["D"], g["h0"] = dA, dD, dh0
    return y, hs[-1], g


def _sigmoid(z):
    return 0.5 * (1.0 + np.tanh(0.5 * z))


def _rms_norm_backward(v, dn, eps):
    """Gradient through n = v / sqrt(mean(v^2) + eps) (rows on the last
    axis): with s = (mean(v^2) + eps)^(-1/2), dn_i/dv_j = s delta_ij -
    s^3 v_i v_j / N, so dv = s (dn - n mean(dn * n))."""
    v = np.asarray(v, np.float64)
    s = 1.0 / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps)
    n = v * s
    return s * (dn - n * np.mean(dn * n, axis=-1, keepdims=True))


def prologue_backward(inp: dict, grads: dict, dtype: str, *, dt_softplus=False, bc_norm=False, dt_bias=None):
    """Chain the gradients with respect to the scan's inputs (after the
    fused prologue) back to the raw inputs the caller passed: dt through
    softplus(dt + dt_bias[h]) (derivative sigmoid), B, C and the carried
    prev_B through the RMS norm of each row.  Adds "dt_bias" (summed over
    batch and tokens per head).  ``inp`` holds the raw inputs."""
    from . import BC_NORM_EPS, _widen

    g = dict(grads)
    if dt_softplus:
        bias = np.zeros(np.shape(inp["dt"])[-1]) if dt_bias is None else np.asarray(dt_bias, np.float64)
        z = _widen(inp["dt"], dtype) + bias
        g["dt"] = grads["dt"] * _sigmoid(z)
        g["dt_bias"] = g["dt"].reshape(-1, z.shape[-1]).sum(axis=0)
    if bc_norm:
        for k in ("B", "C", "prev_B"):
            if inp.get(k) is not None:
                g[k] = _rms_norm_backward(_widen(inp[k], dtype), grads[k], BC_NORM_EPS)
    return g


def prefill_backward(inp: dict, dy, *, batch, L, H, P, N, R, dtype, h0=None, prev_B=None, prev_x=None,
                     dh_final=None, dt_softplus=False, bc_norm=False, dt_bias=None):
    """See _prefill_backward.  With dt_softplus / bc_norm the inputs are raw
    (the fused prologue applies softplus(dt + dt_bias) and the RMS norm of
    B, C and prev_B rows, as the library's prologue flags do) and the
    gradients are with respect to them (plus "dt_bias")."""
    if not (dt_softplus or bc_norm):
        return _prefill_backward(inp, dy, batch=batch, L=L, H=H, P=P, N=N, R=R, dtype=dtype, h0=h0,
                                 prev_B=prev_B, prev_x=prev_x, dh_final=dh_final)
    from . import _widen, apply_prologue

    raw = dict(inp, prev_B=prev_B)
    post = apply_prologue(raw, dtype, dt_softplus=dt_softplus, bc_norm=bc_norm, dt_bias=dt_bias)
    y, hf, grads = _prefill_backward(post, dy, batch=batch, L=L, H=H, P=P, N=N, R=R, dtype="f64", h0=h0,
                                     prev_B=post["prev_B"], prev_x=None if prev_x is None else _widen(prev_x, dtype),
                                     dh_final=dh_final)
    return y, hf, prologue_backward(raw, grads, dtype, dt_softplus=dt_softplus, bc_norm=bc_norm, dt_bias=dt_bias)


def _prefill_backward(inp: dict, dy, *, batch, L, H, P, N, R, dtype, h0=None, prev_B=None, prev_x=None,
                      dh_final=None):
    """Gradients of sum(dy * y) + sum(dh_final * h_final) for a fixed-length
    batch (the oracle's layouts: x [b][L][H][R][P], B/C [b][L][G][R][N],
    dt/lam [b][L][H], theta [b][L][H][N/2], A/D [H]; h0 [b][H][N/2][P][2],
    prev_B [b][H][R][N], prev_x [b][H][R][P]; dh_final like h0).  lam and
    theta given as None are 1 and 0.  Returns (y, h_final, grads): grads
    holds an array like each input (dB and dC summed over the heads of a
    group, dA and dD over batch and tokens)."""
    from . import _widen

    K = N // 2
    w = {k: (None if inp.get(k) is None else _widen(inp[k], dtype)) for k in ("x", "B", "C", "dt", "lam", "theta")}
    if w["lam"] is None:
        w["lam"] = np.ones_like(w["dt"])
    if w["theta"] is None:
        w["theta"] = np.zeros(w["dt"].shape + (K,))
    G = w["B"].shape[2]
    A = np.asarray(inp["A"], np.float64)
    D = np.asarray(inp["D"], np.float64)
    h0c = np.zeros((batch, H, K, P), complex) if h0 is None else \
        np.asarray(h0, np.float64)[..., 0] + 1j * np.asarray(h0, np.float64)[..., 1]
    pB = np.zeros((batch, H, R, N)) if prev_B is None else _widen(prev_B, dtype)
    px = np.zeros((batch, H, R, P)) if prev_x is None else _widen(prev_x, dtype)
    dy = np.asarray(dy, np.float64)
    y = np.zeros((batch, L, H, R, P))
    hf = np.zeros((batch, H, K, P, 2))
    grads = {"x": np.zeros_like(w["x"]), "B": np.zeros_like(w["B"]), "C": np.zeros_like(w["C"]),
             "dt": np.zeros_like(w["dt"]), "lam": np.zeros_like(w["lam"]), "theta": np.zeros_like(w["theta"]),
             "A": np.zeros(H), "D": np.zeros(H), "h0": np.zeros((batch, H, K, P, 2)),
             "prev_B": np.zeros_like(pB), "prev_x": np.zeros_like(px)}
    for b in range(batch):
        for hd in range(H):
            gi = hd // (H // G)
            dhf = None if dh_final is None else \
                np.asarray(dh_final, np.float64)[b, hd, ..., 0] + 1j * np.asarray(dh_final, np.float64)[b, hd, ..., 1]
            yu, hu, g = unit_backward(w["x"][b, :, hd], w["B"][b, :, gi], w["C"][b, :, gi], w["dt"][b, :, hd],
                                      w["lam"][b, :, hd], w["theta"][b, :, hd], A[hd], D[hd], h0c[b, hd],
                                      pB[b, hd], px[b, hd], dy[b, :, hd], dhf)
            y[b, :, hd] = yu
            hf[b, hd, ..., 0], hf[b, hd, ..., 1] = hu.real, hu.imag
            grads["x"][b, :, hd] = g["x"]
            grads["B"][b, :, gi] += g["B"]
            grads["C"][b, :, gi] += g["C"]
            grads["dt"][b, :, hd] = g["dt"]
            grads["lam"][b, :, hd] = g["lam"]
            grads["theta"][b, :, hd] = g["theta"]
            grads["A"][hd] += g["A"]
            grads["D"][hd] += g["D"]
            grads["h0"][b, hd, ..., 0], grads["h0"][b, hd, ..., 1] = g["h0"].real, g["h0"].imag
            grads["prev_B"][b, hd] = g["prev_B"]
            grads["prev_x"][b, hd] = g["prev_x"]
    return y, hf, grads
