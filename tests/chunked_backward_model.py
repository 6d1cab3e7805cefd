"""A double-precision model of the chunked backward algorithm (test
infrastructure: the plan a tensor-core backward kernel follows, checked
against the oracle's token-by-token adjoint in tests/test_chunked_backward_model.py).

It uses the forward kernel's formulation per (sequence, head) unit:
rotated operands Bt = Bhat e^{-i Phi}, Ct = Chat e^{-i Phi} (Phi the running
phase from the sequence start), per chunk the masked weights
M_tj = Re(Ct_t^H Bt_j) e^{Lam_t - Lam_j} w_tj (w_tj = wp_j = gamma_j +
beta'_{j+1} for j < t, gamma_t on the diagonal, Lam the chunk-local sum of
dt A), the inter-chunk output e^{Lam_t} Re(Ct_t^H G'), and the state in
the rotating frame G' <- e^{Lam_end} G' + sum_j e^{Lam_end - Lam_j} wp_j
Bt_j x_j^T (h_final = e^{i Phi_end} G').  The backward walks the chunks in
reverse with the adjoint of G' and needs, per chunk, the forward's
contractions transposed (dY X^T, M^T dY, dS Bt, dS^T Ct, the state terms),
plus row and column sums of dM * M for the decay and per-token sums of
Im(conj(dBt) Bt) + Im(conj(dCt) Ct) for the phase.  Complex gradients are
kept as G_z = dL/dRe z + i dL/dIm z.
"""
import numpy as np


def _pairs(v):
    return v[..., 0::2] + 1j * v[..., 1::2]


def _unpairs(z):
    out = np.empty(z.shape[:-1] + (2 * z.shape[-1],))
    out[..., 0::2] = z.real
    out[..., 1::2] = z.imag
    return out


def chunked_unit_backward(x, B, C, dt, lam, theta, A, D, h0, prev_B, prev_x, dy, dh_final, Q):
    """Same arguments as oracle.unit_backward plus the chunk length Q."""
    T = len(dt)
    Bh, Ch = _pairs(B), _pairs(C)                      # [T][R][K]
    gam, bet = lam * dt, (1.0 - lam) * dt
    wp = gam + np.append(bet[1:], 0.0)                 # gamma_j + beta'_{j+1}
    Phi = np.cumsum(dt[:, None] * theta, axis=0)       # [T][K]
    rho = np.exp(1j * Phi)
    Bt, Ct = Bh * np.conj(rho)[:, None, :], Ch * np.conj(rho)[:, None, :]
    u_m1 = np.einsum("rk,rp->kp", _pairs(prev_B), prev_x)
    chunks = [(c0, min(c0 + Q, T)) for c0 in range(0, T, Q)]

    def chunk_terms(c0, c1):
        n = c1 - c0
        Lam = np.cumsum(dt[c0:c1] * A)
        ii = np.arange(n)
        low = ii[:, None] >= ii[None, :]
        E = np.where(low, np.exp(np.where(low, Lam[:, None] - Lam[None, :], 0.0)), 0.0)
        W = np.where(ii[:, None] > ii[None, :], wp[c0:c1][None, :], 0.0) + np.diag(gam[c0:c1])
        S = np.einsum("trk,jsk->trjs", np.conj(Ct[c0:c1]), Bt[c0:c1]).real
        return Lam, ii, E, W, S

    # forward: keep the state at each chunk start
    G = np.asarray(h0, complex) + bet[0] * u_m1       # G'_{-1}: phase 0 before the first token
    G_start, y = [], np.zeros_like(x)
    for c0, c1 in chunks:
        G_start.append(G)
        Lam, ii, E, W, S = chunk_terms(c0, c1)
        M = S * (E * W)[:, None, :, None]
        y[c0:c1] = (np.einsum("trjs,jsp->trp", M, x[c0:c1])
                    + np.exp(Lam)[:, None, None] * np.einsum("trk,kp->trp", np.conj(Ct[c0:c1]), G).real
                    + D * x[c0:c1])
        f = np.exp(Lam[-1] - Lam) * wp[c0:c1]
        G = np.exp(Lam[-1]) * G + np.einsum("j,jrk,jrp->kp", f, Bt[c0:c1], x[c0:c1])
    h_final = rho[-1][:, None] * G

    # backward
    dBt, dCt = np.zeros_like(Bt), np.zeros_like(Ct)
    dx = D * dy
    dPhi = np.zeros_like(Phi)
    ddt, dA = np.zeros(T), 0.0
    dwp, dgam, dbet = np.zeros(T), np.zeros(T), np.zeros(T)
    dhf = np.zeros_like(h_final) if dh_final is None else np.asarray(dh_final, complex)
    dG = np.conj(rho[-1])[:, None] * dhf               # h_final = e^{i Phi_end} G'
    dPhi[-1] += -np.sum(np.imag(np.conj(dhf) * h_final), axis=1)
    for (c0, c1), Gs in reversed(list(zip(chunks, G_start))):
        Lam, ii, E, W, S = chunk_terms(c0, c1)
        dLam = np.zeros(c1 - c0)
        # state: G_end = e^{Lam_end} Gs + sum_j f_j Bt_j x_j^T
        V = np.einsum("jrk,jrp->jkp", Bt[c0:c1], x[c0:c1])
        f = np.exp(Lam[-1] - Lam) * wp[c0:c1]
        q = np.real(np.sum(np.conj(dG)[None] * V, axis=(1, 2)))
        dwp[c0:c1] += np.exp(Lam[-1] - Lam) * q
        dLam[-1] += np.real(np.sum(np.conj(dG) * np.exp(Lam[-1]) * Gs)) + np.sum(f * q)
        dLam -= f * q
        dBt[c0:c1] += f[:, None, None] * np.einsum("kp,jrp->jrk", dG, x[c0:c1])
        dx[c0:c1] += f[:, None, None] * np.real(np.einsum("jrk,kp->jrp", np.conj(Bt[c0:c1]), dG))
        dGs = np.exp(Lam[-1]) * dG
        # inter-chunk output: e^{Lam_t} Re(Ct_t^H Gs)
        eL = np.exp(Lam)
        Yi = np.real(np.einsum("trk,kp->trp", np.conj(Ct[c0:c1]), Gs))
        dLam += eL * np.sum(dy[c0:c1] * Yi, axis=(1, 2))
        dCt[c0:c1] += eL[:, None, None] * np.einsum("trp,kp->trk", dy[c0:c1], Gs)
        dGs += np.einsum("t,trp,trk->kp", eL, dy[c0:c1], Ct[c0:c1])
        # intra-chunk output: sum_j M_tj x_j, M = S * E * W
        EW = E * W
        M = S * EW[:, None, :, None]
        dM = np.einsum("trp,jsp->trjs", dy[c0:c1], x[c0:c1])
        dx[c0:c1] += np.einsum("trjs,trp->jsp", M, dy[c0:c1])
        dS = dM * EW[:, None, :, None]
        dEW = np.sum(dM * S, axis=(1, 3))
        dLam += np.sum(dEW * EW, axis=1) - np.sum(dEW * EW, axis=0)
        dwp[c0:c1] += np.sum(np.where(ii[:, None] > ii[None, :], dEW * E, 0.0), axis=0)
        dgam[c0:c1] += np.diag(dEW)
        dCt[c0:c1] += np.einsum("trjs,jsk->trk", dS, Bt[c0:c1])
        dBt[c0:c1] += np.einsum("trjs,trk->jsk", dS, Ct[c0:c1])
        # Lam_i = sum_{m <= i} dt_m A inside the chunk
        rc = np.cumsum(dLam[::-1])[::-1]
        ddt[c0:c1] += A * rc
        dA += float(np.sum(dt[c0:c1] * rc))
        dG = dGs
    # G'_{-1} = h0 + beta'_0 u_{-1}
    dh0 = dG
    du_m1 = bet[0] * dG
    dbet[0] += np.real(np.sum(np.conj(dG) * u_m1))
    # the rotation e^{-i Phi} of B and C, and Phi = running sum of dt theta
    dPhi += np.sum(np.imag(np.conj(dBt) * Bt) + np.imag(np.conj(dCt) * Ct), axis=1)
    rcPhi = np.cumsum(dPhi[::-1], axis=0)[::-1]
    ddt += np.sum(theta * rcPhi, axis=1)
    dtheta = dt[:, None] * rcPhi
    dBh, dCh = rho[:, None, :] * dBt, rho[:, None, :] * dCt
    # wp_j = gamma_j + beta'_{j+1}; gamma = lam dt, beta' = (1 - lam) dt
    dgam += dwp
    dbet[1:] += dwp[:-1]
    ddt += lam * dgam + (1.0 - lam) * dbet
    dlam = dt * dgam - dt * dbet
    g = dict(x=dx, B=_unpairs(dBh), C=_unpairs(dCh), dt=ddt, lam=dlam, theta=dtheta, A=dA,
             D=float(np.sum(dy * x)), h0=dh0,
             prev_B=_unpairs(np.einsum("kp,rp->rk", du_m1, prev_x)),
             prev_x=np.real(np.einsum("kp,rk->rp", du_m1, np.conj(_pairs(prev_B)))))
    return y, h_final, g
