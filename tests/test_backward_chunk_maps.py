"""The chunk maps of the adjoint recurrence (CPU only, fp64).

The backward of the recurrence can run chunk-parallel over the tokens: its
adjoint state is (dS, dA, dn), and over a chunk of tokens each part is an
affine function of its value at the chunk's end:
  - dn: the identity plus the chunk's sum of dden_t phi(q_t);
  - dS: dS_start = dS_end Phi_c + Psi_c, Phi_c the product of the chunk's
    transitions (I - alpha_t k_hat_t^T) of section 3.1 ("Variational Linear
    Attention: Stable Associative Memory for Long-Context Transformers"),
    Psi_c the chunk's readout terms carried to its start;
  - dA: only its symmetric part feeds back (the gradients read dA through
    z^T dA z and (dA + dA^T) z), and that part moves two-sided,
    X_{t-1} = K_t (X_t + sym(dg_t k_hat_t^T)) K_t^T with K_t = I - beta_t u_t z_t^T,
    so Xs_start = Q_c Xs_end Q_c^T + Omega_c with Q_c = K_first .. K_last;
    the antisymmetric part of dA0 is a plain sum over the tokens.
This file writes that chunked backward out with plain NumPy (fp64) and checks
it against the autograd oracle for several chunk lengths, ragged ones
included: the identities a chunk-parallel backward kernel implements."""

import numpy as np
import pytest

from oracle import backward as ob
from synthetic import normals

EPS = 1e-6


def _phi(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def _dphi(x):
    return np.where(x > 0, 1.0, np.exp(np.minimum(x, 0.0)))


def _sym(X):
    return 0.5 * (X + X.T)


def _asym(X):
    return 0.5 * (X - X.T)


def _records(q, k, v, u, S0, A0, n0):
    """Token-by-token forward of one unit, keeping what the adjoint reads."""
    S, A, n = S0.copy(), A0.copy(), n0.copy()
    rec = []
    for t in range(q.shape[0]):
        kn = np.linalg.norm(k[t])
        kh = k[t] / max(kn, EPS)
        z = A @ u[t]
        beta = 1.0 / (1.0 + u[t] @ z)
        A_prev, A = A, A - beta * np.outer(z, z)
        g = A @ kh
        gn = np.linalg.norm(g)
        al = g / max(gn, EPS)
        S_prev, r = S, v[t] - S @ kh
        S = S + np.outer(r, al)
        n = n + _phi(kh)
        fq = _phi(q[t])
        den = fq @ n + EPS
        rec.append(dict(kh=kh, kn=kn, z=z, beta=beta, gn=gn, al=al, r=r, fq=fq, n=n.copy(), den=den,
                        o=S @ fq / den, S=S.copy(), S_prev=S_prev, A=A.copy(), A_prev=A_prev, q=q[t], u=u[t]))
    return rec


def chunked_backward(q, k, v, u, dO, dS_T, dA_T, dn_T, S0, A0, n0, m):
    T, d = q.shape
    R = _records(q, k, v, u, S0, A0, n0)
    chunks = [range(c, min(T, c + m)) for c in range(0, T, m)]
    I = np.eye(d)
    dden = [-(dO[t] @ R[t]["o"]) / R[t]["den"] for t in range(T)]
    K = [I - R[t]["beta"] * np.outer(R[t]["u"], R[t]["z"]) for t in range(T)]

    # per chunk, from the records alone: dn sums; dS maps (Phi, Psi); Q
    dn_sum, Phi, Psi, Q = [], [], [], []
    for ch in chunks:
        P, H, Qc = I.copy(), np.zeros((d, d)), I.copy()
        for t in reversed(ch):
            H = H + np.outer(dO[t] / R[t]["den"], R[t]["fq"])
            H = H - np.outer(H @ R[t]["al"], R[t]["kh"])
            P = P - np.outer(P @ R[t]["al"], R[t]["kh"])
            Qc = K[t] @ Qc
        dn_sum.append(sum(dden[t] * R[t]["fq"] for t in ch))
        Phi.append(P)
        Psi.append(H)
        Q.append(Qc)
    # chains along the chunks (from the last): dS, dn at every chunk's end
    dS_end, dn_end = [None] * len(chunks), [None] * len(chunks)
    D, dn = dS_T.copy(), dn_T.copy()
    for c in reversed(range(len(chunks))):
        dS_end[c], dn_end[c] = D.copy(), dn.copy()
        D, dn = D @ Phi[c] + Psi[c], dn + dn_sum[c]
    dS0, dn0 = D, dn

    # per chunk with the exact dS: the S part, the gate terms dg, and Omega
    dq, dv, dkh, dg = (np.zeros_like(q) for _ in range(4))
    Om = []
    for c, ch in enumerate(chunks):
        D, dn = dS_end[c].copy(), dn_end[c].copy()
        for t in reversed(ch):
            Rt = R[t]
            dnum = dO[t] / Rt["den"]
            D = D + np.outer(dnum, Rt["fq"])
            dq[t] = (Rt["S"].T @ dnum + dden[t] * Rt["n"]) * _dphi(Rt["q"])
            dn = dn + dden[t] * Rt["fq"]
            dr = D @ Rt["al"]
            dv[t] = dr
            dal = D.T @ Rt["r"]
            D = D - np.outer(dr, Rt["kh"])
            dkh[t] = -Rt["S_prev"].T @ dr + dn * _dphi(Rt["kh"])
            dg[t] = (dal - Rt["al"] * (Rt["al"] @ dal)) / Rt["gn"]
        X = np.zeros((d, d))
        for t in reversed(ch):
            X = K[t] @ (X + _sym(np.outer(dg[t], R[t]["kh"]))) @ K[t].T
        Om.append(X)
    Xs_end = [None] * len(chunks)
    X = _sym(dA_T)
    for c in reversed(range(len(chunks))):
        Xs_end[c] = X.copy()
        X = Q[c] @ X @ Q[c].T + Om[c]
    dA0 = X + _asym(dA_T)

    # per chunk with the exact symmetric dA: dz, du, dk; the antisymmetric sum
    du, dk = np.zeros_like(q), np.zeros_like(q)
    for c, ch in enumerate(chunks):
        X = Xs_end[c].copy()
        for t in reversed(ch):
            Rt = R[t]
            Xp = X + _sym(np.outer(dg[t], Rt["kh"]))
            ds1 = Rt["beta"] ** 2 * (Rt["z"] @ Xp @ Rt["z"])
            dz = -2.0 * Rt["beta"] * (Xp @ Rt["z"]) + ds1 * Rt["u"]
            du[t] = ds1 * Rt["z"] + Rt["A_prev"] @ dz
            dA0 = dA0 + _asym(np.outer(dg[t], Rt["kh"]) + np.outer(dz, Rt["u"]))
            X = K[t] @ Xp @ K[t].T
            dkt = dkh[t] + Rt["A"] @ dg[t]
            dk[t] = (dkt - Rt["kh"] * (Rt["kh"] @ dkt)) / Rt["kn"]
    return dict(dq=dq, dk=dk, dv=dv, du=du, dS0=dS0, dA0=dA0, dn0=dn0)


@pytest.mark.parametrize("T,d,m", [(50, 4, 8), (64, 6, 16), (37, 5, 37), (40, 4, 1), (33, 8, 7)])
def test_chunked_adjoint_equals_the_oracle(T, d, m):
    seed = 700 + T + d + m
    g = lambda stream, shape, s=1.0: s * normals(seed, stream, int(np.prod(shape))).reshape(shape)  # noqa: E731
    q, k, v, dO = g(1, (T, d)), g(2, (T, d)), g(3, (T, d)), g(4, (T, d))
    u = g(5, (T, d), 0.5)
    dS_T, dA_T, dn_T = g(6, (d, d)), g(7, (d, d)), g(8, (d,))
    S0 = g(9, (d, d), 0.3)
    B = g(10, (d, d))
    A0 = np.linalg.inv(0.8 * np.eye(d) + 0.1 * B @ B.T)
    n0 = np.abs(g(11, (d,)))
    ref = ob.backward(q, k, v, u, 0.8, dO, dS_T=dS_T, dA_T=dA_T, dn_T=dn_T, S0=S0, A0=A0, n0=n0)
    got = chunked_backward(q, k, v, u, dO, dS_T, dA_T, dn_T, S0, A0, n0, m)
    for key, val in got.items():
        want = np.asarray(ref[key]).reshape(val.shape)
        err = np.linalg.norm(val - want) / np.linalg.norm(want)
        assert err < 1e-12, (key, err)
