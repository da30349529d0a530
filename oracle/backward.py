"""fp64 CPU oracle for the gradients of the VLA forward recurrence.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``).  The forward pass
is written out with plain PyTorch CPU ops in fp64, token by token, in the
order of "Variational Linear Attention: Stable Associative Memory for
Long-Context Transformers", sections 2.2-2.3 (same readings as the C
oracle: z_t = A_{t-1} u_t, A_0 = I / lambda0, eps = 1e-6, ELU+1 readout
o_t = S_t phi(q_t) / (phi(q_t)^T n_t + eps)).  The gradients are those of
PyTorch's autograd through that literal forward; ``tests/test_backward_pins.py``
pins them against central finite differences and the forward against the C
oracle.

The loss whose gradients are returned is
    L = sum_t <dO_t, o_t> + <dS_T, S_T> + <dA_T, A_T> + <dn_T, n_T>
(each upstream term optional).  At ||k|| <= eps or ||g|| <= eps the
max(., eps) guards contribute the gradient of the constant branch.
"""

from __future__ import annotations

import numpy as np
import torch

EPS = 1e-6


def _phi(x):
    # ELU(x) + 1: x + 1 for x > 0, exp(x) otherwise (section 2.3)
    return torch.where(x > 0, x + 1.0, torch.exp(torch.clamp(x, max=0.0)))


def forward_torch(q, k, v, u, lambda0: float, S0=None, A0=None, n0=None):
    """Literal recurrence on [N, T, d] fp64 tensors (N independent units).

    Returns o [N, T, d], S_T, A_T [N, d, d], n_T [N, d]."""
    N, T, d = q.shape
    dt = q.dtype
    eye = torch.eye(d, dtype=dt).expand(N, d, d)
    A = A0 if A0 is not None else eye / lambda0
    S = S0 if S0 is not None else torch.zeros(N, d, d, dtype=dt)
    n = n0 if n0 is not None else torch.zeros(N, d, dtype=dt)
    outs = []
    for t in range(T):
        kt, ut, vt, qt = k[:, t], u[:, t], v[:, t], q[:, t]
        kn = torch.linalg.vector_norm(kt, dim=-1, keepdim=True)
        khat = kt / torch.clamp(kn, min=EPS)
        # step 1: A_t = A_{t-1} - z z^T / (1 + u^T z), z = A_{t-1} u
        z = torch.einsum("nij,nj->ni", A, ut)
        den = 1.0 + (ut * z).sum(-1)
        A = A - torch.einsum("ni,nj->nij", z, z) / den[:, None, None]
        # step 2: alpha = A_t k_hat / |A_t k_hat|
        g = torch.einsum("nij,nj->ni", A, khat)
        gn = torch.linalg.vector_norm(g, dim=-1, keepdim=True)
        alpha = g / torch.clamp(gn, min=EPS)
        # step 3: S_t = S_{t-1} + (v - S_{t-1} k_hat) alpha^T
        r = vt - torch.einsum("nij,nj->ni", S, khat)
        S = S + torch.einsum("ni,nj->nij", r, alpha)
        # readout
        n = n + _phi(khat)
        fq = _phi(qt)
        num = torch.einsum("nij,nj->ni", S, fq)
        rden = (fq * n).sum(-1, keepdim=True) + EPS
        outs.append(num / rden)
    return torch.stack(outs, dim=1), S, A, n


def backward(q, k, v, u, lambda0: float, dO, dS_T=None, dA_T=None, dn_T=None, S0=None, A0=None,
             n0=None) -> dict:
    """Gradients in fp64 of the loss above.

    Array arguments are ``[..., T, d]`` (q, k, v, u, dO) and ``[..., d, d]`` /
    ``[..., d]`` (states); any float dtype (widened exactly).  Returns numpy
    arrays dq, dk, dv, du (shape of q), dS0, dA0 ([..., d, d]) and dn0
    ([..., d]), plus the forward outputs o, S_T, A_T, n_T.
    """
    q = np.asarray(q)
    lead = q.shape[:-2]
    T, d = q.shape[-2:]
    N = int(np.prod(lead)) if lead else 1

    def t64(a, shape, grad=True):
        x = torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.float64)).reshape(shape))
        return x.requires_grad_(grad)

    tok = (N, T, d)
    qt, kt, vt, ut = (t64(a, tok) for a in (q, k, v, u))
    S0t = t64(S0, (N, d, d)) if S0 is not None else torch.zeros(N, d, d, dtype=torch.float64, requires_grad=True)
    A0t = t64(A0, (N, d, d)) if A0 is not None else (
        torch.eye(d, dtype=torch.float64).expand(N, d, d) / lambda0).clone().requires_grad_(True)
    n0t = t64(n0, (N, d)) if n0 is not None else torch.zeros(N, d, dtype=torch.float64, requires_grad=True)
    o, S, A, n = forward_torch(qt, kt, vt, ut, lambda0, S0t, A0t, n0t)
    loss = (o * t64(dO, tok, False)).sum()
    if dS_T is not None:
        loss = loss + (S * t64(dS_T, (N, d, d), False)).sum()
    if dA_T is not None:
        loss = loss + (A * t64(dA_T, (N, d, d), False)).sum()
    if dn_T is not None:
        loss = loss + (n * t64(dn_T, (N, d), False)).sum()
    loss.backward()

    def out(x, shape):
        return x.detach().numpy().reshape(lead + shape)

    return {"dq": out(qt.grad, (T, d)), "dk": out(kt.grad, (T, d)), "dv": out(vt.grad, (T, d)),
            "du": out(ut.grad, (T, d)), "dS0": out(S0t.grad, (d, d)), "dA0": out(A0t.grad, (d, d)),
            "dn0": out(n0t.grad, (d,)), "o": out(o, (T, d)), "S_T": out(S, (d, d)),
            "A_T": out(A, (d, d)), "n_T": out(n, (d,))}
