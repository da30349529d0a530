"""Pins for the fp64 gradient oracle (CPU only).

The autograd gradients of oracle/backward.py are checked against central
finite differences of the loss computed with the C oracle's forward
(oracle/vla_oracle.c), an implementation that shares nothing with the
PyTorch forward; and the PyTorch forward itself against the C oracle."""

import numpy as np
import pytest

import oracle
from oracle import backward as ob
from synthetic import make_inputs, normals


def _rand(shape, seed, stream):
    return normals(seed, stream, int(np.prod(shape))).reshape(shape)


def _loss_c(q, k, v, u, lam, dO, dS, dA, dn, S0=None, A0=None, n0=None):
    r = oracle.forward(q, k, v, u, lam, S0=S0, A0=A0, n0=n0, nthreads=1)
    return (np.sum(r["o"] * dO) + np.sum(r["S_T"] * dS) + np.sum(r["A_T"] * dA)
            + np.sum(r["n_T"] * dn))


def test_torch_forward_matches_c_oracle():
    x = make_inputs(2, 2, 23, 6, "f32", seed=90, lambda0=0.7)
    q, k, v, u = (x.as_f64(n) for n in "qkvu")
    S0 = _rand((2, 2, 6, 6), 90, 20)
    A0 = np.linalg.inv(np.eye(6) * 0.7 + np.einsum("bhi,bhj->bhij", _rand((2, 2, 6), 90, 21), _rand((2, 2, 6), 90, 21)))
    n0 = np.abs(_rand((2, 2, 6), 90, 22))
    c = oracle.forward(q, k, v, u, 0.7, S0=S0, A0=A0, n0=n0)
    t = ob.backward(q, k, v, u, 0.7, np.zeros_like(q), S0=S0, A0=A0, n0=n0)
    for key in ("o", "S_T", "A_T", "n_T"):
        assert np.allclose(t[key], c[key], rtol=1e-12, atol=1e-13), key


@pytest.mark.parametrize("with_state", [False, True])
def test_gradients_match_central_differences_of_the_c_oracle(with_state):
    N, T, d, lam = 2, 6, 4, 0.8
    q, k, v, u = (_rand((N, T, d), 91, s) for s in range(4))
    dO = _rand((N, T, d), 91, 4)
    dS = _rand((N, d, d), 91, 5)
    dA = _rand((N, d, d), 91, 6)
    dn = _rand((N, d), 91, 7)
    st = {}
    if with_state:
        st = oracle.forward(_rand((N, 9, d), 92, 0), _rand((N, 9, d), 92, 1), _rand((N, 9, d), 92, 2),
                            _rand((N, 9, d), 92, 3), lam)
        st = {"S0": st["S_T"], "A0": st["A_T"], "n0": st["n_T"]}
    g = ob.backward(q, k, v, u, lam, dO, dS, dA, dn, **st)
    base = dict(q=q, k=k, v=v, u=u, **st)
    if not with_state:
        base.update(S0=np.zeros((N, d, d)), A0=np.tile(np.eye(d) / lam, (N, 1, 1)), n0=np.zeros((N, d)))
    h = 1e-6
    for stream, (name, gname) in enumerate((("q", "dq"), ("k", "dk"), ("v", "dv"), ("u", "du"),
                                             ("S0", "dS0"), ("A0", "dA0"), ("n0", "dn0"))):
        V = _rand(base[name].shape, 93, 100 + stream)
        plus = dict(base)
        minus = dict(base)
        plus[name] = base[name] + h * V
        minus[name] = base[name] - h * V
        Lp = _loss_c(plus["q"], plus["k"], plus["v"], plus["u"], lam, dO, dS, dA, dn,
                     S0=plus["S0"], A0=plus["A0"], n0=plus["n0"])
        Lm = _loss_c(minus["q"], minus["k"], minus["v"], minus["u"], lam, dO, dS, dA, dn,
                     S0=minus["S0"], A0=minus["A0"], n0=minus["n0"])
        fd = (Lp - Lm) / (2 * h)
        an = float(np.sum(g[gname] * V))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_elementwise_gradient_entries_match_differences():
    """Single-entry differences for a few coordinates of k and u (the inputs
    that reach A and the gate)."""
    N, T, d, lam = 1, 4, 3, 1.2
    q, k, v, u = (_rand((N, T, d), 94, s) for s in range(4))
    dO = _rand((N, T, d), 94, 4)
    z = np.zeros((N, d, d))
    g = ob.backward(q, k, v, u, lam, dO)
    h = 1e-6
    for arr_name, gname in (("k", "dk"), ("u", "du")):
        for (t, j) in ((0, 0), (1, 2), (3, 1)):
            args = {"q": q, "k": k, "v": v, "u": u}
            p = args[arr_name].copy()
            m = args[arr_name].copy()
            p[0, t, j] += h
            m[0, t, j] -= h
            ap = dict(args, **{arr_name: p})
            am = dict(args, **{arr_name: m})
            fd = (_loss_c(ap["q"], ap["k"], ap["v"], ap["u"], lam, dO, z, z, np.zeros((N, d)))
                  - _loss_c(am["q"], am["k"], am["v"], am["u"], lam, dO, z, z, np.zeros((N, d)))) / (2 * h)
            assert abs(fd - g[gname][0, t, j]) <= 1e-6 * max(1.0, abs(fd)), (arr_name, t, j)
