"""Pins for the fp64 oracle (CPU only).

Each test ties the oracle to something other than itself: an explicit matrix
inverse, a closed form, a textbook special case (the delta rule, recursive
least squares = ridge regression), an invariant of the method, or a library
routine.  Section numbers refer to "Variational Linear Attention: Stable
Associative Memory for Long-Context Transformers" (web summaries, sections
2.1-2.3, 3.1-3.2, 5).
"""

import numpy as np
import pytest
import torch

import oracle
from synthetic import make_config, make_inputs, normals

EPS = 1e-6


def _rand(shape, seed, stream=40):
    return normals(seed, stream, int(np.prod(shape))).reshape(shape)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _phi_lib(x):
    """ELU+1 via the library routine (torch.nn.functional.elu)."""
    return torch.nn.functional.elu(torch.from_numpy(np.asarray(x, dtype=np.float64))).numpy() + 1.0


def _prefix_states(q, k, v, u, lam, T):
    """S_t, A_t after every prefix length t = 0..T (oracle runs on prefixes)."""
    d = q.shape[-1]
    Ss, As = [np.zeros((d, d))], [np.eye(d) / lam]
    for t in range(1, T + 1):
        r = oracle.forward(q[:t], k[:t], v[:t], u[:t], lam, nthreads=1)
        Ss.append(r["S_T"])
        As.append(r["A_T"])
    return Ss, As


# --- A_t: section 2.2 (A_t = M_t^{-1}, Sherman-Morrison), section 2.3 step 1 ---

@pytest.mark.parametrize("lam", [1.0, 0.37, 2.5])
def test_A_equals_explicit_inverse_of_penalty(lam):
    d, T = 6, 14
    q, k, v = (_rand((T, d), 1, s) for s in (1, 2, 3))
    u = _rand((T, d), 1, 4)
    _, As = _prefix_states(q, k, v, u, lam, T)
    for t in range(T + 1):
        M = lam * np.eye(d) + u[:t].T @ u[:t]
        Ainv = np.linalg.inv(M)
        A = As[t]
        assert np.abs(A - Ainv).max() <= 1e-12 * np.abs(Ainv).max()
        assert np.abs(A - A.T).max() <= 1e-15 * np.abs(A).max()  # symmetric
        np.linalg.cholesky(A)  # positive definite
        assert np.abs(A @ M - np.eye(d)).max() < 1e-12


def test_A_given_A0_continues_the_penalty():
    d, T = 5, 9
    q, k, v, u = (_rand((T, d), 2, s) for s in range(4))
    M0 = 0.8 * np.eye(d) + np.outer(_rand((d,), 2, 9), _rand((d,), 2, 9))
    r = oracle.forward(q, k, v, u, 1.0, A0=np.linalg.inv(M0))
    M = M0 + u.T @ u
    assert np.allclose(r["A_T"], np.linalg.inv(M), rtol=0, atol=1e-12)


# --- unit vectors: section 2.3 (k_hat, alpha_hat unit length) ---

def test_gate_is_unit_and_aligned_with_key():
    x = make_inputs(2, 3, 64, 16, "f32", seed=7)
    r = oracle.forward_inputs(x, trace=True)
    nrm = np.linalg.norm(r["alpha"], axis=-1)
    assert np.abs(nrm - 1.0).max() < 1e-14
    # c_t = alpha_hat . k_hat lies in (0, 1] because A_t is positive definite
    assert r["c"].min() > 0.0 and r["c"].max() <= 1.0 + 1e-14
    kh = _unit(x.as_f64("k"))
    c = np.einsum("bhti,bhti->bht", r["alpha"], kh)
    assert np.abs(c - r["c"]).max() < 1e-14


def test_gate_direction_is_A_t_times_unit_key():
    d, T, lam = 5, 8, 0.6
    q, k, v, u = (_rand((T, d), 3, s) for s in range(4))
    r = oracle.forward(q, k, v, u, lam, trace=True)
    kh = _unit(k)
    for t in range(T):
        A_t = np.linalg.inv(lam * np.eye(d) + u[: t + 1].T @ u[: t + 1])
        g = A_t @ kh[t]
        assert np.allclose(r["alpha"][t], g / np.linalg.norm(g), atol=1e-13)


# --- S_t: section 2.3 step 3 ---

def test_residual_shrinks_by_one_minus_c():
    """v_t - S_t k_hat_t = (1 - c_t) (v_t - S_{t-1} k_hat_t), c_t = alpha_hat_t . k_hat_t."""
    d, T = 6, 12
    q, k, v, u = (_rand((T, d), 4, s) for s in range(4))
    r = oracle.forward(q, k, v, u, 1.0, trace=True)
    Ss, _ = _prefix_states(q, k, v, u, 1.0, T)
    kh = _unit(k)
    for t in range(T):
        pre = v[t] - Ss[t] @ kh[t]
        post = v[t] - Ss[t + 1] @ kh[t]
        assert np.allclose(post, (1.0 - r["c"][t]) * pre, atol=1e-12)


@pytest.mark.parametrize("gamma", [1.0, 0.3])
def test_orthonormal_keys_closed_form_exact_recall(gamma):
    """Orthonormal keys, u_t = gamma k_hat_t, S_0 = 0: alpha_hat_t = k_hat_t,
    S_n = sum_i v_i k_i^T, exact recall S_n k_i = v_i (section 3.2)."""
    d, n, lam = 8, 6, 0.9
    Q, _ = np.linalg.qr(_rand((d, n), 5, 1))
    keys = Q.T  # n orthonormal rows
    vals = _rand((n, d), 5, 2)
    q = _rand((n, d), 5, 3)
    r = oracle.forward(q, keys * 2.5, vals, gamma * keys, lam, trace=True)
    assert np.allclose(r["alpha"], keys, atol=1e-13)
    assert np.allclose(r["c"], 1.0, atol=1e-13)
    S = r["S_T"]
    assert np.allclose(S, vals.T @ keys, atol=1e-13)
    assert np.allclose((S @ keys.T).T, vals, atol=1e-13)
    assert abs(np.sum(S * S) - np.sum(vals * vals)) < 1e-11
    P = keys.T @ keys
    A_expect = (np.eye(d) - P) / lam + P / (lam + gamma ** 2)
    assert np.allclose(r["A_T"], A_expect, atol=1e-13)


def test_zero_penalty_direction_reduces_to_delta_rule():
    """u == 0: A stays lambda0^{-1} I, alpha_hat = k_hat, and S follows the
    delta rule S_t = S_{t-1} + (v_t - S_{t-1} k_t) k_t^T (unit step)."""
    d, T, lam = 7, 20, 1.7
    q, k, v = (_rand((T, d), 6, s) for s in range(3))
    r = oracle.forward(q, k, v, np.zeros((T, d)), lam, trace=True)
    assert np.allclose(r["A_T"], np.eye(d) / lam, atol=1e-15)
    kh = _unit(k)
    assert np.allclose(r["alpha"], kh, atol=1e-14)
    S = np.zeros((d, d))
    for t in range(T):
        S = S + np.outer(v[t] - S @ kh[t], kh[t])
    assert np.allclose(r["S_T"], S, atol=1e-12)


@pytest.mark.parametrize("lam", [1.0, 0.25])
def test_unnormalised_gate_is_ridge_regression(lam):
    """With the gate A_t k_hat_t left unnormalised and u_t = k_hat_t the rule is
    recursive least squares (section 5): S_t solves the ridge problem
    S_t (lambda0 I + sum k k^T) = sum v k^T."""
    d, T = 6, 25
    q, k, v = (_rand((T, d), 7, s) for s in range(3))
    kh = _unit(k)
    r = oracle.forward(q, k, v, kh, lam, unnormalised_gate=True)
    G = lam * np.eye(d) + kh.T @ kh
    C = v.T @ kh
    S_ridge = np.linalg.solve(G.T, C.T).T
    assert np.allclose(r["S_T"], S_ridge, atol=1e-11)


# --- metamorphic relations ---

def test_scale_invariance_lambda_and_u():
    """(lambda0, u) -> (1, u / sqrt(lambda0)) leaves alpha_hat, S, o unchanged and
    A(lambda0) = A(1, u/sqrt(lambda0)) / lambda0."""
    x = make_inputs(1, 2, 40, 8, "f32", seed=8)
    lam = 0.3
    q, k, v, u = (x.as_f64(n) for n in "qkvu")
    a = oracle.forward(q, k, v, u, lam, trace=True)
    b = oracle.forward(q, k, v, u / np.sqrt(lam), 1.0, trace=True)
    for key in ("o", "S_T", "alpha"):
        assert np.allclose(a[key], b[key], atol=1e-11)
    assert np.allclose(a["A_T"], b["A_T"] / lam, atol=1e-12)


def test_rotation_equivariance():
    """An orthogonal Q on keys and penalty directions maps A -> Q A Q^T and
    S -> S Q^T."""
    d, T = 8, 30
    q, k, v, u = (_rand((T, d), 9, s) for s in range(4))
    Q, _ = np.linalg.qr(_rand((d, d), 9, 7))
    a = oracle.forward(q, k, v, u, 0.8)
    b = oracle.forward(q, k @ Q.T, v, u @ Q.T, 0.8)
    assert np.allclose(b["A_T"], Q @ a["A_T"] @ Q.T, atol=1e-12)
    assert np.allclose(b["S_T"], a["S_T"] @ Q.T, atol=1e-11)


def test_permutation_equivariance_including_readout():
    """Permuting key coordinates (q, k, u together) leaves o unchanged because
    phi acts elementwise; permuting value coordinates permutes o and the rows of S."""
    d, T = 9, 33
    q, k, v, u = (_rand((T, d), 10, s) for s in range(4))
    pk = np.array([3, 0, 8, 1, 5, 2, 7, 6, 4])
    pv = np.array([8, 7, 6, 5, 4, 3, 2, 1, 0])
    a = oracle.forward(q, k, v, u, 1.0)
    b = oracle.forward(q[:, pk], k[:, pk], v[:, pv], u[:, pk], 1.0)
    assert np.allclose(b["o"], a["o"][:, pv], atol=1e-12)
    assert np.allclose(b["S_T"], a["S_T"][np.ix_(pv, pk)], atol=1e-12)
    assert np.allclose(b["A_T"], a["A_T"][np.ix_(pk, pk)], atol=1e-13)
    assert np.allclose(b["n_T"], a["n_T"][pk], atol=1e-12)


def test_split_stream_equals_single_call():
    """Streaming (section 5): [0, t) then [t, T) with (S, A, n) handed over."""
    x = make_inputs(2, 2, 50, 8, "f32", seed=12)
    q, k, v, u = (x.as_f64(n) for n in "qkvu")
    full = oracle.forward(q, k, v, u, 0.7)
    t = 19
    a = oracle.forward(q[..., :t, :], k[..., :t, :], v[..., :t, :], u[..., :t, :], 0.7)
    b = oracle.forward(q[..., t:, :], k[..., t:, :], v[..., t:, :], u[..., t:, :], 0.7,
                       S0=a["S_T"], A0=a["A_T"], n0=a["n_T"])
    assert np.allclose(np.concatenate([a["o"], b["o"]], axis=-2), full["o"], atol=1e-13)
    for key in ("S_T", "A_T", "n_T"):
        assert np.allclose(b[key], full[key], atol=1e-12)


def test_empty_stream_returns_initial_state():
    d = 4
    S0 = _rand((1, d, d), 13, 1)
    A0 = np.eye(d)[None] * 0.5
    n0 = np.abs(_rand((1, d), 13, 2))
    e = np.zeros((1, 0, d))
    r = oracle.forward(e, e, e, e, 1.0, S0=S0, A0=A0, n0=n0)
    assert r["o"].shape == (1, 0, d)
    assert np.array_equal(r["S_T"], S0) and np.array_equal(r["A_T"], A0)
    assert np.array_equal(r["n_T"], n0)
    r = oracle.forward(e, e, e, e, 0.25)
    assert np.array_equal(r["A_T"][0], 4.0 * np.eye(d)) and not r["S_T"].any()


# --- readout: section 2.3 (ratio of recurrences with the ELU+1 feature map) ---

def test_readout_decomposes_into_library_routines():
    """o_t (phi(q_t)^T n_t + eps) = S_t phi(q_t), n_t = cumsum phi(k_hat),
    with phi = ELU + 1 from torch and S_t from the delta-rule special case."""
    d, T, lam = 6, 18, 1.0
    q, k, v = (_rand((T, d), 14, s) for s in range(3))
    r = oracle.forward(q, k, v, np.zeros((T, d)), lam)
    kh = _unit(k)
    n = np.cumsum(_phi_lib(kh), axis=0)
    fq = _phi_lib(q)
    S = np.zeros((d, d))
    for t in range(T):
        S = S + np.outer(v[t] - S @ kh[t], kh[t])  # textbook delta rule (u = 0)
        num = S @ fq[t]
        den = fq[t] @ n[t] + EPS
        assert np.allclose(r["o"][t], num / den, atol=1e-13)
    assert np.allclose(r["n_T"], n[-1], atol=1e-13)


def test_readout_general_inputs_against_prefix_states():
    d, T = 5, 16
    q, k, v, u = (_rand((T, d), 15, s) for s in range(4))
    r = oracle.forward(q, k, v, u, 0.5)
    Ss, _ = _prefix_states(q, k, v, u, 0.5, T)
    n = np.cumsum(_phi_lib(_unit(k)), axis=0)
    fq = _phi_lib(q)
    for t in range(T):
        den = fq[t] @ n[t] + EPS
        assert den > 0.0
        assert np.allclose(r["o"][t] * den, Ss[t + 1] @ fq[t], atol=1e-12)


def test_scalar_head_closed_form():
    """d = 1: k_hat = sign(k), alpha_hat = k_hat, S_t = v_t k_hat_t,
    A_t = 1 / (lambda0 + sum u^2), n_t = sum phi(k_hat), with phi(1) = 2 and
    phi(-1) = exp(-1)."""
    T, lam = 12, 0.4
    k = np.array([0.5, -2.0, 3.0, -0.1, 1.0, 7.0, -3.0, -0.5, 2.0, 0.25, -1.5, 4.0])[:, None]
    v = np.arange(1, T + 1, dtype=float)[:, None] * 0.5 - 2.0
    u = np.linspace(-1.0, 1.5, T)[:, None]
    q = np.linspace(-2.0, 2.0, T)[:, None]
    r = oracle.forward(q, k, v, u, lam, trace=True)
    s = np.sign(k[:, 0])
    assert np.allclose(r["alpha"][:, 0], s, atol=0)
    n = np.cumsum(np.where(s > 0, 2.0, np.exp(-1.0)))
    fq = np.where(q[:, 0] > 0, q[:, 0] + 1.0, np.exp(q[:, 0]))
    o = v[:, 0] * s * fq / (fq * n + EPS)
    assert np.allclose(r["o"][:, 0], o, rtol=1e-14, atol=1e-15)
    assert np.isclose(r["A_T"][0, 0], 1.0 / (lam + np.sum(u ** 2)), rtol=1e-14)
    assert np.isclose(r["S_T"][0, 0], v[-1, 0] * s[-1], rtol=1e-14)


# --- Proposition 1 (section 3.1): bounded state vs linear attention's growth ---

def test_state_norm_plateaus_while_linear_attention_grows():
    x = make_inputs(1, 4, 2048, 32, "f32", seed=11, u_scale=0.5)
    r = oracle.forward_inputs(x, trace=True)
    sn = r["snorm"][0]
    kh = _unit(x.as_f64("k"))[0]
    v = x.as_f64("v")[0]
    la = np.cumsum(np.einsum("hti,htj->htij", v, kh), axis=1)
    lan = np.linalg.norm(la, axis=(-2, -1))
    T = 2048
    vla_ratio = sn[:, T - 1] / sn[:, T // 4 - 1]
    la_ratio = lan[:, T - 1] / lan[:, T // 4 - 1]
    # zero-mean writes: linear attention grows like sqrt(T) (x2 over a x4
    # span); the VLA state stays on its plateau.
    assert np.all(vla_ratio < 1.15), vla_ratio
    assert np.all(la_ratio > 1.7), la_ratio
    assert np.all(sn[:, -1] < lan[:, -1] / 4)


def test_recall_stream_exact_recall_before_distractors():
    """Synthetic recall stream: right after the 2n write tokens every stored
    pair is recalled exactly (n <= d orthonormal keys, u = k_hat)."""
    x = make_config("recall24", B=2, H=1)
    n = 24
    r = oracle.forward(x.as_f64("q")[..., : 2 * n, :], x.as_f64("k")[..., : 2 * n, :],
                       x.as_f64("v")[..., : 2 * n, :], x.as_f64("u")[..., : 2 * n, :], 1.0)
    rec = np.einsum("bhij,bhnj->bhni", r["S_T"], x.keys)
    assert np.abs(rec - x.values).max() < 1e-5  # fp32-rounded orthonormal keys


# --- regression fixture written by tests/golden/make_golden.py (oracle only) ---

def test_golden_regression_fixture():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_d4_T6.txt")
    data = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, vals = line.split(":", 1)
            data[name.strip()] = np.array([float(t) for t in vals.split()])
    d, T = 4, 6
    q, k, v, u = (data[n].reshape(T, d) for n in "qkvu")
    r = oracle.forward(q, k, v, u, float(data["lambda0"][0]))
    assert np.allclose(r["o"].ravel(), data["o"], rtol=1e-13, atol=1e-15)
    assert np.allclose(r["S_T"].ravel(), data["S_T"], rtol=1e-13, atol=1e-15)
    assert np.allclose(r["A_T"].ravel(), data["A_T"], rtol=1e-13, atol=1e-15)
