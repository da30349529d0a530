"""GPU parity of the backward pass (vla_backward, through the C ABI) against
the fp64 autograd oracle (oracle/backward.py).  Gradients are fp32 on the
GPU; bar: relative Frobenius error <= 1e-3 per gradient tensor (fp32
arithmetic through T reverse steps and two normalisations; measured errors
are printed)."""

import numpy as np
import pytest
import torch

import rls_associative_memory_gb300 as vla
from oracle import backward as ob
from synthetic import make_inputs, normals
from vla_testutil import rel_fro, to_device

pytestmark = pytest.mark.gpu

GTOL = 1e-3
KEYS = ("dq", "dk", "dv", "du", "dS0", "dA0", "dn0")


def _rand(shape, seed, stream, scale=1.0):
    return normals(seed, stream, int(np.prod(shape))).reshape(shape) * scale


def _dev(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda").to(dtype)


def _run(x, dO, st=None, up=None):
    q, k, v, u = to_device(x)
    io = torch.bfloat16 if x.dtype == "bf16" else torch.float32
    kw = {}
    if st:
        kw.update(S0=_dev(st["S_T"]), A0=_dev(st["A_T"]), n0=_dev(st["n_T"]))
    if up:
        kw.update(dS_T=_dev(up[0]), dA_T=_dev(up[1]), dn_T=_dev(up[2]))
    g = vla.vla_backward(q, k, v, u, _dev(dO, io), x.lambda0, **kw)
    torch.cuda.synchronize()
    return {key: val.cpu().numpy().astype(np.float64) for key, val in g.items()}


def _dO_exact(dO, dtype):
    # the oracle sees exactly the dO bits the GPU gets
    t = torch.from_numpy(np.ascontiguousarray(dO, dtype=np.float32))
    if dtype == "bf16":
        t = t.bfloat16().float()
    return t.double().numpy()


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 17, 100, 200])
def test_backward_small(d, dtype, T):
    x = make_inputs(1, 3, T, d, dtype, seed=500 + d + T, lambda0=0.9)
    dO = _dO_exact(_rand(x.q.shape, 501, 7), dtype)
    got = _run(x, dO)
    ref = ob.backward(x.as_f64("q"), x.as_f64("k"), x.as_f64("v"), x.as_f64("u"), x.lambda0, dO)
    errs = {key: rel_fro(got[key], ref[key]) for key in KEYS}
    print("\nbackward d=%d %s T=%d %s" % (d, dtype, T, {k_: "%.2e" % e for k_, e in errs.items()}))
    assert all(e <= GTOL for e in errs.values()), errs


@pytest.mark.parametrize("d", [32, 64, 128])
def test_backward_with_state_and_state_gradients(d):
    pre = make_inputs(1, 2, 30, d, "f32", seed=510, lambda0=1.3)
    import oracle
    st = oracle.forward_inputs(pre)
    x = make_inputs(1, 2, 150, d, "f32", seed=511, lambda0=1.3)
    dO = _rand(x.q.shape, 512, 1)
    up = (_rand((1, 2, d, d), 512, 2, 0.1), _rand((1, 2, d, d), 512, 3, 10.0), _rand((1, 2, d), 512, 4, 0.1))
    got = _run(x, dO, st, up)
    ref = ob.backward(x.as_f64("q"), x.as_f64("k"), x.as_f64("v"), x.as_f64("u"), x.lambda0, dO,
                      dS_T=up[0], dA_T=up[1], dn_T=up[2], S0=st["S_T"], A0=st["A_T"], n0=st["n_T"])
    errs = {key: rel_fro(got[key], ref[key]) for key in KEYS}
    print("\nbackward with state d=%d %s" % (d, {k_: "%.2e" % e for k_, e in errs.items()}))
    assert all(e <= GTOL for e in errs.values()), errs


def test_backward_long_stream_sampled_heads():
    """B=4 H=8 T=4096 d=64 bf16 (the heads32 workload's shape): the GPU runs
    all 32 units; the oracle checks two of them over the full stream."""
    x = make_inputs(4, 8, 4096, 64, "bf16", seed=2, lambda0=1.0)
    dO = _dO_exact(_rand(x.q.shape, 520, 1), "bf16")
    got = _run(x, dO)
    for (b, h) in ((0, 0), (3, 7)):
        ref = ob.backward(x.as_f64("q")[b, h], x.as_f64("k")[b, h], x.as_f64("v")[b, h], x.as_f64("u")[b, h],
                          x.lambda0, dO[b, h])
        errs = {key: rel_fro(got[key][b, h], ref[key]) for key in KEYS}
        print("\nbackward 4x8x4096 unit (%d,%d) %s" % (b, h, {k_: "%.2e" % e for k_, e in errs.items()}))
        assert all(e <= GTOL for e in errs.values()), errs


def test_backward_d128_many_units_sampled():
    """d = 128 (the sequential form with S and dS in shared memory): 2 x 4 x 300
    bf16 streams (300 tokens cross four checkpoints and end mid-interval); the
    oracle checks two of the eight units."""
    x = make_inputs(2, 4, 300, 128, "bf16", seed=530, lambda0=0.7)
    dO = _dO_exact(_rand(x.q.shape, 531, 1), "bf16")
    got = _run(x, dO)
    for (b, h) in ((0, 1), (1, 3)):
        ref = ob.backward(x.as_f64("q")[b, h], x.as_f64("k")[b, h], x.as_f64("v")[b, h], x.as_f64("u")[b, h],
                          x.lambda0, dO[b, h])
        errs = {key: rel_fro(got[key][b, h], ref[key]) for key in KEYS}
        print("\nbackward d=128 2x4x300 unit (%d,%d) %s" % (b, h, {k_: "%.2e" % e for k_, e in errs.items()}))
        assert all(e <= GTOL for e in errs.values()), errs


@pytest.mark.parametrize("case", ["zero_keys", "u0", "u10", "lambda0_small"])
def test_backward_d128_edge_inputs(case):
    """The method's special cases at d = 128: keys at and below the norm guard,
    no penalty updates (u = 0: A stays lambda0^-1 I), strong penalty
    directions, and a small lambda0."""
    kw = {"u0": dict(u_scale=0.0), "u10": dict(u_scale=10.0)}.get(case, {})
    lam = 0.05 if case == "lambda0_small" else 1.0
    x = make_inputs(1, 2, 90, 128, "f32", seed=540, lambda0=lam, **kw)
    if case == "zero_keys":
        for t in (0, 5, 64, 89):
            x.k[:, :, t, :] = 0.0
        x.k[:, :, 30, :] *= 1e-8
    dO = _rand(x.q.shape, 541, 1)
    got = _run(x, dO)
    ref = ob.backward(x.as_f64("q"), x.as_f64("k"), x.as_f64("v"), x.as_f64("u"), x.lambda0, dO)
    errs = {key: rel_fro(got[key], ref[key]) for key in KEYS}
    print("\nbackward d=128 %s %s" % (case, {k_: "%.2e" % e for k_, e in errs.items()}))
    assert all(e <= GTOL for e in errs.values()), errs
