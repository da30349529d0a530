"""The sequential kernel at d_h = 32 (three warps per (b, h): inputs, the A
chain and the S chain, handing 8-token slots on through a ring of four)
against the fp64 oracle: stream lengths around the slot and ring boundaries,
more units than one wave, the method's special cases, a stream split over two
calls, and the bounded waits' failure path.  Bar: relative Frobenius error
<= 1e-4 (fp32 I/O) and <= 5e-3 (bf16 I/O) per output."""

import numpy as np
import pytest
import torch

import rls_associative_memory_gb300 as vla
from synthetic import make_inputs
from vla_testutil import TOL, compare, oracle_ref, rel_fro, run_gpu, to_device

pytestmark = pytest.mark.gpu

SEQ = vla.VLA_KERNEL_SEQ


def _one_launch(got):
    assert vla.vla_last_launch_count() == 1
    return got


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 7, 8, 9, 31, 32, 33, 40, 65, 257])
def test_slot_and_ring_boundaries(T, dtype):
    x = make_inputs(2, 2, T, 32, dtype, seed=500 + T, lambda0=0.9)
    compare(_one_launch(run_gpu(x, SEQ)), oracle_ref(x), dtype)


def test_more_units_than_one_wave():
    """1100 units: more CTAs than the 7 a SM holds on 152 SMs."""
    x = make_inputs(275, 4, 40, 32, "f32", seed=511, lambda0=0.7)
    got = run_gpu(x, SEQ)
    for i in np.linspace(0, 275 * 4 - 1, 24).round().astype(int):
        b, h = divmod(int(i), 4)
        ref = oracle_ref(x.slice_heads(slice(b, b + 1), slice(h, h + 1)))
        compare({k: v[b:b + 1, h:h + 1] for k, v in got.items()}, ref, "f32")


def test_zero_and_tiny_keys():
    x = make_inputs(1, 3, 120, 32, "f32", seed=512, lambda0=1.0)
    for t in (0, 7, 8, 31, 32, 119):
        x.k[:, :, t, :] = 0.0
    for t in (3, 40, 100):
        x.k[:, :, t, :] *= 1e-8
    compare(run_gpu(x, SEQ), oracle_ref(x), "f32")


@pytest.mark.parametrize("u_scale", [0.0, 0.01, 10.0], ids=["u0", "u0.01", "u10"])
def test_penalty_scale(u_scale):
    x = make_inputs(1, 3, 200, 32, "f32", seed=513, u_scale=u_scale, lambda0=1.0)
    compare(run_gpu(x, SEQ), oracle_ref(x), "f32")


@pytest.mark.parametrize("lambda0", [0.01, 100.0])
def test_lambda0_extremes(lambda0):
    x = make_inputs(1, 3, 200, 32, "f32", seed=514, lambda0=lambda0)
    compare(run_gpu(x, SEQ), oracle_ref(x), "f32")


def test_given_initial_state_bf16():
    pre = make_inputs(2, 2, 50, 32, "bf16", seed=515, lambda0=0.8)
    st = oracle_ref(pre)
    x = make_inputs(2, 2, 70, 32, "bf16", seed=516, lambda0=0.8)
    ref = oracle_ref(x, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"])
    compare(run_gpu(x, SEQ, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"]), ref, "bf16")


def test_split_stream():
    """Two calls with the state handed over (in place) equal the oracle's one call."""
    x = make_inputs(3, 2, 90, 32, "f32", seed=517, lambda0=0.6)
    q, k, v, u = to_device(x)
    t = 37  # splits a slot
    sl = lambda a, lo, hi: a[:, :, lo:hi].contiguous()  # noqa: E731
    o1, S, A, n = vla.vla_forward(sl(q, 0, t), sl(k, 0, t), sl(v, 0, t), sl(u, 0, t), x.lambda0, kernel=SEQ)
    o2, S2, A2, n2 = vla.vla_forward(sl(q, t, 90), sl(k, t, 90), sl(v, t, 90), sl(u, t, 90), x.lambda0,
                                     S0=S, A0=A, n0=n, S_T=S, A_T=A, n_T=n, kernel=SEQ)
    torch.cuda.synchronize()
    ref = oracle_ref(x)
    o = torch.cat([o1, o2], dim=2).cpu().numpy()
    assert rel_fro(o, ref["o"]) < TOL["f32"]
    for key, got in (("S_T", S), ("A_T", A), ("n_T", n)):
        assert rel_fro(got.cpu().numpy(), ref[key]) < TOL["f32"], key


def test_empty_stream_copies_state():
    d, dev = 32, "cuda"
    e = torch.empty((2, 1, 0, d), dtype=torch.float32, device=dev)
    S0 = torch.randn(2, 1, d, d, device=dev)
    A0 = torch.eye(d, device=dev).expand(2, 1, d, d).contiguous() * 0.25
    n0 = torch.rand(2, 1, d, device=dev)
    o, S, A, n = vla.vla_forward(e, e, e, e, 1.0, S0=S0, A0=A0, n0=n0, kernel=SEQ)
    torch.cuda.synchronize()
    assert torch.equal(S, S0) and torch.equal(A, A0) and torch.equal(n, n0)


def test_bounded_wait_expiry_at_d32():
    """Test hook: the first input slot never fills, so the A and S chains'
    bounded waits expire (1 ms), the device error word is set and the kernel
    returns; the next call is normal."""
    x = make_inputs(1, 2, 64, 32, "f32", seed=518)
    q, k, v, u = to_device(x)
    assert vla.vla_debug_inject(1, 1_000_000) == vla.VLA_OK
    try:
        vla.vla_forward(q, k, v, u, 1.0, kernel=SEQ)
        assert vla.vla_device_status() == vla.VLA_ERR_TIMEOUT
    finally:
        vla.vla_debug_inject(0)
    assert vla.vla_device_status() == vla.VLA_OK
    compare(run_gpu(x, SEQ), oracle_ref(x), "f32")
