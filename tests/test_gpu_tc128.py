"""The tensor-core path at d_h = 128 (bf16 I/O, one chunk per (b, h) unit:
block-Woodbury gates from A0, then the UT-transform state pass on S itself,
which writes o) against the fp64 oracle.  Shapes with whole and ragged
64-token sub-blocks, a given initial state, and the method's special cases
(zero and sub-eps keys, u = 0, large and small u, small and large lambda0).
Every call asserts that the tensor-core queue kernel ran (one launch: the
gates and the state pass of every unit, handed to the SMs from a queue).  Bar:
relative Frobenius error <= 5e-3 per output (bf16 I/O, fp32 state).

The stress cases stay inside the path's conditioning envelope: with one chunk
per unit the block downdates of A accumulate over the whole stream in fp32,
and the first ones are small differences of large terms when the penalty
directions outweigh lambda0 (u_t^T A_0 u_t up to ~4e3 here: u x4 at
lambda0 = 0.5, unit u at lambda0 = 0.05).  Beyond it (u x10 at lambda0 = 0.5,
u_t^T A_0 u_t ~ 2.6e4) S_T and A_T drift to ~7e-3 while the token-sequential
kernel holds 8e-4."""

import numpy as np
import pytest
import torch

import rls_associative_memory_gb300 as vla
from synthetic import make_inputs
from synthetic.generator import f32_to_bf16_bits
from vla_testutil import compare, oracle_ref, to_device

pytestmark = pytest.mark.gpu

TC = vla.VLA_KERNEL_CHUNK_TC


def _run(x, S0=None, A0=None, n0=None):
    """One chunk per unit: chunk = T rounded up to a multiple of 64."""
    q, k, v, u = to_device(x)
    dev = q.device
    T = x.q.shape[2]
    chunk = max(64, (T + 63) // 64 * 64)

    def st(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)

    o, S_T, A_T, n_T = vla.vla_forward(q, k, v, u, x.lambda0, S0=st(S0), A0=st(A0), n0=st(n0), kernel=TC,
                                       chunk=chunk)
    torch.cuda.synchronize()
    assert vla.vla_device_status() == vla.VLA_OK
    assert vla.vla_last_launch_count() == 1, "the d = 128 tensor-core queue kernel did not run"
    return {"o": o.float().cpu().numpy().astype(np.float64), "S_T": S_T.cpu().numpy().astype(np.float64),
            "A_T": A_T.cpu().numpy().astype(np.float64), "n_T": n_T.cpu().numpy().astype(np.float64)}


@pytest.mark.parametrize("T", [1, 17, 64, 100, 333, 1000])
def test_shapes(T):
    x = make_inputs(2, 2, T, 128, "bf16", seed=300 + T, lambda0=0.5)
    compare(_run(x), oracle_ref(x), "bf16")


def test_given_initial_state():
    pre = make_inputs(1, 3, 150, 128, "bf16", seed=71, lambda0=0.7)
    st = oracle_ref(pre)
    x = make_inputs(1, 3, 500, 128, "bf16", seed=72, lambda0=0.7)
    ref = oracle_ref(x, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"])
    compare(_run(x, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"]), ref, "bf16")


def test_zero_and_tiny_keys():
    x = make_inputs(1, 3, 600, 128, "bf16", seed=73, lambda0=0.5)
    k = x.as_f32("k")
    for t in (0, 1, 63, 64, 127, 128, 599):
        k[:, :, t, :] = 0.0
    for t in (2, 65, 300):
        k[:, :, t, :] *= 1e-8
    x.k = f32_to_bf16_bits(k)
    compare(_run(x), oracle_ref(x), "bf16")


@pytest.mark.parametrize("u_scale", [0.0, 0.01, 4.0], ids=["u0", "u0.01", "u4"])
def test_penalty_scale(u_scale):
    x = make_inputs(1, 3, 600, 128, "bf16", seed=74, u_scale=u_scale, lambda0=0.5)
    compare(_run(x), oracle_ref(x), "bf16")


@pytest.mark.parametrize("lambda0", [0.05, 100.0])
def test_lambda0_extremes(lambda0):
    x = make_inputs(1, 3, 600, 128, "bf16", seed=75, lambda0=lambda0)
    compare(_run(x), oracle_ref(x), "bf16")


def test_auto_takes_the_tensor_core_path_for_many_units():
    """AUTO at d = 128 with bf16 I/O and 128 units: the single-chunk tensor-core path."""
    x = make_inputs(8, 16, 300, 128, "bf16", seed=76, lambda0=0.5)
    q, k, v, u = to_device(x)
    o, S_T, A_T, n_T = vla.vla_forward(q, k, v, u, x.lambda0)
    torch.cuda.synchronize()
    assert vla.vla_device_status() == vla.VLA_OK
    assert vla.vla_last_launch_count() == 1
    got = {"o": o.float().cpu().numpy(), "S_T": S_T.cpu().numpy(), "A_T": A_T.cpu().numpy(),
           "n_T": n_T.cpu().numpy()}
    compare(got, oracle_ref(x), "bf16")


@pytest.mark.parametrize("T,init", [(1, False), (70, False), (130, True)])
def test_queue_launch_many_units(T, init):
    """300 units: more jobs than the 152 queue CTAs, so most CTAs run several
    units' passes one after another (gates first, then state passes that wait
    on their unit's flag).  Sampled units against the oracle."""
    B, H = 75, 4
    x = make_inputs(B, H, T, 128, "bf16", seed=77 + T, lambda0=0.6)
    S0 = A0 = n0 = None
    if init:  # a state from a short earlier stream (the oracle's, for every unit)
        full = oracle_ref(make_inputs(B, H, 40, 128, "bf16", seed=78, lambda0=0.6))
        S0, A0, n0 = full["S_T"], full["A_T"], full["n_T"]
    got = _run(x, S0=S0, A0=A0, n0=n0)
    for i in np.linspace(0, B * H - 1, 12).round().astype(int):
        b, h = divmod(int(i), H)
        sub = x.slice_heads(slice(b, b + 1), slice(h, h + 1))
        kw = {}
        if init:
            kw = dict(S0=S0[b:b + 1, h:h + 1], A0=A0[b:b + 1, h:h + 1], n0=n0[b:b + 1, h:h + 1])
        ref = oracle_ref(sub, **kw)
        compare({k: v[b:b + 1, h:h + 1] for k, v in got.items()}, ref, "bf16")


def test_bounded_wait_expiry_in_queue_launch():
    """Test hook: the gates jobs of the queue launch leave their flags unset,
    so every state pass's bounded wait expires (1 ms), sets the device error
    word and skips its job; the launch still ends, and the next call is
    normal."""
    x = make_inputs(1, 4, 200, 128, "bf16", seed=521, lambda0=0.5)
    q, k, v, u = to_device(x)
    assert vla.vla_debug_inject(1, 1_000_000) == vla.VLA_OK
    try:
        vla.vla_forward(q, k, v, u, x.lambda0, kernel=TC, chunk=256)
        assert vla.vla_last_launch_count() == 1
        assert vla.vla_device_status() == vla.VLA_ERR_TIMEOUT
    finally:
        vla.vla_debug_inject(0)
    assert vla.vla_device_status() == vla.VLA_OK
    compare(_run(x), oracle_ref(x), "bf16")
