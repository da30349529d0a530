"""GPU parity of the streaming decode step (one or a few tokens per call,
state read from and written back to HBM in place) against the fp64 oracle
run on the whole stream."""

import numpy as np
import pytest
import torch

import oracle
import rls_associative_memory_gb300 as vla
from synthetic import make_config, make_inputs
from vla_testutil import TOL, compare, oracle_ref, rel_fro, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_token_by_token_decode_matches_the_stream(d, dtype):
    T = 37
    x = make_inputs(2, 3, T, d, dtype, seed=300 + d, lambda0=0.9)
    q, k, v, u = to_device(x)
    B, H = 2, 3
    S = torch.zeros(B, H, d, d, device="cuda")
    A = (torch.eye(d, device="cuda") / x.lambda0).expand(B, H, d, d).contiguous()
    n = torch.zeros(B, H, d, device="cuda")
    outs = []
    for t in range(T):
        sl = lambda a: a[:, :, t:t + 1].contiguous()  # noqa: E731
        o, _, _, _ = vla.vla_forward(sl(q), sl(k), sl(v), sl(u), x.lambda0, S0=S, A0=A, n0=n, S_T=S, A_T=A,
                                     n_T=n, kernel=vla.VLA_KERNEL_AUTO)
        outs.append(o)
    torch.cuda.synchronize()
    assert vla.vla_device_status() == vla.VLA_OK
    ref = oracle_ref(x)
    got = {"o": torch.cat(outs, dim=2).float().cpu().numpy(), "S_T": S.cpu().numpy(),
           "A_T": A.cpu().numpy(), "n_T": n.cpu().numpy()}
    compare(got, ref, dtype)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 9])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_kernel_few_tokens(T, d):
    x = make_inputs(3, 2, T, d, "bf16", seed=400 + T, lambda0=1.1)
    pre = make_inputs(3, 2, 20, d, "bf16", seed=401 + T, lambda0=1.1)
    st = oracle_ref(pre)
    got = run_gpu(x, vla.VLA_KERNEL_DECODE, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"])
    ref = oracle_ref(x, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"])
    compare(got, ref, "bf16")


def test_decode_workload_full_size():
    """The benchmarked decode workload (B=32 H=64 d=64 bf16, one token) from a
    non-trivial state: every unit first streams 32 tokens through the oracle."""
    x = make_config("decode")
    B, H, _, d = x.q.shape
    pre = make_inputs(B, H, 32, d, "bf16", seed=61, lambda0=x.lambda0)
    st = oracle_ref(pre)
    got = run_gpu(x, vla.VLA_KERNEL_AUTO, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"])
    ref = oracle_ref(x, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"])
    errs = compare(got, ref, "bf16")
    print("\ndecode full-size errs", errs)


@pytest.mark.parametrize("given", ["both", "A0", "S0"])
def test_decode_many_units_in_place(given):
    """More units than resident CTAs (8 x 80 = 640): each CTA walks several
    units while the next units' initial state lands in shared memory; the
    state is updated in place, and with only A0 or only S0 given the other
    starts from its default (I / lambda0, 0)."""
    B, H, d, T = 8, 80, 64, 2
    pre = make_inputs(B, H, 12, d, "bf16", seed=500, lambda0=0.8)
    st = oracle_ref(pre)
    x = make_inputs(B, H, T, d, "bf16", seed=501, lambda0=0.8)
    q, k, v, u = to_device(x)
    dev = q.device
    S = torch.from_numpy(st["S_T"]).float().to(dev).contiguous() if given in ("both", "S0") else None
    A = torch.from_numpy(st["A_T"]).float().to(dev).contiguous() if given in ("both", "A0") else None
    n = torch.from_numpy(st["n_T"]).float().to(dev).contiguous()
    S_T = S if S is not None else torch.empty(B, H, d, d, device=dev)
    A_T = A if A is not None else torch.empty(B, H, d, d, device=dev)
    o, S_out, A_out, n_out = vla.vla_forward(q, k, v, u, x.lambda0, S0=S, A0=A, n0=n, S_T=S_T, A_T=A_T, n_T=n,
                                             kernel=vla.VLA_KERNEL_DECODE)
    torch.cuda.synchronize()
    assert vla.vla_device_status() == vla.VLA_OK
    ref = oracle_ref(x, S0=st["S_T"] if S is not None else None, A0=st["A_T"] if A is not None else None,
                     n0=st["n_T"])
    got = {"o": o.float().cpu().numpy(), "S_T": S_out.cpu().numpy(), "A_T": A_out.cpu().numpy(),
           "n_T": n_out.cpu().numpy()}
    compare(got, ref, "bf16")
