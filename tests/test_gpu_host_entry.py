"""vla_forward_host: the same kernels as vla_forward on staged copies, so the
results are bit-identical; its uploads run on a second stream."""

import pytest
import torch

import rls_associative_memory_gb300 as vla
from synthetic import make_inputs
from vla_testutil import compare, oracle_ref, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kernel,T,dtype", [(vla.VLA_KERNEL_CHUNK_TC, 1000, "bf16"), (vla.VLA_KERNEL_SEQ, 77, "f32"),
                                            (vla.VLA_KERNEL_CHUNK, 300, "bf16"), (vla.VLA_KERNEL_AUTO, 3, "bf16")])
def test_host_entry_matches_device_entry(kernel, T, dtype):
    x = make_inputs(1, 3, T, 64, dtype, seed=61 + T, u_scale=0.5)
    q, k, v, u = to_device(x)
    o_ref, S_ref, A_ref, n_ref = vla.vla_forward(q, k, v, u, x.lambda0, kernel=kernel)
    torch.cuda.synchronize()

    hq, hk, hv, hu = (t.cpu().pin_memory() for t in (q, k, v, u))
    dq, dk, dv, du = (torch.empty_like(t) for t in (q, k, v, u))
    o = torch.empty_like(q)
    ho = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    B, H, _, d = q.shape
    S_T = torch.empty((B, H, d, d), device="cuda")
    A_T = torch.empty_like(S_T)
    n_T = torch.empty((B, H, d), device="cuda")
    hS, hA = torch.empty(S_T.shape).pin_memory(), torch.empty(A_T.shape).pin_memory()
    hn = torch.empty(n_T.shape).pin_memory()
    need = vla.vla_workspace_bytes(B, H, T, d, vla.VLA_BF16 if dtype == "bf16" else vla.VLA_F32, kernel)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    stream, copy_stream = torch.cuda.current_stream(), torch.cuda.Stream()
    vla.vla_forward_host(hq, hk, hv, hu, x.lambda0, dq, dk, dv, du, o, ho, S_T, A_T, n_T, hS, hA, hn,
                         kernel=kernel, workspace=ws, stream=stream, copy_stream=copy_stream)
    stream.synchronize()
    assert torch.equal(ho, o_ref.cpu())
    assert torch.equal(hS, S_ref.cpu()) and torch.equal(hA, A_ref.cpu()) and torch.equal(hn, n_ref.cpu())
    got = {"o": ho.float().numpy(), "S_T": hS.numpy(), "A_T": hA.numpy(), "n_T": hn.numpy()}
    compare(got, oracle_ref(x), dtype)
