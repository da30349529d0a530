"""vla_forward_host: the same kernels as vla_forward on staged copies, so the
results are bit-identical to vla_forward run on each staged range of units
with that range's chunk lengths (on the tensor-core path at d = 64 the ranges
are problems of their own, vla_host_ranges); its uploads run on a second
stream, and o comes back on the compute or copy stream, or on a third one when
given."""

import pytest
import torch

import rls_associative_memory_gb300 as vla
from synthetic import make_inputs
from vla_testutil import compare, oracle_ref, to_device

pytestmark = pytest.mark.gpu


def _device_reference(q, k, v, u, lam, kernel, S0=None, A0=None, n0=None):
    """vla_forward as the host entry runs it: per staged range with the range's
    chunk lengths where the call stages ranges of its own, else in one call."""
    B, H, T, d = q.shape
    io = vla.VLA_BF16 if q.dtype == torch.bfloat16 else vla.VLA_F32
    ranges = vla.vla_host_ranges(B, H, T, d, io, kernel)
    if not ranges:
        return vla.vla_forward(q, k, v, u, lam, S0=S0, A0=A0, n0=n0, kernel=kernel)
    flat = lambda t: None if t is None else t.reshape(B * H, *t.shape[2:])  # noqa: E731
    outs = []
    for lo, n, C, CA in ranges:
        assert CA == C, "an explicit chunk length sets both"
        sl = lambda t: None if t is None else flat(t)[lo:lo + n].unsqueeze(0).contiguous()  # noqa: E731
        outs.append(vla.vla_forward(sl(q), sl(k), sl(v), sl(u), lam, S0=sl(S0), A0=sl(A0), n0=sl(n0),
                                    kernel=kernel, chunk=C))
    return tuple(torch.cat([o[i][0] for o in outs]).reshape(B, H, *outs[0][i].shape[2:]) for i in range(4))


@pytest.mark.parametrize("kernel,B,H,T,dtype,init", [
    (vla.VLA_KERNEL_CHUNK_TC, 1, 3, 1000, "bf16", False),  # ranges of units 1 | 1 | 1
    (vla.VLA_KERNEL_CHUNK_TC, 1, 2, 700, "bf16", False),   # 1 | 1 (two ranges)
    (vla.VLA_KERNEL_CHUNK_TC, 2, 4, 1000, "bf16", True),   # 4 | 2 | 2, A0 inverted per range
    (vla.VLA_KERNEL_CHUNK_TC, 1, 5, 640, "bf16", False),   # 2 | 1 | 2
    (vla.VLA_KERNEL_CHUNK_TC, 2, 8, 2048, "bf16", True),   # 8 | 4 | 4 with their own chunk lengths
    (vla.VLA_KERNEL_SEQ, 1, 3, 77, "f32", False), (vla.VLA_KERNEL_CHUNK, 1, 3, 300, "bf16", False),
    (vla.VLA_KERNEL_AUTO, 1, 3, 3, "bf16", False)])
@pytest.mark.parametrize("download", [False, True], ids=["two_streams", "download_stream"])
def test_host_entry_matches_device_entry(kernel, B, H, T, dtype, init, download):
    x = make_inputs(B, H, T, 64, dtype, seed=61 + T, u_scale=0.5)
    q, k, v, u = to_device(x)
    S0 = A0 = n0 = None
    ref0 = {}
    if init:
        pre = make_inputs(B, H, 90, 64, dtype, seed=60 + T, u_scale=0.5)
        st = oracle_ref(pre)
        S0, A0, n0 = (torch.from_numpy(st[n]).float().cuda().contiguous() for n in ("S_T", "A_T", "n_T"))
        ref0 = dict(S0=st["S_T"], A0=st["A_T"], n0=st["n_T"])
    o_ref, S_ref, A_ref, n_ref = _device_reference(q, k, v, u, x.lambda0, kernel, S0=S0, A0=A0, n0=n0)
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
                         S0=S0, A0=A0, n0=n0, kernel=kernel, workspace=ws, stream=stream, copy_stream=copy_stream,
                         download_stream=torch.cuda.Stream() if download else None)
    stream.synchronize()
    assert torch.equal(ho, o_ref.cpu())
    assert torch.equal(hS, S_ref.cpu()) and torch.equal(hA, A_ref.cpu()) and torch.equal(hn, n_ref.cpu())
    got = {"o": ho.float().numpy(), "S_T": hS.numpy(), "A_T": hA.numpy(), "n_T": hn.numpy()}
    compare(got, oracle_ref(x, **ref0), dtype)


def _host_call(x, kernel, S0=None, A0=None, n0=None, in_place=False):
    q, k, v, u = to_device(x)
    B, H, T, d = q.shape
    hq, hk, hv, hu = (t.cpu().pin_memory() for t in (q, k, v, u))
    dq, dk, dv, du = (torch.empty_like(t) for t in (q, k, v, u))
    o = torch.empty_like(q)
    ho = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    if in_place:
        S_T, A_T, n_T = S0, A0, n0
    else:
        S_T = torch.empty((B, H, d, d), device="cuda")
        A_T = torch.empty_like(S_T)
        n_T = torch.empty((B, H, d), device="cuda")
    hS, hA = torch.empty(S_T.shape).pin_memory(), torch.empty(A_T.shape).pin_memory()
    hn = torch.empty(n_T.shape).pin_memory()
    io = vla.VLA_BF16 if q.dtype == torch.bfloat16 else vla.VLA_F32
    need = vla.vla_workspace_bytes(B, H, T, d, io, kernel)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    vla.vla_forward_host(hq, hk, hv, hu, x.lambda0, dq, dk, dv, du, o, ho, S_T, A_T, n_T, hS, hA, hn, S0=S0, A0=A0,
                         n0=n0, kernel=kernel, workspace=ws, stream=stream, copy_stream=torch.cuda.Stream())
    stream.synchronize()
    return {"o": ho.float().numpy(), "S_T": hS.numpy(), "A_T": hA.numpy(), "n_T": hn.numpy()}


@pytest.mark.parametrize("kernel", [vla.VLA_KERNEL_CHUNK_TC, vla.VLA_KERNEL_SEQ])
def test_host_entry_given_initial_state(kernel):
    """Streaming continuation through the host entry (A0 given adds the chunked
    path's A0 inversion before the passes that read u and k)."""
    pre = make_inputs(1, 3, 150, 64, "bf16", seed=71, lambda0=0.9, u_scale=0.5)
    st = oracle_ref(pre)
    x = make_inputs(1, 3, 1000, 64, "bf16", seed=72, lambda0=0.9, u_scale=0.5)
    S0, A0, n0 = (torch.from_numpy(st[n]).float().cuda() for n in ("S_T", "A_T", "n_T"))
    got = _host_call(x, kernel, S0=S0, A0=A0, n0=n0)
    compare(got, oracle_ref(x, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"]), "bf16")


def test_host_entry_single_unit():
    """One (b, h) unit: no halves to split into."""
    x = make_inputs(1, 1, 2000, 64, "bf16", seed=73, u_scale=0.5)
    compare(_host_call(x, vla.VLA_KERNEL_CHUNK_TC), oracle_ref(x), "bf16")


def test_host_entry_decode_in_place():
    """Decode steps with the state updated in place on the device."""
    pre = make_inputs(2, 4, 100, 64, "bf16", seed=74)
    st = oracle_ref(pre)
    x = make_inputs(2, 4, 2, 64, "bf16", seed=75)
    S, A, n = (torch.from_numpy(st[k]).float().cuda().contiguous() for k in ("S_T", "A_T", "n_T"))
    got = _host_call(x, vla.VLA_KERNEL_DECODE, S0=S, A0=A, n0=n, in_place=True)
    compare(got, oracle_ref(x, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"]), "bf16")


def test_host_entry_one_stream():
    """copy_stream == stream: the ranges run one after another, same results."""
    x = make_inputs(1, 3, 700, 64, "bf16", seed=76, u_scale=0.5)
    q, k, v, u = to_device(x)
    o_ref, S_ref, A_ref, n_ref = _device_reference(q, k, v, u, x.lambda0, vla.VLA_KERNEL_CHUNK_TC)
    torch.cuda.synchronize()
    hq, hk, hv, hu = (t.cpu().pin_memory() for t in (q, k, v, u))
    dq, dk, dv, du = (torch.empty_like(t) for t in (q, k, v, u))
    o = torch.empty_like(q)
    ho = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    S_T, A_T, n_T = torch.empty_like(S_ref), torch.empty_like(A_ref), torch.empty_like(n_ref)
    hS, hA, hn = (torch.empty(t.shape).pin_memory() for t in (S_T, A_T, n_T))
    B, H, T, d = q.shape
    ws = torch.empty(vla.vla_workspace_bytes(B, H, T, d, vla.VLA_BF16, vla.VLA_KERNEL_CHUNK_TC), dtype=torch.uint8,
                     device="cuda")
    stream = torch.cuda.current_stream()
    vla.vla_forward_host(hq, hk, hv, hu, x.lambda0, dq, dk, dv, du, o, ho, S_T, A_T, n_T, hS, hA, hn,
                         kernel=vla.VLA_KERNEL_CHUNK_TC, workspace=ws, stream=stream, copy_stream=stream)
    stream.synchronize()
    assert torch.equal(ho, o_ref.cpu())
    assert torch.equal(hS, S_ref.cpu()) and torch.equal(hA, A_ref.cpu()) and torch.equal(hn, n_ref.cpu())


@pytest.mark.parametrize("B,H,T", [(1, 2, 200), (2, 80, 130), (5, 64, 70)])
@pytest.mark.parametrize("download", [False, True], ids=["two_streams", "download_stream"])
def test_host_entry_d128_one_chunk_per_unit(B, H, T, download):
    """d = 128 with one chunk per unit: ranges of at most 152 units (one wave),
    u and k up first with each range's gates, then q and v with each range's
    state pass; bit-identical to vla_forward."""
    x = make_inputs(B, H, T, 128, "bf16", seed=90 + T, lambda0=0.5)
    q, k, v, u = to_device(x)
    chunk = (T + 63) // 64 * 64
    kern = vla.VLA_KERNEL_CHUNK_TC
    o_ref, S_ref, A_ref, n_ref = vla.vla_forward(q, k, v, u, x.lambda0, kernel=kern, chunk=chunk)
    torch.cuda.synchronize()
    assert vla.vla_last_launch_count() == 1  # the queue kernel; the ranges below run the two passes apart
    hq, hk, hv, hu = (t.cpu().pin_memory() for t in (q, k, v, u))
    dq, dk, dv, du = (torch.empty_like(t) for t in (q, k, v, u))
    o = torch.empty_like(q)
    ho = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    d = 128
    S_T = torch.empty((B, H, d, d), device="cuda")
    A_T = torch.empty_like(S_T)
    n_T = torch.empty((B, H, d), device="cuda")
    hS, hA = torch.empty(S_T.shape).pin_memory(), torch.empty(A_T.shape).pin_memory()
    hn = torch.empty(n_T.shape).pin_memory()
    ws = torch.empty(vla.vla_workspace_bytes(B, H, T, d, vla.VLA_BF16, kern, chunk), dtype=torch.uint8, device="cuda")
    stream, copy_stream = torch.cuda.current_stream(), torch.cuda.Stream()
    vla.vla_forward_host(hq, hk, hv, hu, x.lambda0, dq, dk, dv, du, o, ho, S_T, A_T, n_T, hS, hA, hn, kernel=kern,
                         chunk=chunk, workspace=ws, stream=stream, copy_stream=copy_stream,
                         download_stream=torch.cuda.Stream() if download else None)
    stream.synchronize()
    nr = min(4, (B * H + 151) // 152)
    assert vla.vla_last_launch_count() == 2 * nr
    assert torch.equal(ho, o_ref.cpu())
    assert torch.equal(hS, S_ref.cpu()) and torch.equal(hA, A_ref.cpu()) and torch.equal(hn, n_ref.cpu())


@pytest.mark.parametrize("download", [False, True], ids=["two_streams", "download_stream"])
@pytest.mark.parametrize("B,H,T", [(8, 4, 130), (1, 2, 40)])
def test_host_entry_sequential_ranges(B, H, T, download):
    """The sequential kernel (d = 32 here) staged in ranges of units: each
    range's inputs up, its launch over the range's slices, its o back;
    bit-identical to vla_forward."""
    x = make_inputs(B, H, T, 32, "f32", seed=95 + T, lambda0=0.8)
    q, k, v, u = to_device(x)
    kern = vla.VLA_KERNEL_SEQ
    o_ref, S_ref, A_ref, n_ref = vla.vla_forward(q, k, v, u, x.lambda0, kernel=kern)
    torch.cuda.synchronize()
    hq, hk, hv, hu = (t.cpu().pin_memory() for t in (q, k, v, u))
    dq, dk, dv, du = (torch.empty_like(t) for t in (q, k, v, u))
    o = torch.empty_like(q)
    ho = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    d = 32
    S_T = torch.empty((B, H, d, d), device="cuda")
    A_T = torch.empty_like(S_T)
    n_T = torch.empty((B, H, d), device="cuda")
    hS, hA = torch.empty(S_T.shape).pin_memory(), torch.empty(A_T.shape).pin_memory()
    hn = torch.empty(n_T.shape).pin_memory()
    stream, copy_stream = torch.cuda.current_stream(), torch.cuda.Stream()
    vla.vla_forward_host(hq, hk, hv, hu, x.lambda0, dq, dk, dv, du, o, ho, S_T, A_T, n_T, hS, hA, hn, kernel=kern,
                         stream=stream, copy_stream=copy_stream,
                         download_stream=torch.cuda.Stream() if download else None)
    stream.synchronize()
    assert vla.vla_last_launch_count() == min(4, B * H)
    assert torch.equal(ho, o_ref.cpu())
    assert torch.equal(hS, S_ref.cpu()) and torch.equal(hA, A_ref.cpu()) and torch.equal(hn, n_ref.cpu())
    compare({"o": ho.numpy(), "S_T": hS.numpy(), "A_T": hA.numpy(), "n_T": hn.numpy()}, oracle_ref(x), "f32")


@pytest.mark.parametrize("init", [False, True], ids=["default_state", "given_state"])
def test_host_entry_halves_with_their_own_chunks(init):
    """1 x 16 x 65536 (the long stream's shape): the first half (8 units) at the
    whole problem's chunk length, then two ranges of 4 at the second half's
    own, each bit-identical to vla_forward on its units with its chunk length;
    the last unit of every range against the oracle.  With a given state each
    half inverts its own A0 before its front."""
    x = make_inputs(1, 16, 65536, 64, "bf16", seed=77, u_scale=0.5)
    q, k, v, u = to_device(x)
    S0 = A0 = n0 = None
    ref0 = {}
    if init:
        pre = make_inputs(1, 16, 200, 64, "bf16", seed=78, u_scale=0.5)
        st = oracle_ref(pre)
        S0, A0, n0 = (torch.from_numpy(st[nm]).float().cuda().contiguous() for nm in ("S_T", "A_T", "n_T"))
        ref0 = dict(S0=st["S_T"], A0=st["A_T"], n0=st["n_T"])
    ranges = vla.vla_host_ranges(1, 16, 65536, 64, vla.VLA_BF16, vla.VLA_KERNEL_AUTO)
    assert len({r[2] for r in ranges}) == 2, ranges  # the halves do not share one chunk length
    o_ref, S_ref, A_ref, n_ref = _device_reference(q, k, v, u, x.lambda0, vla.VLA_KERNEL_AUTO, S0=S0, A0=A0, n0=n0)
    torch.cuda.synchronize()
    got = _host_call(x, vla.VLA_KERNEL_AUTO, S0=S0, A0=A0, n0=n0)
    assert (got["o"] == o_ref.float().cpu().numpy()).all()
    assert (got["S_T"] == S_ref.cpu().numpy()).all() and (got["A_T"] == A_ref.cpu().numpy()).all()
    for lo, n, C, CA in ranges:
        b, h = divmod(lo + n - 1, 16)
        sub0 = {key: val[b:b + 1, h:h + 1] for key, val in ref0.items()}
        ref = oracle_ref(x.slice_heads(slice(b, b + 1), slice(h, h + 1)), **sub0)  # the range's last unit
        compare({key: val[b:b + 1, h:h + 1] for key, val in got.items()}, ref, "bf16")
