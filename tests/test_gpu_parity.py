"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.  Bar: relative Frobenius error per tensor (o, S_T,
A_T, n_T) <= 1e-4 for fp32 I/O and <= 5e-3 for bf16 I/O with fp32 state."""

import numpy as np
import pytest
import torch

import oracle
import rls_associative_memory_gb300 as vla
from synthetic import make_config, make_inputs
from vla_testutil import TOL, compare, oracle_ref, rel_fro, run_gpu, to_device, window_errors

pytestmark = pytest.mark.gpu

KERNELS = [vla.VLA_KERNEL_SEQ, vla.VLA_KERNEL_CHUNK, vla.VLA_KERNEL_CHUNK_TC]
# (kernel, chunk length): the chunked path with a short explicit chunk spans
# many chunks and a ragged last chunk even on small streams.  CHUNK_TC runs
# its tensor-core state passes at d = 64 with bf16 I/O (chunks of 64 and 128
# tokens: one and two sub-blocks) and the plain chunked path elsewhere.
VARIANTS = [(vla.VLA_KERNEL_SEQ, 0), (vla.VLA_KERNEL_CHUNK, 32), (vla.VLA_KERNEL_CHUNK, 0),
            (vla.VLA_KERNEL_CHUNK_TC, 0), (vla.VLA_KERNEL_CHUNK_TC, 128)]


def _kid(k):
    return {vla.VLA_KERNEL_SEQ: "seq", vla.VLA_KERNEL_CHUNK: "chunk", vla.VLA_KERNEL_CHUNK_TC: "chunk_tc",
            vla.VLA_KERNEL_AUTO: "auto"}[k]


def _vid(v):
    return "%s%s" % (_kid(v[0]), ("-c%d" % v[1]) if v[1] else "")


# --- small shapes: several tiles, ragged tails, every d and dtype ---

@pytest.mark.parametrize("variant", VARIANTS, ids=_vid)
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 17, 100, 333])
def test_small_parity(variant, d, dtype, T):
    kernel, chunk = variant
    x = make_inputs(2, 3, T, d, dtype, seed=1000 + d + T, lambda0=0.8)
    compare(run_gpu(x, kernel, chunk=chunk), oracle_ref(x), dtype)


@pytest.mark.parametrize("variant", VARIANTS, ids=_vid)
@pytest.mark.parametrize("d", [32, 64, 128])
def test_given_initial_state(variant, d):
    """S0, A0, n0 supplied (streaming continuation)."""
    kernel, chunk = variant
    pre = make_inputs(1, 2, 40, d, "f32", seed=7, lambda0=1.3)
    st = oracle_ref(pre)
    x = make_inputs(1, 2, 77, d, "f32", seed=8, lambda0=1.3)
    ref = oracle_ref(x, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"])
    got = run_gpu(x, kernel, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"], chunk=chunk)
    compare(got, ref, "f32")


@pytest.mark.parametrize("chunk", [16, 48, 64, 128, 256])
def test_chunk_lengths(chunk):
    """Every chunk length gives the same result (one ragged last chunk)."""
    x = make_inputs(1, 4, 1000, 64, "bf16", seed=31, u_scale=0.5)
    compare(run_gpu(x, vla.VLA_KERNEL_CHUNK, chunk=chunk), oracle_ref(x), "bf16")


@pytest.mark.parametrize("chunk", [0, 128])
def test_tensor_core_path_given_initial_state(chunk):
    """bf16 streaming continuation on the tensor-core path: the first A-chunk
    starts from the given A0, later ones from the inverse of the prefix."""
    pre = make_inputs(1, 3, 150, 64, "bf16", seed=51, lambda0=0.9, u_scale=0.5)
    st = oracle_ref(pre)
    x = make_inputs(1, 3, 1000, 64, "bf16", seed=52, lambda0=0.9, u_scale=0.5)
    ref = oracle_ref(x, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"])
    got = run_gpu(x, vla.VLA_KERNEL_CHUNK_TC, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"], chunk=chunk)
    compare(got, ref, "bf16")


@pytest.mark.parametrize("chunk", [64, 192, 512])
@pytest.mark.parametrize("T", [64, 1000, 1536])
def test_tensor_core_state_passes(chunk, T):
    """The UT-transform state passes (d = 64, bf16): whole and ragged
    sub-blocks, one to eight sub-blocks per chunk, one or several chunks."""
    x = make_inputs(1, 4, T, 64, "bf16", seed=41 + T, u_scale=0.5)
    compare(run_gpu(x, vla.VLA_KERNEL_CHUNK_TC, chunk=chunk), oracle_ref(x), "bf16")


@pytest.mark.parametrize("kernel", KERNELS, ids=_kid)
def test_split_stream_on_gpu(kernel):
    """Two calls with the state handed over equal one call (in-place state buffers)."""
    x = make_inputs(2, 2, 300, 64, "bf16", seed=21)
    q, k, v, u = to_device(x)
    o_full, S_full, A_full, n_full = vla.vla_forward(q, k, v, u, x.lambda0, kernel=kernel)
    t = 123
    sl = lambda a, lo, hi: a[:, :, lo:hi].contiguous()  # noqa: E731
    o1, S, A, n = vla.vla_forward(sl(q, 0, t), sl(k, 0, t), sl(v, 0, t), sl(u, 0, t), x.lambda0,
                                  kernel=kernel)
    o2, S2, A2, n2 = vla.vla_forward(sl(q, t, 300), sl(k, t, 300), sl(v, t, 300), sl(u, t, 300),
                                     x.lambda0, S0=S, A0=A, n0=n, S_T=S, A_T=A, n_T=n, kernel=kernel)
    torch.cuda.synchronize()
    assert S2.data_ptr() == S.data_ptr()
    ref = oracle_ref(x)
    o_cat = torch.cat([o1, o2], dim=2).float().cpu().numpy()
    assert rel_fro(o_cat, ref["o"]) < TOL["bf16"]
    assert rel_fro(S.cpu().numpy(), ref["S_T"]) < TOL["bf16"]
    assert rel_fro(A.cpu().numpy(), ref["A_T"]) < TOL["bf16"]
    assert rel_fro(n.cpu().numpy(), ref["n_T"]) < TOL["bf16"]
    assert rel_fro(o_cat, o_full.float().cpu().numpy()) < 1e-3


@pytest.mark.parametrize("kernel", KERNELS, ids=_kid)
def test_empty_stream_copies_state(kernel):
    d = 64
    dev = "cuda"
    e = torch.empty((1, 2, 0, d), dtype=torch.float32, device=dev)
    S0 = torch.randn(1, 2, d, d, device=dev)
    A0 = torch.eye(d, device=dev).expand(1, 2, d, d).contiguous() * 0.3
    n0 = torch.rand(1, 2, d, device=dev)
    o, S, A, n = vla.vla_forward(e, e, e, e, 1.0, S0=S0, A0=A0, n0=n0, kernel=kernel)
    torch.cuda.synchronize()
    assert torch.equal(S, S0) and torch.equal(A, A0) and torch.equal(n, n0)
    o, S, A, n = vla.vla_forward(e, e, e, e, 0.5, kernel=kernel)
    torch.cuda.synchronize()
    assert torch.equal(A[0, 0], 2.0 * torch.eye(d, device=dev)) and not S.any() and not n.any()


def test_unsupported_and_misaligned_rejected():
    x = make_inputs(1, 1, 8, 64, "f32", seed=3)
    q, k, v, u = to_device(x)
    with pytest.raises(vla.VLAError) as ei:
        vla.vla_forward(q[..., :48].contiguous(), k[..., :48].contiguous(), v[..., :48].contiguous(),
                        u[..., :48].contiguous(), 1.0)
    assert ei.value.status == vla.VLA_ERR_UNSUPPORTED_DIM
    big = torch.zeros(1 * 1 * 8 * 64 + 1, device="cuda")
    qm = big[1:].view(1, 1, 8, 64)  # 4-byte offset: not 16-byte aligned
    with pytest.raises(vla.VLAError) as ei:
        vla.vla_forward(qm, k, v, u, 1.0)
    assert ei.value.status == vla.VLA_ERR_ALIGN


def test_bounded_wait_expiry_reports_timeout_and_context_survives():
    """Test hook: the first input tile is never requested, so the kernel's
    bounded wait expires (1 ms limit), sets the device error word and
    returns; the host reads VLA_ERR_TIMEOUT and the next call is normal."""
    x = make_inputs(1, 2, 64, 64, "bf16", seed=5)
    q, k, v, u = to_device(x)
    assert vla.vla_debug_inject(1, 1_000_000) == vla.VLA_OK
    try:
        vla.vla_forward(q, k, v, u, 1.0, kernel=vla.VLA_KERNEL_SEQ)
        assert vla.vla_device_status() == vla.VLA_ERR_TIMEOUT
    finally:
        vla.vla_debug_inject(0)
    assert vla.vla_device_status() == vla.VLA_OK
    compare(run_gpu(x, vla.VLA_KERNEL_SEQ), oracle_ref(x), "bf16")


# --- full-size workloads ---

FULL = ["tiny", "heads32", "long", "batched", "recall8", "recall24", "recall48"]


_CACHE = {}


def _full_inputs(name):
    # one generated batch per workload, shared by both kernels
    if name not in _CACHE:
        _CACHE.clear()
        _CACHE[name] = make_config(name)
    return _CACHE[name]


def _sample_heads(x, limit=64):
    B, H = x.q.shape[:2]
    idx = np.linspace(0, B * H - 1, min(limit, B * H)).round().astype(int)
    return np.unique(idx)


@pytest.mark.parametrize("name", FULL)
@pytest.mark.parametrize("kernel", KERNELS, ids=_kid)
def test_full_config_parity(kernel, name):
    x = _full_inputs(name)
    got = run_gpu(x, kernel)
    B, H, T, d = x.q.shape
    heads = _sample_heads(x)
    flat = lambda a: a.reshape((B * H,) + a.shape[2:])  # noqa: E731
    qs, ks, vs, us = (flat(x.as_f64(n))[heads] for n in "qkvu")
    ref = oracle.forward(qs, ks, vs, us, x.lambda0)
    sub = {key: flat(val)[heads] for key, val in got.items()}
    errs = compare(sub, ref, x.dtype)
    print("\n%s %s heads=%d errs=%s" % (name, _kid(kernel), len(heads), errs))
    # o over windows of the stream (the late tokens carry little of the whole
    # tensor's norm under the 1/t decay of the readout)
    win = 4096 if T >= 8192 else max(64, T // 8)
    wins, last = window_errors(sub["o"], ref["o"], win)
    print("o per %d-token window: max %.3g (window %d), last %d tokens %.3g"
          % (win, max(wins), int(np.argmax(wins)), win, last))
    assert max(wins) <= TOL[x.dtype] and last <= TOL[x.dtype], (wins, last)
    if x.keys is not None:
        # recall measurement: |S_T key_i - value_i| from the GPU state vs the oracle's
        keys = flat(x.keys)[heads]
        vals = flat(x.values)[heads]
        rec_gpu = np.linalg.norm(np.einsum("bij,bnj->bni", sub["S_T"], keys) - vals, axis=-1)
        rec_ref = np.linalg.norm(np.einsum("bij,bnj->bni", ref["S_T"], keys) - vals, axis=-1)
        assert abs(rec_gpu.mean() - rec_ref.mean()) <= 1e-3 * max(1.0, rec_ref.mean())
        print("recall error mean gpu=%.5f oracle=%.5f" % (rec_gpu.mean(), rec_ref.mean()))
