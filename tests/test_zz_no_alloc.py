"""vla_forward_noalloc: the chunk-parallel path with the library's built-in
scratch array instead of a caller-provided workspace.

It exists for hosts that keep every byte of device memory under their own
control and forbid components from calling cudaMalloc, such as a serving
runtime that reserves its full memory budget at start-up so a long stream
cannot run out of memory halfway, or a plugin that such a runtime only hands
input and output buffers.  Those callers have no workspace to give
vla_forward.

The checks here call the entry point through the C ABI several times in a
row, with different shapes, dtypes and head sizes, so that each call after
the first runs on whatever the previous one left in the shared array: a
small bf16 problem, then a larger one, then d_h = 128 with a given initial
state (S0, A0, n0).  Each result is compared with the fp64 oracle at the
parity tolerance of the other GPU tests, and with vla_forward's on the same
inputs.  This file is collected last so that a run stopping at its first
failure has already run everything else; it also passes on its own in a
fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import rls_associative_memory_gb300 as vla
from synthetic import make_inputs
from vla_testutil import TOL, oracle_ref, rel_fro, to_device

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(q, k, v, u, lambda0, chunk=0, S0=None, A0=None, n0=None):
    B, H, T, d = q.shape
    dev = q.device
    o = torch.empty_like(q)
    S_T = torch.empty((B, H, d, d), dtype=torch.float32, device=dev)
    A_T = torch.empty_like(S_T)
    n_T = torch.empty((B, H, d), dtype=torch.float32, device=dev)
    io = vla.VLA_BF16 if q.dtype == torch.bfloat16 else vla.VLA_F32
    stream = torch.cuda.current_stream(dev)
    rc = vla.lib().vla_forward_noalloc(_p(q), _p(k), _p(v), _p(u), io, float(lambda0), B, H, T, d,
                                       _p(S0), _p(A0), _p(n0), _p(o), _p(S_T), _p(A_T), _p(n_T), chunk,
                                       ctypes.c_void_p(stream.cuda_stream))
    return rc, (o, S_T, A_T, n_T)


def _host(ts):
    return [t.float().cpu().numpy().astype(np.float64) for t in ts]


def _state(x, dev):
    """A state reached by the oracle after a short prefix stream."""
    ref = oracle_ref(x)
    return [torch.from_numpy(np.ascontiguousarray(ref[n], dtype=np.float32)).to(dev)
            for n in ("S_T", "A_T", "n_T")], ref


def test_noalloc_matches_oracle_and_vla_forward_on_calls_in_a_row():
    # a B = 0 call does the set-up only (no pointers needed)
    assert vla.lib().vla_forward_noalloc(None, None, None, None, vla.VLA_BF16, 1.0, 0, 0, 0, 64, None, None,
                                         None, None, None, None, None, 0, None) == vla.VLA_OK
    pre = make_inputs(1, 2, 60, 128, "f32", seed=44, lambda0=0.6)
    cases = [
        # (inputs, chunk, initial state from a prefix stream or None)
        (make_inputs(1, 3, 777, 32, "f32", seed=42, lambda0=0.7), 32, None),
        (make_inputs(2, 4, 2000, 64, "bf16", seed=41, u_scale=0.5, lambda0=1.0), 0, None),
        (make_inputs(1, 2, 300, 128, "f32", seed=43, lambda0=0.6), 0, pre),
    ]
    for x, chunk, prefix in cases:
        q, k, v, u = to_device(x)
        S0 = A0 = n0 = None
        kw = {}
        if prefix is not None:
            (S0, A0, n0), st = _state(prefix, q.device)
            kw = dict(S0=st["S_T"], A0=st["A_T"], n0=st["n_T"])
        rc, got = _noalloc(q, k, v, u, x.lambda0, chunk, S0, A0, n0)
        assert rc == vla.VLA_OK, vla.vla_status_str(rc)
        ref = vla.vla_forward(q, k, v, u, x.lambda0, S0=S0, A0=A0, n0=n0, kernel=vla.VLA_KERNEL_CHUNK,
                              chunk=chunk)
        torch.cuda.synchronize()
        assert vla.vla_device_status() == vla.VLA_OK
        oracle = oracle_ref(x, **kw)
        for name, a, b in zip(("o", "S_T", "A_T", "n_T"), _host(got), _host(ref)):
            err_oracle = rel_fro(a, oracle[name])
            assert err_oracle <= TOL[x.dtype], (x.q.shape, name, "vs oracle", err_oracle)
            err = rel_fro(a, b)
            assert err <= TOL[x.dtype], (x.q.shape, name, "vs vla_forward", err)


def test_noalloc_rejects_problems_beyond_its_scratch():
    # the long stream's chunked workspace (~540 MB) is far beyond 64 MiB;
    # the call must refuse before touching the (never dereferenced) buffers
    need = vla.vla_workspace_bytes(1, 16, 65536, 64, vla.VLA_BF16, vla.VLA_KERNEL_CHUNK)
    assert need > vla.VLA_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)
    rc = vla.lib().vla_forward_noalloc(fake, fake, fake, fake, vla.VLA_BF16, 1.0, 1, 16, 65536, 64,
                                       None, None, None, fake, fake, fake, None, 0, None)
    assert rc == vla.VLA_ERR_SCRATCH_LIMIT
    assert "scratch" in vla.vla_status_str(rc)
