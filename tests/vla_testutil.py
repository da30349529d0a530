"""Helpers shared by the GPU tests: move synthetic inputs to the device, run
the CUDA path through the binding, and compare with the oracle."""

import numpy as np
import torch

import oracle
import rls_associative_memory_gb300 as vla

# parity bar: relative Frobenius error per tensor
TOL = {"f32": 1e-4, "bf16": 5e-3}


def to_device(x, dev="cuda"):
    out = []
    for n in "qkvu":
        a = getattr(x, n)
        if x.dtype == "bf16":
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
        out.append(t.to(dev))
    return out


def run_gpu(x, kernel=vla.VLA_KERNEL_AUTO, S0=None, A0=None, n0=None, chunk=0):
    q, k, v, u = to_device(x)
    dev = q.device

    def st(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)

    o, S_T, A_T, n_T = vla.vla_forward(q, k, v, u, x.lambda0, S0=st(S0), A0=st(A0), n0=st(n0),
                                       kernel=kernel, chunk=chunk)
    torch.cuda.synchronize()
    assert vla.vla_device_status() == vla.VLA_OK
    return {"o": o.float().cpu().numpy().astype(np.float64), "S_T": S_T.cpu().numpy().astype(np.float64),
            "A_T": A_T.cpu().numpy().astype(np.float64), "n_T": n_T.cpu().numpy().astype(np.float64)}


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    nb = np.linalg.norm(b)
    if nb == 0.0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def compare(gpu, ref, dtype, keys=("o", "S_T", "A_T", "n_T")):
    errs = {k: rel_fro(gpu[k], ref[k]) for k in keys}
    tol = TOL[dtype]
    print("parity errors (tol %g): %s" % (tol, " ".join("%s %.3g" % kv for kv in errs.items())))
    bad = {k: e for k, e in errs.items() if not (e <= tol)}
    assert not bad, "parity failed (tol %g): %s" % (tol, errs)
    return errs


def oracle_ref(x, **kw):
    return oracle.forward_inputs(x, **kw)


def window_errors(o_gpu, o_ref, win):
    """Relative Frobenius error of o over consecutive token windows of `win`
    tokens (the last one ragged) and over the last `win` tokens: under the
    readout's 1/t decay a whole-tensor ratio is dominated by the early
    tokens, these show the late ones."""
    T = o_ref.shape[-2]
    wins = [rel_fro(o_gpu[..., a:min(T, a + win), :], o_ref[..., a:min(T, a + win), :]) for a in range(0, T, win)]
    last = rel_fro(o_gpu[..., max(0, T - win):, :], o_ref[..., max(0, T - win):, :])
    return wins, last
