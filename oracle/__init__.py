"""fp64 CPU oracle for the VLA forward recurrence.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check and by
the benchmark's CPU-baseline and reference legs, never by the product
package.  The arithmetic lives in ``vla_oracle.c`` (plain C, fp64, token by
token, in the order of "Variational Linear Attention: Stable Associative
Memory for Long-Context Transformers", sections 2.2-2.3); this module only
compiles it with gcc and marshals numpy arrays.

Parity is pinned by ``tests/test_oracle_pins.py`` against explicit matrix
inversion, closed forms, textbook special cases (delta rule, recursive least
squares / ridge regression) and invariants.  The readout (ELU+1 ratio) is a
reading of an under-specified passage; its pins are decompositions into
library routines, not values printed by the pages.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vla_oracle.c")
_LIB = os.path.join(_HERE, "libvla_oracle.so")
_lock = threading.Lock()
_lib = None

EPS = 1e-6
FLAG_UNNORMALISED_GATE = 1


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (IEEE fp64: no FMA contraction, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-pthread", "-o", tmp, _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.vla_oracle_forward.argtypes = [dp, dp, dp, dp, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_double, dp, dp, dp,
                                               dp, dp, dp, dp, dp, dp, dp, ctypes.c_int,
                                               ctypes.c_int]
            lib.vla_oracle_forward.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a, shape):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.float64)
    if a.shape != shape:
        a = a.reshape(shape)
    return a


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def forward(q, k, v, u, lambda0: float, S0=None, A0=None, n0=None, trace: bool = False,
            unnormalised_gate: bool = False, nthreads: Optional[int] = None) -> dict:
    """Run the recurrence in fp64.

    q, k, v, u: ``[..., T, d]`` arrays (any float dtype; upcast exactly to
    fp64); the leading dims are independent (batch, head) units.  S0, A0:
    ``[..., d, d]``; n0: ``[..., d]`` (each optional).  Returns a dict with
    ``o [..., T, d]``, ``S_T``, ``A_T [..., d, d]``, ``n_T [..., d]`` and, with
    ``trace``, ``alpha [..., T, d]`` (the gate used at each step), ``c [..., T]``
    (alpha_t . k_hat_t) and ``snorm [..., T]`` (Frobenius norm of S_t).
    """
    q = np.asarray(q)
    lead = q.shape[:-2]
    T, d = q.shape[-2], q.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    tok = (BH, T, d)
    qa, ka, va, ua = (_f64(x, tok) for x in (q, k, v, u))
    S0a = _f64(S0, (BH, d, d))
    A0a = _f64(A0, (BH, d, d))
    n0a = _f64(n0, (BH, d))
    o = np.empty(tok)
    S_T = np.empty((BH, d, d))
    A_T = np.empty((BH, d, d))
    n_T = np.empty((BH, d))
    al = np.empty(tok) if trace else None
    c = np.empty((BH, T)) if trace else None
    sn = np.empty((BH, T)) if trace else None
    flags = FLAG_UNNORMALISED_GATE if unnormalised_gate else 0
    nt = default_threads() if nthreads is None else nthreads
    rc = _load().vla_oracle_forward(_ptr(qa), _ptr(ka), _ptr(va), _ptr(ua), BH, T, d,
                                    float(lambda0), _ptr(S0a), _ptr(A0a), _ptr(n0a), _ptr(o),
                                    _ptr(S_T), _ptr(A_T), _ptr(n_T), _ptr(al), _ptr(c),
                                    _ptr(sn), flags, nt)
    if rc != 0:
        raise ValueError("vla_oracle_forward rejected its arguments (rc=%d)" % rc)
    out = {"o": o.reshape(lead + (T, d)), "S_T": S_T.reshape(lead + (d, d)),
           "A_T": A_T.reshape(lead + (d, d)), "n_T": n_T.reshape(lead + (d,))}
    if trace:
        out["alpha"] = al.reshape(lead + (T, d))
        out["c"] = c.reshape(lead + (T,))
        out["snorm"] = sn.reshape(lead + (T,))
    return out


def forward_inputs(x, S0=None, A0=None, n0=None, **kw) -> dict:
    """``forward`` on a ``synthetic.VLAInputs`` batch (exact fp64 upcast)."""
    return forward(x.as_f64("q"), x.as_f64("k"), x.as_f64("v"), x.as_f64("u"), x.lambda0,
                   S0=S0, A0=A0, n0=n0, **kw)
