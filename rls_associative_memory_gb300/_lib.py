"""ctypes binding of libvla (include/vla.h).  Argument marshalling only.

The functions here carry the C names.  ``vla_forward`` accepts torch CUDA
tensors, allocates missing outputs and the workspace with torch (device
memory is PyTorch's job here), and passes raw device pointers and the
current CUDA stream to the C entry point.  Every step of the recurrence runs
in the library's kernels; there is no CPU fallback, and a missing or
unloadable library raises.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

from . import build as _build

VLA_OK = 0
VLA_ERR_ARG = -1
VLA_ERR_UNSUPPORTED_DIM = -2
VLA_ERR_ALIGN = -3
VLA_ERR_WORKSPACE = -4
VLA_ERR_CUDA = -5
VLA_ERR_TIMEOUT = -6
VLA_ERR_SCRATCH_LIMIT = -7
VLA_NOALLOC_SCRATCH_BYTES = 64 << 20

VLA_F32 = 0
VLA_BF16 = 1

VLA_KERNEL_AUTO = 0
VLA_KERNEL_SEQ = 1
VLA_KERNEL_CHUNK = 2
VLA_KERNEL_DECODE = 3
VLA_KERNEL_CHUNK_TC = 4

# every symbol include/vla.h declares, with (restype, argtypes)
_vp = ctypes.c_void_p
_i = ctypes.c_int
_SIGS = {
    "vla_forward": (_i, [_vp, _vp, _vp, _vp, _i, ctypes.c_float, _i, _i, _i, _i, _vp, _vp, _vp, _vp,
                         _vp, _vp, _vp, _i, _i, _vp, ctypes.c_size_t, _vp]),
    "vla_workspace_bytes": (ctypes.c_size_t, [_i, _i, _i, _i, _i, _i, _i]),
    "vla_select_kernel": (_i, [_i, _i, _i, _i, _i]),
    "vla_chunk_lengths": (_i, [_i] * 7 + [ctypes.POINTER(_i)] * 2),
    "vla_host_ranges": (_i, [_i] * 7 + [ctypes.POINTER(_i)] * 4),
    "vla_status_str": (ctypes.c_char_p, [_i]),
    "vla_last_cuda_error": (_i, []),
    "vla_device_status": (_i, [_vp]),
    "vla_debug_inject": (_i, [_i, ctypes.c_longlong]),
    "vla_set_launch_events": (_i, [ctypes.POINTER(_vp), _i]),
    "vla_forward_noalloc": (_i, [_vp, _vp, _vp, _vp, _i, ctypes.c_float, _i, _i, _i, _i, _vp, _vp, _vp,
                                 _vp, _vp, _vp, _vp, _i, _vp]),
    "vla_forward_host": (_i, [_vp, _vp, _vp, _vp, _i, ctypes.c_float, _i, _i, _i, _i, _vp, _vp, _vp]
                         + [_vp] * 12 + [_i, _i, _vp, ctypes.c_size_t, _vp, _vp, _vp, _vp, _vp]),
    "vla_last_launch_count": (_i, []),
    "vla_backward": (_i, [_vp] * 5 + [_i, ctypes.c_float, _i, _i, _i, _i] + [_vp] * 14 + [ctypes.c_size_t, _vp]),
    "vla_backward_workspace_bytes": (ctypes.c_size_t, [_i, _i, _i, _i]),
    "vla_version": (_i, []),
}

_lock = threading.Lock()
_lib = None


class VLAError(RuntimeError):
    def __init__(self, status: int, where: str = "vla_forward"):
        self.status = status
        msg = lib().vla_status_str(status).decode()
        if status == VLA_ERR_CUDA:
            msg += " (cudaError %d)" % lib().vla_last_cuda_error()
        super().__init__("%s failed: %s [%d]" % (where, msg, status))


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded CDLL (building it with nvcc first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError("libvla.so was not built")
            L = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def vla_status_str(status: int) -> str:
    return lib().vla_status_str(int(status)).decode()


def vla_workspace_bytes(B, H, T, d_h, io_dtype=VLA_BF16, kernel=VLA_KERNEL_AUTO, chunk=0) -> int:
    return int(lib().vla_workspace_bytes(B, H, T, d_h, io_dtype, kernel, chunk))


def vla_select_kernel(B, H, T, d_h, io_dtype=VLA_BF16) -> int:
    return int(lib().vla_select_kernel(B, H, T, d_h, io_dtype))


def vla_chunk_lengths(B, H, T, d_h, io_dtype=VLA_BF16, kernel=VLA_KERNEL_AUTO, chunk=0):
    """(C, CA): the S- and A-chunk lengths vla_forward uses ((0, 0) off the chunked paths)."""
    C, CA = ctypes.c_int(0), ctypes.c_int(0)
    rc = lib().vla_chunk_lengths(B, H, T, d_h, io_dtype, kernel, chunk, ctypes.byref(C), ctypes.byref(CA))
    if rc != VLA_OK:
        raise VLAError(rc, "vla_chunk_lengths")
    return C.value, CA.value


def vla_host_ranges(B, H, T, d_h, io_dtype=VLA_BF16, kernel=VLA_KERNEL_AUTO, chunk=0):
    """The ranges vla_forward_host stages on the tensor-core path at d_h = 64:
    a list of (first unit, units, C, CA), empty when it does not stage so."""
    n = ctypes.c_int(0)
    lo, C, CA = (ctypes.c_int * 4)(), (ctypes.c_int * 3)(), (ctypes.c_int * 3)()
    rc = lib().vla_host_ranges(B, H, T, d_h, io_dtype, kernel, chunk, ctypes.byref(n), lo, C, CA)
    if rc != VLA_OK:
        raise VLAError(rc, "vla_host_ranges")
    return [(lo[r], lo[r + 1] - lo[r], C[r], CA[r]) for r in range(n.value)]


def vla_device_status(stream=None) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(lib().vla_device_status(ctypes.c_void_p(s.cuda_stream)))


def vla_debug_inject(mode: int, wait_limit_ns: int = 0) -> int:
    return int(lib().vla_debug_inject(int(mode), int(wait_limit_ns)))


def vla_set_launch_events(events) -> int:
    """Register torch.cuda.Event objects (or raw cudaEvent_t ints) that
    vla_forward records around each of its launches; None turns it off."""
    if not events:
        return int(lib().vla_set_launch_events(None, 0))
    handles = []
    for e in events:
        if hasattr(e, "cuda_event"):
            if not e.cuda_event:
                raise ValueError("record each torch.cuda.Event once before registering it")
            handles.append(e.cuda_event)
        else:
            handles.append(int(e))
    arr = (ctypes.c_void_p * len(handles))(*handles)
    return int(lib().vla_set_launch_events(arr, len(handles)))


def vla_last_launch_count() -> int:
    return int(lib().vla_last_launch_count())


def vla_backward_workspace_bytes(B, H, T, d_h) -> int:
    return int(lib().vla_backward_workspace_bytes(B, H, T, d_h))


def vla_backward(q, k, v, u, dO, lambda0: float, S0=None, A0=None, n0=None, dS_T=None, dA_T=None, dn_T=None,
                 workspace=None, stream=None):
    """Gradients of sum <dO, o> + <dS_T, S_T> + <dA_T, A_T> + <dn_T, n_T>.

    Inputs as for vla_forward plus dO (same shape and dtype as q).  Returns
    a dict of fp32 CUDA tensors dq, dk, dv, du, dS0, dA0, dn0.
    """
    import torch
    B, H, T, d = q.shape
    for t in (k, v, u, dO):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError("q, k, v, u, dO must share shape and dtype and be contiguous")
    io = VLA_BF16 if q.dtype == torch.bfloat16 else VLA_F32
    dev = q.device
    f32 = dict(dtype=torch.float32, device=dev)
    g = {n: torch.empty((B, H, T, d), **f32) for n in ("dq", "dk", "dv", "du")}
    g["dS0"] = torch.empty((B, H, d, d), **f32)
    g["dA0"] = torch.empty((B, H, d, d), **f32)
    g["dn0"] = torch.empty((B, H, d), **f32)
    need = vla_backward_workspace_bytes(B, H, T, d)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = torch.cuda.current_stream(dev) if stream is None else stream
    rc = lib().vla_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(u), _ptr(dO), io, float(lambda0), B, H, T, d,
                            _ptr(S0), _ptr(A0), _ptr(n0), _ptr(dS_T), _ptr(dA_T), _ptr(dn_T),
                            _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["du"]), _ptr(g["dS0"]),
                            _ptr(g["dA0"]), _ptr(g["dn0"]), _ptr(workspace), ws_bytes, ctypes.c_void_p(s.cuda_stream))
    if rc != VLA_OK:
        raise VLAError(rc, "vla_backward")
    return g


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def vla_forward(q, k, v, u, lambda0: float, S0=None, A0=None, n0=None, o=None, S_T=None, A_T=None,
                n_T=None, kernel: int = VLA_KERNEL_AUTO, chunk: int = 0, workspace=None,
                stream=None, want_n: bool = True):
    """Run the VLA forward recurrence on the GPU.

    q, k, v, u: contiguous CUDA tensors ``[B, H, T, d]``, all float32 or all
    bfloat16.  S0, A0 ``[B, H, d, d]`` and n0 ``[B, H, d]`` float32, optional.
    Returns ``(o, S_T, A_T, n_T)``; ``n_T`` is None when ``want_n`` is False
    and no ``n_T`` buffer was passed.  Launches asynchronously on ``stream``
    (default: torch's current stream).
    """
    import torch
    if q.dim() != 4:
        raise ValueError("q must be [B, H, T, d]")
    B, H, T, d = q.shape
    for t in (k, v, u):
        if t.shape != q.shape or t.dtype != q.dtype or t.device != q.device:
            raise ValueError("q, k, v, u must share shape, dtype and device")
    for t in (q, k, v, u):
        if not t.is_contiguous():
            raise ValueError("inputs must be contiguous")
    if not q.is_cuda:
        raise ValueError("inputs must be CUDA tensors")
    if q.dtype == torch.float32:
        io = VLA_F32
    elif q.dtype == torch.bfloat16:
        io = VLA_BF16
    else:
        raise ValueError("io dtype must be float32 or bfloat16")
    dev = q.device
    if o is None:
        o = torch.empty_like(q)
    if S_T is None:
        S_T = torch.empty((B, H, d, d), dtype=torch.float32, device=dev)
    if A_T is None:
        A_T = torch.empty((B, H, d, d), dtype=torch.float32, device=dev)
    if n_T is None and want_n:
        n_T = torch.empty((B, H, d), dtype=torch.float32, device=dev)
    need = vla_workspace_bytes(B, H, T, d, io, kernel, chunk)
    if need > 0 and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = torch.cuda.current_stream(dev) if stream is None else stream
    rc = lib().vla_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(u), io, float(lambda0), B, H, T, d,
                           _ptr(S0), _ptr(A0), _ptr(n0), _ptr(o), _ptr(S_T), _ptr(A_T), _ptr(n_T),
                           int(kernel), int(chunk), _ptr(workspace), ws_bytes,
                           ctypes.c_void_p(s.cuda_stream))
    if rc != VLA_OK:
        raise VLAError(rc)
    return o, S_T, A_T, n_T


def vla_forward_host(hq, hk, hv, hu, lambda0: float, q, k, v, u, o, ho, S_T, A_T, n_T=None, hS_T=None,
                     hA_T=None, hn_T=None, S0=None, A0=None, n0=None, kernel: int = VLA_KERNEL_AUTO,
                     chunk: int = 0, workspace=None, stream=None, copy_stream=None, ev_uk=None, ev_qv=None,
                     download_stream=None):
    """vla_forward on host inputs: copies hq, hk, hv, hu (CPU tensors, ideally
    pinned) into the device buffers q, k, v, u (u and k first on
    ``copy_stream``, overlapped with the passes that read only them), runs the
    recurrence on ``stream`` and copies o (and the final state for the given
    host tensors) back.  ``ev_uk``, ``ev_qv``: torch.cuda.Event objects the call
    records (created here when None).  ``download_stream``: optional third
    stream on which o comes back range by range on the staged paths.
    Asynchronous; returns None."""
    import torch
    B, H, T, d = q.shape
    for t in (hq, hk, hv, hu, ho):
        if t.shape != q.shape or t.dtype != q.dtype or t.is_cuda or not t.is_contiguous():
            raise ValueError("host tensors must be contiguous CPU tensors shaped and typed like q")
    io = VLA_BF16 if q.dtype == torch.bfloat16 else VLA_F32
    dev = q.device
    s = torch.cuda.current_stream(dev) if stream is None else stream
    cs = s if copy_stream is None else copy_stream
    evs = []
    for ev in (ev_uk, ev_qv):
        ev = torch.cuda.Event() if ev is None else ev
        if not ev.cuda_event:  # torch creates the event at its first record
            ev.record(s)
        evs.append(ev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().vla_forward_host(_ptr(hq), _ptr(hk), _ptr(hv), _ptr(hu), io, float(lambda0), B, H, T, d,
                                _ptr(S0), _ptr(A0), _ptr(n0), _ptr(q), _ptr(k), _ptr(v), _ptr(u), _ptr(o),
                                _ptr(ho), _ptr(S_T), _ptr(A_T), _ptr(n_T), _ptr(hS_T), _ptr(hA_T), _ptr(hn_T),
                                int(kernel), int(chunk), _ptr(workspace), ws_bytes,
                                ctypes.c_void_p(s.cuda_stream), ctypes.c_void_p(cs.cuda_stream),
                                ctypes.c_void_p(evs[0].cuda_event), ctypes.c_void_p(evs[1].cuda_event),
                                ctypes.c_void_p(None if download_stream is None else download_stream.cuda_stream))
    if rc != VLA_OK:
        raise VLAError(rc, "vla_forward_host")
