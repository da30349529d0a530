"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/vla.h declares, and rejects bad arguments on the host
before any CUDA call."""

import ctypes
import os
import re

import pytest

import rls_associative_memory_gb300 as vla
from rls_associative_memory_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vla.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(vla_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("vla_forward", "vla_workspace_bytes", "vla_status_str", "vla_device_status"):
        assert must in names
    assert set(names) == set(_lib._SIGS), "binding signatures must cover exactly the header"


def test_library_loads_and_exports_every_declared_symbol():
    L = vla.lib()
    raw = ctypes.CDLL(vla.lib_path())
    for name in declared_functions():
        assert hasattr(raw, name), name
    assert L.vla_version() >= 100


def test_status_strings():
    for st in (vla.VLA_OK, vla.VLA_ERR_ARG, vla.VLA_ERR_UNSUPPORTED_DIM, vla.VLA_ERR_ALIGN,
               vla.VLA_ERR_WORKSPACE, vla.VLA_ERR_CUDA, vla.VLA_ERR_TIMEOUT):
        assert vla.vla_status_str(st) and vla.vla_status_str(st) != "unknown status"
    assert vla.vla_status_str(12345) == "unknown status"


def _call(**kw):
    """vla_forward through the raw C ABI with fake (never dereferenced) pointers."""
    base = 1 << 20
    args = dict(q=base, k=base, v=base, u=base, io=vla.VLA_BF16, lam=1.0, B=1, H=1, T=4, d=64, S0=None,
                A0=None, n0=None, o=base, S_T=base, A_T=base, n_T=None, kernel=0, chunk=0, ws=None,
                ws_bytes=0, stream=None)
    args.update(kw)
    return vla.lib().vla_forward(args["q"], args["k"], args["v"], args["u"], args["io"], args["lam"],
                                 args["B"], args["H"], args["T"], args["d"], args["S0"], args["A0"],
                                 args["n0"], args["o"], args["S_T"], args["A_T"], args["n_T"],
                                 args["kernel"], args["chunk"], args["ws"], args["ws_bytes"],
                                 args["stream"])


@pytest.mark.parametrize("kw,rc", [
    (dict(d=48), vla.VLA_ERR_UNSUPPORTED_DIM),
    (dict(d=256), vla.VLA_ERR_UNSUPPORTED_DIM),
    (dict(lam=0.0), vla.VLA_ERR_ARG),
    (dict(lam=-1.0), vla.VLA_ERR_ARG),
    (dict(lam=float("nan")), vla.VLA_ERR_ARG),
    (dict(lam=float("inf")), vla.VLA_ERR_ARG),
    (dict(io=7), vla.VLA_ERR_ARG),
    (dict(kernel=9), vla.VLA_ERR_ARG),
    (dict(kernel=5), vla.VLA_ERR_ARG),
    (dict(kernel=-1), vla.VLA_ERR_ARG),
    (dict(B=-1), vla.VLA_ERR_ARG),
    (dict(T=-3), vla.VLA_ERR_ARG),
    (dict(chunk=-1), vla.VLA_ERR_ARG),
    (dict(chunk=24), vla.VLA_ERR_ARG),
    (dict(q=None), vla.VLA_ERR_ARG),
    (dict(o=None), vla.VLA_ERR_ARG),
    (dict(S_T=None), vla.VLA_ERR_ARG),
    (dict(A_T=None), vla.VLA_ERR_ARG),
    (dict(k=(1 << 20) + 8), vla.VLA_ERR_ALIGN),
    (dict(S0=(1 << 20) + 4), vla.VLA_ERR_ALIGN),
    (dict(n_T=(1 << 20) + 2), vla.VLA_ERR_ALIGN),
])
def test_bad_arguments_rejected_on_host(kw, rc):
    assert _call(**kw) == rc


def test_chunked_path_needs_workspace():
    assert _call(kernel=vla.VLA_KERNEL_CHUNK, T=4096) == vla.VLA_ERR_WORKSPACE
    need = vla.vla_workspace_bytes(1, 1, 4096, 64, vla.VLA_BF16, vla.VLA_KERNEL_CHUNK)
    assert _call(kernel=vla.VLA_KERNEL_CHUNK, T=4096, ws=1 << 20, ws_bytes=need - 1) == vla.VLA_ERR_WORKSPACE
    assert _call(kernel=vla.VLA_KERNEL_CHUNK, T=4096, ws=(1 << 20) + 8, ws_bytes=need) == vla.VLA_ERR_ALIGN


def test_empty_problem_is_a_no_op():
    assert _call(B=0) == vla.VLA_OK
    assert _call(H=0, q=None, k=None, v=None, u=None, o=None, S_T=None, A_T=None) == vla.VLA_OK


def test_workspace_query_and_kernel_selection():
    assert vla.vla_workspace_bytes(1, 16, 4096, 64, vla.VLA_BF16, vla.VLA_KERNEL_SEQ) == 0
    ws = vla.vla_workspace_bytes(1, 16, 4096, 64, vla.VLA_BF16, vla.VLA_KERNEL_CHUNK, 256)
    # gates (T d fp32 per head) plus four d x d fp32 matrices per chunk per head, and more
    assert ws >= 16 * (4096 * 64 * 4 + 16 * 4 * 64 * 64 * 4)
    assert vla.vla_workspace_bytes(1, 16, 4096, 64, vla.VLA_BF16, vla.VLA_KERNEL_CHUNK, 24) == 0
    assert vla.vla_workspace_bytes(1, 16, 0, 64, vla.VLA_BF16, vla.VLA_KERNEL_CHUNK) == 0
    assert vla.vla_select_kernel(1, 16, 65536, 64) == vla.VLA_KERNEL_CHUNK_TC
    assert vla.vla_select_kernel(256, 4, 512, 32, vla.VLA_F32) == vla.VLA_KERNEL_SEQ
    # d = 128: the tensor-core path (one chunk per unit) with bf16 I/O and enough units,
    # the sequential kernel with fp32 I/O or few units on short streams
    assert vla.vla_select_kernel(32, 16, 2048, 128, vla.VLA_BF16) == vla.VLA_KERNEL_CHUNK_TC
    assert vla.vla_select_kernel(32, 16, 2048, 128, vla.VLA_F32) == vla.VLA_KERNEL_SEQ
    assert vla.vla_select_kernel(2, 16, 512, 128, vla.VLA_BF16) == vla.VLA_KERNEL_SEQ
    assert vla.vla_select_kernel(32, 64, 1, 64) == vla.VLA_KERNEL_DECODE
    assert vla.vla_select_kernel(32, 64, 4, 64) == vla.VLA_KERNEL_DECODE
    assert vla.vla_select_kernel(32, 64, 5, 64) == vla.VLA_KERNEL_SEQ
    assert vla.vla_workspace_bytes(32, 64, 1, 64, vla.VLA_BF16, vla.VLA_KERNEL_DECODE) == 0
    assert vla.vla_workspace_bytes(1, 16, 4096, 48, vla.VLA_BF16, vla.VLA_KERNEL_SEQ) == 0
    assert vla.vla_select_kernel(1, 16, 4096, 64) in (vla.VLA_KERNEL_SEQ, vla.VLA_KERNEL_CHUNK_TC)
    assert vla.vla_select_kernel(1, 16, 4096, 40) == vla.VLA_ERR_UNSUPPORTED_DIM
    assert vla.vla_select_kernel(1, 16, 4096, 64, 7) == vla.VLA_ERR_ARG


def test_single_chunk_layout_at_d128():
    """d = 128 with the tensor-core path and enough units: one chunk per unit, so
    the workspace is the unit gates plus a few d x d matrices per unit."""
    B, H, T, d = 32, 16, 2048, 128
    ws = vla.vla_workspace_bytes(B, H, T, d, vla.VLA_BF16, vla.VLA_KERNEL_CHUNK_TC)
    gates = B * H * T * d * 4
    assert gates <= ws <= gates + B * H * 8 * d * d * 4 + (1 << 20)
    # the same shape on the plain chunked path keeps its multi-chunk default
    assert vla.vla_workspace_bytes(B, H, T, d, vla.VLA_BF16, vla.VLA_KERNEL_CHUNK) > ws


def test_tensor_core_chunk_defaults():
    """Default chunk lengths of the tensor-core path come from a wave model of
    its passes (two CTAs per SM on 152 SMs): 16 units x 65536 tokens take
    1728-token chunks (38 per unit, 608 CTAs: two full waves, and one full
    wave for each half of the units), and 32 units x 4096 tokens 256. The
    explicit length equal to the default gives the same layout."""
    TC = vla.VLA_KERNEL_CHUNK_TC
    assert vla.vla_chunk_lengths(1, 16, 65536, 64, vla.VLA_BF16, TC) == (1728, 1728)
    assert vla.vla_chunk_lengths(1, 32, 4096, 64, vla.VLA_BF16, TC)[0] == 256
    assert vla.vla_chunk_lengths(1, 16, 65536, 64, vla.VLA_BF16, TC, 512) == (512, 512)
    ws = lambda BH, T, c: vla.vla_workspace_bytes(1, BH, T, 64, vla.VLA_BF16, TC, c)  # noqa: E731
    assert ws(16, 65536, 0) != ws(16, 65536, 512)
    # the float path keeps its own lengths (no tensor-core passes, no staged ranges)
    f32 = vla.vla_workspace_bytes(1, 16, 65536, 64, vla.VLA_F32, TC, 0)
    assert f32 == vla.vla_workspace_bytes(1, 16, 65536, 64, vla.VLA_F32, vla.VLA_KERNEL_CHUNK, 0)
    assert vla.vla_host_ranges(1, 16, 65536, 64, vla.VLA_F32, TC) == []
    assert vla.vla_chunk_lengths(1, 16, 65536, 64, vla.VLA_BF16, vla.VLA_KERNEL_SEQ) == (0, 0)


def test_host_entry_ranges():
    """The host entry's ranges on the tensor-core path: half the units, then the
    rest in two.  Each half is a problem of its own: the first with the whole
    problem's default chunk length, the second with that of a lone pass over
    its last range (the wave model at two CTAs per SM on 152 SMs plus the chain
    along the chunks) when that is at least 512 tokens.  16 units x 65536
    tokens run 8 units at 1728 tokens (one full wave), then two ranges of 4 at
    896 (74 chunks a unit, 296 CTAs: one wave of 14 sub-blocks instead of 27);
    32 units x 4096 tokens keep 256 throughout (the lone pass would take 128).
    An explicit chunk length holds for every range.  The workspace covers the
    two halves' layouts side by side."""
    TC, BF = vla.VLA_KERNEL_CHUNK_TC, vla.VLA_BF16
    assert vla.vla_host_ranges(1, 16, 65536, 64, BF, TC) == [(0, 8, 1728, 1728), (8, 4, 896, 896),
                                                             (12, 4, 896, 896)]
    assert vla.vla_host_ranges(1, 16, 65536, 64, BF, TC, 1728) == [(0, 8, 1728, 1728), (8, 4, 1728, 1728),
                                                                   (12, 4, 1728, 1728)]
    assert [r[:2] for r in vla.vla_host_ranges(1, 2, 4096, 64, BF, TC)] == [(0, 1), (1, 1)]
    assert [r[:2] for r in vla.vla_host_ranges(1, 3, 4096, 64, BF, TC)] == [(0, 1), (1, 1), (2, 1)]
    assert vla.vla_host_ranges(1, 32, 4096, 64, BF, TC) == [(0, 16, 256, 256), (16, 8, 256, 256), (24, 8, 256, 256)]
    for lo, n, C, CA in vla.vla_host_ranges(4, 8, 4096, 64, BF, TC):
        assert C % 64 == 0 and CA % 64 == 0 and C % CA == 0
    # no staging at one unit, at d = 128 (its own schedule) or on the sequential kernel
    assert vla.vla_host_ranges(1, 1, 65536, 64, BF, TC) == []
    assert vla.vla_host_ranges(32, 16, 2048, 128, BF, TC) == []
    assert vla.vla_host_ranges(1, 16, 65536, 64, BF, vla.VLA_KERNEL_SEQ) == []
    # the workspace holds every range's layout: at least the whole problem's
    whole = vla.vla_workspace_bytes(1, 1, 65536, 64, BF, TC, 1728) * 16
    assert vla.vla_workspace_bytes(1, 16, 65536, 64, BF, TC) >= whole
    assert vla.vla_workspace_bytes(1, 16, 65536, 64, BF, TC) <= whole * 1.1
    with pytest.raises(vla.VLAError):
        vla.vla_host_ranges(1, 16, 65536, 48, BF, TC)


def test_backward_argument_checks():
    f = 1 << 20
    L = vla.lib()
    args = lambda **kw: [kw.get(n, f) for n in ("q", "k", "v", "u", "dO")] + [  # noqa: E731
        kw.get("io", vla.VLA_BF16), 1.0, 1, 2, 16, kw.get("d", 64)] + [None] * 6 + [f] * 7 + [
        kw.get("ws", None), kw.get("wsb", 0), None]
    assert L.vla_backward(*args(d=96)) == vla.VLA_ERR_UNSUPPORTED_DIM
    assert L.vla_backward(*args()) == vla.VLA_ERR_WORKSPACE
    assert L.vla_backward(*args(d=128)) == vla.VLA_ERR_WORKSPACE
    assert L.vla_backward(*args(dO=None)) == vla.VLA_ERR_ARG
    assert L.vla_backward(*args(k=f + 4)) == vla.VLA_ERR_ALIGN
    assert vla.vla_backward_workspace_bytes(1, 2, 16, 96) == 0
    # d = 128: always the sequential form (records and one checkpoint per 64 tokens)
    assert vla.vla_backward_workspace_bytes(1, 2, 16, 128) == 2 * (16 * 516 + 1 * (2 * 128 * 128 + 128)) * 4
    assert vla.vla_backward_workspace_bytes(2, 3, 200, 128) == 6 * (200 * 516 + 4 * (2 * 128 * 128 + 128)) * 4
    assert vla.vla_backward_workspace_bytes(1, 2, 16, 64) == 2 * (16 * 260 + 1 * (2 * 64 * 64 + 64)) * 4
    # streams of two or more of its chunks: the chunk-parallel backward carves a chunked
    # forward's workspace (its unit gates alone are B H T d fp32 words; no o, its output pass
    # is skipped), the per-token records and dg / dk_hat parts, the checkpoints and the maps
    BH, T, d = 16, 65536, 64
    need = vla.vla_backward_workspace_bytes(1, BH, T, d)
    least = BH * T * d * 4 + BH * T * ((4 * d + 4) + 2 * d) * 4 + BH * (T // 64) * (2 * d * d + d) * 4
    assert least <= need <= 1.2 * least


def test_debug_hook_is_host_state_only():
    assert vla.vla_debug_inject(2) == vla.VLA_ERR_ARG
    assert vla.vla_debug_inject(1, 1000) == vla.VLA_OK
    assert vla.vla_debug_inject(0) == vla.VLA_OK


def test_host_entry_argument_checks():
    """vla_forward_host rejects bad arguments before queuing any copy or
    launch (no CUDA call is reached here)."""
    L = vla.lib()
    f = 1 << 20
    dev = [f + 0x1000 * i for i in range(12)]  # aligned stand-ins, never dereferenced

    def call(ev=(f, f + 16), hq=f + 0x100000, hn=None, n_T=None, io=vla.VLA_BF16, d=64, T=64):
        return L.vla_forward_host(hq, hq, hq, hq, io, 1.0, 1, 1, T, d, None, None, None,
                                  dev[0], dev[1], dev[2], dev[3], dev[4], hq, dev[5], dev[6], n_T,
                                  None, None, hn, vla.VLA_KERNEL_SEQ, 0, None, 0, None, None, ev[0], ev[1], None)

    assert call(ev=(None, f)) == vla.VLA_ERR_ARG
    assert call(ev=(f, None)) == vla.VLA_ERR_ARG
    assert call(hq=None) == vla.VLA_ERR_ARG
    assert call(hq=f + 0x100000 + 4) == vla.VLA_ERR_ALIGN
    assert call(hn=f + 0x200000) == vla.VLA_ERR_ARG  # a host n_T needs the device n_T
    assert call(d=48) == vla.VLA_ERR_UNSUPPORTED_DIM
    assert call(io=9) == vla.VLA_ERR_ARG


def test_launch_event_hook_limit():
    """The measurement hook takes up to 64 event handles (the host entry's
    staged ranges launch up to 18 kernels); more is an argument error."""
    assert vla.vla_set_launch_events([1] * 65) == vla.VLA_ERR_ARG
    assert vla.vla_set_launch_events([1] * 64) == vla.VLA_OK
    assert vla.vla_set_launch_events(None) == vla.VLA_OK
