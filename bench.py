#!/usr/bin/env python3
"""Benchmark of the VLA forward recurrence on GB300.

One step = one vla_forward call over one batch of synthetic inputs (all of
the recurrence: key normalisation, Sherman-Morrison update, unit gate, state
write, ELU+1 readout, final state).  Prints ONE JSON line on rank 0.

Default workload: the long stream, B=1 H=16 T=65536 d_h=64, bf16 inputs, fp32
state, u scaled by 0.5, lambda0=1.  Its inputs (537 MB) and output (134 MB)
exceed the 129 MB L2, so no flush is needed between steps; smaller
workloads are flushed by writing a 256 MB buffer between timed steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                  [--kernel auto|seq|chunk] [--impl ours|reference]

Multi-GPU (torchrun): every rank runs its own batch of the same shape
(independent (batch, head) units, no collective on the data path; weak
scaling); value = all units / max-over-ranks time.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "VLA forward tokens·heads/sec at d_h=64 and % of roofline on 1 GB300"
UNIT = "tokens*heads/s"
L2_BYTES = 129 * 1024 * 1024
N_SM = 152
SM_MAX_GHZ = 2.070
# FP32 SIMT peak: 152 SMs x 128 FP32 lanes x 2 flop per FMA x max SM clock.
FP32_PEAK_TFLOPS = N_SM * 128 * 2 * SM_MAX_GHZ / 1e3

# DRAM traffic per launch of the dominant kernel, from ncu captures
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by (kernel,
# workload).  Reported only while the kernel source still hashes to the value
# it was captured from; otherwise null.  (An edit of the shared header that
# adds only host declarations re-keys the records without a new capture.)
TRAFFIC = {
    # sequential kernel, long stream: 135.3 + 18.9 MB at T=16384, scaled x4 to T=65536
    ("seq", "long", "seq_kernel"): {"bytes": 4 * (135.000064e6 + 19.173888e6), "src_sha": "8029d371d74d05f3"},
    # sequential kernel at d = 32, recall8 workload: one full-size launch (one ncu pass)
    ("seq", "recall8", "seq32_kernel"): {"bytes": 268.476160e6 + 50.967040e6, "src_sha": "c6686e0ee56813b5"},
    # tensor-core path at d = 64, long stream (two launches): one full-size launch each
    # (T=65536; one ncu pass)
    ("chunk_tc", "long", "gates_tc_kernel"): {"bytes": 278.221824e6 + 101.037824e6, "src_sha": "2bd40b3ddad0f1e0"},
    ("chunk_tc", "long", "rows_tc_kernel"): {"bytes": 537.165824e6 + 246.693120e6, "src_sha": "9e62ca08836996eb"},
    # d = 64 queue launch of both passes, 4x8x4096 (heads32): one launch at full size (one ncu pass)
    ("chunk_tc", "heads32", "tc64_queue_kernel"): {"bytes": 78.998784e6 + 17.412352e6, "src_sha": "9bc481f16332c96c"},
    # decode step, state in place: one launch at full size (one ncu pass)
    ("decode", "decode", "decode_kernel"): {"bytes": 68.697600e6 + 12.946432e6, "src_sha": "377e9a67c43a05a7"},
    # d = 128 queue launch, batched workload: at B=8 (128 units), scaled x4 to B=32 (the bytes
    # of a unit's two passes do not depend on how many units a launch holds)
    ("chunk_tc", "batched", "tc128_queue_kernel"): {"bytes": 4 * (402.768640e6 + 127.273472e6),
                                                     "src_sha": "d9e92a2f261757b3"},
}


# The sources of each kernel a traffic record is kept for (with the headers
# every kernel includes): a capture stays valid while they are unchanged.
KERNEL_SOURCES = {
    "seq_kernel": ["vla_seq.cu"],
    "seq32_kernel": ["vla_seq32.cu"],
    "gates_tc_kernel": ["vla_gates_tc.cu", "vla_gates_tc.cuh", "vla_tc_common.cuh", "vla_tma.cuh"],
    "rows_tc_kernel": ["vla_chunk_tc.cu", "vla_rows_tc.cuh", "vla_tc_common.cuh"],
    "tc64_queue_kernel": ["vla_tc64_queue.cu", "vla_gates_tc.cuh", "vla_rows_tc.cuh", "vla_tc_common.cuh",
                          "vla_tma.cuh"],
    "tc128_queue_kernel": ["vla_gates_tc128.cuh", "vla_rows_tc128.cuh", "vla_tc128.cu", "vla_tc_common.cuh", "vla_tma.cuh"],
    "decode_kernel": ["vla_decode.cu"],
}


def kernel_src_hash(kernel_name: str) -> str:
    """Hash of a kernel's sources, code only (comments and blank space stripped)."""
    fns = KERNEL_SOURCES[kernel_name] + ["vla_internal.cuh"]
    h = hashlib.sha256()
    for fn in fns:
        path = os.path.join(ROOT, "rls_associative_memory_gb300", "csrc", fn)
        if not os.path.exists(path):
            return ""
        # the code only: comments and blank space do not invalidate a capture
        src = open(path).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


# Kernels of one step, in launch order, with the share of the algorithmic
# work each one performs: every step of the recurrence is assigned to exactly
# one kernel (the chunked form's extra work - Grams, prefix sums, chunk
# transitions, the chain - counts zero), and so is every input and output
# byte.  engine is the pipe the kernel's arithmetic runs on: "alu" (FP32 CUDA
# cores) or "tensor" (bf16 tcgen05; its roofline takes the bf16 tensor peak).
def kernel_plan(kname, d, io_dtype="bf16", units=0, launches=0):
    """[(kernel, algorithmic flops, algorithmic bytes per token-head, engine)] in launch order
    (units: the (b, h) units of the batch; launches: the launches of one step, which tell
    the d = 64 tensor-core path's one queue launch of both passes from two launches)."""
    io = 2 if io_dtype == "bf16" else 4
    full = 12 * d * d + 16 * d
    if kname == "seq":
        return [("seq32_kernel" if d == 32 else "seq_kernel", full, 5 * d * io, "alu")]
    if kname == "decode":
        # one token per call: the state read and written back dominates (added by the caller)
        return [("decode_kernel", full, 5 * d * io, "alu")]
    # gates: key norm, z = A u, rank-1 update, A k_hat, gate norm (a0-a2), reading u and k;
    # output: S k_hat, state write, S phi(q), readout (a3-a4), reading q and v, writing o
    half = 6 * d * d + 8 * d
    gram = "gram_tc_kernel" if (io_dtype == "bf16" and d >= 64) else "gram_kernel"
    gram_e = "tensor" if gram == "gram_tc_kernel" else "alu"
    # chunk_tc at d = 64 with bf16 I/O: gates and state pass on the tensor cores; the
    # state pass does the state write and readout (a3-a4, reading q and v) for the
    # [H; P] rows of each chunk, and the output pass combines them with the chunk-start
    # state (o = S^(c) y + h, writing o)
    # chunk_tc at d = 128 with bf16 I/O and one chunk per unit (enough units): the
    # gates from A0, then the state pass on S itself, which writes o
    if kname == "chunk_tc" and io_dtype == "bf16" and d == 128 and units >= 128:
        # both passes of every unit in one persistent launch (a job queue)
        return [("tc128_queue_kernel", full, 5 * d * io, "tensor")]
    if kname == "chunk_tc" and io_dtype == "bf16" and d == 64:
        head = [("gram_tma_kernel", 0, 0, "tensor"), ("prefix_kernel", 0, 0, "alu")]
        tail = [("chain_kernel", 0, 0, "alu"), ("out_tc_kernel", 0, d * io, "tensor")]
        if launches == 5:
            # the gates (a0-a2, reading u and k) and the state pass (a3-a4, reading q and
            # v) in one persistent launch fed by a job queue (when the passes' last waves
            # would be part full)
            return head + [("tc64_queue_kernel", full, 4 * d * io, "tensor")] + tail
        return head + [("gates_tc_kernel", half, 2 * d * io, "tensor"),
                       ("rows_tc_kernel", half, 2 * d * io, "tensor")] + tail
    return [(gram, 0, 0, gram_e), ("prefix_kernel", 0, 0, "alu"), ("gates_kernel", half, 2 * d * io, "alu"),
            ("rows_kernel<summary>", 0, 0, "alu"), ("chain_kernel", 0, 0, "alu"),
            ("rows_kernel<output>", half, 3 * d * io, "alu")]


def state_bytes(B, H, d):
    """fp32 state words read and written per call: S, A (d x d) and n (d)."""
    return B * H * 2 * (2 * d * d + d) * 4


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """Slowest rank's value (the job finishes when the last rank does)."""
    if dist is None or not dist.is_initialized():
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, units_per_rank: int, ms_max: float) -> float:
    """Whole-job throughput: every rank processes its own batch (weak scaling)."""
    return world * units_per_rank / (ms_max / 1e3)


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def algorithmic_work(B, H, T, d, io_bytes):
    """Per-launch algorithmic flops and bytes of the recurrence.

    flops: 12 d^2 + 16 d per token-head (A u, A k_hat, S k_hat, S phi(q)
    matrix-vector products; the rank-1 updates of A and S; O(d) norms, phi,
    divisions).  bytes: q, k, v, u read and o written (5 d io_bytes per
    token-head) plus S_T and A_T written (8 d^2 per head).
    """
    units = B * H * T
    flops = units * (12 * d * d + 16 * d)
    byts = units * 5 * d * io_bytes + B * H * 8 * d * d
    return flops, byts


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region."""

    FIELDS = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None, interval_ms: int = 100):
        self.bus_id = bus_id
        self.proc = None
        self.interval_ms = interval_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            time.sleep(0.4)
        except Exception as e:  # pragma: no cover
            log("clock sampling unavailable:", e)
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:  # pragma: no cover
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if self.bus_id and parts[0].lower()[-12:] != self.bus_id.lower()[-12:]:
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


def bus_id_of(dev_index):
    import torch
    try:
        p = torch.cuda.get_device_properties(dev_index)
        return "%08x:%02x:%02x.0" % (getattr(p, "pci_domain_id"), getattr(p, "pci_bus_id"),
                                      getattr(p, "pci_device_id"))
    except Exception:
        return None


def make_host_inputs(cfg_name, rank, overrides):
    from synthetic import make_config
    kw = dict(overrides)
    if rank:
        from synthetic.generator import CONFIGS
        kw["seed"] = CONFIGS[cfg_name]["seed"] + 7919 * rank
    return make_config(cfg_name, **kw)


def to_torch_host(x, pin=True):
    import torch
    out = []
    for n in "qkvu":
        a = getattr(x, n)
        if x.dtype == "bf16":
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
        out.append(t.pin_memory() if pin else t)
    return out


def oracle_sample(x, max_heads=64):
    """The oracle (as it stands) on the first heads of the workload, full T."""
    import oracle
    B, H, T, d = x.q.shape
    nh = min(B * H, max_heads)
    flat = lambda a: a.reshape((B * H, T, d))[:nh]  # noqa: E731
    args = [flat(x.as_f64(n)) for n in "qkvu"]
    threads = min(oracle.default_threads(), nh)
    t0 = time.perf_counter()
    ref = oracle.forward(*args, x.lambda0, nthreads=threads)
    dt = time.perf_counter() - t0
    return ref, nh, threads, dt


def run_reference(args):
    """--impl reference: the fp64 oracle timed on the host cores, one bounded
    sample of the workload per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from synthetic.generator import CONFIGS
    x = make_host_inputs(args.config, 0, parse_overrides(args))
    B, H, T, d = x.q.shape
    for _ in range(args.warmup):
        oracle_sample(x, args.ref_heads)
    times = []
    nh = threads = 0
    for _ in range(args.steps):
        _, nh, threads, dt = oracle_sample(x, args.ref_heads)
        times.append(dt)
    ms = 1e3 * float(np.mean(times))
    value = nh * T / (ms / 1e3)
    sample = "first %d of %d (b,h) units, all %d tokens, d_h=%d, per step" % (nh, B * H, T, d)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(args.config, x, "oracle"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_block(name, x, kernel):
    B, H, T, d = x.q.shape
    io_bytes = 2 if x.dtype == "bf16" else 4
    in_bytes = 4 * B * H * T * d * io_bytes
    return {"workload": "%s: B=%d H=%d T=%d d_h=%d %s inputs, fp32 state, lambda0=%g" % (
        name, B, H, T, d, x.dtype, x.lambda0), "B": B, "H": H, "T": T, "d_h": d,
        "io_dtype": x.dtype, "lambda0": x.lambda0, "kernel": kernel,
        "l2": ("inputs larger than L2 (%d MB)" % (in_bytes >> 20)) if in_bytes > L2_BYTES
        else "L2 flushed (256 MB write) between timed steps"}


def parse_overrides(args):
    ov = {}
    for item in args.set or []:
        k, v = item.split("=", 1)
        ov[k] = type_of(v)
    return ov


def type_of(v):
    for f in (int, float):
        try:
            return f(v)
        except ValueError:
            pass
    return v


def run_backward(args):
    """--pass backward: gradients of sum <dO, o> for one batch of the workload
    (vla_backward: in parallel over the chunked forward's chunks when the
    stream has two or more, else one sequential launch per step)."""
    import torch
    import rls_associative_memory_gb300 as vla
    dev = torch.device("cuda", 0)
    x = make_host_inputs(args.config, 0, parse_overrides(args))
    B, H, T, d = x.q.shape
    hq, hk, hv, hu = to_torch_host(x, pin=False)
    q, k, v, u = (t.to(dev) for t in (hq, hk, hv, hu))
    gen = torch.Generator(device="cpu").manual_seed(7)
    dO = torch.randn(q.shape, generator=gen).to(q.dtype).to(dev)
    ws = torch.empty(vla.vla_backward_workspace_bytes(B, H, T, d), dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        vla.vla_backward(q, k, v, u, dO, x.lambda0, workspace=ws)
    torch.cuda.synchronize(dev)
    st = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        st[i].record()
        vla.vla_backward(q, k, v, u, dO, x.lambda0, workspace=ws)
        en[i].record()
    torch.cuda.synchronize(dev)
    launches = vla.vla_last_launch_count()
    ms = float(np.mean([a.elapsed_time(b) for a, b in zip(st, en)]))
    units = B * H * T
    # forward recompute (12 d^2) + reverse sweep (28 d^2: four matrix-vector
    # products, three column sums, six rank-1 updates, two state undos)
    flops = units * (40 * d * d + 64 * d)
    tf = flops / (ms / 1e3) / 1e12
    line = {"metric": "VLA backward tokens*heads/sec", "value": units / (ms / 1e3), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "dtype": "f32", "data": "synthetic", "config": config_block(args.config, x, "backward"),
            "roofline": {"bound": "alu", "achieved": tf, "peak": FP32_PEAK_TFLOPS, "unit": "TFLOP/s",
                         "frac": tf / FP32_PEAK_TFLOPS, "traffic": None,
                         "kernel": ("chunked backward (%d launches)" % launches if launches > 1
                                    else ("backward128_kernel<%s>" % x.dtype if d == 128
                                          else "backward_kernel<%d,%s>" % (d, x.dtype))),
                         "algorithmic_flops": flops},
            "gpu_launches": args.steps * launches}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="long")
    ap.add_argument("--kernel", default="auto", choices=["auto", "seq", "chunk", "chunk_tc", "decode"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--set", action="append", help="workload override, e.g. T=4096")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--ref-heads", type=int, default=64)
    ap.add_argument("--pass", dest="which", default="forward", choices=["forward", "backward"])
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        log("note: fewer than 3 warm-up steps")
    if args.impl == "reference":
        return run_reference(args)
    if args.which == "backward":
        return run_backward(args)

    import torch
    import rls_associative_memory_gb300 as vla

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kernel = {"auto": vla.VLA_KERNEL_AUTO, "seq": vla.VLA_KERNEL_SEQ, "chunk": vla.VLA_KERNEL_CHUNK,
              "chunk_tc": vla.VLA_KERNEL_CHUNK_TC, "decode": vla.VLA_KERNEL_DECODE}[args.kernel]

    t_gen = time.perf_counter()
    x = make_host_inputs(args.config, rank, parse_overrides(args))
    B, H, T, d = x.q.shape
    log("inputs %s generated in %.1fs" % (x.q.shape, time.perf_counter() - t_gen))
    io_bytes = 2 if x.dtype == "bf16" else 4
    hq, hk, hv, hu = to_torch_host(x)
    q, k, v, u = (t.to(dev) for t in (hq, hk, hv, hu))
    resolved = kernel if kernel != vla.VLA_KERNEL_AUTO else vla.vla_select_kernel(
        B, H, T, d, vla.VLA_BF16 if x.dtype == "bf16" else vla.VLA_F32)
    kname = {vla.VLA_KERNEL_SEQ: "seq", vla.VLA_KERNEL_CHUNK: "chunk", vla.VLA_KERNEL_CHUNK_TC: "chunk_tc",
             vla.VLA_KERNEL_DECODE: "decode"}[resolved]
    o = torch.empty_like(q)
    S_T = torch.empty((B, H, d, d), dtype=torch.float32, device=dev)
    A_T = torch.empty_like(S_T)
    n_T = torch.empty((B, H, d), dtype=torch.float32, device=dev)
    # decode steps carry the state in place from call to call
    in_place = kname == "decode"
    if in_place:
        S_T.zero_()
        n_T.zero_()
        A_T.copy_((torch.eye(d, device=dev) / x.lambda0).expand(B, H, d, d))
    need = vla.vla_workspace_bytes(B, H, T, d, vla.VLA_BF16 if x.dtype == "bf16" else vla.VLA_F32, resolved)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    in_bytes = 4 * B * H * T * d * io_bytes
    flush = in_bytes <= L2_BYTES
    scratch = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev) if flush else None
    stream = torch.cuda.current_stream(dev)

    def step():
        st = (S_T, A_T, n_T) if in_place else (None, None, None)
        vla.vla_forward(q, k, v, u, x.lambda0, S0=st[0], A0=st[1], n0=st[2], o=o, S_T=S_T, A_T=A_T, n_T=n_T,
                        kernel=resolved, workspace=ws if need else None, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = vla.vla_device_status(stream)
    if st != vla.VLA_OK:
        raise RuntimeError("device status after warm-up: " + vla.vla_status_str(st))
    plan = kernel_plan(kname, d, x.dtype, B * H, vla.vla_last_launch_count())
    nb = len(plan) + 1  # launch boundaries per step
    bounds = [[torch.cuda.Event(enable_timing=True) for _ in range(nb)] for _ in range(args.steps)]
    for evs in bounds:
        for ev in evs:
            ev.record(stream)  # creates the underlying cudaEvent_t
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(bus_id_of(dev.index)) if rank == 0 else None
    if sampler:
        sampler.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    launches = 0
    for i in range(args.steps):
        if flush:
            scratch.fill_(float(i))
        vla.vla_set_launch_events(bounds[i])
        starts[i].record(stream)
        step()
        ends[i].record(stream)
        launches += vla.vla_last_launch_count()
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    wall = time.perf_counter() - wall0
    vla.vla_set_launch_events(None)
    if launches != args.steps * len(plan):
        raise RuntimeError("expected %d launches per step, saw %d in total" % (len(plan), launches))
    per_kernel_ms = [float(np.mean([bounds[i][j].elapsed_time(bounds[i][j + 1]) for i in range(args.steps)]))
                     for j in range(len(plan))]
    clocks = sampler.stop() if sampler else None
    st = vla.vla_device_status(stream)
    if st != vla.VLA_OK:
        raise RuntimeError("device status after timed steps: " + vla.vla_status_str(st))
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = max_over_ranks(float(np.mean(step_ms)), dist, dev)
    units = B * H * T
    value = job_value(world, units, ms)

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hS = torch.empty(S_T.shape, dtype=torch.float32).pin_memory()
        hA = torch.empty(A_T.shape, dtype=torch.float32).pin_memory()
        hn = torch.empty(n_T.shape, dtype=torch.float32).pin_memory()

        # a decode step returns o; its state stays resident on the device

        copy_stream, download_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_uk, ev_qv = torch.cuda.Event(), torch.cuda.Event()

        def e2e_step():
            # the public host-buffer entry: uploads u, k first on a second stream, q, v
            # while the passes that read only u, k run, the results back after the kernels
            st = (S_T, A_T, n_T) if in_place else (None, None, None)
            hs = (None, None, None) if in_place else (hS, hA, hn)
            vla.vla_forward_host(hq, hk, hv, hu, x.lambda0, q, k, v, u, o, ho, S_T, A_T, n_T, hs[0], hs[1], hs[2],
                                 S0=st[0], A0=st[1], n0=st[2], kernel=resolved, workspace=ws if need else None,
                                 stream=stream, copy_stream=copy_stream, ev_uk=ev_uk, ev_qv=ev_qv,
                                 download_stream=download_stream)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize(dev)
        es = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        if dist:
            dist.barrier()
        for i in range(args.steps):
            es[i].record(stream)
            e2e_step()
            ee[i].record(stream)
        torch.cuda.synchronize(dev)
        e2e_steps = [s.elapsed_time(e) for s, e in zip(es, ee)]
        e2e_ms = max_over_ranks(float(np.mean(e2e_steps)), dist, dev)
        h2d = 4 * units * d * io_bytes
        d2h = units * d * io_bytes + (0 if in_place else B * H * (2 * d * d + d) * 4)
        e2e = {"value": job_value(world, units, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               # this rank's spread over the timed steps (the value is the mean)
               "ms_min": float(np.min(e2e_steps)), "ms_median": float(np.median(e2e_steps)),
               "ms_max": float(np.max(e2e_steps))}

    # ---- roofline of the dominant kernel (and of the whole step) ----
    flops, byts = algorithmic_work(B, H, T, d, io_bytes)
    if in_place:
        byts += state_bytes(B, H, d) - B * H * 8 * d * d  # the state is read and written each call
    dom = int(np.argmax(per_kernel_ms))
    kernel_ms = per_kernel_ms[dom]
    k_name, k_fpt, k_bpt, k_eng = plan[dom]
    tr = TRAFFIC.get((kname, args.config, k_name))
    traffic = tr["bytes"] if tr and tr.get("src_sha") == kernel_src_hash(k_name) else None
    k_flops = units * k_fpt
    k_bytes = byts if len(plan) == 1 else units * k_bpt  # a one-kernel path owns all bytes (state included)
    hbm = measured_hbm_gbs()
    fpeak, fsrc = flop_peak(k_eng)
    t_f, t_q = k_flops / (fpeak * 1e12), k_bytes / (hbm * 1e9)
    if t_f >= t_q:
        bound, achieved, peak, unit, alg, peak_src = ("alu" if k_eng == "alu" else "tensor"), \
            k_flops / (kernel_ms / 1e3) / 1e12, fpeak, "TFLOP/s", k_flops, fsrc
    else:
        bound, achieved, peak, unit, alg, peak_src = "hbm", k_bytes / (kernel_ms / 1e3) / 1e9, hbm, "GB/s", \
            k_bytes, "MEASURED_PEAKS.json hbm_gbs (of measured)"
    # whole step: the slower of its algorithmic flops at the peak of the pipe they run on and its
    # algorithmic bytes at the measured HBM bandwidth
    s_peak, s_src = flop_peak("tensor" if any(e == "tensor" for _, f, _, e in plan if f > 0) else "alu")
    t_roof = max(flops / (s_peak * 1e12), byts / (hbm * 1e9))
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                "traffic": traffic, "kernel": "%s<%d,%s>" % (k_name, d, x.dtype), "kernel_ms": kernel_ms,
                "algorithmic_per_launch": alg, "peak_source": peak_src,
                "step": {"algorithmic_flops": flops, "algorithmic_bytes": byts,
                         "roofline_ms": t_roof * 1e3, "frac": t_roof / (ms / 1e3),
                         "flop_peak_source": s_src,
                         "alu_frac": flops / (ms / 1e3) / 1e12 / FP32_PEAK_TFLOPS,
                         "alu_peak_tflops": FP32_PEAK_TFLOPS,
                         "alu_peak_source": "derived, not measured: 152 SMs x 128 FP32 lanes x 2 flop/FMA "
                                            "x 2.070 GHz (alu_frac is of derived)",
                         "hbm_frac_of_measured": (byts / (ms / 1e3) / 1e9) / hbm},
                "kernels": [{"name": nm, "ms": t, "share": t / sum(per_kernel_ms)}
                            for (nm, _, _, _), t in zip(plan, per_kernel_ms)]}

    cpu = None
    parity = None
    recall = None
    if rank == 0 and world == 1 and not args.no_cpu:
        ref, nh, threads, dt = oracle_sample(x, args.ref_heads)
        cpu = {"value": nh * T / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": "first %d of %d (b,h) units, all %d tokens (%.1f s)" % (nh, B * H, T, dt),
               "host_cores": os.cpu_count()}
        flat = lambda a: a.reshape((B * H,) + tuple(a.shape[2:]))[:nh]  # noqa: E731
        if in_place:
            # the timed calls advanced the state; redo one call from the initial state
            o2, S2, A2, n2 = vla.vla_forward(q, k, v, u, x.lambda0, kernel=resolved)
            torch.cuda.synchronize(dev)
        else:
            o2, S2, A2, n2 = o, S_T, A_T, n_T
        got = {"o": flat(o2.float().cpu().numpy()), "S_T": flat(S2.cpu().numpy()),
               "A_T": flat(A2.cpu().numpy()), "n_T": flat(n2.cpu().numpy())}
        parity = {key: rel_err(got[key], ref[key]) for key in got}
        # o over windows of the stream: the readout decays like 1/t, so the whole-tensor
        # ratio is dominated by the early tokens; these show the late ones
        win = 4096 if T >= 8192 else max(64, T // 8)
        wins = [rel_err(got["o"][:, a:a + win], ref["o"][:, a:a + win]) for a in range(0, T, win)]
        parity["o_window_tokens"] = win
        parity["o_window_max"] = max(wins)
        parity["o_window_argmax"] = int(np.argmax(wins))
        parity["o_last_window"] = rel_err(got["o"][:, max(0, T - win):], ref["o"][:, max(0, T - win):])
        if x.keys is not None:
            recall = recall_report(vla, x, q, k, v, u, resolved, got, ref, nh, dev,
                                   S2.cpu().numpy().reshape(B * H, d, d))

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "precision": precision_block(kname, x.dtype, d),
                "data": "synthetic",
                "config": config_block(args.config, x, kname), "roofline": roofline, "e2e": e2e,
                "gpu_launches": launches, "clocks": clocks,
                "cpu_baseline": cpu, "parity_rel_fro": parity, "wall_s_timed": wall}
        if recall is not None:
            line["recall"] = recall
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def rel_err(a, b):
    """Relative Frobenius error |a - b| / |b|."""
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def precision_block(kname, io_dtype, d):
    """What the step computes in: I/O, state and accumulation types, and how the
    tensor-core products take their fp32 operands."""
    blk = {"io": io_dtype, "state": "f32", "accumulate": "f32"}
    if kname == "chunk_tc" and io_dtype == "bf16" and d == 128:
        blk["tensor_products"] = ("tcgen05 kind::f16, fp32 operands as bf16 parts: A, AK, W and the "
                                  "downdate's Z in three (about 2^-24 relative), the rest as hi/lo pairs "
                                  "(hi*hi + hi*lo + lo*hi, about 2^-16); fp32 accumulation; the bf16 inputs "
                                  "enter exactly")
        blk["cuda_core"] = "f32 (eliminations, triangular inverses, norms)"
    elif kname == "chunk_tc" and io_dtype == "bf16" and d == 64:
        blk["tensor_products"] = ("tcgen05 kind::f16, fp32 operands as bf16 hi/lo pairs, products "
                                  "hi*hi + hi*lo + lo*hi (about 2^-16 relative), fp32 accumulation; "
                                  "the bf16 inputs enter exactly")
        blk["cuda_core"] = "f32 (eliminations, triangular inverses, norms, chain)"
    else:
        blk["cuda_core"] = "f32 (every step)"
    return blk


def recall_report(vla, x, q, k, v, u, kernel, got, ref, nh, dev, S_all):
    """The key-value recall streams: recall error |S_T key_i - value_i| from
    the GPU's final state (every unit, and the oracle's on the sampled units),
    and the recall error and |S_t|_F at t = 2n (right after the writes), T/8,
    T/4, T/2, T from split-stream calls (the state handed from call to call in
    place), the norms against plain additive linear attention,
    S^LA_t = sum_{s <= t} v_s k_hat_s^T, formed on the host from the same inputs."""
    import torch
    B, H, T, d = x.q.shape
    keys = x.keys.reshape(B * H, -1, d)
    vals = x.values.reshape(B * H, -1, d)

    def rec(S):
        return np.linalg.norm(np.einsum("bij,bnj->bni", S, keys[:S.shape[0]]) - vals[:S.shape[0]], axis=-1)

    r_gpu = rec(S_all)
    r_gpu_s = rec(got["S_T"])
    r_ref = rec(ref["S_T"])
    # split-stream calls through vla_forward: the state right after the 2n write
    # tokens, and after T/8, T/4, T/2, T tokens
    npairs = keys.shape[1]
    cuts = sorted({2 * npairs, T // 8, T // 4, T // 2, T})
    S = A = n = None
    lo = 0
    vla_norm, rec_t = [], []
    for hi in cuts:
        sl = lambda a: a[:, :, lo:hi].contiguous()  # noqa: E731
        _, S, A, n = vla.vla_forward(sl(q), sl(k), sl(v), sl(u), x.lambda0, S0=S, A0=A, n0=n, S_T=S, A_T=A,
                                     n_T=n, kernel=kernel)
        torch.cuda.synchronize(dev)
        vla_norm.append(float(torch.linalg.matrix_norm(S.reshape(B * H, d, d)).mean().item()))
        rec_t.append(float(rec(S.reshape(B * H, d, d).cpu().numpy().astype(np.float64)).mean()))
        lo = hi
    if vla.vla_device_status() != vla.VLA_OK:
        raise RuntimeError("device status after the split-stream calls")
    kk = x.as_f64("k").reshape(B * H, T, d)
    kh = kk / np.maximum(np.linalg.norm(kk, axis=-1, keepdims=True), 1e-6)
    vv = x.as_f64("v").reshape(B * H, T, d)
    la_norm = [float(np.linalg.norm(np.einsum("bti,btj->bij", vv[:, :t], kh[:, :t]), axis=(1, 2)).mean())
               for t in cuts]
    return {"n_pairs": int(keys.shape[1]),
            "recall_error_gpu": {"mean": float(r_gpu.mean()), "max": float(r_gpu.max()),
                                 "units": int(S_all.shape[0])},
            "recall_error_sampled": {"gpu_mean": float(r_gpu_s.mean()), "oracle_mean": float(r_ref.mean()),
                                     "abs_diff_mean": float(abs(r_gpu_s.mean() - r_ref.mean())),
                                     "max_abs_diff": float(np.max(np.abs(r_gpu_s - r_ref))), "units": int(nh)},
            "recall_error_gpu_mean_at_t": rec_t,
            "state_norm_t": cuts,
            "state_norm_vla_gpu": vla_norm,
            "state_norm_linear_attention_host": la_norm,
            "note": "mean over units of |S_t|_F; VLA from split-stream vla_forward calls, additive linear "
                    "attention sum v k_hat^T on the host"}


def flop_peak(engine):
    """(TFLOP/s, source) for the pipe a kernel's arithmetic runs on."""
    if engine == "tensor":
        try:
            return float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"]), \
                "MEASURED_PEAKS.json bf16_tflops, burst (of measured)"
        except Exception:
            return 1900.0, "fallback bf16 1.9 PFLOP/s (of fallback)"
    return FP32_PEAK_TFLOPS, "derived: 152 SMs x 128 FP32 lanes x 2 flop/FMA x 2.070 GHz (of derived)"


def measured_hbm_gbs():
    try:
        return float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["hbm_gbs"])
    except Exception:
        return 6800.0


if __name__ == "__main__":
    sys.exit(main())
