// vla_api.cu -- the extern "C" boundary of libvla: argument validation,
// kernel selection, launch on the caller's stream, status reporting.
//
// Nothing here allocates or synchronises except vla_device_status (which
// synchronises the given stream by contract).
#include <math.h>
#include <stdint.h>

#include "../../include/vla.h"
#include "vla_internal.cuh"

namespace {

__device__ int g_vla_dev_err;  // device error word, set by bounded waits on expiry

thread_local int t_last_cuda_error = 0;

long long g_wait_limit_ns = 1000000000LL;  // 1 s bound on every device-side wait
int g_inject = 0;
void *g_events[64];
int g_n_events = 0;
thread_local int t_last_launches = 0;

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return VLA_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int *device_err_word() {
    // Per device: the symbol's address in the current device's context.
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_vla_dev_err) != cudaSuccess) return nullptr;
    return static_cast<int *>(ptr);
}

int check_common(int io_dtype, float lambda0, int B, int H, int T, int d_h, int kernel) {
    if (B < 0 || H < 0 || T < 0) return VLA_ERR_ARG;
    if (io_dtype != VLA_F32 && io_dtype != VLA_BF16) return VLA_ERR_ARG;
    if (!(lambda0 > 0.f) || !isfinite(lambda0)) return VLA_ERR_ARG;
    if (kernel != VLA_KERNEL_AUTO && kernel != VLA_KERNEL_SEQ && kernel != VLA_KERNEL_CHUNK &&
        kernel != VLA_KERNEL_DECODE && kernel != VLA_KERNEL_CHUNK_TC)
        return VLA_ERR_ARG;
    if (d_h != 32 && d_h != 64 && d_h != 128) return VLA_ERR_UNSUPPORTED_DIM;
    // element offsets are computed in size_t; counts themselves must fit the kernels' int math
    if ((long long)B * H > 0x7fffffffLL) return VLA_ERR_ARG;
    if ((long long)T * d_h > 0x7fffffffLL) return VLA_ERR_ARG;
    return VLA_OK;
}

// AUTO: the decode step for a handful of tokens; at d = 128 with bf16 I/O and
// enough units to fill the GPU, the tensor-core path with one chunk per unit;
// the chunk-parallel path (with the tensor-core passes where they apply) when
// there are too few (b, h) units to fill the GPU with one CTA each and the
// stream is long enough to cut; otherwise the sequential kernel.
int resolve_kernel(int B, int H, int T, int d_h, int io_dtype, int kernel) {
    if (kernel != VLA_KERNEL_AUTO) return kernel;
    const long long BH = (long long)B * H;
    if (T >= 1 && T <= 4) return VLA_KERNEL_DECODE;
    if (d_h == 128 && io_dtype == VLA_BF16 && BH >= 128 && T >= 256) return VLA_KERNEL_CHUNK_TC;
    if (BH < 2 * 152 && T >= 1024) return VLA_KERNEL_CHUNK_TC;
    return VLA_KERNEL_SEQ;
}

// Workspace bytes vla_forward itself needs (the chunked paths' layout).
size_t forward_ws_bytes(int B, int H, int T, int d_h, int io_dtype, int kernel, int chunk) {
    if (check_common(io_dtype, 1.f, B, H, T, d_h, kernel) != VLA_OK) return 0;
    if (chunk < 0 || (chunk > 0 && chunk % 16 != 0)) return 0;
    const int kk = resolve_kernel(B, H, T, d_h, io_dtype, kernel);
    if ((kk != VLA_KERNEL_CHUNK && kk != VLA_KERNEL_CHUNK_TC) || T == 0 || (long long)B * H == 0) return 0;
    return vla::chunk_layout(B * H, T, d_h, chunk, kk == VLA_KERNEL_CHUNK_TC && io_dtype == VLA_BF16).total;
}


}  // namespace

namespace vla {
// Shared with the library's other C-ABI translation units.
int api_check_common(int io_dtype, float lambda0, int B, int H, int T, int d_h, int kernel) {
    return check_common(io_dtype, lambda0, B, H, T, d_h, kernel);
}
int *api_device_err_word() { return device_err_word(); }
long long api_wait_limit_ns() { return g_wait_limit_ns; }
int api_cuda_fail(cudaError_t e) { return cuda_fail(e); }
}  // namespace vla

extern "C" {

int vla_version(void) { return 100; }

const char *vla_status_str(int status) {
    switch (status) {
        case VLA_OK: return "ok";
        case VLA_ERR_ARG: return "invalid argument";
        case VLA_ERR_UNSUPPORTED_DIM: return "unsupported head dimension (d_h must be 32, 64 or 128)";
        case VLA_ERR_ALIGN: return "pointer not 16-byte aligned";
        case VLA_ERR_WORKSPACE: return "workspace missing or too small";
        case VLA_ERR_CUDA: return "CUDA runtime error (see vla_last_cuda_error)";
        case VLA_ERR_TIMEOUT: return "a bounded device-side wait expired";
        case VLA_ERR_SCRATCH_LIMIT:
            return "problem needs more scratch than vla_forward_noalloc's built-in array holds "
                   "(VLA_NOALLOC_SCRATCH_BYTES)";
        default: return "unknown status";
    }
}

int vla_last_cuda_error(void) { return t_last_cuda_error; }

int vla_set_launch_events(void *const *events, int n) {
    if (n < 0 || n > 64) return VLA_ERR_ARG;
    if (!events) n = 0;
    for (int i = 0; i < n; ++i) g_events[i] = events[i];
    g_n_events = n;
    return VLA_OK;
}

int vla_last_launch_count(void) { return t_last_launches; }

int vla_select_kernel(int B, int H, int T, int d_h, int io_dtype) {
    const int rc = check_common(io_dtype, 1.f, B, H, T, d_h, VLA_KERNEL_AUTO);
    if (rc != VLA_OK) return rc;
    return resolve_kernel(B, H, T, d_h, io_dtype, VLA_KERNEL_AUTO);
}

int vla_chunk_lengths(int B, int H, int T, int d_h, int io_dtype, int kernel, int chunk, int *C, int *CA) {
    const int rc = check_common(io_dtype, 1.f, B, H, T, d_h, kernel);
    if (rc != VLA_OK) return rc;
    if (!C || !CA || chunk < 0 || (chunk > 0 && chunk % 16 != 0)) return VLA_ERR_ARG;
    *C = *CA = 0;
    const int kk = resolve_kernel(B, H, T, d_h, io_dtype, kernel);
    if ((kk != VLA_KERNEL_CHUNK && kk != VLA_KERNEL_CHUNK_TC) || T == 0 || (long long)B * H == 0) return VLA_OK;
    const vla::ChunkLayout L =
        vla::chunk_layout(B * H, T, d_h, chunk, kk == VLA_KERNEL_CHUNK_TC && io_dtype == VLA_BF16);
    *C = L.C;
    *CA = L.CA;
    return VLA_OK;
}

int vla_host_ranges(int B, int H, int T, int d_h, int io_dtype, int kernel, int chunk, int *n, int *lo, int *C,
                    int *CA) {
    const int rc = check_common(io_dtype, 1.f, B, H, T, d_h, kernel);
    if (rc != VLA_OK) return rc;
    if (!n || !lo || !C || !CA || chunk < 0 || (chunk > 0 && chunk % 16 != 0)) return VLA_ERR_ARG;
    *n = 0;
    const int kk = resolve_kernel(B, H, T, d_h, io_dtype, kernel);
    const long long BH = (long long)B * H;
    if (kk != VLA_KERNEL_CHUNK_TC || io_dtype != VLA_BF16 || d_h != 64 || BH < 2 || T == 0) return VLA_OK;
    if (vla::chunk_layout((int)BH, T, d_h, chunk, true).C % 64 != 0) return VLA_OK;
    const vla::TcHostPlan plan = vla::tc_host_plan((int)BH, T, chunk);
    for (int s = 0; s < 2; ++s)
        if (plan.L[s].C % 64 != 0 || plan.L[s].CA % 64 != 0) return VLA_OK;
    *n = plan.n;
    for (int r = 0; r <= plan.n; ++r) lo[r] = plan.lo[r];
    for (int r = 0; r < plan.n; ++r) {
        C[r] = plan.L[plan.part[r]].C;
        CA[r] = plan.L[plan.part[r]].CA;
    }
    return VLA_OK;
}

size_t vla_workspace_bytes(int B, int H, int T, int d_h, int io_dtype, int kernel, int chunk) {
    const size_t fwd = forward_ws_bytes(B, H, T, d_h, io_dtype, kernel, chunk);
    if (fwd == 0) return 0;
    // vla_forward_host on the tensor-core path at d = 64 runs its ranges of units
    // with layouts of their own, side by side in the workspace
    const int kk = resolve_kernel(B, H, T, d_h, io_dtype, kernel);
    if (kk == VLA_KERNEL_CHUNK_TC && io_dtype == VLA_BF16 && d_h == 64 && (long long)B * H >= 2) {
        const size_t host = vla::tc_host_plan(B * H, T, chunk).total;
        return host > fwd ? host : fwd;
    }
    return fwd;
}

size_t vla_backward_workspace_bytes(int B, int H, int T, int d_h) {
    if (check_common(VLA_F32, 1.f, B, H, T, d_h, VLA_KERNEL_AUTO) != VLA_OK) return 0;
    const size_t seq = vla::backward_workspace_floats(B * H, T, d_h) * sizeof(float);
    const size_t chunked = vla::backward_chunk_bytes(B * H, T, d_h);
    return seq > chunked ? seq : chunked;
}

int vla_backward(const void *q, const void *k, const void *v, const void *u, const void *dO, int io_dtype,
                 float lambda0, int B, int H, int T, int d_h, const float *S0, const float *A0, const float *n0,
                 const float *dS_T, const float *dA_T, const float *dn_T, float *dq, float *dk, float *dv,
                 float *du, float *dS0, float *dA0, float *dn0, void *workspace, size_t ws_bytes, void *stream) {
    int rc = check_common(io_dtype, lambda0, B, H, T, d_h, VLA_KERNEL_AUTO);
    if (rc != VLA_OK) return rc;
    const long long BH = (long long)B * H;
    if (BH > 0 && T > 0 && (!q || !k || !v || !u || !dO)) return VLA_ERR_ARG;
    const void *ptrs[] = {q, k, v, u, dO, S0, A0, n0, dS_T, dA_T, dn_T, dq, dk, dv, du, dS0, dA0, dn0, workspace};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return VLA_ERR_ALIGN;
    const size_t need = vla_backward_workspace_bytes(B, H, T, d_h);
    if (need > 0 && (!workspace || ws_bytes < need)) return VLA_ERR_WORKSPACE;
    if (BH == 0) return VLA_OK;
    vla::BwdParams p{};
    p.q = q; p.k = k; p.v = v; p.u = u; p.dO = dO;
    p.S0 = S0; p.A0 = A0; p.n0 = n0; p.dS_T = dS_T; p.dA_T = dA_T; p.dn_T = dn_T;
    p.dq = dq; p.dk = dk; p.dv = dv; p.du = du; p.dS0 = dS0; p.dA0 = dA0; p.dn0 = dn0;
    p.BH = (int)BH; p.T = T; p.d = d_h; p.io_bf16 = (io_dtype == VLA_BF16); p.lambda0 = lambda0;
    p.ws = static_cast<float *>(workspace);
    int launches = 0;
    p.launches = &launches;
    const cudaError_t e = vla::launch_backward(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    t_last_launches = launches;
    return VLA_OK;
}

int vla_debug_inject(int mode, long long wait_limit_ns) {
    if (mode != 0 && mode != 1) return VLA_ERR_ARG;
    g_inject = mode;
    if (mode == 0) {
        g_wait_limit_ns = 1000000000LL;
    } else {
        long long l = wait_limit_ns;
        if (l < 100000LL) l = 100000LL;
        if (l > 10000000000LL) l = 10000000000LL;
        g_wait_limit_ns = l;
    }
    return VLA_OK;
}

int vla_device_status(void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    int host = 0;
    e = cudaMemcpyFromSymbol(&host, g_vla_dev_err, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
    if (host != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_vla_dev_err, &zero, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e);
        return VLA_ERR_TIMEOUT;
    }
    return VLA_OK;
}

}  // extern "C"

namespace {

// vla_forward's checks and parameter block. Returns VLA_OK with p (and, for
// the chunked paths, L) filled in, or the error status; queues nothing.
int prepare_forward(const void *q, const void *k, const void *v, const void *u, int io_dtype, float lambda0, int B,
                    int H, int T, int d_h, const float *S0, const float *A0, const float *n0, void *o, float *S_T,
                    float *A_T, float *n_T, int kernel, int chunk, void *workspace, size_t ws_bytes,
                    vla::FwdParams &p, vla::ChunkLayout &L, int &kk) {
    int rc = check_common(io_dtype, lambda0, B, H, T, d_h, kernel);
    if (rc != VLA_OK) return rc;
    if (chunk < 0 || (chunk > 0 && chunk % 16 != 0)) return VLA_ERR_ARG;
    const long long BH = (long long)B * H;
    if (BH > 0) {
        if (!S_T || !A_T) return VLA_ERR_ARG;
        if (T > 0 && (!q || !k || !v || !u || !o)) return VLA_ERR_ARG;
    }
    const void *ptrs[] = {q, k, v, u, o, S0, A0, n0, S_T, A_T, n_T, workspace};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return VLA_ERR_ALIGN;
    kk = resolve_kernel(B, H, T, d_h, io_dtype, kernel);
    const size_t need = forward_ws_bytes(B, H, T, d_h, io_dtype, kk, chunk);
    if (need > 0 && (!workspace || ws_bytes < need)) return VLA_ERR_WORKSPACE;
    p = vla::FwdParams{};
    L = vla::ChunkLayout{};
    if (BH == 0) return VLA_OK;
    int *err = device_err_word();
    if (!err) return cuda_fail(cudaGetLastError());
    p.q = q; p.k = k; p.v = v; p.u = u; p.o = o;
    p.S0 = S0; p.A0 = A0; p.n0 = n0;
    p.S_T = S_T; p.A_T = A_T; p.n_T = n_T;
    p.BH = (int)BH; p.T = T; p.d = d_h;
    p.io_bf16 = (io_dtype == VLA_BF16);
    p.lambda0 = lambda0;
    p.err = err;
    p.wait_limit_ns = g_wait_limit_ns;
    p.inject = g_inject;
    p.ws = workspace; p.ws_bytes = ws_bytes; p.chunk = chunk;
    p.events = g_n_events > 0 ? g_events : nullptr;
    p.n_events = g_n_events;
    if ((kk == VLA_KERNEL_CHUNK || kk == VLA_KERNEL_CHUNK_TC) && T > 0) {
        const bool tc = (kk == VLA_KERNEL_CHUNK_TC);
        L = vla::chunk_layout((int)BH, T, d_h, chunk, tc && io_dtype == VLA_BF16);
        p.rows_tc = tc;
    }
    return VLA_OK;
}

// p restricted to the units [lo, lo + n): every tensor from its slice (`unit`
// bytes of an input per unit), BH = n.  The workspace fields are left as in p.
vla::FwdParams range_params(const vla::FwdParams &p, long long lo, long long n, size_t unit) {
    vla::FwdParams pr = p;
    const size_t dd = (size_t)p.d * p.d;
    const size_t ub = unit * (size_t)lo, sb = dd * (size_t)lo, nb = (size_t)p.d * (size_t)lo;
    pr.q = static_cast<const unsigned char *>(p.q) + ub;
    pr.k = static_cast<const unsigned char *>(p.k) + ub;
    pr.v = static_cast<const unsigned char *>(p.v) + ub;
    pr.u = static_cast<const unsigned char *>(p.u) + ub;
    pr.o = static_cast<unsigned char *>(p.o) + ub;
    if (p.S0) pr.S0 = p.S0 + sb;
    if (p.A0) pr.A0 = p.A0 + sb;
    if (p.n0) pr.n0 = p.n0 + nb;
    pr.S_T = p.S_T + sb;
    pr.A_T = p.A_T + sb;
    if (p.n_T) pr.n_T = p.n_T + nb;
    pr.BH = (int)n;
    return pr;
}

// vla_forward's launches; wait_qv (a cudaEvent_t or null) is waited for before
// the first pass that reads q or v.
cudaError_t launch_forward(vla::FwdParams &p, const vla::ChunkLayout &L, int kk, cudaStream_t st, void *wait_qv) {
    cudaError_t e = cudaSuccess;
    if ((kk == VLA_KERNEL_CHUNK || kk == VLA_KERNEL_CHUNK_TC) && p.T > 0) {
        p.wait_qv = wait_qv;
        e = vla::launch_chunk(p, L, st);
    } else {
        // one kernel reads every input
        if (wait_qv) e = cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(wait_qv), 0);
        if (e == cudaSuccess) {
            if (kk == VLA_KERNEL_DECODE) e = vla::launch_decode(p, st);
            else e = vla::launch_seq(p, st);  // (also T == 0: the state copy, for either choice)
        }
    }
    return e;
}

}  // namespace

extern "C" {

int vla_forward(const void *q, const void *k, const void *v, const void *u, int io_dtype, float lambda0,
                int B, int H, int T, int d_h, const float *S0, const float *A0, const float *n0, void *o,
                float *S_T, float *A_T, float *n_T, int kernel, int chunk, void *workspace,
                size_t ws_bytes, void *stream) {
    vla::FwdParams p;
    vla::ChunkLayout L;
    int kk = 0;
    const int rc = prepare_forward(q, k, v, u, io_dtype, lambda0, B, H, T, d_h, S0, A0, n0, o, S_T, A_T, n_T, kernel,
                                   chunk, workspace, ws_bytes, p, L, kk);
    if (rc != VLA_OK || p.BH == 0) return rc;
    int launches = 0;
    p.launches = &launches;
    const cudaError_t e = launch_forward(p, L, kk, static_cast<cudaStream_t>(stream), nullptr);
    if (e != cudaSuccess) return cuda_fail(e);
    t_last_launches = launches;
    return VLA_OK;
}

int vla_forward_host(const void *hq, const void *hk, const void *hv, const void *hu, int io_dtype, float lambda0,
                     int B, int H, int T, int d_h, const float *S0, const float *A0, const float *n0, void *q,
                     void *k, void *v, void *u, void *o, void *ho, float *S_T, float *A_T, float *n_T,
                     float *hS_T, float *hA_T, float *hn_T, int kernel, int chunk, void *workspace,
                     size_t ws_bytes, void *stream, void *copy_stream, void *ev_uk, void *ev_qv,
                     void *download_stream) {
    int rc = check_common(io_dtype, lambda0, B, H, T, d_h, kernel);
    if (rc != VLA_OK) return rc;
    if (!ev_uk || !ev_qv) return VLA_ERR_ARG;
    const size_t n_io = (size_t)B * H * (size_t)T * d_h * (io_dtype == VLA_BF16 ? 2 : 4);
    if (n_io > 0 && (!hq || !hk || !hv || !hu || !ho)) return VLA_ERR_ARG;
    const void *hptrs[] = {hq, hk, hv, hu, ho, hS_T, hA_T, hn_T};
    for (const void *ptr : hptrs)
        if (ptr && !aligned16(ptr)) return VLA_ERR_ALIGN;
    if (hn_T && !n_T) return VLA_ERR_ARG;
    // the device call's own checks (pointers, alignment, workspace) before anything is queued
    vla::FwdParams p;
    vla::ChunkLayout L;
    int kk = 0;
    rc = prepare_forward(q, k, v, u, io_dtype, lambda0, B, H, T, d_h, S0, A0, n0, o, S_T, A_T, n_T, kernel, chunk,
                         workspace, ws_bytes, p, L, kk);
    if (rc != VLA_OK) return rc;
    const long long BH = (long long)B * H;
    if (BH == 0) return VLA_OK;
    int launches = 0;
    p.launches = &launches;

    cudaStream_t st = static_cast<cudaStream_t>(stream), cs = static_cast<cudaStream_t>(copy_stream);
    cudaStream_t ds = static_cast<cudaStream_t>(download_stream);  // may be NULL
    cudaEvent_t e_uk = static_cast<cudaEvent_t>(ev_uk), e_qv = static_cast<cudaEvent_t>(ev_qv);
    const size_t unit = n_io / (size_t)BH;  // bytes of one (b, h) unit of an input
    auto up = [&](void *dst, const void *src, long long lo, long long n) {
        return cudaMemcpyAsync(static_cast<unsigned char *>(dst) + unit * (size_t)lo,
                               static_cast<const unsigned char *>(src) + unit * (size_t)lo, unit * (size_t)n,
                               cudaMemcpyHostToDevice, cs);
    };
    auto down_o = [&](long long lo, long long n, cudaStream_t s) {
        return cudaMemcpyAsync(static_cast<unsigned char *>(ho) + unit * (size_t)lo,
                               static_cast<const unsigned char *>(o) + unit * (size_t)lo, unit * (size_t)n,
                               cudaMemcpyDeviceToHost, s);
    };
    auto fail = [&](cudaError_t e) { return cuda_fail(e); };
    cudaError_t e;
    bool staged = n_io > 0 && BH >= 2 && kk == VLA_KERNEL_CHUNK_TC && vla::chunk_tc_parts_supported(p, L);
    // the tensor-core path's ranges, each a problem of its own over its units'
    // slices of every tensor, with its layout at its own place in the workspace
    vla::TcHostPlan plan{};
    vla::FwdParams sub[2];
    if (staged) {
        plan = vla::tc_host_plan((int)BH, T, chunk);
        if (ws_bytes < plan.total) return VLA_ERR_WORKSPACE;
        for (int s = 0; s < 2; ++s) {
            sub[s] = range_params(p, plan.sub_lo[s], plan.sub_lo[s + 1] - plan.sub_lo[s], unit);
            sub[s].ws = static_cast<unsigned char *>(workspace) + plan.off[s];
            sub[s].ws_bytes = plan.L[s].total;
            sub[s].chunk = plan.L[s].C;
            staged = staged && vla::chunk_tc_parts_supported(sub[s], plan.L[s]);
        }
    }
    // the uploads overwrite the staging buffers: after `stream`'s earlier work
    if ((e = cudaEventRecord(e_qv, st)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(cs, e_qv, 0)) != cudaSuccess) return fail(e);
    const bool staged128 = n_io > 0 && BH >= 2 && kk == VLA_KERNEL_CHUNK_TC && vla::chunk_tc128_parts_supported(p, L);
    const bool staged_seq = n_io > 0 && BH >= 2 && p.T > 0 && kk == VLA_KERNEL_SEQ;
    long long o_lo = 0;  // o from this unit on comes back on `stream`
    if (staged_seq) {
        // the sequential kernel reads every input of a unit in one pass and works
        // per unit, so it runs in ranges of units (at most four) as their inputs land:
        // q, k, v, u of a range on copy_stream, then its launch on `stream` over
        // the range's slices of every tensor; its o comes back on download_stream
        // when one is given, else on `stream` after the range's pass
        long long nr = BH < 4 ? BH : 4;
        long long r[5];
        for (long long i = 0; i <= nr; ++i) r[i] = BH * i / nr;
        for (long long j = 0; j < nr; ++j) {
            const long long lo = r[j], n = r[j + 1] - r[j];
            if ((e = up(q, hq, lo, n)) != cudaSuccess) return fail(e);
            if ((e = up(k, hk, lo, n)) != cudaSuccess) return fail(e);
            if ((e = up(v, hv, lo, n)) != cudaSuccess) return fail(e);
            if ((e = up(u, hu, lo, n)) != cudaSuccess) return fail(e);
            if ((e = cudaEventRecord(e_uk, cs)) != cudaSuccess) return fail(e);
            if ((e = cudaStreamWaitEvent(st, e_uk, 0)) != cudaSuccess) return fail(e);
            vla::FwdParams pr = range_params(p, lo, n, unit);
            int lc = 0;
            pr.launches = &lc;
            if ((e = vla::launch_seq(pr, st)) != cudaSuccess) return fail(e);
            launches += lc;
            if (ds) {
                if ((e = cudaEventRecord(e_qv, st)) != cudaSuccess) return fail(e);
                if ((e = cudaStreamWaitEvent(ds, e_qv, 0)) != cudaSuccess) return fail(e);
                if ((e = down_o(lo, n, ds)) != cudaSuccess) return fail(e);
            } else if (j + 1 < nr && (e = down_o(lo, n, st)) != cudaSuccess) {
                return fail(e);
            }
        }
        o_lo = ds ? BH : r[nr - 1];
    } else if (staged128) {
        // d = 128, one chunk per unit: both passes are per unit, one CTA per unit at
        // one CTA per SM, so the ranges are waves of 152 units (at most four
        // ranges). u and k go up range by range, each followed by its gates; then
        // q and v, each range followed by its state pass and the download of its
        // o, all on `stream`: the downloads run against the later uploads (the
        // link carries both directions at once), and a range's state pass waits
        // for its q and v longer than the previous range's o takes to come back.
        long long nr = (BH + 151) / 152;
        if (nr > 4) nr = 4;
        long long r[5];
        for (long long i = 0; i <= nr; ++i) r[i] = BH * i / nr;
        for (long long i = 0; i < nr; ++i) {
            if ((e = up(u, hu, r[i], r[i + 1] - r[i])) != cudaSuccess) return fail(e);
            if ((e = up(k, hk, r[i], r[i + 1] - r[i])) != cudaSuccess) return fail(e);
            if ((e = cudaEventRecord(e_uk, cs)) != cudaSuccess) return fail(e);
            if ((e = cudaStreamWaitEvent(st, e_uk, 0)) != cudaSuccess) return fail(e);
            if ((e = vla::launch_chunk_tc128_part(p, L, 0, (int)r[i], (int)(r[i + 1] - r[i]), st)) != cudaSuccess)
                return fail(e);
        }
        for (long long j = 0; j < nr; ++j) {
            if ((e = up(q, hq, r[j], r[j + 1] - r[j])) != cudaSuccess) return fail(e);
            if ((e = up(v, hv, r[j], r[j + 1] - r[j])) != cudaSuccess) return fail(e);
            if ((e = cudaEventRecord(e_uk, cs)) != cudaSuccess) return fail(e);
            if ((e = cudaStreamWaitEvent(st, e_uk, 0)) != cudaSuccess) return fail(e);
            if ((e = vla::launch_chunk_tc128_part(p, L, 1, (int)r[j], (int)(r[j + 1] - r[j]), st)) != cudaSuccess)
                return fail(e);
            if (ds) {  // the range's o on download_stream, beside the later passes
                if ((e = cudaEventRecord(e_qv, st)) != cudaSuccess) return fail(e);
                if ((e = cudaStreamWaitEvent(ds, e_qv, 0)) != cudaSuccess) return fail(e);
                if ((e = down_o(r[j], r[j + 1] - r[j], ds)) != cudaSuccess) return fail(e);
            } else if (j + 1 < nr && (e = down_o(r[j], r[j + 1] - r[j], st)) != cudaSuccess) {
                return fail(e);
            }
        }
        o_lo = ds ? BH : r[nr - 1];
    } else if (staged) {
        // Every pass of the tensor-core path is per (b, h) unit, so the call runs
        // the units as two problems of their own (vla::tc_host_plan), the first
        // half and the rest, as their inputs land on copy_stream: u and k of each
        // half, followed by its front (Grams, prefix, gates); then q and v in two
        // or three ranges (the first half, then the rest in one or two), each
        // followed by its back (state pass, chain, output pass). The second half
        // takes the chunk length of its smaller back ranges, so the back of the
        // last range, which runs after the last upload, is short. The o of all
        // ranges but the last comes back on copy_stream once its uploads are all
        // queued; the last range's o and the final state come back on `stream`,
        // which at the end also waits for copy_stream. The two events are
        // reused: each wait is queued right after the record it refers to,
        // before that event is recorded again.
        const int nr = plan.n;
        long long r[4];
        for (int i = 0; i <= nr; ++i) r[i] = plan.lo[i];
        for (int s = 0; s < 2; ++s) {
            const long long lo = plan.sub_lo[s], n = plan.sub_lo[s + 1] - plan.sub_lo[s];
            if ((e = up(u, hu, lo, n)) != cudaSuccess) return fail(e);
            if ((e = up(k, hk, lo, n)) != cudaSuccess) return fail(e);
            if ((e = cudaEventRecord(e_uk, cs)) != cudaSuccess) return fail(e);
            if ((e = cudaStreamWaitEvent(st, e_uk, 0)) != cudaSuccess) return fail(e);
            if ((e = vla::launch_chunk_tc_part(sub[s], plan.L[s], 0, 0, sub[s].BH, st)) != cudaSuccess)
                return fail(e);
        }
        for (int j = 0; j < nr; ++j) {
            if ((e = up(q, hq, r[j], r[j + 1] - r[j])) != cudaSuccess) return fail(e);
            if ((e = up(v, hv, r[j], r[j + 1] - r[j])) != cudaSuccess) return fail(e);
            if ((e = cudaEventRecord(e_uk, cs)) != cudaSuccess) return fail(e);
            if (j == nr - 1 && !ds) {
                // all uploads are queued: the earlier ranges' o leave on copy_stream
                // (e_qv holds "range 0 done", recorded on `stream` after its back)
                if ((e = cudaStreamWaitEvent(cs, e_qv, 0)) != cudaSuccess) return fail(e);
                if ((e = down_o(r[0], r[1] - r[0], cs)) != cudaSuccess) return fail(e);
                if (nr == 3) {
                    // `stream`'s last queued work is range 1's back
                    if ((e = cudaEventRecord(e_qv, st)) != cudaSuccess) return fail(e);
                    if ((e = cudaStreamWaitEvent(cs, e_qv, 0)) != cudaSuccess) return fail(e);
                    if ((e = down_o(r[1], r[2] - r[1], cs)) != cudaSuccess) return fail(e);
                }
            }
            if ((e = cudaStreamWaitEvent(st, e_uk, 0)) != cudaSuccess) return fail(e);
            const int s = plan.part[j];
            if ((e = vla::launch_chunk_tc_part(sub[s], plan.L[s], 1, (int)(r[j] - plan.sub_lo[s]),
                                               (int)(r[j + 1] - r[j]), st)) != cudaSuccess)
                return fail(e);
            if (ds) {  // the range's o on download_stream, beside the later passes
                if ((e = cudaEventRecord(e_qv, st)) != cudaSuccess) return fail(e);
                if ((e = cudaStreamWaitEvent(ds, e_qv, 0)) != cudaSuccess) return fail(e);
                if ((e = down_o(r[j], r[j + 1] - r[j], ds)) != cudaSuccess) return fail(e);
            } else if (j == 0 && (e = cudaEventRecord(e_qv, st)) != cudaSuccess) {
                return fail(e);
            }
        }
        // copy_stream's downloads done: `stream` waits for it after its own copies
        // (with download_stream, copy_stream's last work, an upload, is already
        // behind `stream`)
        if (!ds && (e = cudaEventRecord(e_uk, cs)) != cudaSuccess) return fail(e);
        o_lo = ds ? BH : r[nr - 1];
    } else {
        // u and k first: on the chunked paths the Grams, the prefix and the gates
        // read only those; the kernels wait for q and v before their first pass
        // that reads them
        if (n_io > 0) {
            if ((e = up(u, hu, 0, BH)) != cudaSuccess) return fail(e);
            if ((e = up(k, hk, 0, BH)) != cudaSuccess) return fail(e);
        }
        if ((e = cudaEventRecord(e_uk, cs)) != cudaSuccess) return fail(e);
        if ((e = cudaStreamWaitEvent(st, e_uk, 0)) != cudaSuccess) return fail(e);
        if (n_io > 0) {
            if ((e = up(q, hq, 0, BH)) != cudaSuccess) return fail(e);
            if ((e = up(v, hv, 0, BH)) != cudaSuccess) return fail(e);
        }
        if ((e = cudaEventRecord(e_qv, cs)) != cudaSuccess) return fail(e);
        if ((e = launch_forward(p, L, kk, st, ev_qv)) != cudaSuccess) return fail(e);
    }
    t_last_launches = launches;
    const size_t n_dd = (size_t)BH * d_h * d_h * 4, n_d = (size_t)BH * d_h * 4;
    if (n_io > 0 && o_lo < BH && (e = down_o(o_lo, BH - o_lo, st)) != cudaSuccess) return fail(e);
    if (hS_T && n_dd && (e = cudaMemcpyAsync(hS_T, S_T, n_dd, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
        return fail(e);
    if (hA_T && n_dd && (e = cudaMemcpyAsync(hA_T, A_T, n_dd, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
        return fail(e);
    if (hn_T && n_d && (e = cudaMemcpyAsync(hn_T, n_T, n_d, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
        return fail(e);
    if (staged && !ds && (e = cudaStreamWaitEvent(st, e_uk, 0)) != cudaSuccess) return fail(e);
    if (ds && (staged || staged128 || staged_seq)) {  // download_stream's copies done before `stream` is
        if ((e = cudaEventRecord(e_qv, ds)) != cudaSuccess) return fail(e);
        if ((e = cudaStreamWaitEvent(st, e_qv, 0)) != cudaSuccess) return fail(e);
    }
    return VLA_OK;
}

}  // extern "C"
