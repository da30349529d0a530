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
void *g_events[16];
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

// AUTO: the decode step for a handful of tokens; the chunk-parallel path
// (with the tensor-core state passes where they apply) when there are too
// few (b, h) units to fill the GPU with one CTA each and the stream is long
// enough to cut; otherwise the sequential kernel.
int resolve_kernel(int B, int H, int T, int d_h, int kernel) {
    (void)d_h;
    if (kernel != VLA_KERNEL_AUTO) return kernel;
    const long long BH = (long long)B * H;
    if (T >= 1 && T <= 4) return VLA_KERNEL_DECODE;
    if (BH < 2 * 152 && T >= 1024) return VLA_KERNEL_CHUNK_TC;
    return VLA_KERNEL_SEQ;
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
    if (n < 0 || n > 16) return VLA_ERR_ARG;
    if (!events) n = 0;
    for (int i = 0; i < n; ++i) g_events[i] = events[i];
    g_n_events = n;
    return VLA_OK;
}

int vla_last_launch_count(void) { return t_last_launches; }

int vla_select_kernel(int B, int H, int T, int d_h) {
    const int rc = check_common(VLA_F32, 1.f, B, H, T, d_h, VLA_KERNEL_AUTO);
    if (rc != VLA_OK) return rc;
    return resolve_kernel(B, H, T, d_h, VLA_KERNEL_AUTO);
}

size_t vla_workspace_bytes(int B, int H, int T, int d_h, int io_dtype, int kernel, int chunk) {
    if (check_common(io_dtype, 1.f, B, H, T, d_h, kernel) != VLA_OK) return 0;
    if (chunk < 0 || (chunk > 0 && chunk % 16 != 0)) return 0;
    const int kk = resolve_kernel(B, H, T, d_h, kernel);
    if ((kk != VLA_KERNEL_CHUNK && kk != VLA_KERNEL_CHUNK_TC) || T == 0 || (long long)B * H == 0) return 0;
    return vla::chunk_layout(B * H, T, d_h, chunk, kk == VLA_KERNEL_CHUNK_TC && io_dtype == VLA_BF16).total;
}

size_t vla_backward_workspace_bytes(int B, int H, int T, int d_h) {
    if (check_common(VLA_F32, 1.f, B, H, T, d_h, VLA_KERNEL_AUTO) != VLA_OK) return 0;
    if (d_h != 32 && d_h != 64) return 0;
    return vla::backward_workspace_floats(B * H, T, d_h) * sizeof(float);
}

int vla_backward(const void *q, const void *k, const void *v, const void *u, const void *dO, int io_dtype,
                 float lambda0, int B, int H, int T, int d_h, const float *S0, const float *A0, const float *n0,
                 const float *dS_T, const float *dA_T, const float *dn_T, float *dq, float *dk, float *dv,
                 float *du, float *dS0, float *dA0, float *dn0, void *workspace, size_t ws_bytes, void *stream) {
    int rc = check_common(io_dtype, lambda0, B, H, T, d_h, VLA_KERNEL_AUTO);
    if (rc != VLA_OK) return rc;
    if (d_h != 32 && d_h != 64) return VLA_ERR_UNSUPPORTED_DIM;
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
    const cudaError_t e = vla::launch_backward(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    t_last_launches = 1;
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

// vla_forward's body; wait_qv (a cudaEvent_t or null) is waited for before the
// first pass that reads q or v; wait_qv2 (or null) before the state pass of the
// units from qv_split on (every pass that reads q or v on the other paths).
// When the tensor-core path runs its later passes per half, done_first is
// recorded after the first half's o is written and *did_split set to 1.
int forward_impl(const void *q, const void *k, const void *v, const void *u, int io_dtype, float lambda0, int B,
                 int H, int T, int d_h, const float *S0, const float *A0, const float *n0, void *o, float *S_T,
                 float *A_T, float *n_T, int kernel, int chunk, void *workspace, size_t ws_bytes, void *stream,
                 void *wait_qv, void *wait_qv2, int qv_split, void *done_first, int *did_split) {
    int rc = check_common(io_dtype, lambda0, B, H, T, d_h, kernel);
    if (rc != VLA_OK) return rc;
    if (chunk < 0 || (chunk > 0 && chunk % 16 != 0)) return VLA_ERR_ARG;
    const long long BH = (long long)B * H;
    if (BH > 0) {
        if (!S_T || !A_T) return VLA_ERR_ARG;
        if (T > 0 && (!q || !k || !v || !u || !o)) return VLA_ERR_ARG;
    }
    const void *ptrs[] = {q, k, v, u, o, S0, A0, n0, S_T, A_T, n_T, workspace};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return VLA_ERR_ALIGN;
    const int kk = resolve_kernel(B, H, T, d_h, kernel);
    const size_t need = vla_workspace_bytes(B, H, T, d_h, io_dtype, kk, chunk);
    if (need > 0 && (!workspace || ws_bytes < need)) return VLA_ERR_WORKSPACE;
    if (BH == 0) return VLA_OK;

    int *err = device_err_word();
    if (!err) return cuda_fail(cudaGetLastError());

    vla::FwdParams p{};
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
    int launches = 0;
    p.launches = &launches;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if ((kk == VLA_KERNEL_CHUNK || kk == VLA_KERNEL_CHUNK_TC) && T > 0) {
        const bool tc = (kk == VLA_KERNEL_CHUNK_TC);
        const vla::ChunkLayout L = vla::chunk_layout((int)BH, T, d_h, chunk, tc && io_dtype == VLA_BF16);
        p.rows_tc = tc;
        p.wait_qv = wait_qv;
        p.wait_qv2 = wait_qv2;
        p.qv_split = qv_split;
        p.done_first = done_first;
        p.did_split = did_split;
        e = vla::launch_chunk(p, L, st);
    } else {
        // one kernel reads every input
        if (wait_qv) e = cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(wait_qv), 0);
        if (e == cudaSuccess && wait_qv2) e = cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(wait_qv2), 0);
        if (e == cudaSuccess) {
            if (kk == VLA_KERNEL_DECODE) e = vla::launch_decode(p, st);
            else e = vla::launch_seq(p, st);  // (also T == 0: the state copy, for either choice)
        }
    }
    if (e != cudaSuccess) return cuda_fail(e);
    t_last_launches = launches;
    return VLA_OK;
}

}  // namespace

extern "C" {

int vla_forward(const void *q, const void *k, const void *v, const void *u, int io_dtype, float lambda0,
                int B, int H, int T, int d_h, const float *S0, const float *A0, const float *n0, void *o,
                float *S_T, float *A_T, float *n_T, int kernel, int chunk, void *workspace,
                size_t ws_bytes, void *stream) {
    return forward_impl(q, k, v, u, io_dtype, lambda0, B, H, T, d_h, S0, A0, n0, o, S_T, A_T, n_T, kernel, chunk,
                        workspace, ws_bytes, stream, nullptr, nullptr, 0, nullptr, nullptr);
}

int vla_forward_host(const void *hq, const void *hk, const void *hv, const void *hu, int io_dtype, float lambda0,
                     int B, int H, int T, int d_h, const float *S0, const float *A0, const float *n0, void *q,
                     void *k, void *v, void *u, void *o, void *ho, float *S_T, float *A_T, float *n_T,
                     float *hS_T, float *hA_T, float *hn_T, int kernel, int chunk, void *workspace,
                     size_t ws_bytes, void *stream, void *copy_stream, void *ev_uk, void *ev_qv) {
    int rc = check_common(io_dtype, lambda0, B, H, T, d_h, kernel);
    if (rc != VLA_OK) return rc;
    if (!ev_uk || !ev_qv) return VLA_ERR_ARG;
    const size_t n_io = (size_t)B * H * (size_t)T * d_h * (io_dtype == VLA_BF16 ? 2 : 4);
    if (n_io > 0 && (!hq || !hk || !hv || !hu || !ho)) return VLA_ERR_ARG;
    const void *hptrs[] = {hq, hk, hv, hu, ho, hS_T, hA_T, hn_T};
    for (const void *p : hptrs)
        if (p && !aligned16(p)) return VLA_ERR_ALIGN;
    // the device call's own checks (pointers, alignment, workspace) before anything is queued
    {
        const long long BH = (long long)B * H;
        if (chunk < 0 || (chunk > 0 && chunk % 16 != 0)) return VLA_ERR_ARG;
        if (BH > 0 && (!S_T || !A_T)) return VLA_ERR_ARG;
        if (BH > 0 && T > 0 && (!q || !k || !v || !u || !o)) return VLA_ERR_ARG;
        const void *ptrs[] = {q, k, v, u, o, S0, A0, n0, S_T, A_T, n_T, workspace};
        for (const void *p : ptrs)
            if (p && !aligned16(p)) return VLA_ERR_ALIGN;
        const int kk = resolve_kernel(B, H, T, d_h, kernel);
        const size_t need = vla_workspace_bytes(B, H, T, d_h, io_dtype, kk, chunk);
        if (need > 0 && (!workspace || ws_bytes < need)) return VLA_ERR_WORKSPACE;
        if ((hn_T && !n_T)) return VLA_ERR_ARG;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream), cs = static_cast<cudaStream_t>(copy_stream);
    cudaEvent_t e_uk = static_cast<cudaEvent_t>(ev_uk), e_qv = static_cast<cudaEvent_t>(ev_qv);
    cudaError_t e;
    // the uploads overwrite the staging buffers: after `stream`'s earlier work
    if ((e = cudaEventRecord(e_qv, st)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamWaitEvent(cs, e_qv, 0)) != cudaSuccess) return cuda_fail(e);
    if (n_io > 0) {
        // u and k first: the Grams, the prefix and the gates read only those
        if ((e = cudaMemcpyAsync(u, hu, n_io, cudaMemcpyHostToDevice, cs)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaMemcpyAsync(k, hk, n_io, cudaMemcpyHostToDevice, cs)) != cudaSuccess) return cuda_fail(e);
    }
    if ((e = cudaEventRecord(e_uk, cs)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamWaitEvent(st, e_uk, 0)) != cudaSuccess) return cuda_fail(e);
    // q and v in two halves of the (b, h) units: the state pass of the first half
    // starts while the second uploads (ev_uk is reused: the wait above has taken
    // its first record)
    const long long BH = (long long)B * H;
    const int split = BH >= 2 ? (int)(BH / 2) : 0;
    const size_t unit = BH > 0 ? n_io / (size_t)BH : 0, first = unit * (size_t)split;
    if (n_io > 0 && split > 0) {
        const unsigned char *hq8 = static_cast<const unsigned char *>(hq), *hv8 = static_cast<const unsigned char *>(hv);
        unsigned char *q8 = static_cast<unsigned char *>(q), *v8 = static_cast<unsigned char *>(v);
        if ((e = cudaMemcpyAsync(q8, hq8, first, cudaMemcpyHostToDevice, cs)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaMemcpyAsync(v8, hv8, first, cudaMemcpyHostToDevice, cs)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaEventRecord(e_uk, cs)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaMemcpyAsync(q8 + first, hq8 + first, n_io - first, cudaMemcpyHostToDevice, cs)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaMemcpyAsync(v8 + first, hv8 + first, n_io - first, cudaMemcpyHostToDevice, cs)) != cudaSuccess)
            return cuda_fail(e);
    } else if (n_io > 0) {
        if ((e = cudaMemcpyAsync(q, hq, n_io, cudaMemcpyHostToDevice, cs)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaMemcpyAsync(v, hv, n_io, cudaMemcpyHostToDevice, cs)) != cudaSuccess) return cuda_fail(e);
    }
    if ((e = cudaEventRecord(e_qv, cs)) != cudaSuccess) return cuda_fail(e);
    const bool two = n_io > 0 && split > 0;
    int did_split = 0;
    rc = forward_impl(q, k, v, u, io_dtype, lambda0, B, H, T, d_h, S0, A0, n0, o, S_T, A_T, n_T, kernel, chunk,
                      workspace, ws_bytes, stream, two ? ev_uk : ev_qv, two ? ev_qv : nullptr, two ? split : 0, ev_uk,
                      &did_split);
    if (rc != VLA_OK) return rc;
    const size_t n_dd = (size_t)B * H * d_h * d_h * 4, n_d = (size_t)B * H * d_h * 4;
    size_t o_from = 0;
    if (did_split) {
        // the first half's o leaves on copy_stream while the second half computes; `stream`
        // then waits for that copy, so that it covers the whole call
        if ((e = cudaStreamWaitEvent(cs, e_uk, 0)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaMemcpyAsync(ho, o, first, cudaMemcpyDeviceToHost, cs)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaEventRecord(e_qv, cs)) != cudaSuccess) return cuda_fail(e);
        o_from = first;
    }
    if (n_io > o_from &&
        (e = cudaMemcpyAsync(static_cast<unsigned char *>(ho) + o_from, static_cast<const unsigned char *>(o) + o_from,
                             n_io - o_from, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
        return cuda_fail(e);
    if (hS_T && n_dd && (e = cudaMemcpyAsync(hS_T, S_T, n_dd, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
        return cuda_fail(e);
    if (hA_T && n_dd && (e = cudaMemcpyAsync(hA_T, A_T, n_dd, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
        return cuda_fail(e);
    if (hn_T && n_d && (e = cudaMemcpyAsync(hn_T, n_T, n_d, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
        return cuda_fail(e);
    if (did_split && (e = cudaStreamWaitEvent(st, e_qv, 0)) != cudaSuccess) return cuda_fail(e);
    return VLA_OK;
}

}  // extern "C"
