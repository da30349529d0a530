// vla_noalloc.cu -- vla_forward_noalloc: the chunk-parallel path with its
// workspace in a scratch array compiled into the library, for callers that
// are not allowed to allocate device memory (see include/vla.h).
//
// The scratch is one file-scope static __device__ array.  Its name, used in
// host code, is only a host-side stand-in for the symbol: passing it to a
// kernel would hand the kernel a host address.  The device address is
// looked up with cudaGetSymbolAddress, with the device current, at set-up,
// and that pointer is what the kernels receive.  Set-up runs once per device
// and context: the address is kept together with the id of the driver
// context it was taken in, and a call made in another context (after a
// cudaDeviceReset, or from a context that is not the device's primary one)
// repeats the set-up instead of using a stale address.
#include <cuda.h>

#include <mutex>

#include "../../include/vla.h"
#include "vla_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[VLA_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

template <typename Fn>
Fn driver_fn(const char *name) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}

// Unique id of the calling thread's current driver context, 0 when there is
// none yet (ids are never reused within a process, so a reset device gets a
// new one).
int current_context_id(unsigned long long *id) {
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    *id = 0;
    if (!get_current || !get_id) return VLA_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return VLA_ERR_CUDA;
    if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return VLA_ERR_CUDA;
    return VLA_OK;
}

constexpr int kMaxDevices = 64;
struct ScratchSlot {
    unsigned long long ctx_id;  // context the address belongs to (0: none yet)
    void *ptr;                  // device address of g_noalloc_scratch in that context
};
std::mutex g_setup_mu;
ScratchSlot g_slot[kMaxDevices];

// The array's device address for the current device.  Set-up: with the
// device current, cudaGetSymbolAddress once per device and context.
int scratch_for_current_device(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return vla::api_cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return VLA_ERR_ARG;
    unsigned long long id = 0;
    int rc = current_context_id(&id);
    if (rc != VLA_OK) return rc;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    ScratchSlot &s = g_slot[dev];
    if (id == 0 || s.ctx_id != id || !s.ptr) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);  // makes the context current if needed
        if (e != cudaSuccess) return vla::api_cuda_fail(e);
        if (!ptr) return VLA_ERR_CUDA;
        if ((rc = current_context_id(&id)) != VLA_OK) return rc;
        if (id == 0) return VLA_ERR_CUDA;
        s.ctx_id = id;
        s.ptr = ptr;
    }
    *out = s.ptr;
    return VLA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int vla_forward_noalloc(const void *q, const void *k, const void *v, const void *u,
                                   int io_dtype, float lambda0, int B, int H, int T, int d_h,
                                   const float *S0, const float *A0, const float *n0, void *o,
                                   float *S_T, float *A_T, float *n_T, int chunk, void *stream) {
    int rc = vla::api_check_common(io_dtype, lambda0, B, H, T, d_h, VLA_KERNEL_CHUNK);
    if (rc != VLA_OK) return rc;
    if (chunk < 0 || (chunk > 0 && chunk % 16 != 0)) return VLA_ERR_ARG;
    const long long BH = (long long)B * H;
    if (BH > 0) {
        if (!S_T || !A_T) return VLA_ERR_ARG;
        if (T > 0 && (!q || !k || !v || !u || !o)) return VLA_ERR_ARG;
    }
    const void *ptrs[] = {q, k, v, u, o, S0, A0, n0, S_T, A_T, n_T};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return VLA_ERR_ALIGN;

    vla::ChunkLayout L{};
    if (BH > 0 && T > 0) {
        L = vla::chunk_layout((int)BH, T, d_h, chunk);
        if (L.total > (size_t)VLA_NOALLOC_SCRATCH_BYTES) return VLA_ERR_SCRATCH_LIMIT;
    }
    // set-up (also for an empty problem, which does nothing else)
    void *scratch = nullptr;
    rc = scratch_for_current_device(&scratch);
    if (rc != VLA_OK) return rc;
    if (BH == 0) return VLA_OK;
    int *err = vla::api_device_err_word();
    if (!err) return vla::api_cuda_fail(cudaGetLastError());

    vla::FwdParams p{};
    p.q = q; p.k = k; p.v = v; p.u = u; p.o = o;
    p.S0 = S0; p.A0 = A0; p.n0 = n0;
    p.S_T = S_T; p.A_T = A_T; p.n_T = n_T;
    p.BH = (int)BH; p.T = T; p.d = d_h;
    p.io_bf16 = (io_dtype == VLA_BF16);
    p.lambda0 = lambda0;
    p.err = err;
    p.wait_limit_ns = vla::api_wait_limit_ns();
    p.inject = 0;
    p.ws = scratch;
    p.ws_bytes = VLA_NOALLOC_SCRATCH_BYTES;
    p.chunk = chunk;
    p.events = nullptr;
    p.n_events = 0;
    p.launches = nullptr;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // T == 0 only copies the initial state (no scratch needed).
    const cudaError_t e = (T > 0) ? vla::launch_chunk(p, L, st) : vla::launch_seq(p, st);
    if (e != cudaSuccess) return vla::api_cuda_fail(e);
    return VLA_OK;
}
