// vla_tc128.cu -- the kernels of the tensor-core path at d = 128 with bf16 I/O
// and one chunk per (b, h) unit: the gates (vla_gates_tc128.cuh) and the state
// pass (vla_rows_tc128.cuh) as two launches, one CTA per unit each, or both in
// one persistent launch that hands the units' passes to the SMs from a queue.
//
// Each pass of a unit is one CTA's work at one CTA per SM (both take all 512
// TMEM columns and most of the shared memory), so two launches over n units
// run ceil(n / 152) rounds each on the 152 SMs of a GB300, the last one part
// full (n = 512: four rounds of which the last holds 56 units).  The queue
// kernel runs one CTA per SM; each takes the next job from a counter in global
// memory: first the gates of every unit (jobs 0 .. n - 1), then their state
// passes (jobs n .. 2 n - 1), so both passes pack into about 2 n / 152 job
// times.  A state pass waits (bounded) for a flag that its unit's gates set
// after their last store.  The wait depends only on a job that a running CTA
// has already taken, so it never waits for a CTA that has not started.
#include "vla_gates_tc128.cuh"
#include "vla_rows_tc128.cuh"

namespace vla {
namespace {

constexpr int kT128Threads = 256;
static_assert(g128::kThreads == kT128Threads && r128::kThreads == kT128Threads, "one block shape");
constexpr size_t kGatesSmem = g128::G2Layout::total + 1024;  // + alignment slack
constexpr size_t kRowsSmem = r128::R2Layout::total + 1024;
constexpr size_t kQueueSmem = kGatesSmem > kRowsSmem ? kGatesSmem : kRowsSmem;
static_assert(kQueueSmem <= 227 * 1024, "one CTA per SM");

__global__ void __launch_bounds__(kT128Threads, 1) gates_tc128_kernel(ChunkArgs a, const __grid_constant__ CUtensorMap tm_u,
                                                                   const __grid_constant__ CUtensorMap tm_k) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    g128::gates_tc128_body(a, a.bh_lo + (int)blockIdx.x, smem_raw, &tm_u, &tm_k);
}

__global__ void __launch_bounds__(kT128Threads, 1) rows_tc128_kernel(ChunkArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    r128::rows_tc128_body(a, a.bh_lo + (int)blockIdx.x, smem_raw);
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Waits until *flag is set, giving up after limit_ns (then sets the device
// error word and returns false).
__device__ bool wait_flag(const unsigned *flag, long long limit_ns, int *err) {
    if (ld_acquire_gpu(flag)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        __nanosleep(200);
        if (ld_acquire_gpu(flag)) return true;
        if ((long long)(globaltimer_ns() - t0) > limit_ns) {
            atomicExch(err, kDevErrTimeout);
            return false;
        }
    }
}

// ctl[0]: the next job; ctl[1 + j]: unit bh_lo + j's gates are published.  Both
// zero at launch.
__global__ void __launch_bounds__(kT128Threads, 1) tc128_queue_kernel(ChunkArgs a, unsigned *ctl,
                                                                   const __grid_constant__ CUtensorMap tm_u,
                                                                   const __grid_constant__ CUtensorMap tm_k) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the job and the wait's outcome in the last 16 bytes of the allocation, past
    // any job's region (each body aligns its start within the 1024 bytes of slack)
    volatile int *s_job = reinterpret_cast<volatile int *>(smem_raw + kQueueSmem - 16);
    volatile int *s_ok = s_job + 1;
    const int n = a.bh_n;
    for (;;) {
        if (threadIdx.x == 0) *s_job = (int)atomicAdd(ctl, 1u);
        __syncthreads();
        const int job = *s_job;
        if (job >= 2 * n) break;
        if (job < n) {
            g128::gates_tc128_body(a, a.bh_lo + job, smem_raw, &tm_u, &tm_k);
            __threadfence();  // this thread's stores of the gates, before the flag
            __syncthreads();
            // (test hook: with inject set the flag stays unset, so the state pass's
            // bounded wait expires and sets the error word)
            if (threadIdx.x == 0 && !a.p.inject) st_release_gpu(ctl + 1 + job, 1u);
        } else {
            if (threadIdx.x == 0) *s_ok = wait_flag(ctl + 1 + (job - n), a.p.wait_limit_ns, a.p.err) ? 1 : 0;
            __syncthreads();
            if (*s_ok) r128::rows_tc128_body(a, a.bh_lo + job - n, smem_raw);
        }
        __syncthreads();  // s_job and s_ok are rewritten for the next job
    }
}

}  // namespace

cudaError_t launch_gates_tc128(const ChunkArgs &a, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(gates_tc128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kGatesSmem);
    if (e != cudaSuccess) return e;
    const int n = a.bh_n > 0 ? a.bh_n : a.p.BH;
    CUtensorMap tm_u, tm_k;
    if (!make_tile_map(&tm_u, a.p.u, a.p.BH, a.p.T, 128) || !make_tile_map(&tm_k, a.p.k, a.p.BH, a.p.T, 128))
        return cudaErrorInvalidValue;
    gates_tc128_kernel<<<(unsigned)n, kT128Threads, kGatesSmem, stream>>>(a, tm_u, tm_k);
    return cudaGetLastError();
}

cudaError_t launch_rows_tc128(const ChunkArgs &a, cudaStream_t stream) {
    cudaError_t e =
        cudaFuncSetAttribute(rows_tc128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRowsSmem);
    if (e != cudaSuccess) return e;
    const int n = a.bh_n > 0 ? a.bh_n : a.p.BH;
    rows_tc128_kernel<<<(unsigned)n, kT128Threads, kRowsSmem, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_tc128_queue(const ChunkArgs &a0, cudaStream_t stream) {
    ChunkArgs a = a0;
    a.bh_lo = 0;
    a.bh_n = a.p.BH;
    unsigned *ctl = reinterpret_cast<unsigned *>(static_cast<unsigned char *>(a.p.ws) + a.L.off_q);
    cudaError_t e = cudaMemsetAsync(ctl, 0, ((size_t)a.p.BH + 1) * sizeof(unsigned), stream);
    if (e != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(tc128_queue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kQueueSmem)) != cudaSuccess)
        return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc128_queue_kernel, kT128Threads, kQueueSmem)) !=
        cudaSuccess)
        return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long long grid = (long long)sms * per_sm;
    if (grid > 2LL * a.p.BH) grid = 2LL * a.p.BH;
    CUtensorMap tm_u, tm_k;
    if (!make_tile_map(&tm_u, a.p.u, a.p.BH, a.p.T, 128) || !make_tile_map(&tm_k, a.p.k, a.p.BH, a.p.T, 128))
        return cudaErrorInvalidValue;
    tc128_queue_kernel<<<(unsigned)grid, kT128Threads, kQueueSmem, stream>>>(a, ctl, tm_u, tm_k);
    return cudaGetLastError();
}

}  // namespace vla
