// vla_tc64_queue.cu -- the gates (vla_gates_tc.cuh) and the state pass
// (vla_rows_tc.cuh) of the tensor-core chunk path at d = 64 in one persistent
// launch.
//
// As two launches each pass runs its CTAs in waves of two per SM on the 152
// SMs of a GB300, and a pass whose CTA count is not a whole number of waves
// ends with a part-full one (32 units of 4096 tokens: 512 CTAs a pass, 1.68
// waves).  Here two CTAs per SM take jobs from a counter in global memory:
// first the gates of every A-chunk, then the state pass of every S-chunk, so
// the two passes pack into (gates jobs x their length + state-pass jobs x
// theirs) / 304 job times.  A state pass waits (bounded) for the flags of the
// A-chunks its S-chunk covers, which their gates set after their last store.
// Jobs are handed out in order, so a state pass only ever waits for gates jobs
// that a running CTA has already taken, and the launch needs no co-residency
// guarantee.
#include "vla_gates_tc.cuh"
#include "vla_rows_tc.cuh"

namespace vla {
namespace {

constexpr int kQThreads = 256;
static_assert(g64::kThreads == kQThreads && r64::kThreads == kQThreads, "one block shape");
constexpr size_t kQGates = g64::GtLayout::total + 1024;  // + alignment slack
constexpr size_t kQRows = r64::TcLayout::total + 1024;
constexpr size_t kQBodies = kQGates > kQRows ? kQGates : kQRows;
constexpr size_t kQSmem = kQBodies + 16;  // the job, the wait's outcome and the TMEM slot past every body's region
static_assert(2 * (kQSmem + 1024) <= 228 * 1024, "two CTAs per SM");

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

// ctl[0]: the next job; ctl[1 + u NCA + c]: A-chunk c of unit bh_lo + u has its
// gates published.  All zero at launch.
__global__ void __launch_bounds__(kQThreads, 2) tc64_queue_kernel(ChunkArgs a, unsigned *ctl,
                                                                  const __grid_constant__ CUtensorMap tm_u,
                                                                  const __grid_constant__ CUtensorMap tm_k) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    volatile int *s_job = reinterpret_cast<volatile int *>(smem_raw + kQBodies);
    volatile int *s_ok = s_job + 1;
    // 256 TMEM columns for every job of this CTA.  The permit is given up at
    // once: a CTA that keeps it holds back the SM's other CTA at its own
    // allocation until this one exits.
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem_raw + kQBodies + 8);
    if (threadIdx.x < 32) tmem_alloc(tslot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const int n = a.bh_n, NCA = a.L.NCA, NC = a.L.NC;
    const int per = a.L.C / a.L.CA;  // A-chunks an S-chunk covers
    const int G = n * NCA, R = n * NC;
    for (;;) {
        if (threadIdx.x == 0) *s_job = (int)atomicAdd(ctl, 1u);
        __syncthreads();
        const int job = *s_job;
        if (job >= G + R) break;
        if (job < G) {
            const int u = job / NCA, c = job % NCA;
            g64::gates_tc_body(a, c, a.bh_lo + u, smem_raw, &tm_u, &tm_k, tbase);
            __threadfence();  // this thread's stores of the gates (and A_T), before the flag
            __syncthreads();
            // (test hook: with inject set the flag stays unset, so the state pass's
            // bounded wait expires and sets the error word)
            if (threadIdx.x == 0 && !a.p.inject) st_release_gpu(ctl + 1 + job, 1u);
        } else {
            const int u = (job - G) / NC, c = (job - G) % NC;
            if (threadIdx.x == 0) {
                bool ok = true;
                for (int j = 0; j < per && ok; ++j) {
                    const int ca = c * per + j;
                    if (ca < NCA) ok = wait_flag(ctl + 1 + (size_t)u * NCA + ca, a.p.wait_limit_ns, a.p.err);
                }
                *s_ok = ok ? 1 : 0;
            }
            __syncthreads();
            if (*s_ok) r64::rows_tc_body(a, c, a.bh_lo + u, smem_raw, tbase);
        }
        __syncthreads();  // s_job and s_ok are rewritten for the next job
    }
    tc_fence_after();  // every body ended with its TMEM reads fenced and the CTA synchronised
    if (threadIdx.x < 32) tmem_dealloc(tbase, 256);
}

}  // namespace

cudaError_t launch_tc64_queue(const ChunkArgs &a0, cudaStream_t stream) {
    ChunkArgs a = a0;
    const int n = a.bh_n > 0 ? a.bh_n : a.p.BH;
    a.bh_n = n;
    const long long jobs = (long long)n * (a.L.NCA + a.L.NC);
    if (jobs > 0x7fffffffLL || a.L.C % a.L.CA != 0) return cudaErrorInvalidConfiguration;
    unsigned *ctl = reinterpret_cast<unsigned *>(static_cast<unsigned char *>(a.p.ws) + a.L.off_q);
    cudaError_t e = cudaMemsetAsync(ctl, 0, ((size_t)n * a.L.NCA + 1) * sizeof(unsigned), stream);
    if (e != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(tc64_queue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kQSmem)) !=
        cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(tc64_queue_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  (int)cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
        return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc64_queue_kernel, kQThreads, kQSmem)) !=
        cudaSuccess)
        return e;
    // Two per SM as the launch bounds ask.  CTAs beyond what is resident take
    // no job until they start (by then the counter may be spent), so a grid
    // larger than the residency is only slower, never stuck.
    long long grid = (long long)sms * (per_sm > 2 ? per_sm : 2);
    if (grid > jobs) grid = jobs;
    CUtensorMap tm_u, tm_k;
    if (!make_tile_map(&tm_u, a.p.u, a.p.BH, a.p.T) || !make_tile_map(&tm_k, a.p.k, a.p.BH, a.p.T))
        return cudaErrorInvalidValue;
    tc64_queue_kernel<<<(unsigned)grid, kQThreads, kQSmem, stream>>>(a, ctl, tm_u, tm_k);
    return cudaGetLastError();
}

}  // namespace vla
