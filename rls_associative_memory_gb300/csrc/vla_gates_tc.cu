// vla_gates_tc.cu -- the gates pass of the tensor-core chunk path at d = 64
// (its body, with the method's account, is in vla_gates_tc.cuh): one CTA per
// A-chunk of every (b, h) unit.
#include "vla_gates_tc.cuh"

namespace vla {
namespace {

constexpr size_t kBody = g64::GtLayout::total + 1024;  // + alignment slack; then the TMEM slot

__global__ void __launch_bounds__(g64::kThreads, 2) gates_tc_kernel(ChunkArgs a, const __grid_constant__ CUtensorMap tm_u,
                                                                    const __grid_constant__ CUtensorMap tm_k) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 256 TMEM columns; the permit is given up at once, so that the SM's other
    // CTA can allocate its own while this one holds them
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem_raw + kBody);
    if (threadIdx.x < 32) tmem_alloc(tslot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const unsigned NCA = (unsigned)a.L.NCA;
    g64::gates_tc_body(a, (int)(blockIdx.x % NCA), a.bh_lo + (int)(blockIdx.x / NCA), smem_raw, &tm_u, &tm_k, tbase);
    tc_fence_after();  // the body ended with its TMEM reads fenced and the CTA synchronised
    if (threadIdx.x < 32) tmem_dealloc(tbase, 256);
}

}  // namespace

bool gates_tc_supported(const FwdParams &p, const ChunkLayout &L) {
    return p.d == tc::kD && p.io_bf16 && L.CA % tc::kSB == 0 && L.yh && tile_maps_available();
}

cudaError_t launch_gates_tc(const ChunkArgs &a, cudaStream_t stream) {
    constexpr size_t bytes = kBody + 16;
    cudaError_t e = cudaFuncSetAttribute(gates_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    const long long grid = (long long)a.L.NCA * (a.bh_n > 0 ? a.bh_n : a.p.BH);
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    CUtensorMap tm_u, tm_k;
    if (!make_tile_map(&tm_u, a.p.u, a.p.BH, a.p.T) || !make_tile_map(&tm_k, a.p.k, a.p.BH, a.p.T))
        return cudaErrorInvalidValue;
    gates_tc_kernel<<<(unsigned)grid, g64::kThreads, bytes, stream>>>(a, tm_u, tm_k);
    return cudaGetLastError();
}

}  // namespace vla
