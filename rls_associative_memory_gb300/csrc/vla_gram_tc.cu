// vla_gram_tc.cu -- chunk Grams of the tensor-core chunk path (d = 64, bf16
// I/O): G_c = U_c^T U_c over each A-chunk and the chunk sums of
// phi(k_hat), the inputs of the prefix form M^(c) = lambda0 I + sum of the
// earlier Grams of section 2.2's M_t = M_{t-1} + u_t u_t^T ("Variational
// Linear Attention: Stable Associative Memory for Long-Context
// Transformers"), and of the readout's n_t (section 2.3).
//
// Tiles of 64 tokens of u and k arrive by TMA tensor copies
// (cp.async.bulk.tensor) in the 128-byte swizzle, three stages deep (a stage
// is refilled one iteration after its product was issued).  The
// token-major u tile is both operands of the product, read MN-major (tile
// rows = K = tokens), so no transposition is needed; bf16 x bf16 products
// are exact in fp32 and only the accumulation (in TMEM) rounds.  Two
// threads a token (32 features each) sum phi(k_hat) on the CUDA cores.  The 3-D
// tensor maps (features, tokens, b*h) fill tokens past T with zeros.
#include "vla_tma.cuh"

namespace vla {
namespace {

using namespace tc;

constexpr int kGThreads = 128;
constexpr int kStages = 3;  // 50 KB a CTA: four CTAs per SM (608 Grams of the long stream in one wave)

struct GrLayout {
    static constexpr size_t ctrl = 0;                     // full[4], done[4] mbarriers, TMEM slot, abort flag
    static constexpr size_t tiles = 1024;                 // [stage]: u tile, k tile (8 KB each)
    static constexpr size_t nred = tiles;                 // [128 threads][33] fp32, over the tiles once all are used
    static constexpr size_t total = tiles + (size_t)kStages * 2 * kTile;
};
static_assert(128 * 33 * 4 <= kStages * 2 * kTile, "the reduction buffer fits over the tiles");

__global__ void __launch_bounds__(kGThreads) gram_tma_kernel(ChunkArgs a, const __grid_constant__ CUtensorMap tm_u,
                                                            const __grid_constant__ CUtensorMap tm_k) {
    using L = GrLayout;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::ctrl);
    uint64_t *done = full + kStages;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L::ctrl + 16 * kStages);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::ctrl + 16 * kStages + 4);
    float *nred = reinterpret_cast<float *>(smem + L::nred);

    const int NCA = a.L.NCA, CA = a.L.CA, T = a.p.T;
    const int c = (int)(blockIdx.x % (unsigned)NCA), bh = a.bh_lo + (int)(blockIdx.x / (unsigned)NCA);
    const int t0 = c * CA, ntok = min(CA, T - t0), nst = (ntok + kSB - 1) / kSB;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    auto su = [&](int b) { return smem + L::tiles + (size_t)b * 2 * kTile; };
    auto sk = [&](int b) { return smem + L::tiles + (size_t)b * 2 * kTile + kTile; };

    if (tid == 0) {
        for (int b = 0; b < kStages; ++b) {
            mbar_init(&full[b], 1);
            mbar_init(&done[b], 1);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0) tmem_alloc(tslot, 64);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;

    auto issue = [&](int st) {
        const int b = st % kStages;
        mbar_arrive_expect_tx(&full[b], 2 * kTile);
        tma_load_3d(su(b), &tm_u, 0, t0 + st * kSB, bh, &full[b]);
        tma_load_3d(sk(b), &tm_k, 0, t0 + st * kSB, bh, &full[b]);
    };
    int issued = 0, committed = 0, landed = 0;  // (thread 0's bookkeeping)
    if (tid == 0) {
        for (int st = 0; st < kStages && st < nst; ++st) issue(st);
        issued = min(kStages, nst);
    }
    // phi(k_hat) sums: thread (token position pt = tid / 2 of every tile,
    // features 32 ph .. 32 ph + 31)
    const int pt = tid >> 1, ph = tid & 1;
    float nk[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) nk[j] = 0.f;
    bool ok = true;
    for (int st = 0; st < nst; ++st) {
        const int b = st % kStages;
        if (!mbar_wait_bounded(&full[b], (uint32_t)((st / kStages) & 1), a.p.wait_limit_ns, a.p.err))
            *abort_flag = 1;
        else
            landed = st + 1;
        __syncthreads();
        if (*abort_flag) {
            ok = false;
            break;
        }
        if (tid == 0) {  // G += U^T U over these 64 tokens (both operands the u tile, MN-major)
            tc_fence_after();
            mma_k64<true, true>(tbase, smem_u32(su(b)), smem_u32(su(b)), idesc_bf16_f32(64, 64), st > 0);
            umma_commit(&done[b]);
            committed = st + 1;
        }
        // phi(k_hat) of this tile's tokens inside the chunk
        {
            float kf[32];
#pragma unroll
            for (int g = 0; g < 4; ++g)
                unpack8(*reinterpret_cast<const uint4 *>(sk(b) + toff(pt, 32 * ph + 8 * g)), kf + 8 * g);
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) ss = fmaf(kf[j], kf[j], ss);
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            const float ks = 1.f / fmaxf(sqrtf(ss), kEps);
            if (pt < min(kSB, ntok - st * kSB)) {
#pragma unroll
                for (int j = 0; j < 32; ++j) nk[j] += phi_fast(kf[j] * ks);
            }
        }
        __syncthreads();  // everyone is done with the k tile
        // refill the previous tile's stage: its product was issued an iteration
        // ago (waiting on it does not stall on the one just issued)
        if (tid == 0 && st >= 1 && st + kStages - 1 < nst) {
            const int sp = st - 1;
            if (!mbar_wait_bounded(&done[sp % kStages], (uint32_t)((sp / kStages) & 1), a.p.wait_limit_ns, a.p.err)) {
                *abort_flag = 1;
            } else {
                issue(sp + kStages);
                issued = sp + kStages + 1;
            }
        }
    }
    // the last product, then the accumulator
    if (ok && tid == 0 && committed > 0) {
        const int l = committed - 1;
        if (!mbar_wait_bounded(&done[l % kStages], (uint32_t)((l / kStages) & 1), a.p.wait_limit_ns, a.p.err))
            *abort_flag = 1;
    }
    __syncthreads();
    tc_fence_after();
    if (!ok || *abort_flag) {
        if (tid == 0) {  // let everything issued land before the CTA exits
            if (committed > 0) {  // (a commit covers every earlier product)
                const int l = committed - 1;
                (void)mbar_wait_bounded(&done[l % kStages], (uint32_t)((l / kStages) & 1), a.p.wait_limit_ns,
                                        a.p.err);
            }
            for (int st = landed; st < issued; ++st)
                (void)mbar_wait_bounded(&full[st % kStages], (uint32_t)((st / kStages) & 1), a.p.wait_limit_ns,
                                        a.p.err);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tbase, 64);
        return;
    }
    float *gout = ws_f(a, a.L.off_M) + ((size_t)bh * NCA + c) * kD * kD;
    {
        // M = 64: row r in lane 32 (r / 16) + r % 16 of quarter r / 16
#pragma unroll
        for (int cb = 0; cb < 64; cb += 32) {
            float v[32];
            tmem_ld32(tbase + ((uint32_t)(32 * warp) << 16) + (uint32_t)cb, v);
            if (lane < 16) {
                float4 *dst = reinterpret_cast<float4 *>(gout + (size_t)(16 * warp + lane) * kD + cb);
#pragma unroll
                for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) nred[tid * 33 + j] = nk[j];  // (33: conflict-free columns below)
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 64);
    if (tid < 64) {  // feature tid: the 64 threads with ph = tid / 32
        const int f = tid & 31, h = tid >> 5;
        float s = 0.f;
        for (int p = 0; p < 64; ++p) s += nred[(2 * p + h) * 33 + f];
        ws_f(a, a.L.off_n)[((size_t)bh * (NCA + 1) + c) * kD + tid] = s;
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

}  // namespace

bool tile_maps_available() { return encode_fn() != nullptr; }

bool make_tile_map(CUtensorMap *m, const void *base, int BH, int T, int d) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || (d != 64 && d != 128)) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)T * d * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kD, (cuuint32_t)kSB, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool gram_tma_supported(const FwdParams &p, const ChunkLayout &L) {
    return p.d == kD && p.io_bf16 && L.CA % kSB == 0 && L.yh && encode_fn() != nullptr;
}

cudaError_t launch_gram_tma(const ChunkArgs &a, cudaStream_t stream) {
    CUtensorMap tm_u, tm_k;
    if (!make_tile_map(&tm_u, a.p.u, a.p.BH, a.p.T) || !make_tile_map(&tm_k, a.p.k, a.p.BH, a.p.T))
        return cudaErrorInvalidValue;
    constexpr size_t bytes = GrLayout::total + 1024;  // + alignment slack
    cudaError_t e = cudaFuncSetAttribute(gram_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    const long long grid = (long long)a.L.NCA * (a.bh_n > 0 ? a.bh_n : a.p.BH);
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    gram_tma_kernel<<<(unsigned)grid, kGThreads, bytes, stream>>>(a, tm_u, tm_k);
    return cudaGetLastError();
}

}  // namespace vla
