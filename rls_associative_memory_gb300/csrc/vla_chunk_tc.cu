// vla_chunk_tc.cu -- the tensor-core state pass (its body, and the account of
// both passes, in vla_rows_tc.cuh) and output pass of the chunk-parallel path
// for d = 64 with bf16 I/O ("Variational Linear Attention: Stable Associative
// Memory for Long-Context Transformers", section 2.3).
#include "vla_rows_tc.cuh"

namespace vla {
namespace {

using namespace tc;

constexpr size_t kRowsBody = r64::TcLayout::total + 1024;  // + alignment slack; then the TMEM slot

__global__ void __launch_bounds__(r64::kThreads, 2) rows_tc_kernel(ChunkArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 256 TMEM columns; the permit is given up at once, so that the SM's other
    // CTA can allocate its own while this one holds them
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem_raw + kRowsBody);
    if (threadIdx.x < 32) tmem_alloc(tslot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const unsigned NC = (unsigned)a.L.NC;
    r64::rows_tc_body(a, (int)(blockIdx.x % NC), a.bh_lo + (int)(blockIdx.x / NC), smem_raw, tbase);
    tc_fence_after();  // the body ended with its TMEM reads fenced and the CTA synchronised
    if (threadIdx.x < 32) tmem_dealloc(tbase, 256);
}

// ---------------------------------------------------------------------------
// Output pass: o_t = S_c y_t + h_t for every token, one CTA per chunk.  Per
// sub-block one product D = [Y | H] [S_c | I]^T on the tensor cores (S_c as
// a bf16 hi/lo pair, H against the exact identity), with the sub-block's
// coefficient tiles brought in by bulk copies two sub-blocks ahead.  y_t and
// h_t are stored as single bf16: each o_t is a 64-term sum over them, whose
// rounding errors average out far below o's own bf16 rounding (measured
// against the fp64 recursion: the relative error of o is unchanged, 1.64e-3
// either way, on the long stream's first 8192 tokens).
// ---------------------------------------------------------------------------
constexpr int kOutThreads = 128;

struct OutLayout {
    static constexpr size_t ctrl = 0;                   // mbarriers (2 stages, MMA), TMEM slot, abort flag
    static constexpr size_t stage = 1024;               // 2 x [y | h]
    static constexpr size_t sc_hi = stage + 4 * kTile;  // S_c (row i, column j), hi, lo
    static constexpr size_t sc_lo = sc_hi + kTile;
    static constexpr size_t eye = sc_hi + 2 * kTile;    // identity (bf16)
    static constexpr size_t total = eye + kTile;
};

__global__ void __launch_bounds__(kOutThreads) out_tc_kernel(ChunkArgs a) {
    using L = OutLayout;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::ctrl);  // [2]
    uint64_t *mbar = full + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L::ctrl + 24);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::ctrl + 28);
    unsigned char *st = smem + L::stage, *sc_hi = smem + L::sc_hi, *sc_lo = smem + L::sc_lo, *eye = smem + L::eye;

    // two CTAs a chunk, each over half of its sub-blocks (the output pass has no
    // recurrence left in it; more, shorter CTAs fill the waves better)
    const int NC = a.L.NC, C = a.L.C, T = a.p.T;
    const unsigned blk = blockIdx.x >> 1;
    const int c = (int)(blk % (unsigned)NC), bh = a.bh_lo + (int)(blk / (unsigned)NC);
    const int t0 = c * C, ntok = min(C, T - t0), nsb_chunk = (ntok + kSB - 1) / kSB;
    const int half = (nsb_chunk + 1) / 2, sb0 = (int)(blockIdx.x & 1u) * half;
    const int nsb = min(nsb_chunk, sb0 + half) - sb0;  // this CTA's sub-blocks sb0 .. sb0 + nsb - 1
    if (nsb <= 0) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned char *gyh = static_cast<const unsigned char *>(a.p.ws) + a.L.off_yh +
                               ((size_t)(bh * NC + c) * (C / kSB) + (size_t)sb0) * (2 * kTile);
    __nv_bfloat16 *gout = static_cast<__nv_bfloat16 *>(a.p.o) + ((size_t)bh * T + t0 + (size_t)sb0 * kSB) * kD;
    const int ntok_cta = ntok - sb0 * kSB;  // tokens from this CTA's first sub-block on

    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(mbar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0) tmem_alloc(tslot, 64);
    {  // S_c row i, columns 32 h .. as a hi/lo pair; the identity
        const int i = tid >> 1, h = tid & 1;
        const float4 *src = reinterpret_cast<const float4 *>(ws_f(a, a.L.off_S) + ((size_t)bh * NC + c) * kD * kD +
                                                             (size_t)i * kD + 32 * h);
        float v[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 s4 = src[q];
            v[4 * q] = s4.x; v[4 * q + 1] = s4.y; v[4 * q + 2] = s4.z; v[4 * q + 3] = s4.w;
        }
        put_row32(sc_hi, sc_lo, i, 32 * h, v);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {  // bf16 1.0 = 0x3f80; element k in the low half
                const int k = 32 * h + 8 * g + 2 * e;
                w[e] = (k == i ? 0x3f80u : 0u) | (k + 1 == i ? 0x3f800000u : 0u);
            }
            *reinterpret_cast<uint4 *>(eye + toff(i, 32 * h + 8 * g)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    int issued = min(2, nsb), landed = 0, mma_open = -1;  // (thread 0's bookkeeping)
    if (tid == 0) {
        for (int s = 0; s < issued; ++s) {
            mbar_arrive_expect_tx(&full[s], 2 * kTile);
            bulk_g2s(st + (size_t)s * 2 * kTile, gyh + (size_t)s * 2 * kTile, 2 * kTile, &full[s]);
        }
    }
    constexpr uint32_t id_64 = idesc_bf16_f32(64, 64);
    for (int sb = 0; sb < nsb; ++sb) {
        const int s = sb & 1;
        unsigned char *yh = st + (size_t)s * 2 * kTile;
        if (tid == 0) {
            bool w = mbar_wait_bounded(&full[s], (uint32_t)((sb >> 1) & 1), a.p.wait_limit_ns, a.p.err);
            if (w) {
                landed = sb + 1;
                tc_fence_after();
                // D = Y (S_c hi + S_c lo)^T + H I^T; the coefficient tiles hold a
                // feature per row (MN-major: rows = K, columns = the tokens M)
                mma_k64<true, false>(tbase, smem_u32(yh), smem_u32(sc_hi), id_64, false);
                mma_k64<true, false>(tbase, smem_u32(yh), smem_u32(sc_lo), id_64, true);
                mma_k64<true, false>(tbase, smem_u32(yh + kTile), smem_u32(eye), id_64, true);
                umma_commit(mbar);
                w = mbar_wait_bounded(mbar, (uint32_t)(sb & 1), a.p.wait_limit_ns, a.p.err);
                if (!w) mma_open = sb;
            }
            if (!w) {
                *abort_flag = 1;
            } else if (sb + 2 < nsb) {  // the stage is free again: bring in sub-block sb + 2
                mbar_arrive_expect_tx(&full[s], 2 * kTile);
                bulk_g2s(yh, gyh + (size_t)(sb + 2) * 2 * kTile, 2 * kTile, &full[s]);
                issued = sb + 3;
            }
        }
        __syncthreads();
        tc_fence_after();
        if (*abort_flag) break;
        // o rows: token t = 16 warp + lane (lanes 0..15 hold the M = 64 rows)
        const int t = 16 * warp + lane;
        const bool act = lane < 16 && sb * kSB + t < ntok_cta;
        uint4 *dst = reinterpret_cast<uint4 *>(gout + (size_t)(sb * kSB + (t & 63)) * kD);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v[32];
            tmem_ld32(tbase + ((uint32_t)(32 * warp) << 16) + 32 * h, v);
            if (act) {
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = bf2_bits(__floats2bfloat162_rn(v[8 * g + 2 * e], v[8 * g + 2 * e + 1]));
                    dst[4 * h + g] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
        tc_fence_before();
        __syncthreads();
    }
    if (tid == 0) {  // after an abort: copies and products that may still be in flight
        for (int sb = landed; sb < issued; ++sb)
            (void)mbar_wait_bounded(&full[sb & 1], (uint32_t)((sb >> 1) & 1), a.p.wait_limit_ns, a.p.err);
        if (mma_open >= 0) (void)mbar_wait_bounded(mbar, (uint32_t)(mma_open & 1), a.p.wait_limit_ns, a.p.err);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 64);
}

}  // namespace

bool rows_tc_supported(const FwdParams &p, const ChunkLayout &L) {
    return p.d == kD && p.io_bf16 && L.C % kSB == 0 && L.yh;
}

cudaError_t launch_rows_tc(const ChunkArgs &a, int mode, cudaStream_t stream) {
    const long long grid = (long long)a.L.NC * (a.bh_n > 0 ? a.bh_n : a.p.BH);
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaError_t e;
    if (mode == 0) {
        constexpr size_t bytes = kRowsBody + 16;
        if ((e = cudaFuncSetAttribute(rows_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes)) !=
            cudaSuccess)
            return e;
        rows_tc_kernel<<<(unsigned)grid, r64::kThreads, bytes, stream>>>(a);
    } else {
        constexpr size_t bytes = OutLayout::total + 1024;
        if ((e = cudaFuncSetAttribute(out_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes)) !=
            cudaSuccess)
            return e;
        if (2 * grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        out_tc_kernel<<<(unsigned)(2 * grid), kOutThreads, bytes, stream>>>(a);  // two CTAs a chunk
    }
    return cudaGetLastError();
}

}  // namespace vla
