// vla_gates_tc.cu -- the gates of the chunk-parallel path on the tensor cores
// for d = 64 with bf16 I/O: section 2.2's inverse penalty A (kept by
// Sherman-Morrison) and section 2.3's unit gate alpha_t = A_t k_hat_t /
// |A_t k_hat_t| of "Variational Linear Attention: Stable Associative Memory
// for Long-Context Transformers", 64 tokens at a time in block-Woodbury form.
//
// For a sub-block of c = 64 tokens with A at its start, U = [u_1 .. u_c] and
// K = [k_1 .. k_c]:
//   W = A U,  G = U^T W  (c x c),  I + G = L D L^T  (unit lower L)
//   z_s = A_{s-1} u_s = W x_s with X = L^{-T}, beta_s = 1 / (1 + u_s . z_s) = 1 / D_s
//     (the leading blocks of an LDL^T are the LDL^T of the leading blocks, so
//     these are exactly the quantities of the token-by-token recursion)
//   A_t k_hat_t = A k_hat_t - sum_{s <= t} beta_s z_s (z_s . k_hat_t),
//     z_s . k_hat_t = (X^T U^T A K_hat)[s][t]
//   A_end = A - Z diag(beta) Z^T
// Per sub-block (tensor-core rounds R1..R4; tiles and products as in the
// state passes, bf16 hi/lo pairs for fp32 operands):
//   R1  D1 = [U; K] A                 rows: w_t, A k_t
//   R2  D2 = U [A K ; W]^T            Y = U^T A K, G = U^T W
//   on the CUDA cores: elimination of [I + G | I] -> [D L^T | L^{-1}],
//       L^{-1} = X^T and beta_s = 1 / pivot_s (the trailing block stays
//       symmetric, so the multipliers come from the pivot row)
//   R3  D3 = X^T [W | Y_hat]          Z^T and P = X^T Y_hat, Y_hat = Y diag(1/|k|)
//   R4  D1[k rows] += E'^T Z^T        E'[s][t] = -beta_s P[s][t] |k_t| (s <= t):
//                                      the rows become |k_t| A_t k_hat_t
//       A += -(Z diag(beta)) Z^T      (A held in fp32 in TMEM for the whole
//                                      A-chunk; the product accumulates onto it)
//   alpha_t = that row / |that row|, and the new A's operand tiles.
// A starts each A-chunk from its definition (M^(c))^{-1}, M^(c) = lambda0 I +
// the Grams of the earlier A-chunks: the same elimination on M^(c) gives
// E = L^{-1} and D, then A = E^T D^{-1} E is one product on the tensor cores.
#include "vla_tc_common.cuh"

namespace vla {
namespace {

using namespace tc;

constexpr int kThreads = 256;

struct GtLayout {
    static constexpr size_t ctrl = 0;                       // mbarrier, TMEM slot, abort flag
    static constexpr size_t uk = 1024;                      // [U; K] (128 rows, exact bf16)
    static constexpr size_t ah = uk + 2 * kTile;            // A hi, lo
    static constexpr size_t slots = ah + 2 * kTile;         // six 8 KB slots:
    // R1-R3: AK^T hi, W^T hi, Y_hat hi, AK^T lo, W^T lo, Y_hat lo
    // R4:    (beta Z)^T hi, E' hi, Z^T hi, (beta Z)^T lo, E' lo, Z^T lo
    // elimination: published pivot rows in slot 0 (sub-blocks) or slot 4, scaled
    // pivot rows in slot 3 (sub-blocks) or slot 5
    // chunk start: M^(c) (fp32, 64 x kGS) in slots 0-2, then (1/D) L^{-1} hi, lo in slots 0, 1
    static constexpr size_t xt = slots + 6 * kTile;         // I + G (fp32, 64 x kGS), then X^T hi, lo
    static constexpr size_t ksc = xt + (size_t)64 * kGS * 4;  // [2][64] 1 / max(|k|, eps) (by sub-block parity)
    static constexpr size_t kn = ksc + 512;                 // [2][64] max(|k|, eps)
    static constexpr size_t beta = kn + 512;                // [64]
    static constexpr size_t nrm = beta + 256;               // [2][64] halves of |row|^2
    static constexpr size_t total = nrm + 512;
};

__global__ void __launch_bounds__(kThreads, 2) gates_tc_kernel(ChunkArgs a) {
    using L = GtLayout;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::ctrl);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L::ctrl + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::ctrl + 12);
    unsigned char *uk = smem + L::uk;
    unsigned char *a_hi = smem + L::ah, *a_lo = smem + L::ah + kTile;
    unsigned char *slot = smem + L::slots;  // slot(i) = slot + i * kTile
    unsigned char *xt_hi = smem + L::xt, *xt_lo = smem + L::xt + kTile;
    float *gs = reinterpret_cast<float *>(smem + L::xt);
    float *stage = reinterpret_cast<float *>(slot);
    float *s_ks = reinterpret_cast<float *>(smem + L::ksc);
    float *s_kn = reinterpret_cast<float *>(smem + L::kn);
    float *s_beta = reinterpret_cast<float *>(smem + L::beta);
    float *s_nrm = reinterpret_cast<float *>(smem + L::nrm);
    // R1-R3 operands and R4 operands in the six slots
    unsigned char *akt_hi = slot, *wt_hi = slot + kTile, *yh_hi = slot + 2 * kTile;
    unsigned char *akt_lo = slot + 3 * kTile, *wt_lo = slot + 4 * kTile, *yh_lo = slot + 5 * kTile;
    unsigned char *bz_hi = slot, *ep_hi = slot + kTile, *zt_hi = slot + 2 * kTile;
    unsigned char *bz_lo = slot + 3 * kTile, *ep_lo = slot + 4 * kTile, *zt_lo = slot + 5 * kTile;

    const int NCA = a.L.NCA, CA = a.L.CA, T = a.p.T;
    const int c = (int)(blockIdx.x % (unsigned)NCA), bh = a.bh_lo + (int)(blockIdx.x / (unsigned)NCA);
    const int t0 = c * CA, ntok = min(CA, T - t0), nsb = (ntok + kSB - 1) / kSB;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int qw = warp & 3, hw = warp >> 2;  // TMEM lane quarter, column half
    const int pt = 8 * warp + (lane & 7), pq = lane >> 3;  // staging: token, feature quarter
    const int r64 = 16 * qw + lane;                         // row in an M = 64 accumulator (lanes < 16)
    const bool act64 = lane < 16;
    const int r128 = 32 * qw + lane;                        // row in an M = 128 accumulator
    const size_t tok0 = ((size_t)bh * T + t0) * kD;
    const __nv_bfloat16 *gu = static_cast<const __nv_bfloat16 *>(a.p.u) + tok0;
    const __nv_bfloat16 *gk = static_cast<const __nv_bfloat16 *>(a.p.k) + tok0;
    float *galpha = ws_f(a, a.L.off_alpha) + tok0;

    if (tid == 0) {
        mbar_init(bar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0) tmem_alloc(tslot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t tq = tbase + ((uint32_t)(32 * qw) << 16);  // this warp's lane quarter
    constexpr uint32_t col_d1 = 0, col_d5 = 64, col_d2 = 128;  // D2, then D3

    // ---- A at the chunk start ----
    // c > 0: A = (M^(c))^{-1} = L^{-T} D^{-1} L^{-1}: elimination of M^(c),
    // then one product E^T (diag(1/D) E) on the tensor cores.  c = 0: A0 or
    // I / lambda0 as given.  A stays in fp32 in the TMEM columns of D5 (rows
    // in the M = 64 lane layout) for the whole chunk: each sub-block's last
    // product accumulates onto it.
    {
        float am[32];  // A[r64][32 hw .. 32 hw + 31]
        const int gr = tid >> 2, gp = tid & 3;
        const float *src = nullptr;
        if (c > 0) src = ws_f(a, a.L.off_M) + ((size_t)bh * NCA + c) * kD * kD;
        else if (a.p.A0) src = a.p.A0 + (size_t)bh * kD * kD;
        if (c > 0) {
            const float4 *g4 = reinterpret_cast<const float4 *>(src + gr * kD + 16 * gp);
            float4 *st = reinterpret_cast<float4 *>(stage + gr * kGS + 16 * gp);
#pragma unroll
            for (int q = 0; q < 4; ++q) st[q] = g4[q];
            __syncthreads();
            eliminate64(stage, reinterpret_cast<float *>(slot + 4 * kTile), reinterpret_cast<float *>(slot + 5 * kTile),
                        s_beta, xt_hi, xt_lo, slot, slot + kTile);
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                mma_k64x3<true, true>(tbase + col_d5, smem_u32(slot), smem_u32(slot + kTile), smem_u32(xt_hi),
                                      smem_u32(xt_lo), idesc_bf16_f32(64, 64), false);
                umma_commit(bar);
            }
            const bool w = mbar_wait_bounded(bar, 0, a.p.wait_limit_ns, a.p.err);
            if (!w) *abort_flag = 1;
            __syncthreads();
            tc_fence_after();
            float v[32];
            tmem_ld32(tq + col_d5 + 32 * hw, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) am[j] = act64 ? v[j] : 0.f;
            tc_fence_before();
        } else {
            const float il = 1.f / a.p.lambda0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (act64 && src) v = reinterpret_cast<const float4 *>(src + (size_t)r64 * kD + 32 * hw)[q];
                am[4 * q] = v.x; am[4 * q + 1] = v.y; am[4 * q + 2] = v.z; am[4 * q + 3] = v.w;
            }
            if (!src && act64) {
#pragma unroll
                for (int j = 0; j < 32; ++j) am[j] = (32 * hw + j == r64) ? il : 0.f;
            }
            tmem_st32(tq + col_d5 + 32 * hw, am);
            tc_fence_before();
        }
        __syncthreads();
        if (act64) put_row32(a_hi, a_lo, r64, 32 * hw, am);
    }

    uint4 ru[2], rk[2];  // inputs of the next sub-block (token pt, features 16 pq ..)
    // (always a valid token row, clamped: no select waits on the loads here;
    // tokens past the chunk are zeroed where the values are used)
    auto load_in = [&](int sb) {
        const int t = min(sb * kSB + pt, ntok - 1);
        const size_t off = (size_t)t * kD + 16 * pq;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            ru[h] = reinterpret_cast<const uint4 *>(gu + off)[h];
            rk[h] = reinterpret_cast<const uint4 *>(gk + off)[h];
        }
    };
    uint32_t phase = (c > 0) ? 1u : 0u;  // the chunk-start product used phase 0
    auto round_wait = [&]() -> bool {
        const bool w = mbar_wait_bounded(bar, phase, a.p.wait_limit_ns, a.p.err);
        phase ^= 1u;
        if (!w) *abort_flag = 1;
        __syncthreads();
        tc_fence_after();
        return *abort_flag == 0;
    };

    // [U; K] of sub-block sb into its operand tile and its key norms into the
    // sb-parity half of s_kn, s_ks (the other half still serves sub-block sb - 1);
    // the tile is read by the tensor cores after a proxy fence and a barrier
    auto stage_in = [&](int sb) {
        const int nt = min(kSB, ntok - sb * kSB);
        if (pt >= nt) ru[0] = ru[1] = rk[0] = rk[1] = make_uint4(0, 0, 0, 0);  // past the chunk
        float kf[16];
        unpack8(rk[0], kf);
        unpack8(rk[1], kf + 8);
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) ss = fmaf(kf[m], kf[m], ss);
        ss += __shfl_xor_sync(0xffffffffu, ss, 8);
        ss += __shfl_xor_sync(0xffffffffu, ss, 16);
        const float kn = fmaxf(sqrtf(ss), kEps);
        if (pq == 0) {
            s_kn[64 * (sb & 1) + pt] = kn;
            s_ks[64 * (sb & 1) + pt] = 1.f / kn;
        }
        *reinterpret_cast<uint4 *>(uk + toff(pt, 16 * pq)) = ru[0];
        *reinterpret_cast<uint4 *>(uk + toff(pt, 16 * pq + 8)) = ru[1];
        *reinterpret_cast<uint4 *>(uk + toff(64 + pt, 16 * pq)) = rk[0];
        *reinterpret_cast<uint4 *>(uk + toff(64 + pt, 16 * pq + 8)) = rk[1];
        fence_proxy_async_smem();
    };

    bool ok = true;
    load_in(0);
    if (nsb > 0) stage_in(0);
    __syncthreads();
    for (int sb = 0; sb < nsb; ++sb) {
        const int nt = min(kSB, ntok - sb * kSB);
        const float *kn_sb = s_kn + 64 * (sb & 1), *ks_sb = s_ks + 64 * (sb & 1);
        // ---- R1: D1 = [U; K] A (M = 128) ----
        if (tid == 0) {
            tc_fence_after();
            mma_k64<false, false>(tbase + col_d1, smem_u32(uk), smem_u32(a_hi), idesc_bf16_f32(128, 64), false);
            mma_k64<false, false>(tbase + col_d1, smem_u32(uk), smem_u32(a_lo), idesc_bf16_f32(128, 64), true);
            umma_commit(bar);
        }
        if (!round_wait()) {
            ok = false;
            break;
        }
        // ---- W^T and (A K)^T tiles (token rows) ----
        {
            float v[32];
            tmem_ld32(tq + col_d1 + 32 * hw, v);
            if (qw < 2) put_row32(wt_hi, wt_lo, r128, 32 * hw, v);
            else put_row32(akt_hi, akt_lo, r128 - 64, 32 * hw, v);
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();
        // ---- R2: D2 = U [A K; W]^T (M = 64, N = 128): Y | G ----
        if (tid == 0) {
            tc_fence_after();
            mma_k64<false, false>(tbase + col_d2, smem_u32(uk), smem_u32(akt_hi), idesc_bf16_f32(64, 128), false);
            mma_k64<false, false>(tbase + col_d2, smem_u32(uk), smem_u32(akt_lo), idesc_bf16_f32(64, 128), true);
            umma_commit(bar);
        }
        if (!round_wait()) {
            ok = false;
            break;
        }
        // ---- Y_hat tiles (rows s), I + G (fp32) for the elimination ----
        {
            float v[32];
            tmem_ld32(tq + col_d2 + 32 * hw, v);  // Y[s][t], t = 32 hw ..
            if (act64) {
                const float4 *k4 = reinterpret_cast<const float4 *>(ks_sb + 32 * hw);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 kv = k4[q];
                    v[4 * q] *= kv.x; v[4 * q + 1] *= kv.y; v[4 * q + 2] *= kv.z; v[4 * q + 3] *= kv.w;
                }
                put_row32(yh_hi, yh_lo, r64, 32 * hw, v);
            }
            tmem_ld32(tq + col_d2 + 64 + 32 * hw, v);  // G[s][t]
            if (act64) {
#pragma unroll
                for (int m = 0; m < 32; ++m)
                    if (32 * hw + m == r64) v[m] += 1.f;
                float4 *dst = reinterpret_cast<float4 *>(gs + r64 * kGS + 32 * hw);
#pragma unroll
                for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
        }
        tc_fence_before();
        __syncthreads();
        // ---- elimination of I + G: X^T = L^{-1} and beta_s = 1 / D_s ----
        eliminate64(gs, reinterpret_cast<float *>(akt_hi), reinterpret_cast<float *>(akt_lo), s_beta, xt_hi, xt_lo,
                    nullptr, nullptr);
        fence_proxy_async_smem();
        __syncthreads();
        // ---- R3: D3 = X^T [W | Y_hat] (B MN-major, two atoms 8 KB apart): Z^T | P ----
        if (tid == 0) {
            tc_fence_after();
            mma_k64x3<false, true>(tbase + col_d2, smem_u32(xt_hi), smem_u32(xt_lo), smem_u32(wt_hi), smem_u32(wt_lo),
                                   idesc_bf16_f32(64, 128), false, 16, kTile);
            umma_commit(bar);
        }
        // the next sub-block's inputs: issued after the elimination, so that their
        // registers are not live through it (rounds 3-4 hide the latency)
        load_in(sb + 1);
        if (!round_wait()) {
            ok = false;
            break;
        }
        // ---- Z^T, -(beta Z)^T and E' tiles (rows s) ----
        {
            float v[32];
            tmem_ld32(tq + col_d2 + 32 * hw, v);  // z_s[i], i = 32 hw ..
            const float bs = act64 ? s_beta[r64] : 0.f;
            if (act64) {
                put_row32(zt_hi, zt_lo, r64, 32 * hw, v);
#pragma unroll
                for (int m = 0; m < 32; ++m) v[m] *= -bs;
                put_row32(bz_hi, bz_lo, r64, 32 * hw, v);
            }
            tmem_ld32(tq + col_d2 + 64 + 32 * hw, v);  // P[s][t] = z_s . k_hat_t, t = 32 hw ..
            if (act64) {
                const float4 *n4 = reinterpret_cast<const float4 *>(kn_sb + 32 * hw);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 kv = n4[q];
                    const float kk[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) {
                        const int mm = 4 * q + e4;
                        v[mm] = (32 * hw + mm >= r64) ? -bs * v[mm] * kk[e4] : 0.f;
                    }
                }
                put_row32(ep_hi, ep_lo, r64, 32 * hw, v);
            }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();
        // ---- R4: D1[k rows] += E'^T Z^T (A MN-major, atoms [-(beta Z)^T | E']: M = 128,
        // the first 64 rows land in D1's dead W rows); A += -(Z diag(beta)) Z^T ----
        if (tid == 0) {
            tc_fence_after();
            mma_k64x3<true, true>(tbase + col_d1, smem_u32(bz_hi), smem_u32(bz_lo), smem_u32(zt_hi), smem_u32(zt_lo),
                                  idesc_bf16_f32(128, 64), true, kTile, 16);
            mma_k64x3<true, true>(tbase + col_d5, smem_u32(bz_hi), smem_u32(bz_lo), smem_u32(zt_hi), smem_u32(zt_lo),
                                  idesc_bf16_f32(64, 64), true);
            umma_commit(bar);
        }
        // the next sub-block's [U; K] while round 4 runs ([U; K] was last read by
        // round 2; its loads were issued after round 3's issue)
        if (sb + 1 < nsb) stage_in(sb + 1);
        if (!round_wait()) {
            ok = false;
            break;
        }
        // ---- gates and the A update ----
        {
            float g[32];
            tmem_ld32(tq + col_d1 + 32 * hw, g);  // rows 64 + t: |k_t| A_t k_hat_t, columns 32 hw ..
            const int t = r128 - 64;
            if (qw >= 2) {
                float sq = 0.f;
#pragma unroll
                for (int m = 0; m < 32; ++m) sq = fmaf(g[m], g[m], sq);
                s_nrm[hw * 64 + t] = sq;
            }
            float v[32];
            tmem_ld32(tq + col_d5 + 32 * hw, v);  // the updated A[r64][32 hw ..]
            if (act64) put_row32(a_hi, a_lo, r64, 32 * hw, v);
            tc_fence_before();
            fence_proxy_async_smem();
            __syncthreads();
            if (qw >= 2 && t < nt) {
                // alpha = g / max(|g|, eps) with g = row / |k_t|
                const float nr = sqrtf(s_nrm[t] + s_nrm[64 + t]);
                const float sc = 1.f / fmaxf(nr, kEps * kn_sb[t]);
                float4 *dst = reinterpret_cast<float4 *>(galpha + (size_t)(sb * kSB + t) * kD + 32 * hw);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    dst[q] = make_float4(g[4 * q] * sc, g[4 * q + 1] * sc, g[4 * q + 2] * sc, g[4 * q + 3] * sc);
            }
        }
    }
    if (!ok) {
        if (tid == 0) (void)mbar_wait_bounded(bar, phase ^ 1u, a.p.wait_limit_ns, a.p.err);
    } else if (c == NCA - 1) {
        float am[32];
        tmem_ld32(tq + col_d5 + 32 * hw, am);
        if (act64) {
            float4 *dA = reinterpret_cast<float4 *>(a.p.A_T + (size_t)bh * kD * kD + (size_t)r64 * kD + 32 * hw);
#pragma unroll
            for (int q = 0; q < 8; ++q) dA[q] = make_float4(am[4 * q], am[4 * q + 1], am[4 * q + 2], am[4 * q + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 256);
}

}  // namespace

bool gates_tc_supported(const FwdParams &p, const ChunkLayout &L) {
    return p.d == kD && p.io_bf16 && L.CA % kSB == 0 && L.yh;
}

cudaError_t launch_gates_tc(const ChunkArgs &a, cudaStream_t stream) {
    constexpr size_t bytes = GtLayout::total + 1024;  // + alignment slack
    cudaError_t e = cudaFuncSetAttribute(gates_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    const long long grid = (long long)a.L.NCA * (a.bh_n > 0 ? a.bh_n : a.p.BH);
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    gates_tc_kernel<<<(unsigned)grid, kThreads, bytes, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace vla
