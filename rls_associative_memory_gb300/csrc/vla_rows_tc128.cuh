// vla_rows_tc128.cuh -- the state write and ELU+1 readout of "Variational
// Linear Attention: Stable Associative Memory for Long-Context Transformers"
// (section 2.3, step 3 and the readout) on the tensor cores for d = 128 with
// bf16 I/O, when every (b, h) unit is one chunk: one CTA runs a unit's state
// S (128 rows, fp32 in TMEM) through its whole stream, 64 tokens at a time in
// the UT (WY) form of a product of rank-1 updates, and writes o directly.
//
// Within a sub-block of c = 64 tokens with state X = S at its start (the
// identities of the d = 64 state pass, vla_chunk_tc.cu, with X the state
// itself and the values v):
//   R (I + N) = V - X K_hat,       N = strictly-upper(Al^T K_hat)  (c x c)
//   X_end     = X + R Al^T
//   X_t phi(q_t) = X phi(q_t) + sum_{s <= t} r_s (alpha_s . phi(q_t))
// and o_t = X_t phi(q_t) / (phi(q_t) . n_t + eps).  Per sub-block:
//   1. N^T = K Al^T (own barrier), then [DO^T | D1] = X [Phi; K]^T;
//      T_inv = (I + N)^{-1} on the CUDA cores while the wide product runs
//   2. R = E T_inv (E = V - (X K) diag(1/|k|)),  Qm = Al Phi^T
//   3. [X | DO^T] += R [Al | Qm]   (M = 128, N = 192: three 64-wide atoms)
//   o_t = column t of DO^T / den_t, staged as [t][i] and written by one bulk
//   copy per sub-block.
// Products over the features (K = 128) run as two K = 64 halves.  fp32
// operands are bf16 hi/lo pairs (hi*hi + hi*lo + lo*hi); k, v, q are exact
// bf16.  TMEM 320 columns (512 allocated), ~212 KB of shared memory: one CTA
// per SM.
// The body of one CTA's work for one unit, included by vla_tc128.cu.
#pragma once

#include "vla_tc_common.cuh"

namespace vla {
namespace r128 {

using namespace tc;

constexpr int kD2 = 128;
constexpr int kThreads = 256;
constexpr int kVS2 = 136;  // row stride (bf16) of the v tile

struct R2Layout {
    static constexpr size_t ctrl = 0;                      // mbarriers, TMEM slot, abort flag
    static constexpr size_t xs = 1024;                     // X: hi f0, hi f1, lo f0, lo f1 (128 rows each);
                                                           // E, then R: hi @xs, lo @xs + 2 kTile
    static constexpr size_t phk = xs + 8 * kTile;          // [Phi_hi; K] f0, then f1 (128 rows each)
    static constexpr size_t phl = phk + 4 * kTile;         // Phi_lo f0, f1 (64 rows each)
    static constexpr size_t alq = phl + 2 * kTile;         // Al hi f0 @0, lo f0 @8K, hi f1 @16K, lo f1 @24K,
                                                           // Qm hi @32K, lo @40K: round 3's B operand is
                                                           // three atoms 16 KB apart
    static constexpr uint32_t kAtom3 = 2 * kTile;
    static constexpr size_t ti = alq + 6 * kTile;          // N fp32 (row stride kGS), then T_inv hi, lo
    static constexpr size_t vt = ti + (size_t)64 * kGS * 4;  // v [t][i] bf16
    static constexpr size_t ost = vt + (size_t)64 * kVS2 * 2;  // o [t][i] bf16 (64 x 128), bulk-copied out
    static constexpr size_t ks = ost + (size_t)64 * kD2 * 2;   // [64] 1 / max(|k|, eps)
    static constexpr size_t rden = ks + 256;               // [64] 1 / (phi(q).n + eps)
    static constexpr size_t tot = rden + 256;              // [8][128] warp totals of phi(k_hat), then prefixes
    static constexpr size_t nrun = tot + 8 * kD2 * 4;      // [128] n at the sub-block start
    static constexpr size_t tms = nrun + kD2 * 4;          // triangular-inverse scratch (32 x 36 floats)
    static constexpr size_t total = tms + 32 * 36 * 4;
};
static_assert(R2Layout::phk % 1024 == 0 && R2Layout::alq % 1024 == 0 && R2Layout::ti % 1024 == 0,
              "operand tiles must be 1024-byte aligned");
static_assert(R2Layout::ost % 16 == 0, "bulk-copy source is 16-byte aligned");
static_assert(R2Layout::total + 1024 <= 227 * 1024, "one CTA per SM");

__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// The state pass of unit bh, by one CTA of kThreads threads with
// R2Layout::total + 1024 bytes of dynamic shared memory at smem_raw.
__device__ __forceinline__ void rows_tc128_body(const ChunkArgs &a, int bh, unsigned char *smem_raw) {
    using L = R2Layout;
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::ctrl);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L::ctrl + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::ctrl + 12);
    uint64_t *bar_n = reinterpret_cast<uint64_t *>(smem + L::ctrl + 16);
    unsigned char *xs = smem + L::xs, *phk = smem + L::phk, *phl = smem + L::phl, *alq = smem + L::alq;
    float *ntb = reinterpret_cast<float *>(smem + L::ti);
    unsigned char *ti_hi = smem + L::ti, *ti_lo = smem + L::ti + kTile;
    __nv_bfloat16 *vt = reinterpret_cast<__nv_bfloat16 *>(smem + L::vt);
    __nv_bfloat16 *ost = reinterpret_cast<__nv_bfloat16 *>(smem + L::ost);
    float *s_ks = reinterpret_cast<float *>(smem + L::ks);
    float *s_rden = reinterpret_cast<float *>(smem + L::rden);
    float *s_tot = reinterpret_cast<float *>(smem + L::tot);
    float *s_nrun = reinterpret_cast<float *>(smem + L::nrun);
    unsigned char *qm_hi = alq + 4 * kTile, *qm_lo = alq + 5 * kTile;

    const int T = a.p.T;
    const int nsb = (T + kSB - 1) / kSB;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int qw = warp & 3, hw = warp >> 2;                // TMEM lane quarter, column half
    const int pt = 8 * warp + (lane & 7), pq = lane >> 3;  // staging: token, feature quarter (32 features)
    const int kh = pq >> 1, kc = 32 * (pq & 1);            // staging: feature half, column in the tile
    const int xrow = 32 * qw + lane;                        // state row (value coordinate)
    const size_t tok0 = (size_t)bh * T * kD2;
    const __nv_bfloat16 *gk = static_cast<const __nv_bfloat16 *>(a.p.k) + tok0;
    const __nv_bfloat16 *gv = static_cast<const __nv_bfloat16 *>(a.p.v) + tok0;
    const __nv_bfloat16 *gq = static_cast<const __nv_bfloat16 *>(a.p.q) + tok0;
    __nv_bfloat16 *go = static_cast<__nv_bfloat16 *>(a.p.o) + tok0;
    const __half *gal = reinterpret_cast<const __half *>(static_cast<const unsigned char *>(a.p.ws) + a.L.off_alpha) + tok0;

    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar_n, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (tid < kD2) s_nrun[tid] = a.p.n0 ? a.p.n0[(size_t)bh * kD2 + tid] : 0.f;
    if (warp == 0) tmem_alloc(tslot, 512, false);  // (one CTA per SM; a queue CTA allocates per job)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t tq = tbase + ((uint32_t)(32 * qw) << 16);
    constexpr uint32_t col_x = 0;     // X (fp32 state, 128 columns)
    constexpr uint32_t col_do = 128;  // DO^T (state rows x tokens), right after X
    constexpr uint32_t col_d1 = 192;  // D1 = X K^T, then R
    constexpr uint32_t col_d2 = 256;  // D2 = N^T, then Qm (M = 64)

    // ---- the state S0 (or 0) into TMEM and, as hi/lo tiles, the first round's operand ----
    {
        const float *src = a.p.S0 ? a.p.S0 + (size_t)bh * kD2 * kD2 + (size_t)xrow * kD2 : nullptr;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int c0 = 64 * hw + 32 * half;
            float x[32];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 v = src ? reinterpret_cast<const float4 *>(src + c0)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
                x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
            }
            tmem_st32(tq + col_x + c0, x);
            put_row32(xs + 2 * kTile * hw, xs + 4 * kTile + 2 * kTile * hw, xrow, 32 * half, x);
        }
        tc_fence_before();
    }

    uint4 rk[4], rv[4], rq[4], ra[4];
    auto load_in = [&](int sb) {
        const int t = min(sb * kSB + pt, T - 1);
        const size_t off = (size_t)t * kD2 + 32 * pq;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            rk[h] = reinterpret_cast<const uint4 *>(gk + off)[h];
            rv[h] = reinterpret_cast<const uint4 *>(gv + off)[h];
            rq[h] = reinterpret_cast<const uint4 *>(gq + off)[h];
        }
#pragma unroll
        for (int h = 0; h < 4; ++h) ra[h] = reinterpret_cast<const uint4 *>(gal + off)[h];
    };

    // phase: next parity of bar (three commits per sub-block), phase_n of bar_n
    // (one); pend: after an abort, the parity of bar's last commit
    uint32_t phase = 0, phase_n = 0, pend = 0;
    auto round_wait = [&]() -> bool {
        const bool w = mbar_wait_bounded(bar, phase, a.p.wait_limit_ns, a.p.err);
        pend = phase;
        phase ^= 1u;
        if (!w) *abort_flag = 1;
        __syncthreads();
        tc_fence_after();
        return *abort_flag == 0;
    };
    constexpr uint32_t id_big = idesc_bf16_f32(128, 128);
    constexpr uint32_t id_x64 = idesc_bf16_f32(128, 64);
    constexpr uint32_t id_64 = idesc_bf16_f32(64, 64);
    constexpr uint32_t id_r3 = idesc_bf16_f32(128, 192);

    bool ok = true;
    load_in(0);
    for (int sb = 0; sb < nsb; ++sb) {
        const int nt = min(kSB, T - sb * kSB);
        float fq[32];
        // ---- stage the sub-block's operands ----
        if (pt >= nt) {
#pragma unroll
            for (int h = 0; h < 4; ++h) rk[h] = rv[h] = rq[h] = ra[h] = make_uint4(0, 0, 0, 0);
        }
        {
            float ss = 0.f;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float kf[8];
                unpack8(rk[h], kf);
#pragma unroll
                for (int m = 0; m < 8; ++m) ss = fmaf(kf[m], kf[m], ss);
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 8);
            ss += __shfl_xor_sync(0xffffffffu, ss, 16);
            if (pq == 0) s_ks[pt] = 1.f / fmaxf(sqrtf(ss), kEps);
            unsigned char *pk = phk + 2 * kTile * kh;
            unsigned char *pl = phl + kTile * kh;
            unsigned char *ah_ = alq + 2 * kTile * kh, *al_ = ah_ + kTile;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                *reinterpret_cast<uint4 *>(pk + toff(64 + pt, kc + 8 * h)) = rk[h];
                *reinterpret_cast<uint4 *>(vt + pt * kVS2 + 32 * pq + 8 * h) = rv[h];
                float af[8];
                unpack8_h(ra[h], af);
                uint4 h4, l4;
                split8(af, h4, l4);
                *reinterpret_cast<uint4 *>(ah_ + toff(pt, kc + 8 * h)) = h4;
                *reinterpret_cast<uint4 *>(al_ + toff(pt, kc + 8 * h)) = l4;
                float qf[8];
                unpack8(rq[h], qf);
#pragma unroll
                for (int m = 0; m < 8; ++m) fq[8 * h + m] = phi_fast(qf[m]);
                split8(fq + 8 * h, h4, l4);
                *reinterpret_cast<uint4 *>(pk + toff(pt, kc + 8 * h)) = h4;
                *reinterpret_cast<uint4 *>(pl + toff(pt, kc + 8 * h)) = l4;
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        // ---- round 1: N^T = K Al^T (own barrier), then [DO^T | D1] = X [Phi; K]^T ----
        if (tid == 0) {
            tc_fence_after();
            // K rows are rows 64..127 of the [Phi_hi; K] tiles (8 KB in)
            mma_k64<false, false>(tbase + col_d2, smem_u32(phk + kTile), smem_u32(alq), id_64, false);
            mma_k64<false, false>(tbase + col_d2, smem_u32(phk + 3 * kTile), smem_u32(alq + 2 * kTile), id_64, true);
            mma_k64<false, false>(tbase + col_d2, smem_u32(phk + kTile), smem_u32(alq + kTile), id_64, true);
            mma_k64<false, false>(tbase + col_d2, smem_u32(phk + 3 * kTile), smem_u32(alq + 3 * kTile), id_64, true);
            umma_commit(bar_n);
            // hi.hi and lo.hi for [Phi; K] (K exact), then hi.lo for the Phi part
            mma_k64<false, false>(tbase + col_do, smem_u32(xs), smem_u32(phk), id_big, false);
            mma_k64<false, false>(tbase + col_do, smem_u32(xs + 2 * kTile), smem_u32(phk + 2 * kTile), id_big, true);
            mma_k64<false, false>(tbase + col_do, smem_u32(xs + 4 * kTile), smem_u32(phk), id_big, true);
            mma_k64<false, false>(tbase + col_do, smem_u32(xs + 6 * kTile), smem_u32(phk + 2 * kTile), id_big, true);
            mma_k64<false, false>(tbase + col_do, smem_u32(xs), smem_u32(phl), id_x64, true);
            mma_k64<false, false>(tbase + col_do, smem_u32(xs + 2 * kTile), smem_u32(phl + kTile), id_x64, true);
            umma_commit(bar);
        }
        // ---- readout denominators 1 / (phi(q_t) . n_t + eps), while round 1 runs ----
        float fk[32];
        {
            const float ksc = s_ks[pt];
            const unsigned char *pk = phk + 2 * kTile * kh;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float kf[8];
                unpack8(*reinterpret_cast<const uint4 *>(pk + toff(64 + pt, kc + 8 * h)), kf);
#pragma unroll
                for (int m = 0; m < 8; ++m) fk[8 * h + m] = pt < nt ? phi_fast(kf[m] * ksc) : 0.f;
            }
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) {
#pragma unroll
                for (int m = 0; m < 32; ++m) {
                    const float y = __shfl_up_sync(0xffffffffu, fk[m], off);
                    if ((lane & 7) >= off) fk[m] += y;
                }
            }
            if ((lane & 7) == 7) {
                float4 *dst = reinterpret_cast<float4 *>(s_tot + warp * kD2 + 32 * pq);
#pragma unroll
                for (int h = 0; h < 8; ++h) dst[h] = make_float4(fk[4 * h], fk[4 * h + 1], fk[4 * h + 2], fk[4 * h + 3]);
            }
        }
        __syncthreads();
        if (tid < kD2) {  // per feature: n before each warp's tokens, and n after the sub-block
            float run = s_nrun[tid];
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const float y = s_tot[w * kD2 + tid];
                s_tot[w * kD2 + tid] = run;
                run += y;
            }
            s_nrun[tid] = run;
        }
        __syncthreads();
        {
            const float4 *pw = reinterpret_cast<const float4 *>(s_tot + warp * kD2 + 32 * pq);
            float dp = 0.f;
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const float4 p4 = pw[h];
                const float pv[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) dp = fmaf(fq[4 * h + e], pv[e] + fk[4 * h + e], dp);
            }
            dp += __shfl_xor_sync(0xffffffffu, dp, 8);
            dp += __shfl_xor_sync(0xffffffffu, dp, 16);
            if (pq == 0) s_rden[pt] = 1.f / (dp + kEps);
        }
        {
            const bool w = mbar_wait_bounded(bar_n, phase_n, a.p.wait_limit_ns, a.p.err);
            phase_n ^= 1u;
            if (!w) *abort_flag = 1;
            __syncthreads();
            tc_fence_after();
            if (*abort_flag) {
                pend = phase;  // the wide product's commit is still outstanding
                ok = false;
                break;
            }
        }
        // ---- N (fp32, row-major, for the inverse) ----
        {
            float v[32];
            tmem_ld32(tq + col_d2 + 32 * hw, v);  // D2 row t = 16 qw + lane (M = 64), columns s = 32 hw ..
            if (lane < 16) {
                const int t = 16 * qw + lane;
                const float kt = s_ks[t];
#pragma unroll
                for (int m = 0; m < 32; ++m) {
                    const int sr = 32 * hw + m;
                    ntb[sr * kGS + t] = sr < t ? v[m] * kt : 0.f;
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        // ---- T_inv = (I + N)^{-1}, while the wide product of round 1 runs ----
        tri_inv64(ntb, reinterpret_cast<float *>(smem + L::tms), ti_hi, ti_lo);
        if (!round_wait()) {
            ok = false;
            break;
        }
        // ---- E = V - X K_hat: tiles over X (round 1 has read it) ----
        {
            float v[32];
            tmem_ld32(tq + col_d1 + 32 * hw, v);  // X K, tokens 32 hw ..
            const float4 *ks4 = reinterpret_cast<const float4 *>(s_ks + 32 * hw);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 k4 = ks4[q];
                const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = 4 * q + e, t = 32 * hw + m;
                    v[m] = fmaf(-v[m], kv[e], __bfloat162float(vt[t * kVS2 + xrow]));
                }
            }
            put_row32(xs, xs + 2 * kTile, xrow, 32 * hw, v);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- round 2: R = E T_inv, Qm = Al Phi^T ----
        if (tid == 0) {
            tc_fence_after();
            mma_k64x3<false, true>(tbase + col_d1, smem_u32(xs), smem_u32(xs + 2 * kTile), smem_u32(ti_hi),
                                   smem_u32(ti_lo), id_x64, false);
            mma_k64x3<false, false>(tbase + col_d2, smem_u32(alq), smem_u32(alq + kTile), smem_u32(phk),
                                    smem_u32(phl), id_64, false);
            mma_k64x3<false, false>(tbase + col_d2, smem_u32(alq + 2 * kTile), smem_u32(alq + 3 * kTile),
                                    smem_u32(phk + 2 * kTile), smem_u32(phl + kTile), id_64, true);
            umma_commit(bar);
        }
        load_in(sb + 1);
        if (!round_wait()) {
            ok = false;
            break;
        }
        // ---- R tiles (over E); Qm tiles ----
        {
            float v[32];
            tmem_ld32(tq + col_d1 + 32 * hw, v);
            put_row32(xs, xs + 2 * kTile, xrow, 32 * hw, v);
            tmem_ld32(tq + col_d2 + 32 * hw, v);  // Qm row s = 16 qw + lane, columns t = 32 hw ..
            if (lane < 16) {
                const int srow = 16 * qw + lane;
#pragma unroll
                for (int m = 0; m < 32; ++m)
                    if (32 * hw + m < srow) v[m] = 0.f;
                put_row32(qm_hi, qm_lo, srow, 32 * hw, v);
            }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();
        // ---- round 3: [X | DO^T] += R [Al f0 | Al f1 | Qm] (B MN-major, atoms 16 KB apart) ----
        if (tid == 0) {
            tc_fence_after();
            mma_k64x3<false, true>(tbase + col_x, smem_u32(xs), smem_u32(xs + 2 * kTile), smem_u32(alq),
                                   smem_u32(alq + kTile), id_r3, true, 16, L::kAtom3);
            umma_commit(bar);
            bulk_wait_read();  // the previous sub-block's o copy has read the staging
        }
        if (!round_wait()) {
            ok = false;
            break;
        }
        {
            // the new X: next round 1's operand (features 64 hw ..)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float v[32];
                tmem_ld32(tq + col_x + 64 * hw + 32 * half, v);
                put_row32(xs + 2 * kTile * hw, xs + 4 * kTile + 2 * kTile * hw, xrow, 32 * half, v);
            }
            // o_t[xrow] for tokens 32 hw ..: DO^T / den_t, staged as [t][i]
            float v[32];
            tmem_ld32(tq + col_do + 32 * hw, v);
#pragma unroll
            for (int m = 0; m < 32; ++m) {
                const int t = 32 * hw + m;
                ost[t * kD2 + xrow] = __float2bfloat16_rn(v[m] * s_rden[t]);
            }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) bulk_s2g(go + (size_t)sb * kSB * kD2, ost, (uint32_t)nt * kD2 * 2);
    }
    if (tid == 0) bulk_wait_all();
    if (!ok) {
        if (tid == 0) (void)mbar_wait_bounded(bar, pend, a.p.wait_limit_ns, a.p.err);
    } else {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float x[32];
            tmem_ld32(tq + col_x + 64 * hw + 32 * half, x);
            float4 *dst = reinterpret_cast<float4 *>(a.p.S_T + (size_t)bh * kD2 * kD2 + (size_t)xrow * kD2 + 64 * hw +
                                                     32 * half);
#pragma unroll
            for (int q = 0; q < 8; ++q) dst[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
        }
        if (a.p.n_T && tid < kD2) a.p.n_T[(size_t)bh * kD2 + tid] = s_nrun[tid];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
    if (tid == 0) {  // (a later job of this CTA may lay out its memory otherwise)
        mbar_inval(bar);
        mbar_inval(bar_n);
    }
}

}  // namespace r128
}  // namespace vla
