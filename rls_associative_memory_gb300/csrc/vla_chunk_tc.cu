// vla_chunk_tc.cu -- tensor-core state passes of the chunk-parallel path for
// d = 64 with bf16 I/O: the chunk transitions (mode 0) and the readout
// (mode 1) of the state write and ELU+1 readout of "Variational Linear
// Attention: Stable Associative Memory for Long-Context Transformers",
// section 2.3 (step 3 and the readout), taken 64 tokens at a time in the UT
// (WY) form of a product of rank-1 updates.
//
// Within a sub-block of c = 64 tokens whose state at the start is X, the
// state write x <- x + (value - x.k_hat) alpha^T, applied token by token,
// is equivalent to
//   R (I + N) = Vals - X K_hat,        N = strictly-upper(Al^T K_hat)  (c x c)
//   X_end     = X + R Al^T
//   X_t phi(q_t) = X phi(q_t) + sum_{s <= t} r_s (alpha_s . phi(q_t))
// where R = [r_1 .. r_c] holds the per-token residuals value_t - X_{t-1} k_hat_t
// (the residual of token t is its value minus what the earlier tokens of
// the sub-block left in the state, hence the triangular system).  A
// sub-block is three rounds of tcgen05.mma plus one triangular inverse on
// the CUDA cores:
//   1. D1 = X K^T;  mode 0: D2 = K Al^T (= N^T);  mode 1: D2 = Phi Al^T
//      (= Qm^T, Qm = upper-incl(Al^T Phi)) and DO = Phi X^T
//   2. R  = E T_inv,   E = Vals - (X K) diag(1/|k|),  T_inv = (I + N)^{-1}
//   3. X += R Al^T    and (mode 1)  DO += Qm^T R^T
// T_inv depends on the keys and gates only: mode 0 computes it and stores
// it (bf16 hi/lo operand tiles) in the workspace, and mode 1 loads it with a
// bulk copy.  DO holds the readout numerators token-major (rows = tokens),
// so o leaves as whole 16-byte vectors.
//
// Mode 0 runs the rows [H; P] of the chunk map S_end = S_start P_c + H_c
// (values [v; 0], start [0; I]: M = 128); mode 1 runs S itself from the
// chunk-start state of the chain pass and writes o (M = 64).
//
// Precision: fp32 operands enter the tensor cores as bf16 pairs
// x = hi + lo (hi = bf16(x), lo = bf16(x - hi)), and a product takes
// hi*hi + hi*lo + lo*hi with fp32 accumulation (relative error about
// 2^-16).  k and v are bf16 inputs and exact: the raw key enters once and
// the key norm is applied as a column scale in fp32.
#include "vla_tc_common.cuh"

namespace vla {
namespace {

using namespace tc;

constexpr int kThreads = 256;

template <int MODE>
struct TcLayout {
    static constexpr int XR = MODE == 0 ? 128 : 64;            // state rows
    static constexpr uint32_t ncols = MODE == 0 ? 128 : 256;    // TMEM columns
    static constexpr size_t ctrl = 0;                            // mbarriers (MMA, T_inv load), TMEM slot, abort flag
    // X / E / R tiles (hi, lo) and the gate tiles Al (token rows; hi, lo).  In
    // mode 1 they interleave as [X hi | Al hi | X lo | Al lo], so that [X; Al]
    // is one 128-row operand (Phi [X; Al]^T in one product).
    static constexpr size_t xs_hi = 1024;
    static constexpr size_t xs_lo = MODE == 0 ? xs_hi + 2 * kTile : xs_hi + 2 * kTile;
    static constexpr size_t al_hi = MODE == 0 ? xs_hi + 4 * kTile : xs_hi + kTile;
    static constexpr size_t al_lo = MODE == 0 ? al_hi + kTile : xs_hi + 3 * kTile;
    static constexpr size_t kb = xs_hi + 4 * kTile + (MODE == 0 ? 2 * kTile : 0);  // [K; Phi_hi] (mode 1) or K; then Qm^T hi, lo
    static constexpr size_t kblo = kb + (MODE == 0 ? kTile : 2 * kTile);  // Phi_lo (mode 1)
    static constexpr size_t ti = kblo + (MODE == 0 ? 0 : kTile); // (mode 0) N fp32 (row stride kGS); T_inv hi, lo
    static constexpr int kVS = 72;                               // row stride (bf16) of the v tile
    static constexpr size_t vt = ti + (MODE == 0 ? (size_t)64 * kGS * 4 : 2 * (size_t)kTile);  // v [t][i] bf16
    static constexpr size_t ks = vt + (size_t)64 * kVS * 2;      // [64] 1 / max(|k|, eps)
    static constexpr size_t rden = ks + 256;                     // [64] 1 / (phi(q).n + eps)
    static constexpr size_t tot = rden + 256;                    // [9][64] warp totals of phi(k_hat), then prefixes
    static constexpr size_t total = tot + 9 * 64 * 4;
};

template <int MODE>
__global__ void __launch_bounds__(kThreads, 2) rows_tc_kernel(ChunkArgs a) {
    using L = TcLayout<MODE>;
    constexpr int XR = L::XR;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // swizzled tiles need 1024-byte aligned addresses (one extra KB is allocated)
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::ctrl);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L::ctrl + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::ctrl + 12);
    uint64_t *bar_t = reinterpret_cast<uint64_t *>(smem + L::ctrl + 16);  // T_inv load (mode 1)
    unsigned char *xs_hi = smem + L::xs_hi, *xs_lo = smem + L::xs_lo;
    unsigned char *kb = smem + L::kb, *kblo = smem + L::kblo;
    unsigned char *al_hi = smem + L::al_hi, *al_lo = smem + L::al_lo;
    float *ntb = reinterpret_cast<float *>(smem + L::ti);  // N (mode 0), row stride kGS
    unsigned char *ti_hi = smem + L::ti, *ti_lo = smem + L::ti + kTile;  // T_inv, tile row s = row s
    __nv_bfloat16 *vt = reinterpret_cast<__nv_bfloat16 *>(smem + L::vt);
    float *s_ks = reinterpret_cast<float *>(smem + L::ks);
    float *s_rden = reinterpret_cast<float *>(smem + L::rden);
    float *s_tot = reinterpret_cast<float *>(smem + L::tot);

    const int NC = a.L.NC, C = a.L.C, T = a.p.T;
    const int c = (int)(blockIdx.x % (unsigned)NC), bh = (int)(blockIdx.x / (unsigned)NC);
    const int t0 = c * C, ntok = min(C, T - t0), nsb = (ntok + kSB - 1) / kSB;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int qw = warp & 3, hw = warp >> 2;  // TMEM lane quarter, column half
    // operand staging: token pt (8 consecutive tokens in the 8 lanes of a
    // quarter-warp), features 16 pq .. 16 pq + 15
    const int pt = 8 * warp + (lane & 7), pq = lane >> 3;
    const size_t tok0 = ((size_t)bh * T + t0) * kD;
    const __nv_bfloat16 *gk = static_cast<const __nv_bfloat16 *>(a.p.k) + tok0;
    const __nv_bfloat16 *gv = static_cast<const __nv_bfloat16 *>(a.p.v) + tok0;
    const __nv_bfloat16 *gq = static_cast<const __nv_bfloat16 *>(a.p.q) + tok0;
    const float *gal = ws_f(a, a.L.off_alpha) + tok0;
    __nv_bfloat16 *gout = static_cast<__nv_bfloat16 *>(a.p.o) + tok0;

    unsigned char *gtinv = static_cast<unsigned char *>(a.p.ws) + a.L.off_tinv +
                           (size_t)(bh * NC + c) * (C / kSB) * (2 * kTile);  // this chunk's T_inv tiles
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar_t, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0) tmem_alloc(tslot, L::ncols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t tq = tbase + ((uint32_t)(32 * qw) << 16);  // this warp's lane quarter

    // State rows held in registers: the row and 32 columns this thread reads
    // back from TMEM (M = 128: row 32 qw + lane; M = 64: row 16 qw + lane,
    // lanes 0..15 of each quarter).
    const int xrow = MODE == 0 ? 32 * qw + lane : 16 * qw + lane;
    const bool xact = MODE == 0 || lane < 16;
    float x[32];
    if (MODE == 0) {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = (xrow - 64 == 32 * hw + j) ? 1.f : 0.f;
    } else {
        const float4 *src = reinterpret_cast<const float4 *>(ws_f(a, a.L.off_S) + ((size_t)bh * NC + c) * kD * kD +
                                                             (size_t)(xrow & 63) * kD + 32 * hw);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 v = xact ? src[q] : make_float4(0.f, 0.f, 0.f, 0.f);
            x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
        }
    }
    if (xact) put_row32(xs_hi, xs_lo, xrow, 32 * hw, x);

    // Inputs of the next sub-block, prefetched into registers (token pt,
    // features 16 pq .. 16 pq + 15).
    uint4 rk[2], rv[2], rq[2];
    float4 ra[4];
    // (always a valid token row, clamped: no select waits on the loads here;
    // tokens past the chunk are zeroed where the values are used)
    auto load_in = [&](int sb) {
        const int t = min(sb * kSB + pt, ntok - 1);
        const size_t off = (size_t)t * kD + 16 * pq;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            rk[h] = reinterpret_cast<const uint4 *>(gk + off)[h];
            rv[h] = reinterpret_cast<const uint4 *>(gv + off)[h];
            if (MODE == 1) rq[h] = reinterpret_cast<const uint4 *>(gq + off)[h];
        }
#pragma unroll
        for (int h = 0; h < 4; ++h) ra[h] = reinterpret_cast<const float4 *>(gal + off)[h];
    };
    float nb[16];  // n at the sub-block start, features 16 pq .. (mode 1)
    if (MODE == 1) {
        const float *n0 = ws_f(a, a.L.off_n) + ((size_t)bh * (a.L.NCA + 1) + (size_t)c * (C / a.L.CA)) * kD + 16 * pq;
#pragma unroll
        for (int m = 0; m < 16; ++m) nb[m] = n0[m];
    }

    uint32_t phase = 0;
    auto round_wait = [&]() -> bool {
        const bool w = mbar_wait_bounded(bar, phase, a.p.wait_limit_ns, a.p.err);
        phase ^= 1u;
        if (!w) *abort_flag = 1;
        __syncthreads();
        tc_fence_after();
        return *abort_flag == 0;
    };
    constexpr uint32_t id_x64 = idesc_bf16_f32(XR, 64);                       // X-row products
    constexpr uint32_t id_64 = idesc_bf16_f32(64, 64);
    constexpr int kVS = L::kVS;
    constexpr uint32_t col_d2 = MODE == 1 ? 128 : 64;   // D2, then D3 = R
    constexpr uint32_t col_d4 = 0;                      // D1 = X K^T, then D4 = R Al^T
    constexpr uint32_t col_do = 64;                     // (mode 1) readout numerators, token rows

    bool ok = true;
    int tinv_issued = 0, tinv_done = 0;  // T_inv loads (mode 1)
    load_in(0);
    for (int sb = 0; sb < nsb; ++sb) {
        const int nt = min(kSB, ntok - sb * kSB);
        float fq[16], fk[16];
        if (MODE == 1 && tid == 0) {  // T_inv of this sub-block (the slot is free: round 2 is done)
            mbar_arrive_expect_tx(bar_t, 2 * kTile);
            bulk_g2s(ti_hi, gtinv + (size_t)sb * 2 * kTile, 2 * kTile, bar_t);
        }
        tinv_issued = sb + 1;
        // ---- stage the sub-block's operands ----
        if (pt >= nt) {  // past the chunk: zero inputs
            rk[0] = rk[1] = rv[0] = rv[1] = rq[0] = rq[1] = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int h = 0; h < 4; ++h) ra[h] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        {
            float kf[16];
            unpack8(rk[0], kf);
            unpack8(rk[1], kf + 8);
            float ss = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) ss = fmaf(kf[m], kf[m], ss);
            ss += __shfl_xor_sync(0xffffffffu, ss, 8);
            ss += __shfl_xor_sync(0xffffffffu, ss, 16);
            const float ksc = 1.f / fmaxf(sqrtf(ss), kEps);
            if (pq == 0) s_ks[pt] = ksc;
            *reinterpret_cast<uint4 *>(kb + toff(pt, 16 * pq)) = rk[0];
            *reinterpret_cast<uint4 *>(kb + toff(pt, 16 * pq + 8)) = rk[1];
            *reinterpret_cast<uint4 *>(vt + pt * kVS + 16 * pq) = rv[0];
            *reinterpret_cast<uint4 *>(vt + pt * kVS + 16 * pq + 8) = rv[1];
            float af[16];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                af[4 * h] = ra[h].x; af[4 * h + 1] = ra[h].y; af[4 * h + 2] = ra[h].z; af[4 * h + 3] = ra[h].w;
            }
            uint4 h4, l4;
            split8(af, h4, l4);
            *reinterpret_cast<uint4 *>(al_hi + toff(pt, 16 * pq)) = h4;
            *reinterpret_cast<uint4 *>(al_lo + toff(pt, 16 * pq)) = l4;
            split8(af + 8, h4, l4);
            *reinterpret_cast<uint4 *>(al_hi + toff(pt, 16 * pq + 8)) = h4;
            *reinterpret_cast<uint4 *>(al_lo + toff(pt, 16 * pq + 8)) = l4;
            if (MODE == 1) {
                float qf[16];
                unpack8(rq[0], qf);
                unpack8(rq[1], qf + 8);
#pragma unroll
                for (int m = 0; m < 16; ++m) fq[m] = phi_fast(qf[m]);
                split8(fq, h4, l4);
                *reinterpret_cast<uint4 *>(kb + toff(64 + pt, 16 * pq)) = h4;
                *reinterpret_cast<uint4 *>(kblo + toff(pt, 16 * pq)) = l4;
                split8(fq + 8, h4, l4);
                *reinterpret_cast<uint4 *>(kb + toff(64 + pt, 16 * pq + 8)) = h4;
                *reinterpret_cast<uint4 *>(kblo + toff(pt, 16 * pq + 8)) = l4;
                // phi(k_hat): inclusive scan over this warp's 8 tokens (adjacent lanes)
#pragma unroll
                for (int m = 0; m < 16; ++m) fk[m] = pt < nt ? phi_fast(kf[m] * ksc) : 0.f;
#pragma unroll
                for (int off = 1; off < 8; off <<= 1) {
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        const float y = __shfl_up_sync(0xffffffffu, fk[m], off);
                        if ((lane & 7) >= off) fk[m] += y;
                    }
                }
                if ((lane & 7) == 7) {
                    float4 *dst = reinterpret_cast<float4 *>(s_tot + warp * 64 + 16 * pq);
#pragma unroll
                    for (int h = 0; h < 4; ++h) dst[h] = make_float4(fk[4 * h], fk[4 * h + 1], fk[4 * h + 2], fk[4 * h + 3]);
                }
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        // ---- round 1: D1 = X K^T; D2 = K Al^T (mode 0) or Phi Al^T (mode 1); (mode 1) DO = Phi X^T ----
        if (tid == 0) {
            tc_fence_after();
            mma_k64<false, false>(tbase + col_d4, smem_u32(xs_hi), smem_u32(kb), id_x64, false);
            mma_k64<false, false>(tbase + col_d4, smem_u32(xs_lo), smem_u32(kb), id_x64, true);
            if (MODE == 1) {
                // [DO | D2] = Phi [X; Al]^T: DO at col_do, D2 = Qm^T at col_do + 64 = col_d2
                mma_k64x3<false, false>(tbase + col_do, smem_u32(kb + kTile), smem_u32(kblo), smem_u32(xs_hi),
                                        smem_u32(xs_lo), idesc_bf16_f32(64, 128), false);
            } else {
                mma_k64<false, false>(tbase + col_d2, smem_u32(kb), smem_u32(al_hi), id_64, false);
                mma_k64<false, false>(tbase + col_d2, smem_u32(kb), smem_u32(al_lo), id_64, true);
            }
            umma_commit(bar);
        }
        if (MODE == 1) {  // readout denominators 1 / (phi(q_t) . n_t + eps)
            if (tid < 64) {  // per feature: exclusive prefix of the warp totals, and the total
                float run = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    const float x = s_tot[w * 64 + tid];
                    s_tot[w * 64 + tid] = run;
                    run += x;
                }
                s_tot[8 * 64 + tid] = run;
            }
            __syncthreads();
            const float4 *pw = reinterpret_cast<const float4 *>(s_tot + warp * 64 + 16 * pq);
            const float4 *pa = reinterpret_cast<const float4 *>(s_tot + 8 * 64 + 16 * pq);
            float dp = 0.f;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float4 p4 = pw[h], a4 = pa[h];
                const float pv[4] = {p4.x, p4.y, p4.z, p4.w}, av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = 4 * h + e;
                    dp = fmaf(fq[m], nb[m] + pv[e] + fk[m], dp);
                    nb[m] += av[e];
                }
            }
            dp += __shfl_xor_sync(0xffffffffu, dp, 8);
            dp += __shfl_xor_sync(0xffffffffu, dp, 16);
            if (pq == 0) s_rden[pt] = 1.f / (dp + kEps);
        }
        load_in(sb + 1);
        if (!round_wait()) {
            ok = false;
            break;
        }
        // ---- N (fp32, row-major, for the inverse; mode 0), Qm^T tiles (mode 1), E tiles ----
        {
            float v[32];
            tmem_ld32(tq + col_d2 + 32 * hw, v);  // D2 row t = 16 qw + lane (M = 64), columns s = 32 hw ..
            if (lane < 16) {
                const int t = 16 * qw + lane;
                if (MODE == 1) {
#pragma unroll
                    for (int m = 0; m < 32; ++m)
                        if (32 * hw + m > t) v[m] = 0.f;
                    put_row32(kb, kb + kTile, t, 32 * hw, v);
                } else {  // N[s][t] = alpha_s . k_hat_t (s < t), row-major: lanes t write one row s together
                    const float kt = s_ks[t];
#pragma unroll
                    for (int m = 0; m < 32; ++m) {
                        const int sr = 32 * hw + m;
                        ntb[sr * kGS + t] = sr < t ? v[m] * kt : 0.f;
                    }
                }
            }
            tmem_ld32(tq + col_d4 + 32 * hw, v);  // X K, columns 32 hw ..
            if (xact) {
                const float4 *ks4 = reinterpret_cast<const float4 *>(s_ks + 32 * hw);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 k4 = ks4[q];
                    const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int m = 4 * q + e, t = 32 * hw + m;
                        const float val = (MODE == 1 || xrow < 64) ? __bfloat162float(vt[t * kVS + (xrow & 63)]) : 0.f;
                        v[m] = fmaf(-v[m], kv[e], val);
                    }
                }
                put_row32(xs_hi, xs_lo, xrow, 32 * hw, v);
            }
        }
        tc_fence_before();
        __syncthreads();
        // ---- T_inv = (I + N)^{-1} (mode 0; blocked back substitution) ----
        if (MODE == 0) {
            tri_inv64(ntb, reinterpret_cast<float *>(kb), ti_hi, ti_lo);
        } else {  // mode 1: T_inv of this sub-block, stored by the transition pass
            if (!mbar_wait_bounded(bar_t, (uint32_t)(sb & 1), a.p.wait_limit_ns, a.p.err)) *abort_flag = 1;
            tinv_done = sb + 1;
        }
        fence_proxy_async_smem();
        __syncthreads();
        // ---- round 2: R = E T_inv ----
        if (tid == 0) {
            tc_fence_after();
            mma_k64x3<false, true>(tbase + col_d2, smem_u32(xs_hi), smem_u32(xs_lo), smem_u32(ti_hi),
                                   smem_u32(ti_lo), id_x64, false);
            umma_commit(bar);
        }
        if (MODE == 0) {  // T_inv tiles to the workspace for the readout pass
            const uint4 *src4 = reinterpret_cast<const uint4 *>(ti_hi);
            uint4 *dst4 = reinterpret_cast<uint4 *>(gtinv + (size_t)sb * 2 * kTile);
#pragma unroll
            for (int e = 0; e < 4; ++e) dst4[tid + kThreads * e] = src4[tid + kThreads * e];
        }
        if (!round_wait()) {
            ok = false;
            break;
        }
        {
            float v[32];
            tmem_ld32(tq + col_d2 + 32 * hw, v);
            if (xact) put_row32(xs_hi, xs_lo, xrow, 32 * hw, v);
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();
        // ---- round 3: X += R Al^T; (mode 1) DO += Qm^T R^T ----
        if (tid == 0) {
            tc_fence_after();
            mma_k64x3<false, true>(tbase + col_d4, smem_u32(xs_hi), smem_u32(xs_lo), smem_u32(al_hi), smem_u32(al_lo), id_x64,
                          false);
            if (MODE == 1)
                mma_k64x3<false, false>(tbase + col_do, smem_u32(kb), smem_u32(kb + kTile), smem_u32(xs_hi), smem_u32(xs_lo), id_64, true);
            umma_commit(bar);
        }
        if (!round_wait()) {
            ok = false;
            break;
        }
        {
            float v[32];
            tmem_ld32(tq + col_d4 + 32 * hw, v);
            if (xact) {
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] += v[j];
                put_row32(xs_hi, xs_lo, xrow, 32 * hw, x);
            }
            if (MODE == 1) {
                tmem_ld32(tq + col_do + 32 * hw, v);  // numerators of token 16 qw + lane, columns 32 hw ..
                const int t = 16 * qw + lane;
                if (lane < 16 && t < nt) {
                    const float rd = s_rden[t];
                    uint4 *dst = reinterpret_cast<uint4 *>(gout + (size_t)(sb * kSB + t) * kD + 32 * hw);
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = bf2_bits(__floats2bfloat162_rn(v[8 * g + 2 * e] * rd, v[8 * g + 2 * e + 1] * rd));
                        dst[g] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();
    }
    if (!ok) {
        if (tid == 0) {
            (void)mbar_wait_bounded(bar, phase ^ 1u, a.p.wait_limit_ns, a.p.err);
            if (MODE == 1 && tinv_issued > tinv_done)  // a T_inv copy may still be landing
                (void)mbar_wait_bounded(bar_t, (uint32_t)((tinv_issued - 1) & 1), a.p.wait_limit_ns, a.p.err);
        }
    } else if (MODE == 0) {  // rows 0..63 are H_c, rows 64..127 P_c
        float4 *dst = reinterpret_cast<float4 *>(ws_f(a, xrow < 64 ? a.L.off_H : a.L.off_P) +
                                                 ((size_t)bh * NC + c) * kD * kD + (size_t)(xrow & 63) * kD + 32 * hw);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, L::ncols);
}

template <int MODE>
cudaError_t launch_mode(const ChunkArgs &a, cudaStream_t st) {
    constexpr size_t bytes = TcLayout<MODE>::total + 1024;  // + alignment slack
    cudaError_t e = cudaFuncSetAttribute(rows_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
    if (e != cudaSuccess) return e;
    const long long grid = (long long)a.L.NC * a.p.BH;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    rows_tc_kernel<MODE><<<(unsigned)grid, kThreads, bytes, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool rows_tc_supported(const FwdParams &p, const ChunkLayout &L) {
    return p.d == kD && p.io_bf16 && L.C % kSB == 0 && L.tinv;
}

cudaError_t launch_rows_tc(const ChunkArgs &a, int mode, cudaStream_t stream) {
    return mode == 0 ? launch_mode<0>(a, stream) : launch_mode<1>(a, stream);
}

}  // namespace vla
