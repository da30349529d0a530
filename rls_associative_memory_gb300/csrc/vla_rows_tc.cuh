// vla_rows_tc.cuh -- tensor-core state pass (and the account of the output
// pass, vla_chunk_tc.cu) of the
// chunk-parallel path for d = 64 with bf16 I/O: the state write and ELU+1
// readout of "Variational Linear Attention: Stable Associative Memory for
// Long-Context Transformers", section 2.3 (step 3 and the readout), taken
// 64 tokens at a time in the UT (WY) form of a product of rank-1 updates.
//
// Within a chunk the state write is affine in the chunk-start state S_c:
// S_t = S_c P_t + H_t, where P_t and H_t are the states reached from the
// starts I and 0 (with values 0 and v).  So the readout is
//   o_t = S_c y_t + h_t,   y_t = P_t phi(q_t) / den_t,   h_t = H_t phi(q_t) / den_t
// with den_t = phi(q_t) . n_t + eps.  The state pass runs the 128 rows
// [H; P] of each chunk, writes the chunk map (H_c, P_c) for the chain along
// the chunks and y_t, h_t for every token; the output pass then only forms
// S_c y_t + h_t, with no recurrence left in it.
//
// Within a sub-block of c = 64 tokens whose state at the start is X (128 x
// 64), the token-by-token state write x <- x + (value - x.k_hat) alpha^T is
// equivalent to
//   R (I + N) = Vals - X K_hat,        N = strictly-upper(Al^T K_hat)  (c x c)
//   X_end     = X + R Al^T
//   X_t phi(q_t) = X phi(q_t) + sum_{s <= t} r_s (alpha_s . phi(q_t))
// where R = [r_1 .. r_c] holds the per-token residuals value_t - X_{t-1} k_hat_t
// (the residual of token t is its value minus what the earlier tokens of
// the sub-block left in the state, hence the triangular system).  The
// readout numerators are kept transposed, DO^T (rows = the 128 state rows,
// columns = tokens), so that every product of a round shares its left
// operand and the round is one wide product.  A sub-block is three rounds
// of tcgen05.mma plus one triangular inverse on the CUDA cores (recursive
// doubling on the 8 x 8 block structure):
//   1. [DO^T | D1] = X [Phi; K]^T  (N = 128),  D2 = K Al^T (= N^T)
//   2. R = E T_inv  (E = Vals - (X K) diag(1/|k|), T_inv = (I + N)^{-1}),
//      and Qm = Al Phi^T  (upper-incl: Qm[s][t] = alpha_s . phi(q_t), s <= t)
//   3. [X | DO^T] += R [Al | Qm]  (M = N = 128, accumulated in place)
// X stays in fp32 in TMEM for the whole chunk; its bf16 hi/lo tiles are
// rebuilt for each round 1.
//
// Precision: fp32 operands enter the tensor cores as bf16 pairs
// x = hi + lo (hi = bf16(x), lo = bf16(x - hi)), and a product takes
// hi*hi + hi*lo + lo*hi with fp32 accumulation (relative error about
// 2^-16).  k and v are bf16 inputs and exact: the raw key enters once and
// the key norm is applied as a column scale in fp32.
#pragma once

#include "vla_tc_common.cuh"

namespace vla {
namespace r64 {

using namespace tc;

constexpr int kThreads = 256;

struct TcLayout {
    static constexpr size_t ctrl = 0;  // mbarriers, abort flag
    // X / E / R tiles: 128 rows (0..63 the H rows, 64..127 the P rows), hi then lo
    static constexpr size_t xs_hi = 1024;
    static constexpr size_t xs_lo = xs_hi + 2 * kTile;
    // gates (token rows) hi, lo; then the T_inv tiles, later Qm: [Al | Qm] is
    // round 3's right operand, two MN-major atoms 16 KB apart
    static constexpr size_t al_hi = xs_hi + 4 * kTile;
    static constexpr size_t al_lo = al_hi + kTile;
    static constexpr size_t ti = al_hi + 2 * kTile;          // N fp32 (row stride kGS), then T_inv hi, lo, then Qm
    static constexpr uint32_t kAtom = 2 * kTile;             // Al -> Qm distance
    static constexpr size_t ph_hi = ti + 18 * 1024;          // Phi = phi(Q) hi, directly followed by
    static constexpr size_t kb = ph_hi + kTile;              // K (raw bf16): [Phi_hi; K] is one 128-row operand
    static constexpr size_t ph_lo = kb + kTile;              // Phi lo
    static constexpr int kVS = 72;                           // row stride (bf16) of the v tile
    static constexpr size_t vt = ph_lo + kTile;              // v [t][i] bf16
    static constexpr size_t ks = vt + (size_t)64 * kVS * 2;  // [64] 1 / max(|k|, eps)
    static constexpr size_t rden = ks + 256;                 // [64] 1 / (phi(q).n + eps)
    static constexpr size_t tot = rden + 256;                // [8][64] warp totals of phi(k_hat), then prefixes
    static constexpr size_t nrun = tot + 8 * 64 * 4;         // [64] n at the sub-block start
    static constexpr size_t tms = nrun + 256;                // triangular-inverse scratch (32 x 36 floats)
    static constexpr size_t total = tms + 32 * 36 * 4;
};
static_assert(TcLayout::ti % 1024 == 0 && TcLayout::ph_hi % 1024 == 0, "operand tiles must be 1024-byte aligned");
static_assert(TcLayout::ti + (size_t)64 * kGS * 4 <= TcLayout::ph_hi, "N fits before Phi");
static_assert(TcLayout::al_lo == TcLayout::al_hi + kTile, "the readout coefficients of a sub-block are staged in "
              "the Al tiles (16 KB)");

// 32 consecutive fp32 values as bf16 into row `row`, columns k0 .. k0+31, of a tile.
__device__ __forceinline__ void put_row32_bf16(unsigned char *tile, int row, int k0, const float *v) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = bf2_bits(__floats2bfloat162_rn(v[8 * g + 2 * e], v[8 * g + 2 * e + 1]));
        *reinterpret_cast<uint4 *>(tile + toff(row, k0 + 8 * g)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}
static_assert(TcLayout::tms % 16 == 0, "scratch rows are 16-byte aligned");

// Bulk copy shared -> global (bulk-group completion), its commit, and the
// waits for the group's source reads / for its completion.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// State pass of S-chunk c of unit bh (a CTA of kThreads threads; smem_raw:
// TcLayout::total + 1024 bytes of dynamic shared memory; tbase: 256 TMEM
// columns the caller has allocated).  The mbarriers are invalidated at the end,
// so that a persistent CTA can run further jobs.
__device__ __forceinline__ void rows_tc_body(const ChunkArgs &a, int c, int bh, unsigned char *smem_raw,
                                             uint32_t tbase) {
    using L = TcLayout;
    // swizzled tiles need 1024-byte aligned addresses (one extra KB is allocated)
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::ctrl);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::ctrl + 12);
    uint64_t *bar_n = reinterpret_cast<uint64_t *>(smem + L::ctrl + 16);  // round 1's N^T product alone
    unsigned char *xs_hi = smem + L::xs_hi, *xs_lo = smem + L::xs_lo;
    unsigned char *kb = smem + L::kb, *ph_hi = smem + L::ph_hi, *ph_lo = smem + L::ph_lo;
    unsigned char *al_hi = smem + L::al_hi, *al_lo = smem + L::al_lo;
    float *ntb = reinterpret_cast<float *>(smem + L::ti);  // N, row stride kGS
    unsigned char *ti_hi = smem + L::ti, *ti_lo = smem + L::ti + kTile;  // T_inv (tile row s = row s), then Qm
    __nv_bfloat16 *vt = reinterpret_cast<__nv_bfloat16 *>(smem + L::vt);
    float *s_ks = reinterpret_cast<float *>(smem + L::ks);
    float *s_rden = reinterpret_cast<float *>(smem + L::rden);
    float *s_tot = reinterpret_cast<float *>(smem + L::tot);
    float *s_nrun = reinterpret_cast<float *>(smem + L::nrun);

    const int NC = a.L.NC, C = a.L.C, T = a.p.T;
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
    const __half *gal = reinterpret_cast<const __half *>(static_cast<const unsigned char *>(a.p.ws) + a.L.off_alpha) + tok0;
    // this chunk's readout coefficients: per sub-block [y | h] (bf16), tile row =
    // state row (feature), columns = tokens
    unsigned char *gyh = static_cast<unsigned char *>(a.p.ws) + a.L.off_yh +
                         (size_t)(bh * NC + c) * (C / kSB) * (2 * kTile);

    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar_n, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (tid < 64)  // n at the chunk start (chunks start on A-chunk boundaries)
        s_nrun[tid] = ws_f(a, a.L.off_n)[((size_t)bh * (a.L.NCA + 1) + (size_t)c * (C / a.L.CA)) * kD + tid];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tq = tbase + ((uint32_t)(32 * qw) << 16);  // this warp's lane quarter
    constexpr uint32_t col_x = 0;     // X (fp32 state, M = 128 rows)
    constexpr uint32_t col_do = 64;   // DO^T (state rows x tokens), next to X and to D1
    constexpr uint32_t col_d1 = 128;  // D1 = X K^T, then R
    constexpr uint32_t col_d2 = 192;  // D2 = N^T, then Qm

    // State row 32 qw + lane of [H; P], columns 32 hw .. (H starts at 0, P at I):
    // into TMEM and, as hi/lo tiles, into the first round's operand.
    const int xrow = 32 * qw + lane;
    {
        float x[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = (xrow - 64 == 32 * hw + j) ? 1.f : 0.f;
        tmem_st32(tq + col_x + 32 * hw, x);
        put_row32(xs_hi, xs_lo, xrow, 32 * hw, x);
        tc_fence_before();  // (the first round accumulates onto X after a barrier)
    }

    // Inputs of the next sub-block, prefetched into registers during rounds
    // 2-3 of the current one (token pt, features 16 pq .. 16 pq + 15).
    uint4 rk[2], rv[2], rq[2], ra[2];
    // (always a valid token row, clamped: no select waits on the loads here;
    // tokens past the chunk are zeroed where the values are used)
    auto load_in = [&](int sb) {
        const int t = min(sb * kSB + pt, ntok - 1);
        const size_t off = (size_t)t * kD + 16 * pq;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            rk[h] = reinterpret_cast<const uint4 *>(gk + off)[h];
            rv[h] = reinterpret_cast<const uint4 *>(gv + off)[h];
            rq[h] = reinterpret_cast<const uint4 *>(gq + off)[h];
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) ra[h] = reinterpret_cast<const uint4 *>(gal + off)[h];
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
    constexpr uint32_t id_xw = idesc_bf16_f32(128, 128);  // the 128 state rows x 128 columns
    constexpr uint32_t id_x = idesc_bf16_f32(128, 64);
    constexpr uint32_t id_64 = idesc_bf16_f32(64, 64);
    constexpr int kVS = L::kVS;

    bool ok = true;
    load_in(0);
    for (int sb = 0; sb < nsb; ++sb) {
        const int nt = min(kSB, ntok - sb * kSB);
        float fq[16];
        // ---- stage the sub-block's operands ----
        if (pt >= nt) {  // past the chunk: zero inputs
            rk[0] = rk[1] = rv[0] = rv[1] = rq[0] = rq[1] = ra[0] = ra[1] = make_uint4(0, 0, 0, 0);
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
            unpack8_h(ra[0], af);
            unpack8_h(ra[1], af + 8);
            uint4 h4, l4;
            split8(af, h4, l4);
            *reinterpret_cast<uint4 *>(al_hi + toff(pt, 16 * pq)) = h4;
            *reinterpret_cast<uint4 *>(al_lo + toff(pt, 16 * pq)) = l4;
            split8(af + 8, h4, l4);
            *reinterpret_cast<uint4 *>(al_hi + toff(pt, 16 * pq + 8)) = h4;
            *reinterpret_cast<uint4 *>(al_lo + toff(pt, 16 * pq + 8)) = l4;
            float qf[16];
            unpack8(rq[0], qf);
            unpack8(rq[1], qf + 8);
#pragma unroll
            for (int m = 0; m < 16; ++m) fq[m] = phi_fast(qf[m]);
            split8(fq, h4, l4);
            *reinterpret_cast<uint4 *>(ph_hi + toff(pt, 16 * pq)) = h4;
            *reinterpret_cast<uint4 *>(ph_lo + toff(pt, 16 * pq)) = l4;
            split8(fq + 8, h4, l4);
            *reinterpret_cast<uint4 *>(ph_hi + toff(pt, 16 * pq + 8)) = h4;
            *reinterpret_cast<uint4 *>(ph_lo + toff(pt, 16 * pq + 8)) = l4;
        }
        fence_proxy_async_smem();
        __syncthreads();
        // ---- round 1: [DO^T | D1] = X [Phi; K]^T, D2 = K Al^T ----
        if (tid == 0) {
            tc_fence_after();
            // hi.hi and lo.hi for both (K is exact), then hi.lo for the Phi part
            // N^T = K Al^T first, on its own barrier: the triangular inverse
            // runs on the CUDA cores while the wide product is still going
            mma_k64<false, false>(tbase + col_d2, smem_u32(kb), smem_u32(al_hi), id_64, false);
            mma_k64<false, false>(tbase + col_d2, smem_u32(kb), smem_u32(al_lo), id_64, true);
            umma_commit(bar_n);
            mma_k64<false, false>(tbase + col_do, smem_u32(xs_hi), smem_u32(ph_hi), id_xw, false);
            mma_k64<false, false>(tbase + col_do, smem_u32(xs_lo), smem_u32(ph_hi), id_xw, true);
            mma_k64<false, false>(tbase + col_do, smem_u32(xs_hi), smem_u32(ph_lo), id_x, true);
            umma_commit(bar);
        }
        // ---- readout denominators 1 / (phi(q_t) . n_t + eps), while round 1 runs ----
        // phi(k_hat) of token pt (the raw keys from the K tile), scanned over this
        // warp's 8 tokens (adjacent lanes)
        float fk[16];
        {
            float kf[16];
            unpack8(*reinterpret_cast<const uint4 *>(kb + toff(pt, 16 * pq)), kf);
            unpack8(*reinterpret_cast<const uint4 *>(kb + toff(pt, 16 * pq + 8)), kf + 8);
            const float ksc = s_ks[pt];
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
        __syncthreads();
        if (tid < 64) {  // per feature: n before each warp's tokens, and n after the sub-block
            float run = s_nrun[tid];
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const float y = s_tot[w * 64 + tid];
                s_tot[w * 64 + tid] = run;
                run += y;
            }
            s_nrun[tid] = run;
        }
        __syncthreads();
        {
            const float4 *pw = reinterpret_cast<const float4 *>(s_tot + warp * 64 + 16 * pq);
            float dp = 0.f;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
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
            if (lane < 16) {  // N[s][t] = alpha_s . k_hat_t (s < t), row-major: lanes t write one row s together
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
        // ---- T_inv = (I + N)^{-1} (recursive doubling, in place over N), while the
        // wide product of round 1 runs ----
        tri_inv64(ntb, reinterpret_cast<float *>(smem + L::tms), ti_hi, ti_lo);
        if (!round_wait()) {
            ok = false;
            break;
        }
        // ---- E tiles ----
        {
            float v[32];
            tmem_ld32(tq + col_d1 + 32 * hw, v);  // X K, columns 32 hw ..
            const float4 *ks4 = reinterpret_cast<const float4 *>(s_ks + 32 * hw);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 k4 = ks4[q];
                const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = 4 * q + e, t = 32 * hw + m;
                    const float val = xrow < 64 ? __bfloat162float(vt[t * kVS + xrow]) : 0.f;
                    v[m] = fmaf(-v[m], kv[e], val);
                }
            }
            put_row32(xs_hi, xs_lo, xrow, 32 * hw, v);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- round 2: R = E T_inv, Qm = Al Phi^T ----
        if (tid == 0) {
            tc_fence_after();
            mma_k64x3<false, true>(tbase + col_d1, smem_u32(xs_hi), smem_u32(xs_lo), smem_u32(ti_hi),
                                   smem_u32(ti_lo), id_x, false);
            mma_k64x3<false, false>(tbase + col_d2, smem_u32(al_hi), smem_u32(al_lo), smem_u32(ph_hi),
                                    smem_u32(ph_lo), id_64, false);
            umma_commit(bar);
        }
        // the next sub-block's inputs: issued here, after the inverse, so that
        // their registers are not live through it (rounds 2-3 hide the latency)
        load_in(sb + 1);
        if (!round_wait()) {
            ok = false;
            break;
        }
        // ---- R tiles; Qm tiles over T_inv (round 2 has read it) ----
        {
            float v[32];
            tmem_ld32(tq + col_d1 + 32 * hw, v);
            put_row32(xs_hi, xs_lo, xrow, 32 * hw, v);
            tmem_ld32(tq + col_d2 + 32 * hw, v);  // Qm row s = 16 qw + lane, columns t = 32 hw ..
            if (lane < 16) {
                const int srow = 16 * qw + lane;
#pragma unroll
                for (int m = 0; m < 32; ++m)
                    if (32 * hw + m < srow) v[m] = 0.f;
                put_row32(ti_hi, ti_lo, srow, 32 * hw, v);
            }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();
        // ---- round 3: [X | DO^T] += R [Al | Qm] (B MN-major, two atoms 16 KB apart) ----
        if (tid == 0) {
            tc_fence_after();
            mma_k64x3<false, true>(tbase + col_x, smem_u32(xs_hi), smem_u32(xs_lo), smem_u32(al_hi), smem_u32(al_lo),
                                   id_xw, true, 16, L::kAtom);
            umma_commit(bar);
        }
        if (!round_wait()) {
            ok = false;
            break;
        }
        {
            float v[32];
            tmem_ld32(tq + col_x + 32 * hw, v);  // the new X: next round 1's operand
            put_row32(xs_hi, xs_lo, xrow, 32 * hw, v);
            // readout coefficients of state row xrow for tokens 32 hw .., divided by
            // den_t: y (rows 64..127, tile row xrow - 64) and h (rows 0..63)
            tmem_ld32(tq + col_do + 32 * hw, v);
            const float4 *rd4 = reinterpret_cast<const float4 *>(s_rden + 32 * hw);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 r4 = rd4[q];
                v[4 * q] *= r4.x; v[4 * q + 1] *= r4.y; v[4 * q + 2] *= r4.z; v[4 * q + 3] *= r4.w;
            }
            // staged in the Al tiles (free once round 3 is done) in the global
            // layout [y | h], then one bulk copy
            put_row32_bf16(al_hi + (xrow < 64 ? kTile : 0), xrow & 63, 32 * hw, v);
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            bulk_s2g(gyh + (size_t)sb * (2 * kTile), al_hi, 2 * kTile);
            bulk_wait_read();  // the next sub-block's staging overwrites the source
        }
        __syncthreads();
    }
    if (tid == 0) bulk_wait_all();  // the coefficient copies are complete before the CTA ends
    if (!ok) {
        if (tid == 0) (void)mbar_wait_bounded(bar, pend, a.p.wait_limit_ns, a.p.err);
    } else {  // rows 0..63 are H_c, rows 64..127 P_c
        float x[32];
        tmem_ld32(tq + col_x + 32 * hw, x);
        float4 *dst = reinterpret_cast<float4 *>(ws_f(a, xrow < 64 ? a.L.off_H : a.L.off_P) +
                                                 ((size_t)bh * NC + c) * kD * kD + (size_t)(xrow & 63) * kD + 32 * hw);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // (a later job of this CTA may lay out its memory otherwise)
        mbar_inval(bar);
        mbar_inval(bar_n);
    }
}

}  // namespace r64
}  // namespace vla
