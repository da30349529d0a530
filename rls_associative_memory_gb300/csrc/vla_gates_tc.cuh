// vla_gates_tc.cuh -- the gates of the chunk-parallel path on the tensor cores
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
// Per sub-block (tensor-core rounds R1, R2, R4; tiles and products as in the
// state passes, bf16 hi/lo pairs for fp32 operands):
//   R1  D1 = [U; K] A                 rows: w_t, A k_t
//   R2  D2 = U [A K ; W]^T            Y = U^T A K, G = U^T W
//   on the CUDA cores, in fp32: forward elimination of [I + G | W^T | Y_hat]
//       (Y_hat = Y diag(1/|k|)) -> [D L^T | L^{-1} W^T | L^{-1} Y_hat]: the
//       rows of L^{-1} W^T are z_s^T (X = L^{-T}), P = L^{-1} Y_hat holds
//       z_s . k_hat_t, and beta_s = 1 / pivot_s (the trailing block stays
//       symmetric, so the multipliers come from the pivot row)
//   R4  D1[k rows] += E'^T Z^T        E'[s][t] = -beta_s P[s][t] |k_t| (s <= t):
//                                      the rows become |k_t| A_t k_hat_t
//       A += -(Z diag(beta)) Z^T      (A held in fp32 in TMEM for the whole
//                                      A-chunk; the product accumulates onto
//                                      it with three-way bf16 splits)
//   alpha_t = that row / |that row|, and the new A's operand tiles.
// Precision: Z and P carry most of the cancellation when the sub-block's
// penalty directions outweigh the penalty accumulated so far (A_t k_hat_t is
// then a small difference of large terms; at the start of a stream, or with
// large u or small lambda0).  They come out of the fp32 elimination, not
// out of split products, and the downdate of A, which accumulates over the
// A-chunk, takes three-way splits (x = x0 + x1 + x2, the six products with
// i + j <= 2, about 2^-24 relative); the other products keep hi/lo pairs.
// A starts each A-chunk from its definition (M^(c))^{-1}, M^(c) = lambda0 I +
// the Grams of the earlier A-chunks: the same elimination on M^(c) against
// the identity gives E = L^{-1} and D, then A = E^T D^{-1} E is one product on
// the tensor cores (a sum of positive semi-definite terms, no cancellation).
#pragma once

#include "vla_tma.cuh"

namespace vla {
namespace g64 {

using namespace tc;

constexpr int kThreads = 256;

struct GtLayout {
    static constexpr size_t ctrl = 0;                       // mbarriers, abort flag
    static constexpr size_t uk = 1024;                      // [U; K] (128 rows, exact bf16)
    static constexpr size_t ah = uk + 2 * kTile;            // A hi, lo
    static constexpr size_t work = ah + 2 * kTile;          // 66 KB work area, by phase:
    // R1 -> R2: AK^T hi @0, W^T hi @8K, AK^T lo @16K, W^T lo @24K (R2's B operand, two
    //           64-row tiles stacked), W^T fp32 @kW32
    // R2 -> elimination: Y_hat fp32 @0, I + G fp32 @kG32, W^T fp32 @kW32
    // elimination: 8 KB a block of 8 pivots @0 .. 64K (I + G pivot rows, scaled rows,
    //     W^T and Y_hat pivot rows, 8 x 64 floats each)
    // R4: [-(beta Z)^T | E'] pairs of atoms @0 (parts 0) and @16K (parts 1), Z^T parts
    //     0, 1, 2 @32K, 40K, 48K, -(beta Z)^T part 2 @56K
    // chunk start: diag(1/D) E hi @0, lo @8K, E hi @16K, lo @24K, M^(c) fp32 @32K,
    //     pivot rows @kCrow (2 x 8 x 128 floats), scaled pivot rows @kCsrow
    static constexpr size_t kW32 = 4 * kTile;
    static constexpr size_t kG32 = kW32 + (size_t)64 * kGS * 4;
    static constexpr size_t kCrow = kW32 + (size_t)64 * kGS * 4;
    static constexpr size_t kCsrow = kCrow + (size_t)2 * 8 * 128 * 4;
    static constexpr size_t work_bytes = kG32 + (size_t)64 * kGS * 4;
    static constexpr size_t ksc = work + work_bytes;        // [2][64] 1 / max(|k|, eps) (by sub-block parity)
    static constexpr size_t kn = ksc + 512;                 // [2][64] max(|k|, eps)
    static constexpr size_t beta = kn + 512;                // [64]
    static constexpr size_t nrm = beta + 256;               // [2][64] halves of |row|^2
    static constexpr size_t total = nrm + 512;
};
static_assert(GtLayout::work % 1024 == 0, "operand tiles must be 1024-byte aligned");
static_assert(8 * 8 * 4 * 64 * 4 <= GtLayout::work_bytes, "the elimination's publication buffers fit");
static_assert(8 * kTile <= GtLayout::work_bytes, "R4 tiles fit the work area");
static_assert(GtLayout::kCsrow + 2 * 8 * 64 * 4 <= GtLayout::work_bytes, "chunk-start scratch fits");

// bf16 parts x = x0 + x1 + x2 of two fp32 values (each part the nearest bf16
// of what the earlier parts leave), as packed pairs.
__device__ __forceinline__ void split3_pair(float a, float b, uint32_t &p0, uint32_t &p1, uint32_t &p2) {
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(a, b);
    const float2 f0 = __bfloat1622float2(h0);
    const float ra = a - f0.x, rb = b - f0.y;
    const __nv_bfloat162 h1 = __floats2bfloat162_rn(ra, rb);
    const float2 f1 = __bfloat1622float2(h1);
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(ra - f1.x, rb - f1.y);
    p0 = bf2_bits(h0);
    p1 = bf2_bits(h1);
    p2 = bf2_bits(h2);
}

// Forward elimination of [I + G | W^T | Y_hat] (64 rows s, fp32, row stride
// kGS) without pivoting.  Warp w owns rows 8 w .. 8 w + 7 and lane l columns
// 2 l, 2 l + 1 of each block; the owner of a block of 8 pivots eliminates it
// with shuffles.  Only the I + G part is on the serial chain: the owner runs
// its pivots on I + G alone and publishes their rows and the rows scaled by
// -1 / D_s (whose entries are the multipliers of the later rows), so that the
// next owner can apply them to its I + G rows and start its own pivots at
// once.  The right-hand blocks follow off the chain: each warp applies the
// earlier blocks' pivots to its W^T and Y_hat rows, then its own (multipliers
// read back from its scaled rows), and publishes its pivot rows of those.
// Every element takes the same FMAs in the same pivot order as in a single
// sweep, so the result does not depend on the split.  Each block has its own
// publication buffers in `pub` (8 KB a block: I + G pivot rows, scaled rows,
// W^T and Y_hat pivot rows) and two mbarriers, ebar[b] (the I + G part of
// block b published) and ebar[8 + b] (its right-hand part), each completed by
// the owner's 32 lanes once per call (phase parity `ephase`); every wait is
// bounded, and after a failed one the warp sets the abort flag and waits no
// more (it still publishes and arrives, so nobody else is held).
// Afterwards row s holds z_s^T = (L^{-1} W^T)[s] and P[s] = (L^{-1} Y_hat)[s],
// and rpiv[s] = 1 / D_s.  It writes the operand tiles of round 4 (rows s): Z^T
// and -(beta Z)^T in three bf16 parts, E'[s][t] = -beta_s P[s][t] |k_t|
// (s <= t, else 0) in two.  256 threads; all must call.
__device__ __forceinline__ void eliminate_rhs64(const float *gs, const float *w32, const float *y32, float *pub,
                                                float *rpiv, const float *kn, unsigned char *work, uint64_t *ebar,
                                                uint32_t ephase, const ChunkArgs &a, volatile int *abort_flag) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float2 m[8], z[8], pp[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 8 * warp + i;
        m[i] = *reinterpret_cast<const float2 *>(gs + r * kGS + 2 * lane);
        z[i] = *reinterpret_cast<const float2 *>(w32 + r * kGS + 2 * lane);
        pp[i] = *reinterpret_cast<const float2 *>(y32 + r * kGS + 2 * lane);
    }
    __syncthreads();  // the staging may be overwritten once everyone has its rows
    // block b's buffers: I + G pivot rows, scaled rows, W^T and Y_hat pivot rows (8 x 64 each)
    auto pm = [&](int b) { return pub + b * 2048; };
    auto ps = [&](int b) { return pub + b * 2048 + 512; };
    auto pz = [&](int b) { return pub + b * 2048 + 1024; };
    auto py = [&](int b) { return pub + b * 2048 + 1536; };
    bool live = true;
    auto wait = [&](uint64_t *bar) {
        if (live && !mbar_wait_bounded(bar, ephase, a.p.wait_limit_ns, a.p.err)) {
            live = false;
            *abort_flag = 1;
        }
    };
    // block b's pivots applied to this warp's rows of I + G, or of W^T and Y_hat
    auto apply_m = [&](int b) {
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const float4 fa = *reinterpret_cast<const float4 *>(ps(b) + p * 64 + 8 * warp);
            const float4 fb = *reinterpret_cast<const float4 *>(ps(b) + p * 64 + 8 * warp + 4);
            const float2 pv = *reinterpret_cast<const float2 *>(pm(b) + p * 64 + 2 * lane);
            const float fr[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) m[i] = __ffma2_rn(make_float2(fr[i], fr[i]), pv, m[i]);
        }
    };
    auto apply_zp = [&](int b) {
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const float4 fa = *reinterpret_cast<const float4 *>(ps(b) + p * 64 + 8 * warp);
            const float4 fb = *reinterpret_cast<const float4 *>(ps(b) + p * 64 + 8 * warp + 4);
            const float2 pzv = *reinterpret_cast<const float2 *>(pz(b) + p * 64 + 2 * lane);
            const float2 pyv = *reinterpret_cast<const float2 *>(py(b) + p * 64 + 2 * lane);
            const float fr[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 fi = make_float2(fr[i], fr[i]);
                z[i] = __ffma2_rn(fi, pzv, z[i]);
                pp[i] = __ffma2_rn(fi, pyv, pp[i]);
            }
        }
    };
    // the earlier blocks: I + G as soon as published; the right-hand part of
    // all but the last one in between (the last one's comes after this warp's
    // own pivots, which are on the chain)
#pragma unroll 1
    for (int b = 0; b < warp; ++b) {
        wait(&ebar[b]);
        apply_m(b);
        if (b + 1 < warp) {
            wait(&ebar[8 + b]);
            apply_zp(b);
        }
    }
    // this warp's block: pivots s = 8 warp + p on I + G
    {
        float *bm = pm(warp), *bs = ps(warp);
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            // pivot M[s][s], s = 8 warp + p: lane s / 2, component p mod 2
            const float pv = __shfl_sync(0xffffffffu, (p & 1) ? m[p].y : m[p].x, 4 * warp + (p >> 1));
            // fast reciprocal: the pivots of I + G are >= 1 and its relative
            // error (about 2^-22) is far below the parity bar downstream
            const float rp = __fdividef(1.f, pv);
            if (lane == 0) rpiv[8 * warp + p] = rp;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (i <= p) continue;  // (constant trip count: the rows stay in registers)
                const float mv = __shfl_sync(0xffffffffu, (i & 1) ? m[p].y : m[p].x, 4 * warp + (i >> 1));
                m[i] = __ffma2_rn(make_float2(-mv * rp, -mv * rp), m[p], m[i]);
            }
            *reinterpret_cast<float2 *>(bm + p * 64 + 2 * lane) = m[p];
            *reinterpret_cast<float2 *>(bs + p * 64 + 2 * lane) = __fmul2_rn(m[p], make_float2(-rp, -rp));
        }
        mbar_arrive(&ebar[warp]);
    }
    // the right-hand part: the previous block's pivots, then this block's (their
    // multipliers are the scaled rows just published: entry 8 warp + i of row p)
    if (warp > 0) {
        wait(&ebar[8 + warp - 1]);
        apply_zp(warp - 1);
    }
    __syncwarp();
    {
        const float *bs = ps(warp);
        float *bz = pz(warp), *by = py(warp);
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const float4 fa = *reinterpret_cast<const float4 *>(bs + p * 64 + 8 * warp);
            const float4 fb = *reinterpret_cast<const float4 *>(bs + p * 64 + 8 * warp + 4);
            const float fr[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (i <= p) continue;
                const float2 fi = make_float2(fr[i], fr[i]);
                z[i] = __ffma2_rn(fi, z[p], z[i]);
                pp[i] = __ffma2_rn(fi, pp[p], pp[i]);
            }
            *reinterpret_cast<float2 *>(bz + p * 64 + 2 * lane) = z[p];
            *reinterpret_cast<float2 *>(by + p * 64 + 2 * lane) = pp[p];
        }
        mbar_arrive(&ebar[8 + warp]);
    }
    __syncthreads();  // every block applied: the buffers may be overwritten
    // round 4's tiles, rows s = 8 warp + i, columns 2 lane, 2 lane + 1
    unsigned char *bz0 = work, *ep0 = work + kTile, *bz1 = work + 2 * kTile, *ep1 = work + 3 * kTile;
    unsigned char *zt0 = work + 4 * kTile, *zt1 = work + 5 * kTile, *zt2 = work + 6 * kTile;
    unsigned char *bz2 = work + 7 * kTile;
    const float2 knt = *reinterpret_cast<const float2 *>(kn + 2 * lane);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int s = 8 * warp + i;
        const float bs = rpiv[s];  // written by this warp as the owner of row s
        const uint32_t o = toff(s, 2 * lane);
        uint32_t w0, w1, w2;
        split3_pair(z[i].x, z[i].y, w0, w1, w2);
        *reinterpret_cast<uint32_t *>(zt0 + o) = w0;
        *reinterpret_cast<uint32_t *>(zt1 + o) = w1;
        *reinterpret_cast<uint32_t *>(zt2 + o) = w2;
        split3_pair(-bs * z[i].x, -bs * z[i].y, w0, w1, w2);
        *reinterpret_cast<uint32_t *>(bz0 + o) = w0;
        *reinterpret_cast<uint32_t *>(bz1 + o) = w1;
        *reinterpret_cast<uint32_t *>(bz2 + o) = w2;
        const float ex = (2 * lane >= s) ? -bs * pp[i].x * knt.x : 0.f;
        const float ey = (2 * lane + 1 >= s) ? -bs * pp[i].y * knt.y : 0.f;
        split3_pair(ex, ey, w0, w1, w2);
        *reinterpret_cast<uint32_t *>(ep0 + o) = w0;
        *reinterpret_cast<uint32_t *>(ep1 + o) = w1;
    }
}

// One A-chunk c of unit bh (a CTA of kThreads threads; smem_raw: GtLayout::total
// + 1024 bytes of dynamic shared memory; tbase: 256 TMEM columns the caller has
// allocated).  The mbarriers are invalidated at the end, so that a persistent
// CTA can run further jobs.
__device__ __forceinline__ void gates_tc_body(const ChunkArgs &a, int c, int bh, unsigned char *smem_raw,
                                              const CUtensorMap *tm_u, const CUtensorMap *tm_k, uint32_t tbase) {
    using L = GtLayout;
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::ctrl);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::ctrl + 12);
    uint64_t *ebar = reinterpret_cast<uint64_t *>(smem + L::ctrl + 64);  // the elimination's 16 mbarriers
    uint64_t *tbar = reinterpret_cast<uint64_t *>(smem + L::ctrl + 256);  // [U; K] tensor copies
    unsigned char *uk = smem + L::uk;
    unsigned char *a_hi = smem + L::ah, *a_lo = smem + L::ah + kTile;
    unsigned char *work = smem + L::work;  // work + i * kTile: tile slot i
    float *s_ks = reinterpret_cast<float *>(smem + L::ksc);
    float *s_kn = reinterpret_cast<float *>(smem + L::kn);
    float *s_beta = reinterpret_cast<float *>(smem + L::beta);
    float *s_nrm = reinterpret_cast<float *>(smem + L::nrm);
    // R2's B operand [AK; W] (two stacked tiles, hi then lo) and the elimination's staging
    unsigned char *akt_hi = work, *wt_hi = work + kTile, *akt_lo = work + 2 * kTile, *wt_lo = work + 3 * kTile;
    float *w32 = reinterpret_cast<float *>(work + L::kW32);  // W^T rows (fp32)
    float *g32 = reinterpret_cast<float *>(work + L::kG32);  // I + G (fp32)
    float *y32 = reinterpret_cast<float *>(work);            // Y_hat rows (fp32), once R2 is done
    // R4's operands (written by the elimination)
    unsigned char *bz0 = work, *bz1 = work + 2 * kTile, *bz2 = work + 7 * kTile;
    unsigned char *zt0 = work + 4 * kTile, *zt1 = work + 5 * kTile, *zt2 = work + 6 * kTile;

    const int NCA = a.L.NCA, CA = a.L.CA, T = a.p.T;
    const int t0 = c * CA, ntok = min(CA, T - t0), nsb = (ntok + kSB - 1) / kSB;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int qw = warp & 3, hw = warp >> 2;  // TMEM lane quarter, column half
    const int pt = 8 * warp + (lane & 7), pq = lane >> 3;  // staging: token, feature quarter
    const int r64 = 16 * qw + lane;                         // row in an M = 64 accumulator (lanes < 16)
    const bool act64 = lane < 16;
    const int r128 = 32 * qw + lane;                        // row in an M = 128 accumulator
    const size_t tok0 = ((size_t)bh * T + t0) * kD;
    __half *galpha = reinterpret_cast<__half *>(static_cast<unsigned char *>(a.p.ws) + a.L.off_alpha) + tok0;

    if (tid == 0) {
        mbar_init(bar, 1);
        for (int b = 0; b < 16; ++b) mbar_init(&ebar[b], 32);
        mbar_init(tbar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tq = tbase + ((uint32_t)(32 * qw) << 16);  // this warp's lane quarter
    constexpr uint32_t col_d1 = 0, col_d5 = 64, col_d2 = 128;

    // [U; K] of sub-block sb by two tensor copies into the operand tile (U rows,
    // then K rows; the maps fill tokens past T with zeros, and every A-chunk but
    // the stream's last is whole sub-blocks).  Thread 0 issues; the copy of
    // sub-block sb completes phase sb mod 2 of tbar.
    int tma_issued = -1;  // (thread 0's bookkeeping) the last sub-block whose copy was issued
    auto issue_in = [&](int sb) {
        mbar_arrive_expect_tx(tbar, 2 * kTile);
        tma_load_3d(uk, tm_u, 0, t0 + sb * kSB, bh, tbar);
        tma_load_3d(uk + kTile, tm_k, 0, t0 + sb * kSB, bh, tbar);
        tma_issued = sb;
    };
    if (tid == 0 && nsb > 0) issue_in(0);  // lands while the chunk-start A is formed

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
            float *stage = reinterpret_cast<float *>(work + L::kW32);  // M^(c) (fp32)
            const float4 *g4 = reinterpret_cast<const float4 *>(src + gr * kD + 16 * gp);
            float4 *st = reinterpret_cast<float4 *>(stage + gr * kGS + 16 * gp);
#pragma unroll
            for (int q = 0; q < 4; ++q) st[q] = g4[q];
            __syncthreads();
            // E = L^{-1} hi, lo @16K, 24K; diag(1/D) E hi, lo @0, 8K
            eliminate64(stage, reinterpret_cast<float *>(work + L::kCrow), reinterpret_cast<float *>(work + L::kCsrow),
                        s_beta, work + 2 * kTile, work + 3 * kTile, work, work + kTile);
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                mma_k64x3<true, true>(tbase + col_d5, smem_u32(work), smem_u32(work + kTile), smem_u32(work + 2 * kTile),
                                      smem_u32(work + 3 * kTile), idesc_bf16_f32(64, 64), false);
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

    uint32_t phase = (c > 0) ? 1u : 0u;  // the chunk-start product used phase 0
    auto round_wait = [&]() -> bool {
        const bool w = mbar_wait_bounded(bar, phase, a.p.wait_limit_ns, a.p.err);
        phase ^= 1u;
        if (!w) *abort_flag = 1;
        __syncthreads();
        tc_fence_after();
        return *abort_flag == 0;
    };

    // the key norms of sub-block sb, from its K rows once its copy has landed,
    // into the sb-parity half of s_kn, s_ks (the other half still serves
    // sub-block sb - 1)
    auto norms_in = [&](int sb) {
        if (!mbar_wait_bounded(tbar, (uint32_t)(sb & 1), a.p.wait_limit_ns, a.p.err)) *abort_flag = 1;
        const uint4 k0 = *reinterpret_cast<const uint4 *>(uk + toff(64 + pt, 16 * pq));
        const uint4 k1 = *reinterpret_cast<const uint4 *>(uk + toff(64 + pt, 16 * pq + 8));
        float kf[16];
        unpack8(k0, kf);
        unpack8(k1, kf + 8);
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
    };

    bool ok = true;
    if (nsb > 0) norms_in(0);
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
        // ---- W^T and (A K)^T tiles (token rows); W^T in fp32 for the elimination ----
        {
            float v[32];
            tmem_ld32(tq + col_d1 + 32 * hw, v);
            if (qw < 2) {
                put_row32(wt_hi, wt_lo, r128, 32 * hw, v);
                float4 *dst = reinterpret_cast<float4 *>(w32 + r128 * kGS + 32 * hw);
#pragma unroll
                for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            } else {
                put_row32(akt_hi, akt_lo, r128 - 64, 32 * hw, v);
            }
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
        // round 2 has read [U; K]: the next sub-block's copy lands during the elimination
        if (tid == 0 && sb + 1 < nsb) issue_in(sb + 1);
        // ---- Y_hat rows s and I + G (fp32) for the elimination ----
        {
            float v[32];
            tmem_ld32(tq + col_d2 + 32 * hw, v);  // Y[s][t], t = 32 hw ..
            if (act64) {
                const float4 *k4 = reinterpret_cast<const float4 *>(ks_sb + 32 * hw);
                float4 *dst = reinterpret_cast<float4 *>(y32 + r64 * kGS + 32 * hw);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 kv = k4[q];
                    dst[q] = make_float4(v[4 * q] * kv.x, v[4 * q + 1] * kv.y, v[4 * q + 2] * kv.z, v[4 * q + 3] * kv.w);
                }
            }
            tmem_ld32(tq + col_d2 + 64 + 32 * hw, v);  // G[s][t]
            if (act64) {
#pragma unroll
                for (int m = 0; m < 32; ++m)
                    if (32 * hw + m == r64) v[m] += 1.f;
                float4 *dst = reinterpret_cast<float4 *>(g32 + r64 * kGS + 32 * hw);
#pragma unroll
                for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
        }
        tc_fence_before();
        __syncthreads();
        // ---- elimination of [I + G | W^T | Y_hat]: Z^T, P and beta, and round 4's tiles ----
        eliminate_rhs64(g32, w32, y32, reinterpret_cast<float *>(work), s_beta, kn_sb, work, ebar,
                        (uint32_t)(sb & 1), a, abort_flag);
        fence_proxy_async_smem();
        __syncthreads();
        // ---- R4: D1[k rows] += E'^T Z^T (A MN-major, atoms [-(beta Z)^T | E']: M = 128,
        // the first 64 rows land in D1's dead W rows); A += -(Z diag(beta)) Z^T with
        // three-way splits (parts i + j <= 2) ----
        if (tid == 0) {
            tc_fence_after();
            mma_k64x3<true, true>(tbase + col_d1, smem_u32(bz0), smem_u32(bz1), smem_u32(zt0), smem_u32(zt1),
                                  idesc_bf16_f32(128, 64), true, kTile, 16);
            constexpr uint32_t id64 = idesc_bf16_f32(64, 64);
            mma_k64<true, true>(tbase + col_d5, smem_u32(bz0), smem_u32(zt0), id64, true);
            mma_k64<true, true>(tbase + col_d5, smem_u32(bz0), smem_u32(zt1), id64, true);
            mma_k64<true, true>(tbase + col_d5, smem_u32(bz1), smem_u32(zt0), id64, true);
            mma_k64<true, true>(tbase + col_d5, smem_u32(bz0), smem_u32(zt2), id64, true);
            mma_k64<true, true>(tbase + col_d5, smem_u32(bz1), smem_u32(zt1), id64, true);
            mma_k64<true, true>(tbase + col_d5, smem_u32(bz2), smem_u32(zt0), id64, true);
            umma_commit(bar);
        }
        // the next sub-block's key norms while round 4 runs (its copy has landed by now)
        if (sb + 1 < nsb) norms_in(sb + 1);
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
                uint4 *dst = reinterpret_cast<uint4 *>(galpha + (size_t)(sb * kSB + t) * kD + 32 * hw);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float e[8];
#pragma unroll
                    for (int m = 0; m < 8; ++m) e[m] = g[8 * q + m] * sc;
                    dst[q] = pack8_h(e);
                }
            }
        }
    }
    if (!ok) {
        if (tid == 0) (void)mbar_wait_bounded(bar, phase ^ 1u, a.p.wait_limit_ns, a.p.err);
        // a copy issued for a sub-block that was never reached lands before the CTA ends
        if (tid == 0 && tma_issued >= 0) (void)mbar_wait_bounded(tbar, (uint32_t)(tma_issued & 1), a.p.wait_limit_ns, a.p.err);
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
    if (tid == 0) {  // (a later job of this CTA may lay out its memory otherwise)
        mbar_inval(bar);
        for (int b = 0; b < 16; ++b) mbar_inval(&ebar[b]);
        mbar_inval(tbar);
    }
}

}  // namespace g64
}  // namespace vla
