// vla_gates_tc128.cuh -- the unit gates of "Variational Linear Attention:
// Stable Associative Memory for Long-Context Transformers" (section 2.2's
// inverse penalty A, kept by Sherman-Morrison, and section 2.3's gate
// alpha_t = A_t k_hat_t / |A_t k_hat_t|) on the tensor cores for d = 128 with
// bf16 I/O, when every (b, h) unit is one chunk: one CTA walks a unit's whole
// stream from its initial A, 64 tokens at a time in block-Woodbury form.
//
// The algebra is that of the d = 64 gates (vla_gates_tc.cu): for a sub-block
// of c = 64 tokens with A (d x d) at its start, U, K (d x c):
//   W = A U, G = U^T W (c x c), I + G = L D L^T (unit lower L),
//   z_s = A_{s-1} u_s = (W L^{-T})[:, s], beta_s = 1 / D_s,
//   A_t k_hat_t = A k_hat_t - sum_{s <= t} beta_s z_s (z_s . k_hat_t),
//   A_end = A - Z diag(beta) Z^T,
// with d = 128: every product over the features runs as two K = 64 halves,
// every operand that is 128 wide along M or N as two 64-wide atoms.
//   R1  D1 = [U; K] A               (M = 128 tokens, N = 128, K = 128; A in three
//                                    bf16 parts)
//   R2  D2 = U [A K ; W]^T          (M = 64, N = 128: Y | G; AK and W in three parts)
//   CUDA cores, fp32: forward elimination of [I + G | W^T | Y_hat] gives
//       Z^T, P = L^{-1} Y_hat (z_s . k_hat_t) and beta
//   R4  D1[k rows] += E'^T Z^T      (E'[s][t] = -beta_s P[s][t] |k_t|, s <= t)
//       A += -(Z diag(beta)) Z^T    (three-way bf16 splits: the downdate
//                                    accumulates over the whole stream)
// A stays in fp32 in TMEM (M = 128, 128 columns).  TMEM 384 columns and
// ~196 KB of shared memory: one CTA per SM.
// Precision: a whole stream is one chunk, so the downdates of A accumulate
// over all its sub-blocks, and early in a stream (A_0 = I / lambda0 large
// against the updates) each one is a small difference of large terms.  The
// operands that carry A into the gates and into the next A (A itself in R1,
// AK and W in R2, Z in the downdate) are therefore split in three bf16 parts
// (about 2^-24 relative, with U and K exact); E' and Z in R4's gate product
// keep two.
// The body of one CTA's work for one unit, included by vla_tc128.cu.
#pragma once

#include "vla_tma.cuh"

namespace vla {
namespace g128 {

using namespace tc;

constexpr int kD2 = 128;
constexpr int kThreads = 256;
constexpr int kWS = 132;  // row stride (floats) of the fp32 W^T staging: conflict-free rows

struct G2Layout {
    static constexpr size_t ctrl = 0;                 // mbarrier, TMEM slot, abort flag
    static constexpr size_t uk = 1024;                // [U; K] features 0..63, then 64..127 (128 rows each)
    static constexpr size_t ah = uk + 4 * kTile;      // A: hi f0, hi f1, lo f0, lo f1 (128 rows each)
    static constexpr size_t work = ah + 8 * kTile;    // work area, by phase:
    // before R1: A part 2 (f0, f1) @kW32 (parts 0, 1 in the A tiles)
    // R1 -> R2: [AK; W] part 0 f0 @0, f1 @16K, part 1 f0 @32K, f1 @48K (128 rows each),
    //           part 2 over the A tiles (f0 @ah, f1 @ah + 16K), W^T fp32 @kW32
    // R2 -> elimination: Y_hat fp32 @0, I + G fp32 @kG32, W^T fp32 @kW32
    // elimination: published rows @kPub (2 x 8 x 256 floats), scaled rows @kSrow
    // R4: -(beta Z)^T part 0 @0, part 1 @16K (two atoms 8 KB apart each), E' part 0
    //     @32K, part 1 @48K; Z^T parts 0, 1, 2 and -(beta Z)^T part 2 over the A tiles
    static constexpr size_t kW32 = 8 * kTile;
    static constexpr size_t kG32 = (size_t)64 * kGS * 4;
    static constexpr size_t kPub = 2 * kG32;
    static constexpr size_t kSrow = kPub + (size_t)2 * 8 * 256 * 4;
    static constexpr size_t work_bytes = kW32 + (size_t)64 * kWS * 4;
    static constexpr size_t ksc = work + work_bytes;  // [2][64] 1 / max(|k|, eps) (by sub-block parity)
    static constexpr size_t kn = ksc + 512;           // [2][64] max(|k|, eps)
    static constexpr size_t beta = kn + 512;          // [64]
    static constexpr size_t nrm = beta + 256;         // [2][64] halves of |row|^2
    static constexpr size_t total = nrm + 512;
};
static_assert(G2Layout::work % 1024 == 0, "operand tiles must be 1024-byte aligned");
static_assert(G2Layout::kSrow + 2 * 8 * 64 * 4 <= G2Layout::kW32, "elimination scratch fits below W^T");
static_assert(G2Layout::total + 1024 <= 227 * 1024, "one CTA per SM");

__device__ __forceinline__ void split3_pair2(float a, float b, uint32_t &p0, uint32_t &p1, uint32_t &p2) {
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

// Three bf16 parts of 32 consecutive fp32 values into row `row`, columns
// k0 .. k0 + 31, of three tiles.
__device__ __forceinline__ void put_row32x3(unsigned char *t0, unsigned char *t1, unsigned char *t2, int row, int k0,
                                            const float *v) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint32_t w0[4], w1[4], w2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split3_pair2(v[8 * g + 2 * e], v[8 * g + 2 * e + 1], w0[e], w1[e], w2[e]);
        const uint32_t o = toff(row, k0 + 8 * g);
        *reinterpret_cast<uint4 *>(t0 + o) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
        *reinterpret_cast<uint4 *>(t1 + o) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
        *reinterpret_cast<uint4 *>(t2 + o) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
    }
}

// Forward elimination of [I + G | W^T | Y_hat] (64 rows s; I + G and Y_hat
// with row stride kGS, W^T with row stride kWS), without pivoting, blocked by
// 8 pivots exactly as in the d = 64 gates (warp w owns rows 8 w .. 8 w + 7;
// lane l holds columns 2 l, 2 l + 1 of I + G and of Y_hat, and features
// 2 l, 2 l + 1 and 64 + 2 l, 64 + 2 l + 1 of W^T).  Afterwards it writes
// round 4's operand tiles (rows s): Z^T and -(beta Z)^T in three bf16 parts
// (two 64-feature atoms each), E' in two.  256 threads; all must call.
__device__ __forceinline__ void eliminate_rhs128(const float *gs, const float *w32, const float *y32, float *prow,
                                                 float *srow, float *rpiv, const float *kn, unsigned char *const *zt,
                                                 unsigned char *const *bz, unsigned char *const *ep) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float2 m[8], za[8], zb[8], pp[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 8 * warp + i;
        m[i] = *reinterpret_cast<const float2 *>(gs + r * kGS + 2 * lane);
        za[i] = *reinterpret_cast<const float2 *>(w32 + r * kWS + 2 * lane);
        zb[i] = *reinterpret_cast<const float2 *>(w32 + r * kWS + 64 + 2 * lane);
        pp[i] = *reinterpret_cast<const float2 *>(y32 + r * kGS + 2 * lane);
    }
    __syncthreads();  // the staging may be overwritten once everyone has its rows
#pragma unroll 1
    for (int b = 0; b < 8; ++b) {
        float *pb = prow + (b & 1) * 8 * 256;
        float *sb = srow + (b & 1) * 8 * 64;
        if (warp == b) {
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const float pv = __shfl_sync(0xffffffffu, (p & 1) ? m[p].y : m[p].x, 4 * b + (p >> 1));
                // fast reciprocal: the pivots of I + G are >= 1
                const float rp = __fdividef(1.f, pv);
                if (lane == 0) rpiv[8 * b + p] = rp;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (i <= p) continue;
                    const float mv = __shfl_sync(0xffffffffu, (i & 1) ? m[p].y : m[p].x, 4 * b + (i >> 1));
                    const float2 f = make_float2(-mv * rp, -mv * rp);
                    m[i] = __ffma2_rn(f, m[p], m[i]);
                    za[i] = __ffma2_rn(f, za[p], za[i]);
                    zb[i] = __ffma2_rn(f, zb[p], zb[i]);
                    pp[i] = __ffma2_rn(f, pp[p], pp[i]);
                }
                *reinterpret_cast<float2 *>(pb + p * 256 + 2 * lane) = m[p];
                *reinterpret_cast<float2 *>(pb + p * 256 + 64 + 2 * lane) = za[p];
                *reinterpret_cast<float2 *>(pb + p * 256 + 128 + 2 * lane) = zb[p];
                *reinterpret_cast<float2 *>(pb + p * 256 + 192 + 2 * lane) = pp[p];
                *reinterpret_cast<float2 *>(sb + p * 64 + 2 * lane) = __fmul2_rn(m[p], make_float2(-rp, -rp));
            }
        }
        __syncthreads();
        if (warp > b) {
            const uint32_t nbar = 32u * (uint32_t)(7 - b);
            if (warp > b + 1) asm volatile("bar.sync 1, %0;" ::"r"(nbar) : "memory");
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const float4 fa = *reinterpret_cast<const float4 *>(sb + p * 64 + 8 * warp);
                const float4 fb = *reinterpret_cast<const float4 *>(sb + p * 64 + 8 * warp + 4);
                const float2 pm = *reinterpret_cast<const float2 *>(pb + p * 256 + 2 * lane);
                const float2 pa = *reinterpret_cast<const float2 *>(pb + p * 256 + 64 + 2 * lane);
                const float2 pz = *reinterpret_cast<const float2 *>(pb + p * 256 + 128 + 2 * lane);
                const float2 py = *reinterpret_cast<const float2 *>(pb + p * 256 + 192 + 2 * lane);
                const float fr[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 fi = make_float2(fr[i], fr[i]);
                    m[i] = __ffma2_rn(fi, pm, m[i]);
                    za[i] = __ffma2_rn(fi, pa, za[i]);
                    zb[i] = __ffma2_rn(fi, pz, zb[i]);
                    pp[i] = __ffma2_rn(fi, py, pp[i]);
                }
            }
            if (warp == b + 1) asm volatile("bar.arrive 1, %0;" ::"r"(nbar) : "memory");
        }
    }
    __syncthreads();  // the tiles below overwrite the staging and the pivot scratch
    const float2 knt = *reinterpret_cast<const float2 *>(kn + 2 * lane);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int s = 8 * warp + i;
        const float bs = rpiv[s];
        const uint32_t o = toff(s, 2 * lane);
        uint32_t w0, w1, w2;
        // features 2 l, 2 l + 1 (atom 0) and 64 + 2 l, 64 + 2 l + 1 (atom 1, 8 KB on)
        split3_pair2(za[i].x, za[i].y, w0, w1, w2);
        *reinterpret_cast<uint32_t *>(zt[0] + o) = w0;
        *reinterpret_cast<uint32_t *>(zt[1] + o) = w1;
        *reinterpret_cast<uint32_t *>(zt[2] + o) = w2;
        split3_pair2(zb[i].x, zb[i].y, w0, w1, w2);
        *reinterpret_cast<uint32_t *>(zt[0] + kTile + o) = w0;
        *reinterpret_cast<uint32_t *>(zt[1] + kTile + o) = w1;
        *reinterpret_cast<uint32_t *>(zt[2] + kTile + o) = w2;
        split3_pair2(-bs * za[i].x, -bs * za[i].y, w0, w1, w2);
        *reinterpret_cast<uint32_t *>(bz[0] + o) = w0;
        *reinterpret_cast<uint32_t *>(bz[1] + o) = w1;
        *reinterpret_cast<uint32_t *>(bz[2] + o) = w2;
        split3_pair2(-bs * zb[i].x, -bs * zb[i].y, w0, w1, w2);
        *reinterpret_cast<uint32_t *>(bz[0] + kTile + o) = w0;
        *reinterpret_cast<uint32_t *>(bz[1] + kTile + o) = w1;
        *reinterpret_cast<uint32_t *>(bz[2] + kTile + o) = w2;
        const float ex = (2 * lane >= s) ? -bs * pp[i].x * knt.x : 0.f;
        const float ey = (2 * lane + 1 >= s) ? -bs * pp[i].y * knt.y : 0.f;
        split3_pair2(ex, ey, w0, w1, w2);
        *reinterpret_cast<uint32_t *>(ep[0] + o) = w0;
        *reinterpret_cast<uint32_t *>(ep[1] + o) = w1;
    }
}

// The gates of unit bh, by one CTA of kThreads threads with G2Layout::total +
// 1024 bytes of dynamic shared memory at smem_raw.
__device__ __forceinline__ void gates_tc128_body(const ChunkArgs &a, int bh, unsigned char *smem_raw,
                                                 const CUtensorMap *tm_u, const CUtensorMap *tm_k) {
    using L = G2Layout;
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::ctrl);
    uint64_t *tbar = reinterpret_cast<uint64_t *>(smem + L::ctrl + 64);  // [U; K] tensor copies
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L::ctrl + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::ctrl + 12);
    unsigned char *uk = smem + L::uk;  // + 2 kTile * h: features 64 h ..
    unsigned char *ah = smem + L::ah;  // hi f0, hi f1, lo f0, lo f1 at 2 kTile steps
    unsigned char *work = smem + L::work;
    float *s_ks = reinterpret_cast<float *>(smem + L::ksc);
    float *s_kn = reinterpret_cast<float *>(smem + L::kn);
    float *s_beta = reinterpret_cast<float *>(smem + L::beta);
    float *s_nrm = reinterpret_cast<float *>(smem + L::nrm);
    float *w32 = reinterpret_cast<float *>(work + L::kW32);
    float *g32 = reinterpret_cast<float *>(work + L::kG32);
    float *y32 = reinterpret_cast<float *>(work);
    unsigned char *const a2 = work + L::kW32;  // A part 2: f0, f1 (16 KB each)
    unsigned char *const zt[3] = {ah, ah + 2 * kTile, ah + 4 * kTile};
    unsigned char *const bz[3] = {work, work + 2 * kTile, ah + 6 * kTile};
    unsigned char *const ep[2] = {work + 4 * kTile, work + 6 * kTile};

    const int T = a.p.T;
    const int nsb = (T + kSB - 1) / kSB;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int qw = warp & 3, hw = warp >> 2;                // TMEM lane quarter, column half
    const int pt = 8 * warp + (lane & 7), pq = lane >> 3;  // staging: token, feature quarter (32 features)
    const int r64 = 16 * qw + lane;                         // row in an M = 64 accumulator (lanes < 16)
    const bool act64 = lane < 16;
    const int r128 = 32 * qw + lane;                        // row in an M = 128 accumulator
    const size_t tok0 = (size_t)bh * T * kD2;
    __half *galpha = reinterpret_cast<__half *>(static_cast<unsigned char *>(a.p.ws) + a.L.off_alpha) + tok0;

    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(tbar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0) tmem_alloc(tslot, 512, false);  // (one CTA per SM; a queue CTA allocates per job)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t tq = tbase + ((uint32_t)(32 * qw) << 16);  // this warp's lane quarter
    constexpr uint32_t col_a = 0, col_d1 = 128, col_d2 = 256;

    // [U; K] of sub-block sb by four tiled tensor copies (U, then K, of features
    // 0..63, then of 64..127) into the two feature tiles; the maps fill tokens
    // past T with zeros.  Thread 0 issues; the copies of sub-block sb complete
    // phase sb mod 2 of tbar.
    int tma_issued = -1;  // (thread 0's bookkeeping) the last sub-block whose copies were issued
    auto issue_in = [&](int sb) {
        mbar_arrive_expect_tx(tbar, 4 * kTile);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            tma_load_3d(uk + 2 * kTile * h, tm_u, 64 * h, sb * kSB, bh, tbar);
            tma_load_3d(uk + 2 * kTile * h + kTile, tm_k, 64 * h, sb * kSB, bh, tbar);
        }
        tma_issued = sb;
    };
    if (tid == 0 && nsb > 0) issue_in(0);  // lands while A0 is set up

    // ---- A at the start (A0, or I / lambda0): fp32 in TMEM, bf16 hi/lo tiles ----
    {
        const float il = 1.f / a.p.lambda0;
        const float *src = a.p.A0 ? a.p.A0 + (size_t)bh * kD2 * kD2 + (size_t)r128 * kD2 : nullptr;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int c0 = 64 * hw + 32 * half;
            float am[32];
            if (src) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 v = reinterpret_cast<const float4 *>(src + c0)[q];
                    am[4 * q] = v.x; am[4 * q + 1] = v.y; am[4 * q + 2] = v.z; am[4 * q + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) am[j] = (c0 + j == r128) ? il : 0.f;
            }
            tmem_st32(tq + col_a + c0, am);
            put_row32x3(ah + 2 * kTile * hw, ah + 2 * kTile * hw + 4 * kTile, a2 + 2 * kTile * hw, r128, 32 * half,
                        am);
        }
        tc_fence_before();
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
    // the key norms of sub-block sb, from its K rows once its copies have landed,
    // into the sb-parity halves
    auto norms_in = [&](int sb) {
        if (!mbar_wait_bounded(tbar, (uint32_t)(sb & 1), a.p.wait_limit_ns, a.p.err)) *abort_flag = 1;
        const unsigned char *tile = uk + 2 * kTile * (pq >> 1);
        const int k0 = 32 * (pq & 1);
        float ss = 0.f;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const uint4 rk = *reinterpret_cast<const uint4 *>(tile + toff(64 + pt, k0 + 8 * h));
            float kf[8];
            unpack8(rk, kf);
#pragma unroll
            for (int m = 0; m < 8; ++m) ss = fmaf(kf[m], kf[m], ss);
        }
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
    fence_proxy_async_smem();
    __syncthreads();
    constexpr uint32_t id_r1 = idesc_bf16_f32(128, 128);
    constexpr uint32_t id_r2 = idesc_bf16_f32(64, 128);
    for (int sb = 0; sb < nsb; ++sb) {
        const int nt = min(kSB, T - sb * kSB);
        const float *kn_sb = s_kn + 64 * (sb & 1), *ks_sb = s_ks + 64 * (sb & 1);
        // ---- R1: D1 = [U; K] A (M = 128, N = 128, two feature halves, A as hi + lo) ----
        if (tid == 0) {
            tc_fence_after();
            mma_k64<false, false>(tbase + col_d1, smem_u32(uk), smem_u32(ah), id_r1, false);
            mma_k64<false, false>(tbase + col_d1, smem_u32(uk + 2 * kTile), smem_u32(ah + 2 * kTile), id_r1, true);
            mma_k64<false, false>(tbase + col_d1, smem_u32(uk), smem_u32(ah + 4 * kTile), id_r1, true);
            mma_k64<false, false>(tbase + col_d1, smem_u32(uk + 2 * kTile), smem_u32(ah + 6 * kTile), id_r1, true);
            mma_k64<false, false>(tbase + col_d1, smem_u32(uk), smem_u32(a2), id_r1, true);
            mma_k64<false, false>(tbase + col_d1, smem_u32(uk + 2 * kTile), smem_u32(a2 + 2 * kTile), id_r1, true);
            umma_commit(bar);
        }
        if (!round_wait()) {
            ok = false;
            break;
        }
        // ---- [AK; W] operand tiles (AK rows first), W^T in fp32 for the elimination ----
        {
            // row r128 of D1: W row t = r128 (r128 < 64) or AK row t = r128 - 64, features 64 hw ..
            const int t = r128 & 63;
            const int trow = r128 < 64 ? 64 + t : t;
            unsigned char *t0 = work + 2 * kTile * hw, *t1 = work + 4 * kTile + 2 * kTile * hw;
            unsigned char *t2 = ah + 2 * kTile * hw;  // (the A tiles are free once R1 is done)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float v[32];
                tmem_ld32(tq + col_d1 + 64 * hw + 32 * half, v);
                put_row32x3(t0, t1, t2, trow, 32 * half, v);
                if (r128 < 64) {
                    float4 *dst = reinterpret_cast<float4 *>(w32 + t * kWS + 64 * hw + 32 * half);
#pragma unroll
                    for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
            }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();
        // ---- R2: D2 = U [AK; W]^T (M = 64, N = 128): Y | G ----
        if (tid == 0) {
            tc_fence_after();
            mma_k64<false, false>(tbase + col_d2, smem_u32(uk), smem_u32(work), id_r2, false);
            mma_k64<false, false>(tbase + col_d2, smem_u32(uk + 2 * kTile), smem_u32(work + 2 * kTile), id_r2, true);
            mma_k64<false, false>(tbase + col_d2, smem_u32(uk), smem_u32(work + 4 * kTile), id_r2, true);
            mma_k64<false, false>(tbase + col_d2, smem_u32(uk + 2 * kTile), smem_u32(work + 6 * kTile), id_r2, true);
            mma_k64<false, false>(tbase + col_d2, smem_u32(uk), smem_u32(ah), id_r2, true);
            mma_k64<false, false>(tbase + col_d2, smem_u32(uk + 2 * kTile), smem_u32(ah + 2 * kTile), id_r2, true);
            umma_commit(bar);
        }
        if (!round_wait()) {
            ok = false;
            break;
        }
        // round 2 has read [U; K]: the next sub-block's copies land during the elimination
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
        // ---- elimination: Z^T, P, beta and round 4's tiles ----
        eliminate_rhs128(g32, w32, y32, reinterpret_cast<float *>(work + L::kPub),
                         reinterpret_cast<float *>(work + L::kSrow), s_beta, kn_sb, zt, bz, ep);
        fence_proxy_async_smem();
        __syncthreads();
        // ---- R4: D1[k rows] += E'^T Z^T (A MN-major, atoms [-(beta Z)^T f0 | E'] 32 KB apart: the
        // first 64 rows land in D1's dead W rows; B MN-major, two feature atoms 8 KB apart);
        // A += -(Z diag(beta)) Z^T with three-way splits (parts i + j <= 2) ----
        if (tid == 0) {
            tc_fence_after();
            mma_k64x3<true, true>(tbase + col_d1, smem_u32(bz[0]), smem_u32(bz[1]), smem_u32(zt[0]), smem_u32(zt[1]),
                                  id_r1, true, 4 * kTile, kTile);
            mma_k64<true, true>(tbase + col_a, smem_u32(bz[0]), smem_u32(zt[0]), id_r1, true, kTile, kTile);
            mma_k64<true, true>(tbase + col_a, smem_u32(bz[0]), smem_u32(zt[1]), id_r1, true, kTile, kTile);
            mma_k64<true, true>(tbase + col_a, smem_u32(bz[1]), smem_u32(zt[0]), id_r1, true, kTile, kTile);
            mma_k64<true, true>(tbase + col_a, smem_u32(bz[0]), smem_u32(zt[2]), id_r1, true, kTile, kTile);
            mma_k64<true, true>(tbase + col_a, smem_u32(bz[1]), smem_u32(zt[1]), id_r1, true, kTile, kTile);
            mma_k64<true, true>(tbase + col_a, smem_u32(bz[2]), smem_u32(zt[0]), id_r1, true, kTile, kTile);
            umma_commit(bar);
        }
        if (sb + 1 < nsb) norms_in(sb + 1);  // its copies have landed by now
        if (!round_wait()) {
            ok = false;
            break;
        }
        // ---- gates and the A update ----
        {
            const int t = r128 - 64;
            float sq = 0.f;
            float g[2][32];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tmem_ld32(tq + col_d1 + 64 * hw + 32 * half, g[half]);  // rows 64 + t: |k_t| A_t k_hat_t
#pragma unroll
                for (int m = 0; m < 32; ++m) sq = fmaf(g[half][m], g[half][m], sq);
            }
            if (qw >= 2) s_nrm[hw * 64 + t] = sq;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float v[32];
                tmem_ld32(tq + col_a + 64 * hw + 32 * half, v);  // the updated A, row r128
                put_row32x3(ah + 2 * kTile * hw, ah + 4 * kTile + 2 * kTile * hw, a2 + 2 * kTile * hw, r128,
                            32 * half, v);
            }
            tc_fence_before();
            fence_proxy_async_smem();
            __syncthreads();
            if (qw >= 2 && t < nt) {
                const float nr = sqrtf(s_nrm[t] + s_nrm[64 + t]);
                const float sc = 1.f / fmaxf(nr, kEps * kn_sb[t]);
                uint4 *dst = reinterpret_cast<uint4 *>(galpha + (size_t)(sb * kSB + t) * kD2 + 64 * hw);
#pragma unroll
                for (int half = 0; half < 2; ++half)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float e[8];
#pragma unroll
                        for (int m = 0; m < 8; ++m) e[m] = g[half][8 * q + m] * sc;
                        dst[4 * half + q] = pack8_h(e);
                    }
            }
        }
    }
    if (!ok) {
        if (tid == 0) (void)mbar_wait_bounded(bar, phase ^ 1u, a.p.wait_limit_ns, a.p.err);
        // copies issued for a sub-block that was never reached land before the CTA ends
        if (tid == 0 && tma_issued >= 0) (void)mbar_wait_bounded(tbar, (uint32_t)(tma_issued & 1), a.p.wait_limit_ns, a.p.err);
    } else {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float am[32];
            tmem_ld32(tq + col_a + 64 * hw + 32 * half, am);
            float4 *dA = reinterpret_cast<float4 *>(a.p.A_T + (size_t)bh * kD2 * kD2 + (size_t)r128 * kD2 + 64 * hw +
                                                    32 * half);
#pragma unroll
            for (int q = 0; q < 8; ++q) dA[q] = make_float4(am[4 * q], am[4 * q + 1], am[4 * q + 2], am[4 * q + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
    if (tid == 0) {  // (a later job of this CTA may lay out its memory otherwise)
        mbar_inval(bar);
        mbar_inval(tbar);
    }
}

}  // namespace g128
}  // namespace vla
