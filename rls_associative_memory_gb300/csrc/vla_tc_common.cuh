// vla_tc_common.cuh -- operand tiles and tcgen05 helpers shared by the
// tensor-core passes of the chunk-parallel path (d = 64, bf16 I/O).
#pragma once

#include "vla_internal.cuh"

namespace vla {
namespace tc {

constexpr int kD = 64;        // head dimension of this path
constexpr int kSB = 64;       // tokens per sub-block
constexpr int kTile = 8192;   // bytes of a 64-row, 64-column bf16 operand tile

// Operand tiles: 64 bf16 (128 bytes) per row, rows 128 bytes apart, in the
// 128-byte swizzle: the 16-byte chunk j of row r sits at chunk j ^ (r mod 8)
// (tiles start on 1024-byte boundaries).  Read K-major (row = M/N index,
// 8-row groups SBO = 1024 bytes apart, a K-step of 16 advances 32 bytes) or
// MN-major (row = K index, a K-step of 16 advances two row groups, 2048
// bytes).  The swizzle keeps both the tensor core's reads and the row-wise
// 16-byte stores here free of bank conflicts.
__device__ __forceinline__ uint32_t toff(int r, int k) {
    return (uint32_t)(r * 128 + ((((k >> 3) ^ (r & 7)) << 4) | ((k & 7) * 2)));
}

// Shared-memory descriptor of a tile in that layout: start address, LBO
// (the distance between 64-element atoms of an MN-major operand; unused by
// K-major reads), SBO 1024 bytes, descriptor version of the sm_100 family,
// 128-byte swizzle.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo = 16) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// phi(x) = ELU(x) + 1 with the fast exponential (bf16 I/O only: its relative
// error, about 2^-21, is far below the output rounding).
__device__ __forceinline__ float phi_fast(float x) { return x > 0.f ? x + 1.f : __expf(x); }


__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 h) { return *reinterpret_cast<uint32_t *>(&h); }

// bf16 pairs (hi, lo) of 8 consecutive fp32 values, in element order.
__device__ __forceinline__ void split8(const float *x, uint4 &hi, uint4 &lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 hb = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
        const float2 hf = __bfloat1622float2(hb);
        h[e] = bf2_bits(hb);
        l[e] = bf2_bits(__floats2bfloat162_rn(x[2 * e] - hf.x, x[2 * e + 1] - hf.y));
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// The unit gates between the gates and the state pass travel as fp16: their
// components lie in [-1, 1], where fp16 keeps 11 significant bits (bf16: 8),
// and an fp16 value is exactly a bf16 pair (hi, lo), so the state pass's split
// products see the stored gate without further rounding.
__device__ __forceinline__ uint4 pack8_h(const float *x) {
    uint32_t h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __half2 v = __floats2half2_rn(x[2 * e], x[2 * e + 1]);
        h[e] = *reinterpret_cast<const uint32_t *>(&v);
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

__device__ __forceinline__ void unpack8_h(uint4 w, float *x) {
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&a[e]));
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
    }
}

__device__ __forceinline__ void unpack8(uint4 w, float *x) {
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(a[e] << 16);
        x[2 * e + 1] = __uint_as_float(a[e] & 0xffff0000u);
    }
}

// 32 consecutive fp32 values as (hi, lo) into row `row`, columns k0 .. k0+31.
__device__ __forceinline__ void put_row32(unsigned char *hi, unsigned char *lo, int row, int k0, const float *v) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint4 h, l;
        split8(v + 8 * g, h, l);
        *reinterpret_cast<uint4 *>(hi + toff(row, k0 + 8 * g)) = h;
        *reinterpret_cast<uint4 *>(lo + toff(row, k0 + 8 * g)) = l;
    }
}

// 32 consecutive TMEM columns of this warp's lane quarter (shape 32x32b).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// 32 consecutive TMEM columns of this warp's lane quarter from registers
// (shape 32x32b), waiting until the stores are done.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D (+)= A B^T over K = 64 (four K-steps of 16).  A (M rows) and B (N
// rows) are tiles in the layout above, read K-major, or MN-major when A_MN /
// B_MN (tile rows are then K and each row runs along M / N).  An MN-major
// operand wider than 64 takes its next 64-wide atom lbo bytes further on.
template <bool A_MN, bool B_MN>
__device__ __forceinline__ void mma_k64(uint32_t d, uint32_t a, uint32_t b, uint32_t idesc, bool acc,
                                        uint32_t lbo_a = 16, uint32_t lbo_b = 16) {
    // descriptor address fields count 16-byte units: a K-step adds 32 bytes
    // (K-major) or 2048 bytes (MN-major) to the start address
    const uint64_t ad = desc_sw128(a, lbo_a), bd = desc_sw128(b, lbo_b);
    const uint32_t id = idesc | (A_MN ? (1u << 15) : 0u) | (B_MN ? (1u << 16) : 0u);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
        umma_bf16(d, ad + (uint64_t)((A_MN ? 128 : 2) * ks), bd + (uint64_t)((B_MN ? 128 : 2) * ks), id,
                  (acc || ks > 0) ? 1u : 0u);
}

// Split product D (+)= (Ah + Al)(Bh + Bl)^T without the lo*lo term.
template <bool A_MN, bool B_MN>
__device__ __forceinline__ void mma_k64x3(uint32_t d, uint32_t ah, uint32_t al, uint32_t bh, uint32_t bl,
                                          uint32_t idesc, bool acc, uint32_t lbo_a = 16, uint32_t lbo_b = 16) {
    mma_k64<A_MN, B_MN>(d, ah, bh, idesc, acc, lbo_a, lbo_b);
    mma_k64<A_MN, B_MN>(d, ah, bl, idesc, true, lbo_a, lbo_b);
    mma_k64<A_MN, B_MN>(d, al, bh, idesc, true, lbo_a, lbo_b);
}

constexpr int kGS = 68;  // row stride (floats) of fp32 staging matrices: conflict-free rows

// Gaussian elimination of a 64 x 64 SPD matrix M against the identity,
// without pivoting (the pivots of an SPD matrix are positive): with
// M = L D L^T (unit lower L), it yields E = L^{-1} and the reciprocal pivots
// 1 / D_s.  M is symmetric and stays so in the trailing block, so the
// multiplier of row t for pivot s, M[t][s] / D_s, is the pivot row's entry
// M[s][t] / D_s.  Blocked by 8 pivots: warp w owns rows 8 w .. 8 w + 7 (lane l
// columns 2 l, 2 l + 1).  The owner of a block eliminates it with shuffles and
// publishes its 8 pivot rows of M and E, and the rows of M scaled by -1 / D_s
// that carry the later rows' multipliers (double-buffered); after one barrier
// every later warp applies all 8.  The next owner applies first: the other
// warps wait for it on a named barrier, then apply while it runs its own
// pivot chain, which leaves most issue slots free.  256 threads; all must
// call.
//   ms:   M (fp32, row stride kGS), read once at the start
//   prow: scratch, 2 x 8 x 128 floats (pivot rows of M and E)
//   srow: scratch, 2 x 8 x 64 floats (pivot rows of M scaled by -1 / D_s)
//   rpiv: out, 1 / D_s
//   e_hi, e_lo: out, E as bf16 hi/lo tile pairs (row s, column r)
//   be_hi, be_lo: optional out, diag(1 / D) E likewise (rows scaled)
__device__ __forceinline__ void eliminate64(const float *ms, float *prow, float *srow, float *rpiv,
                                            unsigned char *e_hi, unsigned char *e_lo, unsigned char *be_hi,
                                            unsigned char *be_lo) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float2 m[8], e[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 8 * warp + i;
        m[i] = *reinterpret_cast<const float2 *>(ms + r * kGS + 2 * lane);
        e[i] = make_float2(r == 2 * lane ? 1.f : 0.f, r == 2 * lane + 1 ? 1.f : 0.f);
    }
    __syncthreads();  // ms may be overwritten once everyone has its rows
#pragma unroll 1
    for (int b = 0; b < 8; ++b) {
        float *pb = prow + (b & 1) * 8 * 128;
        float *sb = srow + (b & 1) * 8 * 64;
        if (warp == b) {
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                // pivot M[s][s], s = 8 b + p: lane s / 2, component p mod 2
                const float pv = __shfl_sync(0xffffffffu, (p & 1) ? m[p].y : m[p].x, 4 * b + (p >> 1));
                // fast reciprocal: the pivots are >= the smallest eigenvalue (>= 1
                // for I + G) and its relative error (about 2^-22) is far below
                // the bf16 operand splits downstream
                const float rp = __fdividef(1.f, pv);
                if (lane == 0) rpiv[8 * b + p] = rp;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (i <= p) continue;  // (constant trip count: m, e stay in registers)
                    // multiplier of row 8 b + i: pivot row at column 8 b + i
                    const float mv = __shfl_sync(0xffffffffu, (i & 1) ? m[p].y : m[p].x, 4 * b + (i >> 1));
                    const float2 f = make_float2(-mv * rp, -mv * rp);
                    m[i] = __ffma2_rn(f, m[p], m[i]);
                    e[i] = __ffma2_rn(f, e[p], e[i]);
                }
                *reinterpret_cast<float2 *>(pb + p * 128 + 2 * lane) = m[p];
                *reinterpret_cast<float2 *>(pb + p * 128 + 64 + 2 * lane) = e[p];
                *reinterpret_cast<float2 *>(sb + p * 64 + 2 * lane) = __fmul2_rn(m[p], make_float2(-rp, -rp));
            }
        }
        __syncthreads();
        if (warp > b) {
            // warps after the next owner start once it has applied (named barrier 1:
            // the next owner arrives, the 6 - b warps after it wait)
            const uint32_t nbar = 32u * (uint32_t)(7 - b);
            if (warp > b + 1) asm volatile("bar.sync 1, %0;" ::"r"(nbar) : "memory");
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                // multipliers of this warp's rows: the scaled pivot row at their columns
                const float4 fa = *reinterpret_cast<const float4 *>(sb + p * 64 + 8 * warp);
                const float4 fb = *reinterpret_cast<const float4 *>(sb + p * 64 + 8 * warp + 4);
                const float2 pm = *reinterpret_cast<const float2 *>(pb + p * 128 + 2 * lane);
                const float2 pe = *reinterpret_cast<const float2 *>(pb + p * 128 + 64 + 2 * lane);
                const float fr[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 fi = make_float2(fr[i], fr[i]);
                    m[i] = __ffma2_rn(fi, pm, m[i]);
                    e[i] = __ffma2_rn(fi, pe, e[i]);
                }
            }
            if (warp == b + 1) asm volatile("bar.arrive 1, %0;" ::"r"(nbar) : "memory");
        }
    }
    // E (and diag(1/D) E) rows 8 warp + i, columns 2 lane, 2 lane + 1
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 8 * warp + i;
        const __nv_bfloat162 h = __floats2bfloat162_rn(e[i].x, e[i].y);
        const float2 hf = __bfloat1622float2(h);
        const __nv_bfloat162 l = __floats2bfloat162_rn(e[i].x - hf.x, e[i].y - hf.y);
        *reinterpret_cast<uint32_t *>(e_hi + toff(r, 2 * lane)) = bf2_bits(h);
        *reinterpret_cast<uint32_t *>(e_lo + toff(r, 2 * lane)) = bf2_bits(l);
        if (be_hi) {
            const float rp = rpiv[r];  // written by this warp as owner
            const float bx = e[i].x * rp, by = e[i].y * rp;
            const __nv_bfloat162 bh = __floats2bfloat162_rn(bx, by);
            const float2 bhf = __bfloat1622float2(bh);
            *reinterpret_cast<uint32_t *>(be_hi + toff(r, 2 * lane)) = bf2_bits(bh);
            *reinterpret_cast<uint32_t *>(be_lo + toff(r, 2 * lane)) =
                bf2_bits(__floats2bfloat162_rn(bx - bhf.x, by - bhf.y));
        }
    }
}

// One doubling level of tri_inv64: for each pair of consecutive diagonal
// blocks A, B of size Bk whose inverses T_A, T_B are already in place, the
// off-diagonal block of the inverse of the pair is T_AB = -T_A N_AB T_B,
// written over N_AB.  Step 1 forms M = N_AB T_B into scratch, step 2
// T_AB = -T_A M.  Thread t takes pair t / (8 Bk), row (t / 8) mod Bk and the
// E = Bk / 8 consecutive columns E (t mod 8); zero entries below the
// diagonal make every product a full sum (no divergent trip counts).  Four
// multipliers arrive in one 16-byte load, the rows they scale as float4 /
// float2 / float.
template <int E>
__device__ __forceinline__ void fma_row(float (&acc)[E], float m, const float *row) {
    if constexpr (E == 4) {
        const float4 r = *reinterpret_cast<const float4 *>(row);
        const float2 a = __ffma2_rn(make_float2(m, m), make_float2(r.x, r.y), make_float2(acc[0], acc[1]));
        const float2 b = __ffma2_rn(make_float2(m, m), make_float2(r.z, r.w), make_float2(acc[2], acc[3]));
        acc[0] = a.x; acc[1] = a.y; acc[2] = b.x; acc[3] = b.y;
    } else if constexpr (E == 2) {
        const float2 r = *reinterpret_cast<const float2 *>(row);
        const float2 a = __ffma2_rn(make_float2(m, m), r, make_float2(acc[0], acc[1]));
        acc[0] = a.x; acc[1] = a.y;
    } else {
        acc[0] = fmaf(m, row[0], acc[0]);
    }
}

template <int Bk>
__device__ __forceinline__ void tri_level(float *ts, float *ms) {
    constexpr int E = Bk / 8;   // columns per thread
    constexpr int MS = Bk + 4;  // scratch row stride (16-byte rows)
    const int t = threadIdx.x, j = t / (8 * Bk), i = (t >> 3) % Bk, c0 = E * (t & 7);
    const int a0 = 2 * j * Bk, b0 = a0 + Bk;
    float *mj = ms + j * Bk * MS;
    float acc[E];
#pragma unroll
    for (int q = 0; q < E; ++q) acc[q] = 0.f;
#pragma unroll
    for (int k = 0; k < Bk; k += 4) {
        const float4 n = *reinterpret_cast<const float4 *>(ts + (a0 + i) * kGS + b0 + k);
        fma_row<E>(acc, n.x, ts + (b0 + k) * kGS + b0 + c0);
        fma_row<E>(acc, n.y, ts + (b0 + k + 1) * kGS + b0 + c0);
        fma_row<E>(acc, n.z, ts + (b0 + k + 2) * kGS + b0 + c0);
        fma_row<E>(acc, n.w, ts + (b0 + k + 3) * kGS + b0 + c0);
    }
#pragma unroll
    for (int q = 0; q < E; ++q) mj[i * MS + c0 + q] = acc[q];
    __syncthreads();
#pragma unroll
    for (int q = 0; q < E; ++q) acc[q] = 0.f;
#pragma unroll
    for (int k = 0; k < Bk; k += 4) {
        const float4 ta = *reinterpret_cast<const float4 *>(ts + (a0 + i) * kGS + a0 + k);
        fma_row<E>(acc, ta.x, mj + k * MS + c0);
        fma_row<E>(acc, ta.y, mj + (k + 1) * MS + c0);
        fma_row<E>(acc, ta.z, mj + (k + 2) * MS + c0);
        fma_row<E>(acc, ta.w, mj + (k + 3) * MS + c0);
    }
#pragma unroll
    for (int q = 0; q < E; ++q) ts[(a0 + i) * kGS + b0 + c0 + q] = -acc[q];
    __syncthreads();
}

// The same level with 4 x 4 register blocks (used for Bk = 32, where the
// products are large enough to pay for the idle warps): thread t <
// (32 / Bk) (Bk / 4)^2 takes pair t / (Bk / 4)^2, rows 4 rg .. 4 rg + 3 and
// columns 4 cg .. 4 cg + 3 (cg fastest, so a quarter-warp reads one row of the
// right operand and broadcasts the left one) over the full sum; the other
// threads only join the barriers.
template <int Bk>
__device__ __forceinline__ void tri_level_blk(float *ts, float *ms) {
    constexpr int G = Bk / 4;       // row / column groups per block
    constexpr int MS = Bk + 4;      // scratch row stride (16-byte rows)
    const int t = threadIdx.x;
    const bool act = t < (32 / Bk) * G * G;
    const int j = t / (G * G), rg = (t / G) % G, cg = t % G;
    const int a0 = 2 * j * Bk, b0 = a0 + Bk, r0 = 4 * rg, c0 = 4 * cg;
    float *mj = ms + j * Bk * MS;
    float2 acc[4][2];
    if (act) {
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[r][0] = acc[r][1] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < Bk; k += 4) {
            float4 n[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) n[r] = *reinterpret_cast<const float4 *>(ts + (a0 + r0 + r) * kGS + b0 + k);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float4 tb = *reinterpret_cast<const float4 *>(ts + (b0 + k + kk) * kGS + b0 + c0);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float m = kk == 0 ? n[r].x : kk == 1 ? n[r].y : kk == 2 ? n[r].z : n[r].w;
                    acc[r][0] = __ffma2_rn(make_float2(m, m), make_float2(tb.x, tb.y), acc[r][0]);
                    acc[r][1] = __ffma2_rn(make_float2(m, m), make_float2(tb.z, tb.w), acc[r][1]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
            *reinterpret_cast<float4 *>(mj + (r0 + r) * MS + c0) =
                make_float4(acc[r][0].x, acc[r][0].y, acc[r][1].x, acc[r][1].y);
    }
    __syncthreads();
    if (act) {
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[r][0] = acc[r][1] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < Bk; k += 4) {
            float4 ta[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) ta[r] = *reinterpret_cast<const float4 *>(ts + (a0 + r0 + r) * kGS + a0 + k);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float4 mk = *reinterpret_cast<const float4 *>(mj + (k + kk) * MS + c0);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float m = kk == 0 ? ta[r].x : kk == 1 ? ta[r].y : kk == 2 ? ta[r].z : ta[r].w;
                    acc[r][0] = __ffma2_rn(make_float2(m, m), make_float2(mk.x, mk.y), acc[r][0]);
                    acc[r][1] = __ffma2_rn(make_float2(m, m), make_float2(mk.z, mk.w), acc[r][1]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
            *reinterpret_cast<float4 *>(ts + (a0 + r0 + r) * kGS + b0 + c0) =
                make_float4(-acc[r][0].x, -acc[r][0].y, -acc[r][1].x, -acc[r][1].y);
    }
    __syncthreads();
}

// T = (I + N)^{-1} for a strictly upper triangular 64 x 64 N by recursive
// doubling on the block structure: the inverse of [[I + N_A, N_AB], [0,
// I + N_B]] is [[T_A, -T_A N_AB T_B], [0, T_B]].  Each warp first inverts
// its own 8 x 8 diagonal block (lane c < 8 solves column c by back
// substitution, no barrier), then three levels join pairs of blocks
// 8 -> 16 -> 32 -> 64 with small products spread over all threads.  T is
// built in place over N.  256 threads; all must call.
//   ns:   in N, then T (fp32, row s, stride kGS; below-diagonal entries zero)
//   ms:   scratch, 32 x 36 floats (16-byte aligned)
//   t_hi, t_lo: out, T as bf16 hi/lo tile pairs, tile row s = row s of T
//               (an MN-major operand for products with T on the right); may
//               alias ns
__device__ __forceinline__ void tri_inv64(float *ns, float *ms, unsigned char *t_hi, unsigned char *t_lo) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    {   // diagonal block 8 warp .. 8 warp + 7: column c = lane of its inverse
        const int c = lane & 7;
        float col[8];
#pragma unroll
        for (int r = 7; r >= 0; --r) {
            const float4 n0 = *reinterpret_cast<const float4 *>(ns + (8 * warp + r) * kGS + 8 * warp);
            const float4 n1 = *reinterpret_cast<const float4 *>(ns + (8 * warp + r) * kGS + 8 * warp + 4);
            const float nr[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
            float acc = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int k = 7; k > r; --k) acc = fmaf(-nr[k], col[k], acc);  // col[r + 1] (the latest) last
            col[r] = acc;
        }
        __syncwarp();  // every lane has read the block's N before it is overwritten
        if (lane < 8) {
#pragma unroll
            for (int r = 0; r < 8; ++r) ns[(8 * warp + r) * kGS + 8 * warp + c] = col[r];
        }
    }
    __syncthreads();
    tri_level<8>(ns, ms);
    tri_level<16>(ns, ms);
    tri_level_blk<32>(ns, ms);
    // rows 8 warp + i, columns 2 lane, 2 lane + 1, as bf16 hi/lo
    float2 tr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) tr[i] = *reinterpret_cast<const float2 *>(ns + (8 * warp + i) * kGS + 2 * lane);
    __syncthreads();  // the output may alias ns
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 8 * warp + i;
        const __nv_bfloat162 h = __floats2bfloat162_rn(tr[i].x, tr[i].y);
        const float2 hf = __bfloat1622float2(h);
        *reinterpret_cast<uint32_t *>(t_hi + toff(r, 2 * lane)) = bf2_bits(h);
        *reinterpret_cast<uint32_t *>(t_lo + toff(r, 2 * lane)) =
            bf2_bits(__floats2bfloat162_rn(tr[i].x - hf.x, tr[i].y - hf.y));
    }
}

}  // namespace tc
}  // namespace vla
