// vla_backward128.cu -- gradients of the VLA forward recurrence at d = 128
// ("Variational Linear Attention: Stable Associative Memory for Long-Context
// Transformers", sections 2.2-2.3; the S transition J_t = I - alpha_t
// k_hat_t^T of section 3.1 is the S part of the adjoint).
//
// Same loss, records, checkpoints and per-token adjoint as the sequential
// backward at d = 32 and 64 (vla_backward.cu): phase 1 reruns the forward and
// stores per token k_hat, z, alpha, r and |k|, beta, |g|, 1/den, and every
// kBwdCk tokens the state; phase 2 walks the tokens backwards, rebuilding each
// previous state by undoing the rank-1 updates and re-anchoring it at the
// checkpoints.  At d = 128 four register-resident d x d states do not fit one
// CTA (512 threads x 128 floats, before any temporaries), so the states are
// split by where their transposed products fall:
//   - A and dA stay in registers: thread (row, part) holds row `row`, columns
//     [32 part, 32 part + 32).  A is symmetric, so A x needs no transpose;
//     the one transposed product of the A part, dA'^T z, goes through a
//     64 KB buffer written in row order and summed in column order.
//   - S and dS live in shared memory (fp32, 64 KB each).  Their 16-byte
//     chunks are XOR-swizzled so that both the four threads of a row (row
//     order) and a warp walking 32 columns of one row (column order) hit 32
//     distinct banks.  The S part of a reverse step is then two passes: one
//     in row order that only reads (S'_i . phi(q), dS_i . alpha), and one in
//     column order that undoes the state write, updates dS in place and forms
//     S'^T dnum, dS'^T r and S^T (-dr) on the way:
//       dr_i = (dS + dnum phi(q)^T)_i . alpha = dS_i . alpha + dnum_i (phi(q) . alpha)
// One CTA per (b, h), 512 threads, 208 KB of shared memory.
#include "vla_internal.cuh"

namespace vla {
namespace {

constexpr int D = 128;
constexpr int NT = 512;             // four threads a row
constexpr int NW = NT / 32;
constexpr int VLEN = (D / 32) * kPart;
constexpr int REC = 4 * D + 4;      // floats per token record
constexpr int CKF = 2 * D * D + D;  // floats per checkpoint
constexpr int RQ = NT / D;          // column order: four quarters of the rows
constexpr int RPQ = D / RQ;         // rows a quarter

// Shared memory, in floats.
struct Bw128 {
    static constexpr int S = 0;                      // S, swizzled chunks
    static constexpr int dS = S + D * D;             // dS
    static constexpr int buf = dS + D * D;           // z_i dA'[i][j] (column buffer)
    static constexpr int part = buf + D * D;         // three [RQ][D] column partials
    static constexpr int vec = part + 3 * RQ * D;    // seven part-strided vectors
    static constexpr int sv = vec + 7 * VLEN;        // eight plain vectors of D
    static constexpr int red = sv + 8 * D;           // six block-sum slots of NW float4
    static constexpr int sc = red + 6 * NW * 4;      // four per-token scalars
    static constexpr int total = sc + 4;
};
static_assert(Bw128::vec % 4 == 0 && Bw128::sv % 4 == 0 && Bw128::red % 4 == 0, "float4 alignment");
static_assert(Bw128::total * 4 <= 227 * 1024, "fits one CTA's shared memory");

// Float offset of the 16-byte chunk q (columns 4 q .. 4 q + 3) of row i.  In
// row order a quarter-warp reads chunk 8 part + c of two adjacent rows
// (parts 0..3): the XOR with part and the row's parity spreads the eight over
// all banks.  In column order a warp reads chunks 8 g .. 8 g + 7 of one row:
// the XOR is the same for all eight, a permutation of the banks.
__device__ __forceinline__ int chk(int i, int q) { return i * D + 4 * (q ^ (((q >> 3) & 3) | ((i & 1) << 2))); }
__device__ __forceinline__ int elt(int i, int j) { return chk(i, j >> 2) + (j & 3); }

__device__ __forceinline__ float dphi(float x) { return x > 0.f ? 1.f : expf(x); }

// Block-wide sum of four values over the 16 warps; every thread gets the four
// totals.  Each warp reads the 16 warp partials once (lane l takes component
// l mod 4 of partials l / 4 and l / 4 + 8) and finishes with shuffles: two
// shared-memory passes and seven shuffles a warp, where reading all 16 float4
// partials in every thread took 64 passes a warp.  red: 16 float4, not reused
// before the next block barrier.
__device__ __forceinline__ float4 block_sum4_w16(float v0, float v1, float v2, float v3, float4 *red) {
    static_assert(NW == 16, "16 warps");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float r = warp_reduce4(v0, v1, v2, v3);
    if ((lane & 7) == 0) reinterpret_cast<float *>(red)[warp * 4 + (lane >> 3)] = r;
    __syncthreads();
    const float *rf = reinterpret_cast<const float *>(red);
    float x = rf[lane] + rf[32 + lane];  // component lane & 3 of partials lane / 4 and lane / 4 + 8
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 8);
    x += __shfl_xor_sync(0xffffffffu, x, 16);
    return make_float4(__shfl_sync(0xffffffffu, x, 0), __shfl_sync(0xffffffffu, x, 1),
                       __shfl_sync(0xffffffffu, x, 2), __shfl_sync(0xffffffffu, x, 3));
}

template <typename IO>
__global__ void __launch_bounds__(NT, 1) backward128_kernel(BwdParams p) {
    using L = Bw128;
    extern __shared__ __align__(16) float sm[];
    float *sS = sm + L::S, *sdS = sm + L::dS, *sbuf = sm + L::buf;
    float *pcA = sm + L::part, *pcB = pcA + RQ * D, *pcC = pcB + RQ * D;
    float *v_kh = sm + L::vec, *v_u = v_kh + VLEN, *v_fq = v_u + VLEN, *v_z = v_fq + VLEN;
    float *v_al = v_z + VLEN, *v_dg = v_al + VLEN, *v_dz = v_dg + VLEN;
    float *s_r = sm + L::sv, *s_dO = s_r + D, *s_w = s_dO + D, *s_adz = s_w + D;
    float *s_dkh = s_adz + D, *s_v = s_dkh + D, *s_dnum = s_v + D, *s_dr = s_dnum + D;
    float4 *s_red = reinterpret_cast<float4 *>(sm + L::red);
    float *s_sc = sm + L::sc;

    const int tid = threadIdx.x;
    const int row = tid >> 2, part = tid & 3;      // row order
    const int c0 = part * 32, vo = part * kPart;
    const int cj = tid & (D - 1), rq = tid >> 7;   // column order: column, quarter of the rows
    const int bh = blockIdx.x;
    const int T = p.T;
    const size_t moff = (size_t)bh * D * D + (size_t)row * D + c0;
    const int nck = (T + kBwdCk - 1) / kBwdCk;
    float *rec = p.ws + (size_t)bh * ((size_t)T * REC + (size_t)nck * CKF);
    float *ckp = rec + (size_t)T * REC;
    // this thread's chunk c (columns c0 + 4 c ..) of row `row` of a shared state
    auto rowc = [&](float *M, int c) -> float4 & { return *reinterpret_cast<float4 *>(M + chk(row, part * 8 + c)); };

    float2 a[16];
    if (p.A0) {
        const float4 *src = reinterpret_cast<const float4 *>(p.A0 + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) { const float4 x = src[c]; a[2 * c] = lo2(x); a[2 * c + 1] = hi2(x); }
    } else {
        const float il = 1.f / p.lambda0;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            a[j] = make_float2((c0 + 2 * j == row) ? il : 0.f, (c0 + 2 * j + 1 == row) ? il : 0.f);
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
        rowc(sS, c) = p.S0 ? reinterpret_cast<const float4 *>(p.S0 + moff)[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    float nj = (tid < D && p.n0) ? p.n0[(size_t)bh * D + tid] : 0.f;

    // ---------------- phase 1: forward with records and checkpoints ----------------
    // a token's inputs are loaded one token ahead, so their latency overlaps a token's work
    float nq = 0.f, nk = 0.f, nv = 0.f, nu = 0.f;
    auto fetch_in = [&](int t) {
        if (tid < D && t < T) {
            const size_t tok = ((size_t)bh * T + t) * D;
            nq = io_to_f32(static_cast<const IO *>(p.q)[tok + tid]);
            nk = io_to_f32(static_cast<const IO *>(p.k)[tok + tid]);
            nv = io_to_f32(static_cast<const IO *>(p.v)[tok + tid]);
            nu = io_to_f32(static_cast<const IO *>(p.u)[tok + tid]);
        }
    };
    fetch_in(0);
    for (int t = 0; t < T; ++t) {
        if (t % kBwdCk == 0) {
            float *ck = ckp + (size_t)(t / kBwdCk) * CKF;
            float4 *cs = reinterpret_cast<float4 *>(ck + (size_t)row * D + c0);
            float4 *ca = reinterpret_cast<float4 *>(ck + (size_t)D * D + (size_t)row * D + c0);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                cs[c] = rowc(sS, c);
                ca[c] = make_float4(a[2 * c].x, a[2 * c].y, a[2 * c + 1].x, a[2 * c + 1].y);
            }
            if (tid < D) ck[2 * D * D + tid] = nj;
        }
        float *rt = rec + (size_t)t * REC;
        const float qj = nq, kj = nk, vj = nv, uj = nu;
        fetch_in(t + 1);
        const float4 r1 = block_sum4_w16(kj * kj, 0.f, 0.f, 0.f, s_red);
        const float knorm = sqrtf(r1.x);
        const float ks = 1.f / fmaxf(knorm, kEps);
        float fq = 0.f;
        if (tid < D) {
            const float kh = kj * ks;
            fq = phi_elu1(qj);
            nj += phi_elu1(kh);
            v_kh[vidx(tid)] = kh;
            v_u[vidx(tid)] = uj;
            v_fq[vidx(tid)] = fq;
            s_v[tid] = vj;
            rt[tid] = kh;
        }
        __syncthreads();
        const float4 *up = reinterpret_cast<const float4 *>(v_u + vo);
        const float4 *kp = reinterpret_cast<const float4 *>(v_kh + vo);
        float2 za = f2(0.f), ya = f2(0.f), ka = f2(0.f);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 u4 = up[c], k4 = kp[c], s4 = rowc(sS, c);
            za = fma2(a[2 * c], lo2(u4), za); za = fma2(a[2 * c + 1], hi2(u4), za);
            ya = fma2(a[2 * c], lo2(k4), ya); ya = fma2(a[2 * c + 1], hi2(k4), ya);
            ka = fma2(lo2(s4), lo2(k4), ka); ka = fma2(hi2(s4), hi2(k4), ka);
        }
        float z = hsum2(za), y = hsum2(ya), sk = hsum2(ka);
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
            z += __shfl_xor_sync(0xffffffffu, z, o);
            y += __shfl_xor_sync(0xffffffffu, y, o);
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
        }
        float p1 = 0.f, p2 = 0.f;
        if (part == 0) {
            p1 = v_u[vidx(row)] * z;
            p2 = v_kh[vidx(row)] * z;
            v_z[vidx(row)] = z;
            rt[D + row] = z;
        }
        const float4 r2 = block_sum4_w16(p1, p2, tid < D ? fq * nj : 0.f, 0.f, s_red + NW);
        const float beta = 1.f / (1.f + r2.x);
        const float rden = 1.f / (r2.z + kEps);
        const float g = y - beta * r2.y * z;
        const float4 r3 = block_sum4_w16(part == 0 ? g * g : 0.f, 0.f, 0.f, 0.f, s_red + 2 * NW);
        const float gnorm = sqrtf(r3.x);
        const float inv = 1.f / fmaxf(gnorm, kEps);
        const float r = s_v[row] - sk;
        if (part == 0) {
            v_al[vidx(row)] = g * inv;
            rt[2 * D + row] = g * inv;
            rt[3 * D + row] = r;
        }
        if (tid == 0) {
            rt[4 * D + 0] = knorm;
            rt[4 * D + 1] = beta;
            rt[4 * D + 2] = gnorm;
            rt[4 * D + 3] = rden;
        }
        __syncthreads();
        const float2 mb = f2(-beta), zi = f2(z), r2v = f2(r);
        const float4 *zp = reinterpret_cast<const float4 *>(v_z + vo);
        const float4 *ap = reinterpret_cast<const float4 *>(v_al + vo);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 zz = zp[c], al = ap[c];
            a[2 * c] = fma2(mb, mul2(zi, lo2(zz)), a[2 * c]);
            a[2 * c + 1] = fma2(mb, mul2(zi, hi2(zz)), a[2 * c + 1]);
            float4 &s4 = rowc(sS, c);
            const float2 lo = fma2(r2v, lo2(al), lo2(s4)), hi = fma2(r2v, hi2(al), hi2(s4));
            s4 = make_float4(lo.x, lo.y, hi.x, hi.y);
        }
        __syncthreads();
    }

    // ---------------- phase 2: reverse sweep ----------------
    float2 da[16];
    if (p.dA_T) {
        const float4 *src = reinterpret_cast<const float4 *>(p.dA_T + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) { const float4 x = src[c]; da[2 * c] = lo2(x); da[2 * c + 1] = hi2(x); }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) da[j] = f2(0.f);
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
        rowc(sdS, c) = p.dS_T ? reinterpret_cast<const float4 *>(p.dS_T + moff)[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    float dnj = (tid < D && p.dn_T) ? p.dn_T[(size_t)bh * D + tid] : 0.f;
    __syncthreads();

    // a token's record and inputs are loaded one token ahead, so their latency
    // overlaps a token's work
    float pkh = 0.f, pz = 0.f, pal = 0.f, pr = 0.f, pu = 0.f, pq = 0.f, pdO = 0.f, psc = 0.f;
    auto fetch_rec = [&](int t) {
        if (t < 0) return;
        const size_t tok = ((size_t)bh * T + t) * D;
        const float *rt = rec + (size_t)t * REC;
        if (tid < D) {
            pkh = rt[tid];
            pz = rt[D + tid];
            pal = rt[2 * D + tid];
            pr = rt[3 * D + tid];
            pu = io_to_f32(static_cast<const IO *>(p.u)[tok + tid]);
            pq = io_to_f32(static_cast<const IO *>(p.q)[tok + tid]);
            pdO = io_to_f32(static_cast<const IO *>(p.dO)[tok + tid]);
        }
        if (tid < 4) psc = rt[4 * D + tid];
    };
    fetch_rec(T - 1);
    for (int t = T - 1; t >= 0; --t) {
        if ((t + 1) % kBwdCk == 0 && t + 1 < T) {  // re-anchor: state after token t
            const float *ck = ckp + (size_t)((t + 1) / kBwdCk) * CKF;
            const float4 *cs = reinterpret_cast<const float4 *>(ck + (size_t)row * D + c0);
            const float4 *ca = reinterpret_cast<const float4 *>(ck + (size_t)D * D + (size_t)row * D + c0);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 w = ca[c];
                rowc(sS, c) = cs[c];
                a[2 * c] = lo2(w); a[2 * c + 1] = hi2(w);
            }
            if (tid < D) nj = ck[2 * D * D + tid];
        }
        const size_t tok = ((size_t)bh * T + t) * D;
        const float khj = pkh, zj = pz, alj = pal, uj = pu, qj = pq, fqj = phi_elu1(qj);
        if (tid < D) {
            v_kh[vidx(tid)] = khj;
            v_z[vidx(tid)] = zj;
            v_al[vidx(tid)] = alj;
            v_u[vidx(tid)] = uj;
            v_fq[vidx(tid)] = fqj;
            s_r[tid] = pr;
            s_dO[tid] = pdO;
        }
        if (tid < 4) s_sc[tid] = psc;
        fetch_rec(t - 1);
        __syncthreads();
        const float knorm = s_sc[0], beta = s_sc[1], gnorm = s_sc[2], rden = s_sc[3];
        const float4 *kp = reinterpret_cast<const float4 *>(v_kh + vo);
        const float4 *fp = reinterpret_cast<const float4 *>(v_fq + vo);
        const float4 *alp = reinterpret_cast<const float4 *>(v_al + vo);
        const float4 *zp = reinterpret_cast<const float4 *>(v_z + vo);
        const float4 *up = reinterpret_cast<const float4 *>(v_u + vo);

        // ---- S1 (row order, read only): S'_i . phi(q), dS_i . alpha, phi(q) . alpha ----
        float2 na = f2(0.f), sa = f2(0.f), fa2 = f2(0.f);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 f4 = fp[c], al4 = alp[c], s4 = rowc(sS, c), d4 = rowc(sdS, c);
            na = fma2(lo2(s4), lo2(f4), na); na = fma2(hi2(s4), hi2(f4), na);
            sa = fma2(lo2(d4), lo2(al4), sa); sa = fma2(hi2(d4), hi2(al4), sa);
            fa2 = fma2(lo2(f4), lo2(al4), fa2); fa2 = fma2(hi2(f4), hi2(al4), fa2);
        }
        float num = hsum2(na), dsa = hsum2(sa), fal = hsum2(fa2);
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
            num += __shfl_xor_sync(0xffffffffu, num, o);
            dsa += __shfl_xor_sync(0xffffffffu, dsa, o);
            fal += __shfl_xor_sync(0xffffffffu, fal, o);
        }
        const float dOi = s_dO[row];
        const float dnum = dOi * rden;
        const float ri = s_r[row];
        const float dr = fmaf(dnum, fal, dsa);  // (dS + dnum phi(q)^T)_i . alpha
        if (part == 0) {
            s_dnum[row] = dnum;
            s_dr[row] = dr;
            if (p.dv) p.dv[tok + row] = dr;
        }
        const float o_i = num * rden;
        const float4 R1 = block_sum4_w16(part == 0 ? dOi * o_i : 0.f, part == 0 ? ri * dr : 0.f, 0.f, 0.f,
                                         s_red + 3 * NW);
        // ---- S2 (column order): S'^T dnum, dS'^T r, S^T(-dr); undo the state write; dS ----
        {
            const float alc = v_al[vidx(cj)], fqc = v_fq[vidx(cj)], khc = v_kh[vidx(cj)];
            float ca = 0.f, cb = 0.f, cc = 0.f;
#pragma unroll 8
            for (int ii = 0; ii < RPQ; ++ii) {
                const int i = rq * RPQ + ii;
                const float dn = s_dnum[i], rr = s_r[i], drr = s_dr[i];
                float *ps = sS + elt(i, cj), *pd = sdS + elt(i, cj);
                const float s = *ps;
                ca = fmaf(dn, s, ca);
                const float sn = fmaf(-rr, alc, s);  // S_{t-1} = S_t - r alpha^T
                *ps = sn;
                cc = fmaf(-drr, sn, cc);
                const float ds = fmaf(dn, fqc, *pd);  // dS' = dS + dnum phi(q)^T
                cb = fmaf(rr, ds, cb);
                *pd = fmaf(-drr, khc, ds);            // dS' - dr k_hat^T
            }
            pcA[rq * D + cj] = ca;
            pcB[rq * D + cj] = cb;
            pcC[rq * D + cj] = cc;
        }
        __syncthreads();
        // ---- P2 (columns): dq, dn, dalpha -> dg, dk_hat partials; undo n ----
        if (tid < D) {
            const int j = tid;
            const float colA = (pcA[j] + pcA[D + j]) + (pcA[2 * D + j] + pcA[3 * D + j]);
            const float colB = (pcB[j] + pcB[D + j]) + (pcB[2 * D + j] + pcB[3 * D + j]);
            const float colC = (pcC[j] + pcC[D + j]) + (pcC[2 * D + j] + pcC[3 * D + j]);
            const float dden = -R1.x * rden;
            const float dfq = fmaf(dden, nj, colA);
            if (p.dq) p.dq[tok + j] = dfq * dphi(qj);
            dnj = fmaf(dden, fqj, dnj);
            const float dg = gnorm > kEps ? (colB - alj * R1.y) / gnorm : colB / kEps;
            v_dg[vidx(j)] = dg;
            s_dkh[j] = dnj * dphi(khj) + colC;
            nj -= phi_elu1(khj);
        }
        __syncthreads();
        // ---- P3 (rows): gate -> dA', dk_hat += A' dg; w = dA' z; z_i dA'_i to the buffer ----
        const float4 *gp = reinterpret_cast<const float4 *>(v_dg + vo);
        const float2 dg2 = f2(v_dg[vidx(row)]);
        float2 adg = f2(0.f), wa = f2(0.f);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 k4 = kp[c], g4 = gp[c], z4 = zp[c];
            adg = fma2(a[2 * c], lo2(g4), adg);
            adg = fma2(a[2 * c + 1], hi2(g4), adg);
            da[2 * c] = fma2(dg2, lo2(k4), da[2 * c]);
            da[2 * c + 1] = fma2(dg2, hi2(k4), da[2 * c + 1]);
            wa = fma2(da[2 * c], lo2(z4), wa);
            wa = fma2(da[2 * c + 1], hi2(z4), wa);
        }
        float adgv = hsum2(adg), w = hsum2(wa);
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
            adgv += __shfl_xor_sync(0xffffffffu, adgv, o);
            w += __shfl_xor_sync(0xffffffffu, w, o);
        }
        const float zrow = v_z[vidx(row)];
        if (part == 0) {
            s_dkh[row] += adgv;
            s_w[row] = w;
        }
        const float2 zr2 = f2(zrow);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float2 lo = mul2(zr2, da[2 * c]), hi = mul2(zr2, da[2 * c + 1]);
            rowc(sbuf, c) = make_float4(lo.x, lo.y, hi.x, hi.y);
        }
        const float4 R3 = block_sum4_w16(part == 0 ? zrow * w : 0.f, 0.f, 0.f, 0.f, s_red + 4 * NW);
        // ---- P4 (columns): dA'^T z, dbeta, dz ----
        {
            float acc = 0.f;
#pragma unroll 8
            for (int ii = 0; ii < RPQ; ++ii) acc += sbuf[elt(rq * RPQ + ii, cj)];
            pcA[rq * D + cj] = acc;
        }
        __syncthreads();
        const float ds1 = beta * beta * R3.x;  // ds1 = -beta^2 dbeta, dbeta = -z.w
        float du_part = 0.f;
        if (tid < D) {
            const int j = tid;
            const float datz = (pcA[j] + pcA[D + j]) + (pcA[2 * D + j] + pcA[3 * D + j]);
            const float dz = -beta * (s_w[j] + datz) + ds1 * uj;
            v_dz[vidx(j)] = dz;
            du_part = ds1 * zj;
        }
        __syncthreads();
        // ---- P5 (rows): undo the penalty update, A dz, dA += dz u^T ----
        const float4 *dzp = reinterpret_cast<const float4 *>(v_dz + vo);
        const float2 pb = f2(beta), dz2 = f2(v_dz[vidx(row)]);
        float2 adz = f2(0.f);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 z4 = zp[c], dz4 = dzp[c], u4 = up[c];
            a[2 * c] = fma2(pb, mul2(zr2, lo2(z4)), a[2 * c]);
            a[2 * c + 1] = fma2(pb, mul2(zr2, hi2(z4)), a[2 * c + 1]);
            adz = fma2(a[2 * c], lo2(dz4), adz);
            adz = fma2(a[2 * c + 1], hi2(dz4), adz);
            da[2 * c] = fma2(dz2, lo2(u4), da[2 * c]);
            da[2 * c + 1] = fma2(dz2, hi2(u4), da[2 * c + 1]);
        }
        float adzv = hsum2(adz);
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) adzv += __shfl_xor_sync(0xffffffffu, adzv, o);
        if (part == 0) s_adz[row] = adzv;
        __syncthreads();
        // ---- P6 (columns): du, dk ----
        float dkh = 0.f;
        if (tid < D) {
            if (p.du) p.du[tok + tid] = du_part + s_adz[tid];
            dkh = s_dkh[tid];
        }
        const float4 R4 = block_sum4_w16(tid < D ? khj * dkh : 0.f, 0.f, 0.f, 0.f, s_red + 5 * NW);
        if (tid < D && p.dk)
            p.dk[tok + tid] = knorm > kEps ? (dkh - khj * R4.x) / knorm : dkh / kEps;
        __syncthreads();  // the next token overwrites the shared vectors and partials
    }
    if (p.dS0) {
        float4 *dst = reinterpret_cast<float4 *>(p.dS0 + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) dst[c] = rowc(sdS, c);
    }
    if (p.dA0) {
        float4 *dst = reinterpret_cast<float4 *>(p.dA0 + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) dst[c] = make_float4(da[2 * c].x, da[2 * c].y, da[2 * c + 1].x, da[2 * c + 1].y);
    }
    if (tid < D && p.dn0) p.dn0[(size_t)bh * D + tid] = dnj;
}

template <typename IO>
cudaError_t launch_t(const BwdParams &p, cudaStream_t st) {
    const size_t bytes = (size_t)Bw128::total * sizeof(float);
    const cudaError_t e =
        cudaFuncSetAttribute(backward128_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    backward128_kernel<IO><<<(unsigned)p.BH, NT, bytes, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward128(const BwdParams &p, cudaStream_t stream) {
    if (p.d != D || p.BH <= 0) return p.BH == 0 ? cudaSuccess : cudaErrorInvalidValue;
    return p.io_bf16 ? launch_t<__nv_bfloat16>(p, stream) : launch_t<float>(p, stream);
}

}  // namespace vla
