// vla_backward.cu -- gradients of the VLA forward recurrence ("Variational
// Linear Attention: Stable Associative Memory for Long-Context Transformers",
// sections 2.2-2.3; the recurrence transition J_t = I - alpha_t k_hat_t^T of
// section 3.1 is the S part of the adjoint below).
//
// Loss: L = sum_t <dO_t, o_t> + <dS_T, S_T> + <dA_T, A_T> + <dn_T, n_T>.
// Gradients: dq, dk, dv, du (fp32, [BH, T, d]) and dS0, dA0, dn0.
//
// One CTA per (b, h).  Phase 1 reruns the forward (three block reductions
// per token, as in the decode kernel) and stores, per token, k_hat, z,
// alpha, r and |k|, beta, |g|, 1/den, and every kCk tokens the state (S, A,
// n).  Phase 2 walks the tokens backwards with the state of the current
// step in registers, rebuilding the previous state by undoing the rank-1
// updates (S -= r alpha^T, A += beta z z^T, n -= phi(k_hat)) and reloading it
// from the nearest checkpoint to bound fp32 drift.  Per token (adjoints are
// primed for the step's outputs):
//   readout  dnum = dO / den, dden = -(dO . o) / den, dS' += dnum phi(q)^T,
//            dphi(q) = S'^T dnum + dden n', dn' += dden phi(q)
//   state    dr = dS' alpha, dalpha = dS'^T r, dv = dr,
//            dS = dS' - dr k_hat^T, dk_hat += -S^T dr + dn' phi'(k_hat)
//   gate     dg = (dalpha - alpha (alpha . dalpha)) / |g|,
//            dA' += dg k_hat^T, dk_hat += A' dg
//   penalty  w = dA' z, dbeta = -z . w, ds1 = -beta^2 dbeta,
//            dz = -beta (w + dA'^T z) + ds1 u, du = ds1 z + A dz,
//            dA = dA' + dz u^T
//   key      dk = (dk_hat - k_hat (k_hat . dk_hat)) / |k|
// Rows of S, A, dS, dA live in registers of row-owner threads; the
// transposed products S^T x, dS'^T r and dA'^T z are column sums through
// shared memory.  d in {32, 64} (four d x d register states; d = 128 has a
// kernel of its own, vla_backward128.cu).
#include "vla_internal.cuh"

namespace vla {
namespace {

constexpr int kCk = kBwdCk;  // tokens between state checkpoints

template <int D>
struct BwdCfg {
    static constexpr int TPR = D / 32;
    static constexpr int NT = D * TPR;
    static constexpr int NW = NT / 32;
    static constexpr int VLEN = TPR * kPart;
    static constexpr int REC = 4 * D + 4;   // floats per token record
    static constexpr int CKF = 2 * D * D + D;  // floats per checkpoint
    static constexpr int LDC = D + 4;        // row stride of the column-sum buffers
};

__device__ __forceinline__ float dphi(float x) { return x > 0.f ? 1.f : expf(x); }

template <int D, typename IO>
__global__ void __launch_bounds__(BwdCfg<D>::NT) backward_kernel(BwdParams p) {
    using C = BwdCfg<D>;
    constexpr int TPR = C::TPR, VLEN = C::VLEN, NW = C::NW, REC = C::REC, CKF = C::CKF, LDC = C::LDC;
    __shared__ __align__(16) float v_kh[VLEN], v_u[VLEN], v_fq[VLEN], v_z[VLEN], v_al[VLEN], v_dg[VLEN],
        v_dz[VLEN];
    __shared__ __align__(16) float s_r[D], s_dO[D], s_w[D], s_adz[D], s_dkh[D], s_v[D];
    extern __shared__ __align__(16) float s_dyn[];  // three column-sum buffers [D][LDC]
    float *colA = s_dyn, *colB = s_dyn + D * LDC, *colC = s_dyn + 2 * D * LDC;
    __shared__ __align__(16) float4 s_red[8][NW];
    __shared__ float s_sc[4];

    const int tid = threadIdx.x;
    const int row = tid / TPR, part = tid % TPR;
    const int c0 = part * 32, vo = part * kPart;
    const int bh = blockIdx.x;
    const int T = p.T;
    const size_t moff = (size_t)bh * D * D + (size_t)row * D + c0;
    const int nck = (T + kCk - 1) / kCk;
    float *rec = p.ws + (size_t)bh * ((size_t)T * REC + (size_t)nck * CKF);
    float *ckp = rec + (size_t)T * REC;

    float2 s[16], a[16];
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
    if (p.S0) {
        const float4 *src = reinterpret_cast<const float4 *>(p.S0 + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) { const float4 x = src[c]; s[2 * c] = lo2(x); s[2 * c + 1] = hi2(x); }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) s[j] = f2(0.f);
    }
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
        if (t % kCk == 0) {
            float *ck = ckp + (size_t)(t / kCk) * CKF;
            float4 *cs = reinterpret_cast<float4 *>(ck + (size_t)row * D + c0);
            float4 *ca = reinterpret_cast<float4 *>(ck + (size_t)D * D + (size_t)row * D + c0);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                cs[c] = make_float4(s[2 * c].x, s[2 * c].y, s[2 * c + 1].x, s[2 * c + 1].y);
                ca[c] = make_float4(a[2 * c].x, a[2 * c].y, a[2 * c + 1].x, a[2 * c + 1].y);
            }
            if (tid < D) ck[2 * D * D + tid] = nj;
        }
        float *rt = rec + (size_t)t * REC;
        const float qj = nq, kj = nk, vj = nv, uj = nu;
        fetch_in(t + 1);
        const float4 r1 = block_sum4<NW>(kj * kj, 0.f, 0.f, 0.f, s_red[0]);
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
            const float4 u4 = up[c], k4 = kp[c];
            za = fma2(a[2 * c], lo2(u4), za); za = fma2(a[2 * c + 1], hi2(u4), za);
            ya = fma2(a[2 * c], lo2(k4), ya); ya = fma2(a[2 * c + 1], hi2(k4), ya);
            ka = fma2(s[2 * c], lo2(k4), ka); ka = fma2(s[2 * c + 1], hi2(k4), ka);
        }
        float z = hsum2(za), y = hsum2(ya), sk = hsum2(ka);
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) {
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
        const float4 r2 = block_sum4<NW>(p1, p2, tid < D ? fq * nj : 0.f, 0.f, s_red[1]);
        const float beta = 1.f / (1.f + r2.x);
        const float rden = 1.f / (r2.z + kEps);
        const float g = y - beta * r2.y * z;
        const float4 r3 = block_sum4<NW>(part == 0 ? g * g : 0.f, 0.f, 0.f, 0.f, s_red[2]);
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
            s[2 * c] = fma2(r2v, lo2(al), s[2 * c]);
            s[2 * c + 1] = fma2(r2v, hi2(al), s[2 * c + 1]);
        }
        __syncthreads();
    }

    // ---------------- phase 2: reverse sweep ----------------
    float2 ds[16], da[16];
    if (p.dS_T) {
        const float4 *src = reinterpret_cast<const float4 *>(p.dS_T + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) { const float4 x = src[c]; ds[2 * c] = lo2(x); ds[2 * c + 1] = hi2(x); }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) ds[j] = f2(0.f);
    }
    if (p.dA_T) {
        const float4 *src = reinterpret_cast<const float4 *>(p.dA_T + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) { const float4 x = src[c]; da[2 * c] = lo2(x); da[2 * c + 1] = hi2(x); }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) da[j] = f2(0.f);
    }
    float dnj = (tid < D && p.dn_T) ? p.dn_T[(size_t)bh * D + tid] : 0.f;

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
        if ((t + 1) % kCk == 0 && t + 1 < T) {  // re-anchor: state after token t
            const float *ck = ckp + (size_t)((t + 1) / kCk) * CKF;
            const float4 *cs = reinterpret_cast<const float4 *>(ck + (size_t)row * D + c0);
            const float4 *ca = reinterpret_cast<const float4 *>(ck + (size_t)D * D + (size_t)row * D + c0);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 x = cs[c], w = ca[c];
                s[2 * c] = lo2(x); s[2 * c + 1] = hi2(x);
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

        // ---- P1 (rows): readout and state adjoints ----
        float2 na = f2(0.f);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 f4 = fp[c];
            na = fma2(s[2 * c], lo2(f4), na);
            na = fma2(s[2 * c + 1], hi2(f4), na);
        }
        float num = hsum2(na);
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) num += __shfl_xor_sync(0xffffffffu, num, o);
        const float dOi = s_dO[row];
        const float dnum = dOi * rden;
        const float ri = s_r[row];
        const float2 dn2 = f2(dnum);
        float *cA = colA + row * LDC + c0;
        float *cB = colB + row * LDC + c0;
        float *cC = colC + row * LDC + c0;
        float2 dra = f2(0.f);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 f4 = fp[c], al4 = alp[c];
            // dphi(q) partial: dnum * S'_i
            reinterpret_cast<float4 *>(cA)[c] =
                make_float4(dnum * s[2 * c].x, dnum * s[2 * c].y, dnum * s[2 * c + 1].x, dnum * s[2 * c + 1].y);
            ds[2 * c] = fma2(dn2, lo2(f4), ds[2 * c]);
            ds[2 * c + 1] = fma2(dn2, hi2(f4), ds[2 * c + 1]);
            dra = fma2(ds[2 * c], lo2(al4), dra);
            dra = fma2(ds[2 * c + 1], hi2(al4), dra);
        }
        float dr = hsum2(dra);
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) dr += __shfl_xor_sync(0xffffffffu, dr, o);
        if (part == 0 && p.dv) p.dv[tok + row] = dr;
        const float2 mri = f2(-ri), dsk = f2(-dr);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 al4 = alp[c], k4 = kp[c];
            // dalpha partial: r_i dS'_i; undo the state write; S^T dsk partial
            reinterpret_cast<float4 *>(cB)[c] =
                make_float4(ri * ds[2 * c].x, ri * ds[2 * c].y, ri * ds[2 * c + 1].x, ri * ds[2 * c + 1].y);
            s[2 * c] = fma2(mri, lo2(al4), s[2 * c]);
            s[2 * c + 1] = fma2(mri, hi2(al4), s[2 * c + 1]);
            const float2 s0 = mul2(dsk, s[2 * c]), s1 = mul2(dsk, s[2 * c + 1]);
            reinterpret_cast<float4 *>(cC)[c] = make_float4(s0.x, s0.y, s1.x, s1.y);
            ds[2 * c] = fma2(dsk, lo2(k4), ds[2 * c]);
            ds[2 * c + 1] = fma2(dsk, hi2(k4), ds[2 * c + 1]);
        }
        const float o_i = num * rden;
        const float4 R1 = block_sum4<NW>(part == 0 ? dOi * o_i : 0.f, part == 0 ? ri * dr : 0.f, 0.f, 0.f,
                                         s_red[3]);
        // ---- P2 (columns): dq, dn, dalpha -> dg, dk_hat partials; undo n ----
        if (tid < D) {
            const int j = tid;
            const float dden = -R1.x * rden;
            float dfq = dden * nj, dal = 0.f, stdsk = 0.f;
            for (int i = 0; i < D; ++i) {
                dfq += colA[i * LDC + j];
                dal += colB[i * LDC + j];
                stdsk += colC[i * LDC + j];
            }
            if (p.dq) p.dq[tok + j] = dfq * dphi(qj);
            dnj = fmaf(dden, fqj, dnj);
            const float dg = gnorm > kEps ? (dal - alj * R1.y) / gnorm : dal / kEps;
            v_dg[vidx(j)] = dg;
            s_dkh[j] = dnj * dphi(khj) + stdsk;
            nj -= phi_elu1(khj);
        }
        __syncthreads();
        // ---- P3 (rows): gate -> dA', dk_hat += A' dg; w = dA' z ----
        const float4 *gp = reinterpret_cast<const float4 *>(v_dg + vo);
        const float dgi = v_dg[vidx(row)];
        const float2 dg2 = f2(dgi);
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
        for (int o = 1; o < TPR; o <<= 1) {
            adgv += __shfl_xor_sync(0xffffffffu, adgv, o);
            w += __shfl_xor_sync(0xffffffffu, w, o);
        }
        const float zrow = v_z[vidx(row)];
        if (part == 0) {
            s_dkh[row] += adgv;
            s_w[row] = w;
        }
#pragma unroll
        for (int c = 0; c < 8; ++c)
            reinterpret_cast<float4 *>(cA)[c] = make_float4(zrow * da[2 * c].x, zrow * da[2 * c].y,
                                                             zrow * da[2 * c + 1].x, zrow * da[2 * c + 1].y);
        const float4 R3 = block_sum4<NW>(part == 0 ? zrow * w : 0.f, 0.f, 0.f, 0.f, s_red[4]);
        // ---- P4 (columns): dbeta, dz ----
        const float ds1 = beta * beta * R3.x;  // ds1 = -beta^2 dbeta, dbeta = -z.w
        float du_part = 0.f;
        if (tid < D) {
            const int j = tid;
            float datz = 0.f;
            for (int i = 0; i < D; ++i) datz += colA[i * LDC + j];
            const float dz = -beta * (s_w[j] + datz) + ds1 * uj;
            v_dz[vidx(j)] = dz;
            du_part = ds1 * zj;
        }
        __syncthreads();
        // ---- P5 (rows): undo the penalty update, A dz, dA += dz u^T ----
        const float4 *dzp = reinterpret_cast<const float4 *>(v_dz + vo);
        const float dzi = v_dz[vidx(row)];
        const float2 pb = f2(beta), zr2 = f2(zrow), dz2 = f2(dzi);
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
        for (int o = 1; o < TPR; o <<= 1) adzv += __shfl_xor_sync(0xffffffffu, adzv, o);
        if (part == 0) s_adz[row] = adzv;
        __syncthreads();
        // ---- P6 (columns): du, dk ----
        float dkh = 0.f;
        if (tid < D) {
            if (p.du) p.du[tok + tid] = du_part + s_adz[tid];
            dkh = s_dkh[tid];
        }
        const float4 R4 = block_sum4<NW>(tid < D ? khj * dkh : 0.f, 0.f, 0.f, 0.f, s_red[5]);
        if (tid < D && p.dk)
            p.dk[tok + tid] = knorm > kEps ? (dkh - khj * R4.x) / knorm : dkh / kEps;
        __syncthreads();  // the next token overwrites the shared vectors and column buffers
    }
    if (p.dS0) {
        float4 *dst = reinterpret_cast<float4 *>(p.dS0 + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) dst[c] = make_float4(ds[2 * c].x, ds[2 * c].y, ds[2 * c + 1].x, ds[2 * c + 1].y);
    }
    if (p.dA0) {
        float4 *dst = reinterpret_cast<float4 *>(p.dA0 + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) dst[c] = make_float4(da[2 * c].x, da[2 * c].y, da[2 * c + 1].x, da[2 * c + 1].y);
    }
    if (tid < D && p.dn0) p.dn0[(size_t)bh * D + tid] = dnj;
}

template <int D, typename IO>
cudaError_t launch_backward_t(const BwdParams &p, cudaStream_t st) {
    const size_t dyn = 3 * (size_t)D * BwdCfg<D>::LDC * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(backward_kernel<D, IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)dyn);
    if (e != cudaSuccess) return e;
    backward_kernel<D, IO><<<p.BH, BwdCfg<D>::NT, dyn, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t backward_workspace_floats(int BH, int T, int d) {
    const size_t nck = ((size_t)T + kCk - 1) / kCk;
    return (size_t)BH * ((size_t)T * (4 * d + 4) + nck * (2 * (size_t)d * d + d));
}

cudaError_t launch_backward(const BwdParams &p, cudaStream_t stream) {
    if (p.BH == 0) return cudaSuccess;
    // two or more of the chunked forward's S-chunks: in parallel over the chunks
    bool chunked = false;
    const cudaError_t ec = launch_backward_chunk(p, stream, &chunked);
    if (ec != cudaSuccess || chunked) return ec;
    if (p.launches) *p.launches = 1;
    if (p.d == 128) return launch_backward128(p, stream);
    if (p.io_bf16) {
        switch (p.d) {
            case 32: return launch_backward_t<32, __nv_bfloat16>(p, stream);
            case 64: return launch_backward_t<64, __nv_bfloat16>(p, stream);
        }
    } else {
        switch (p.d) {
            case 32: return launch_backward_t<32, float>(p, stream);
            case 64: return launch_backward_t<64, float>(p, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace vla
