// vla_backward_chunk.cu -- the backward of the VLA recurrence ("Variational
// Linear Attention: Stable Associative Memory for Long-Context Transformers",
// sections 2.2-2.3; the transition J_t = I - alpha_t k_hat_t^T of section
// 3.1) in parallel over chunks of tokens.
//
// Over a chunk, the adjoint state (dS, dA, dn) at the chunk's start is an
// affine function of its value at the chunk's end:
//   dn_start = dn_end + sum_t dden_t phi(q_t)
//   dS_start = dS_end Phi_c + Psi_c,  Phi_c = product of (I - alpha_t k_hat_t^T),
//              Psi_c the chunk's readout terms carried to its start
//   dA: the gradients read dA only through z^T dA z and (dA + dA^T) z, so only
//       its symmetric part X feeds back, and it moves two-sided:
//       X_{t-1} = K_t (X_t + sym(dg_t k_hat_t^T)) K_t^T,  K_t = I - beta_t u_t z_t^T,
//       X_start = Q_c X_end Q_c^T + Omega_c,  Q_c = K_first .. K_last;
//       the antisymmetric part of dA0 is the sum over the tokens of
//       asym(dg_t k_hat_t^T + dz_t u_t^T) plus that of dA_T.
// The chunks are the chunked forward's S-chunks (a multiple of 64 tokens),
// whose start states it already computes: S^(c), n^(c), and A^(c) as the
// inverse of the prefix of Grams M^(c).  Launches (CTA = (unit, chunk) unless
// noted):
//   forward      the chunked forward, into a scratch region of the workspace
//   starts       the chunk-start states into the checkpoint slots
//   fwd_maps     per token records and checkpoints over the chunk (as the
//                sequential backward's forward sweep), the chunk's dn sum, then
//                Phi_c, Psi_c and Q_c^T from the records
//   chain_s      (CTA = unit) dS and dn along the chunks, from the last
//   spart        the reverse sweep of the S part with the exact dS: dq, dv,
//                the gate terms dg_t and the S and n parts of dk_hat (stored),
//                and Omega_c
//   chain_x      (CTA = unit) X along the chunks, from the last
//   final        the reverse sweep of the A part with the exact X: du, dk, and
//                the chunk's antisymmetric sum
//   reduce       (CTA = unit) dA0 = X_start + asym(dA_T) + the antisymmetric sums
// The per-token equations are those of the sequential backward (vla_backward.cu).
#include "vla_internal.cuh"

namespace vla {
namespace {

constexpr int kCkB = 64;  // tokens between state checkpoints

template <int D>
struct Bc {
    static constexpr int TPR = D / 32;
    static constexpr int NT = D * TPR;
    static constexpr int NW = NT / 32;
    static constexpr int VLEN = TPR * kPart;
    // resident CTAs per SM the reverse sweeps are built for (d = 64: 168 registers)
    static constexpr int MINB = D == 64 ? 3 : 1;
    static constexpr int REC = 4 * D + 4;      // per token: k_hat, z, alpha, r, |k|, beta, |g|, 1/den
    static constexpr int CKF = 2 * D * D + D;  // checkpoint: S, A, n
    static constexpr int LDC = D + 4;          // row stride of the column-sum buffers
};

struct BcArgs {
    BwdParams p;
    ChunkLayout L;             // the forward's layout: its S-chunks are the chunks here
    const unsigned char *fws;  // the forward's workspace
    int NCK;                   // checkpoint slots per unit before the final-state slot
    float *rec;                // [BH][T][REC]
    float *ckp;                // [BH][NCK + 1][CKF]
    float *maps;               // [BH][NC][3][D][D]: Phi, Psi, Q^T
    float *dnsum, *dn_end;     // [BH][NC][D]
    float *dS_end;             // [BH][NC][D][D]
    float *om, *xs_end;        // [BH][NC][D][D]
    float *xs0;                // [BH][D][D]
    float *asum;               // [BH][NC][D][D]
    float *tokv;               // [BH][T][2][D]: dg_t, dk_hat_t (S and n parts)
};

// A row slice: 32 consecutive floats of one row as 16 pairs.
__device__ __forceinline__ void ld_row(float2 (&x)[16], const float *src) {
    const float4 *s = reinterpret_cast<const float4 *>(src);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float4 v = s[c];
        x[2 * c] = lo2(v);
        x[2 * c + 1] = hi2(v);
    }
}

__device__ __forceinline__ void st_row(float *dst, const float2 (&x)[16]) {
    float4 *d = reinterpret_cast<float4 *>(dst);
#pragma unroll
    for (int c = 0; c < 8; ++c) d[c] = make_float4(x[2 * c].x, x[2 * c].y, x[2 * c + 1].x, x[2 * c + 1].y);
}

__device__ __forceinline__ void set_diag(float2 (&x)[16], int row, int c0, float diag) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
        x[j] = make_float2((c0 + 2 * j == row) ? diag : 0.f, (c0 + 2 * j + 1 == row) ? diag : 0.f);
}

// Row slice . shared vector (its part at vo), summed over the TPR threads of the row.
template <int TPR>
__device__ __forceinline__ float dot_row(const float2 (&x)[16], const float *vec) {
    const float4 *v = reinterpret_cast<const float4 *>(vec);
    float2 acc = f2(0.f);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float4 w = v[c];
        acc = fma2(x[2 * c], lo2(w), acc);
        acc = fma2(x[2 * c + 1], hi2(w), acc);
    }
    float s = hsum2(acc);
#pragma unroll
    for (int o = 1; o < TPR; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

// x += f * vec (shared vector part at vo).
__device__ __forceinline__ void axpy_row(float2 (&x)[16], float f, const float *vec) {
    const float4 *v = reinterpret_cast<const float4 *>(vec);
    const float2 f2v = f2(f);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float4 w = v[c];
        x[2 * c] = fma2(f2v, lo2(w), x[2 * c]);
        x[2 * c + 1] = fma2(f2v, hi2(w), x[2 * c + 1]);
    }
}

// ---------------------------------------------------------------------------
// chunk-start states into the checkpoint slot of each chunk's first token
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(Bc<D>::NT) bc_starts_kernel(BcArgs a) {
    using K = Bc<D>;
    __shared__ __align__(16) float piv[2 * K::VLEN];
    const BwdParams &p = a.p;
    const int NC = a.L.NC, C = a.L.C;
    const int c = (int)(blockIdx.x % (unsigned)NC), bh = (int)(blockIdx.x / (unsigned)NC);
    const int tid = threadIdx.x, row = tid / K::TPR, part = tid % K::TPR, c0 = part * 32;
    const size_t moff = (size_t)row * D + c0;
    float *ck = a.ckp + ((size_t)bh * (a.NCK + 1) + (size_t)c * C / kCkB) * K::CKF;
    float2 x[16];
    if (c == 0) {  // the given or default initial state
        if (p.S0) ld_row(x, p.S0 + (size_t)bh * D * D + moff);
        else set_diag(x, row, c0, 0.f);
        st_row(ck + moff, x);
        if (p.A0) ld_row(x, p.A0 + (size_t)bh * D * D + moff);
        else set_diag(x, row, c0, 1.f / p.lambda0);
        st_row(ck + (size_t)D * D + moff, x);
        if (tid < D) ck[2 * D * D + tid] = p.n0 ? p.n0[(size_t)bh * D + tid] : 0.f;
        return;
    }
    const float *fS = reinterpret_cast<const float *>(a.fws + a.L.off_S) + ((size_t)bh * NC + c) * D * D;
    ld_row(x, fS + moff);
    st_row(ck + moff, x);
    const int ca = c * (C / a.L.CA);  // the A-chunk that starts with this chunk
    const float *fM = reinterpret_cast<const float *>(a.fws + a.L.off_M) + ((size_t)bh * a.L.NCA + ca) * D * D;
    float y[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) y[j] = fM[moff + j];
    gj_inverse<D, 32>(y, piv, row, part);  // A^(c) = (M^(c))^{-1}
#pragma unroll
    for (int j = 0; j < 32; ++j) ck[(size_t)D * D + moff + j] = y[j];
    if (tid < D)
        ck[2 * D * D + tid] =
            reinterpret_cast<const float *>(a.fws + a.L.off_n)[((size_t)bh * (a.L.NCA + 1) + ca) * D + tid];
}

// ---------------------------------------------------------------------------
// forward sweep of one chunk (records, checkpoints, the dn sum), then its
// maps Phi_c, Psi_c, Q_c^T from the records
// ---------------------------------------------------------------------------
template <int D, typename IO>
__global__ void __launch_bounds__(Bc<D>::NT) bc_fwd_maps_kernel(BcArgs a) {
    using K = Bc<D>;
    constexpr int TPR = K::TPR, VLEN = K::VLEN, NW = K::NW, REC = K::REC, CKF = K::CKF;
    __shared__ __align__(16) float v_kh[VLEN], v_u[VLEN], v_fq[VLEN], v_z[VLEN], v_al[VLEN];
    __shared__ __align__(16) float s_v[D];
    __shared__ __align__(16) float4 s_red[3][NW];
    const BwdParams &p = a.p;
    const int NC = a.L.NC, C = a.L.C, T = p.T;
    const int c = (int)(blockIdx.x % (unsigned)NC), bh = (int)(blockIdx.x / (unsigned)NC);
    const int tid = threadIdx.x, row = tid / TPR, part = tid % TPR, c0 = part * 32, vo = part * kPart;
    const int t0 = c * C, t1 = min(T, t0 + C);
    const size_t moff = (size_t)row * D + c0;
    float *rec = a.rec + (size_t)bh * T * REC;
    float *ckp = a.ckp + (size_t)bh * (a.NCK + 1) * CKF;

    float2 s[16], am[16];
    {
        const float *ck = ckp + (size_t)(t0 / kCkB) * CKF;
        ld_row(s, ck + moff);
        ld_row(am, ck + (size_t)D * D + moff);
    }
    float nj = tid < D ? ckp[(size_t)(t0 / kCkB) * CKF + 2 * D * D + tid] : 0.f;
    float dn_acc = 0.f;  // thread j < D: sum over the chunk of dden_t phi(q_t)_j
    // the inputs are loaded one token ahead, so their latency overlaps a token's work
    float nq = 0.f, nk = 0.f, nv = 0.f, nu = 0.f, ndO = 0.f;
    auto fetch = [&](int t) {
        if (t >= t1) return;
        const size_t tok = ((size_t)bh * T + t) * D;
        if (tid < D) {
            nq = io_to_f32(static_cast<const IO *>(p.q)[tok + tid]);
            nk = io_to_f32(static_cast<const IO *>(p.k)[tok + tid]);
            nv = io_to_f32(static_cast<const IO *>(p.v)[tok + tid]);
            nu = io_to_f32(static_cast<const IO *>(p.u)[tok + tid]);
        }
        ndO = io_to_f32(static_cast<const IO *>(p.dO)[tok + row]);
    };
    fetch(t0);
    for (int t = t0; t < t1; ++t) {
        if (t % kCkB == 0 && t != t0) {
            float *ck = ckp + (size_t)(t / kCkB) * CKF;
            st_row(ck + moff, s);
            st_row(ck + (size_t)D * D + moff, am);
            if (tid < D) ck[2 * D * D + tid] = nj;
        }
        float *rt = rec + (size_t)t * REC;
        const float qj = nq, kj = nk, vj = nv, uj = nu, dOi = ndO;
        fetch(t + 1);
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
        // z = A u, y = A k_hat, S k_hat, S phi(q) (all with the state before token t)
        const float z = dot_row<TPR>(am, v_u + vo);
        const float y = dot_row<TPR>(am, v_kh + vo);
        const float sk = dot_row<TPR>(s, v_kh + vo);
        const float sq = dot_row<TPR>(s, v_fq + vo);
        float p1 = 0.f, p2 = 0.f, p4 = 0.f;
        if (part == 0) {
            p1 = v_u[vidx(row)] * z;
            p2 = v_kh[vidx(row)] * z;
            p4 = dOi * sq;
            v_z[vidx(row)] = z;
            rt[D + row] = z;
        }
        const float4 r2 = block_sum4<NW>(p1, p2, tid < D ? fq * nj : 0.f, p4, s_red[1]);
        const float beta = 1.f / (1.f + r2.x);
        const float rden = 1.f / (r2.z + kEps);
        const float g = y - beta * r2.y * z;
        const float r = s_v[row] - sk;
        const float4 r3 = block_sum4<NW>(part == 0 ? g * g : 0.f, part == 0 ? g * v_fq[vidx(row)] : 0.f,
                                         part == 0 ? dOi * r : 0.f, 0.f, s_red[2]);
        const float gnorm = sqrtf(r3.x);
        const float inv = 1.f / fmaxf(gnorm, kEps);
        // dO . o_t with S_t phi(q) = S_{t-1} phi(q) + r (alpha . phi(q))
        const float dden = -((r2.w + r3.z * (r3.y * inv)) * rden) * rden;
        if (tid < D) dn_acc = fmaf(dden, fq, dn_acc);
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
        for (int cc = 0; cc < 8; ++cc) {
            const float4 zz = zp[cc], al = ap[cc];
            am[2 * cc] = fma2(mb, mul2(zi, lo2(zz)), am[2 * cc]);
            am[2 * cc + 1] = fma2(mb, mul2(zi, hi2(zz)), am[2 * cc + 1]);
            s[2 * cc] = fma2(r2v, lo2(al), s[2 * cc]);
            s[2 * cc + 1] = fma2(r2v, hi2(al), s[2 * cc + 1]);
        }
        __syncthreads();
    }
    if (t1 == T) {  // the final state, for the reverse sweeps of the last chunk
        float *ck = ckp + (size_t)a.NCK * CKF;
        st_row(ck + moff, s);
        st_row(ck + (size_t)D * D + moff, am);
        if (tid < D) ck[2 * D * D + tid] = nj;
    }
    if (tid < D) a.dnsum[((size_t)bh * NC + c) * D + tid] = dn_acc;

    // ---- maps from the records, tokens in reverse ----
    float2 P[16], H[16], Qt[16];
    set_diag(P, row, c0, 1.f);
    set_diag(H, row, c0, 0.f);
    set_diag(Qt, row, c0, 1.f);
    for (int t = t1 - 1; t >= t0; --t) {
        const size_t tok = ((size_t)bh * T + t) * D;
        const float *rt = rec + (size_t)t * REC;
        if (tid < D) {
            v_kh[vidx(tid)] = rt[tid];
            v_z[vidx(tid)] = rt[D + tid];
            v_al[vidx(tid)] = rt[2 * D + tid];
            v_u[vidx(tid)] = io_to_f32(static_cast<const IO *>(p.u)[tok + tid]);
            v_fq[vidx(tid)] = phi_elu1(io_to_f32(static_cast<const IO *>(p.q)[tok + tid]));
        }
        __syncthreads();
        const float beta = rt[4 * D + 1], rden = rt[4 * D + 3];
        const float dnum = io_to_f32(static_cast<const IO *>(p.dO)[tok + row]) * rden;
        // Psi: + dnum phi(q)^T, then times (I - alpha k_hat^T); Phi: times (I - alpha k_hat^T)
        axpy_row(H, dnum, v_fq + vo);
        const float ha = dot_row<TPR>(H, v_al + vo);
        const float pa = dot_row<TPR>(P, v_al + vo);
        const float qz = dot_row<TPR>(Qt, v_z + vo);
        axpy_row(H, -ha, v_kh + vo);
        axpy_row(P, -pa, v_kh + vo);
        // Q^T <- Q^T K_t^T = Q^T (I - beta z u^T)
        axpy_row(Qt, -beta * qz, v_u + vo);
        __syncthreads();
    }
    float *mp = a.maps + ((size_t)bh * NC + c) * 3 * D * D;
    st_row(mp + moff, P);
    st_row(mp + (size_t)D * D + moff, H);
    st_row(mp + 2 * (size_t)D * D + moff, Qt);
}

// Loads the state (S or A, and n) after token t_end - 1 of a chunk: the next
// chunk's start checkpoint, or the final-state slot for the last chunk.
template <int D>
__device__ __forceinline__ const float *end_slot(const BcArgs &a, const float *ckp, int t_end) {
    return ckp + (size_t)(t_end == a.p.T ? a.NCK : t_end / kCkB) * Bc<D>::CKF;
}

// ---------------------------------------------------------------------------
// reverse sweep of one chunk, S part, from the exact dS and dn at its end:
// dq, dv, dg_t and the S and n parts of dk_hat; Omega_c
// ---------------------------------------------------------------------------
template <int D, typename IO>
__global__ void __launch_bounds__(Bc<D>::NT, Bc<D>::MINB) bc_spart_kernel(BcArgs a) {
    using K = Bc<D>;
    constexpr int TPR = K::TPR, VLEN = K::VLEN, NW = K::NW, REC = K::REC, CKF = K::CKF, LDC = K::LDC;
    __shared__ __align__(16) float v_kh[VLEN], v_u[VLEN], v_fq[VLEN], v_z[VLEN], v_al[VLEN], v_dg[VLEN];
    __shared__ __align__(16) float s_r[D], s_dO[D], s_w[D];
    extern __shared__ __align__(16) float s_dyn[];  // three column-sum buffers [D][LDC]
    float *colA = s_dyn, *colB = s_dyn + D * LDC, *colC = s_dyn + 2 * D * LDC;
    __shared__ __align__(16) float4 s_red[3][NW];
    __shared__ float s_sc[4];
    const BwdParams &p = a.p;
    const int NC = a.L.NC, C = a.L.C, T = p.T;
    const int c = (int)(blockIdx.x % (unsigned)NC), bh = (int)(blockIdx.x / (unsigned)NC);
    const int tid = threadIdx.x, row = tid / TPR, part = tid % TPR, c0 = part * 32, vo = part * kPart;
    const int t0 = c * C, t1 = min(T, t0 + C);
    const size_t moff = (size_t)row * D + c0;
    const float *rec = a.rec + (size_t)bh * T * REC;
    const float *ckp = a.ckp + (size_t)bh * (a.NCK + 1) * CKF;
    float *tokv = a.tokv + (size_t)bh * T * 2 * D;

    float2 s[16], ds[16], X[16];
    const float *ce = end_slot<D>(a, ckp, t1);
    ld_row(s, ce + moff);
    float nj = tid < D ? ce[2 * D * D + tid] : 0.f;
    ld_row(ds, a.dS_end + ((size_t)bh * NC + c) * D * D + moff);
    float dnj = tid < D ? a.dn_end[((size_t)bh * NC + c) * D + tid] : 0.f;
    set_diag(X, row, c0, 0.f);

    // the token's record and inputs are loaded one token ahead, so their latency
    // overlaps a token's work
    float nkh = 0.f, nz = 0.f, nal = 0.f, nr = 0.f, nq = 0.f, nu = 0.f, ndO = 0.f, nsc = 0.f;
    auto fetch = [&](int t) {
        if (t < t0) return;
        const size_t tok = ((size_t)bh * T + t) * D;
        const float *rt = rec + (size_t)t * REC;
        if (tid < D) {
            nkh = rt[tid];
            nz = rt[D + tid];
            nal = rt[2 * D + tid];
            nr = rt[3 * D + tid];
            nq = io_to_f32(static_cast<const IO *>(p.q)[tok + tid]);
            nu = io_to_f32(static_cast<const IO *>(p.u)[tok + tid]);
            ndO = io_to_f32(static_cast<const IO *>(p.dO)[tok + tid]);
        }
        if (tid < 4) nsc = rt[4 * D + tid];
    };
    fetch(t1 - 1);
    for (int t = t1 - 1; t >= t0; --t) {
        if ((t + 1) % kCkB == 0 && t + 1 < t1) {  // re-anchor: the state after token t
            const float *ck = ckp + (size_t)((t + 1) / kCkB) * CKF;
            ld_row(s, ck + moff);
            if (tid < D) nj = ck[2 * D * D + tid];
        }
        const size_t tok = ((size_t)bh * T + t) * D;
        const float khj = nkh, alj = nal, qj = nq, fqj = phi_elu1(qj);
        if (tid < D) {
            v_kh[vidx(tid)] = khj;
            v_z[vidx(tid)] = nz;
            v_al[vidx(tid)] = alj;
            v_u[vidx(tid)] = nu;
            v_fq[vidx(tid)] = fqj;
            s_r[tid] = nr;
            s_dO[tid] = ndO;
        }
        if (tid < 4) s_sc[tid] = nsc;
        fetch(t - 1);
        __syncthreads();
        const float beta = s_sc[1], gnorm = s_sc[2], rden = s_sc[3];
        const float4 *kp = reinterpret_cast<const float4 *>(v_kh + vo);
        const float4 *fp = reinterpret_cast<const float4 *>(v_fq + vo);
        const float4 *alp = reinterpret_cast<const float4 *>(v_al + vo);

        // ---- rows: readout and state adjoints ----
        const float num = dot_row<TPR>(s, v_fq + vo);
        const float dOi = s_dO[row];
        const float dnum = dOi * rden;
        const float ri = s_r[row];
        const float2 dn2 = f2(dnum);
        float *cA = colA + row * LDC + c0;
        float *cB = colB + row * LDC + c0;
        float *cC = colC + row * LDC + c0;
        float2 dra = f2(0.f);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
            const float4 f4 = fp[cc], al4 = alp[cc];
            reinterpret_cast<float4 *>(cA)[cc] = make_float4(dnum * s[2 * cc].x, dnum * s[2 * cc].y,
                                                             dnum * s[2 * cc + 1].x, dnum * s[2 * cc + 1].y);
            ds[2 * cc] = fma2(dn2, lo2(f4), ds[2 * cc]);
            ds[2 * cc + 1] = fma2(dn2, hi2(f4), ds[2 * cc + 1]);
            dra = fma2(ds[2 * cc], lo2(al4), dra);
            dra = fma2(ds[2 * cc + 1], hi2(al4), dra);
        }
        float dr = hsum2(dra);
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) dr += __shfl_xor_sync(0xffffffffu, dr, o);
        if (part == 0 && p.dv) p.dv[tok + row] = dr;
        const float2 mri = f2(-ri), dsk = f2(-dr);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
            const float4 al4 = alp[cc], k4 = kp[cc];
            reinterpret_cast<float4 *>(cB)[cc] = make_float4(ri * ds[2 * cc].x, ri * ds[2 * cc].y,
                                                             ri * ds[2 * cc + 1].x, ri * ds[2 * cc + 1].y);
            s[2 * cc] = fma2(mri, lo2(al4), s[2 * cc]);
            s[2 * cc + 1] = fma2(mri, hi2(al4), s[2 * cc + 1]);
            const float2 s0 = mul2(dsk, s[2 * cc]), s1 = mul2(dsk, s[2 * cc + 1]);
            reinterpret_cast<float4 *>(cC)[cc] = make_float4(s0.x, s0.y, s1.x, s1.y);
            ds[2 * cc] = fma2(dsk, lo2(k4), ds[2 * cc]);
            ds[2 * cc + 1] = fma2(dsk, hi2(k4), ds[2 * cc + 1]);
        }
        const float o_i = num * rden;
        const float4 R1 = block_sum4<NW>(part == 0 ? dOi * o_i : 0.f, part == 0 ? ri * dr : 0.f, 0.f, 0.f,
                                         s_red[0]);
        // ---- columns: dq, dn, dalpha -> dg, the S and n parts of dk_hat; undo n ----
        if (tid < D) {
            const int j = tid;
            const float dden = -R1.x * rden;
            float dfq = dden * nj, dal = 0.f, stdsk = 0.f;
            for (int i = 0; i < D; ++i) {
                dfq += colA[i * LDC + j];
                dal += colB[i * LDC + j];
                stdsk += colC[i * LDC + j];
            }
            if (p.dq) p.dq[tok + j] = dfq * (qj > 0.f ? 1.f : expf(qj));
            dnj = fmaf(dden, fqj, dnj);
            const float dg = gnorm > kEps ? (dal - alj * R1.y) / gnorm : dal / kEps;
            v_dg[vidx(j)] = dg;
            tokv[(size_t)t * 2 * D + j] = dg;
            tokv[(size_t)t * 2 * D + D + j] = dnj * (khj > 0.f ? 1.f : expf(khj)) + stdsk;
            nj -= phi_elu1(khj);
        }
        __syncthreads();
        // ---- Omega: X' = X + sym(dg k_hat^T); X <- K X' K^T, K = I - beta u z^T ----
        const float dgi = v_dg[vidx(row)], khi = v_kh[vidx(row)];
        axpy_row(X, 0.5f * dgi, v_kh + vo);
        axpy_row(X, 0.5f * khi, v_dg + vo);
        const float w = dot_row<TPR>(X, v_z + vo);  // X' z (X' symmetric)
        if (part == 0) s_w[row] = w;
        const float4 R2 = block_sum4<NW>(part == 0 ? v_z[vidx(row)] * w : 0.f, 0.f, 0.f, 0.f, s_red[1]);
        const float ui = v_u[vidx(row)];
        // row i of X' - beta u w^T - beta w u^T + beta^2 (z.w) u u^T (s_w in plain layout)
        axpy_row(X, -beta * ui, s_w + c0);
        axpy_row(X, -beta * w + beta * beta * R2.x * ui, v_u + vo);
        __syncthreads();
    }
    st_row(a.om + ((size_t)bh * NC + c) * D * D + moff, X);
}

// ---------------------------------------------------------------------------
// chains along the chunks (CTA = unit), from the last chunk
// ---------------------------------------------------------------------------
// y = x M for the row slices of x (staged in sx, row stride LDC), M in sm (D x D)
template <int D>
__device__ __forceinline__ void row_times(float2 (&y)[16], const float *sx, const float *sm, int row, int c0) {
    constexpr int LDC = Bc<D>::LDC;
#pragma unroll 4
    for (int k = 0; k < D; ++k) {
        const float2 xk = f2(sx[row * LDC + k]);
        const float4 *mr = reinterpret_cast<const float4 *>(sm + k * D + c0);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
            const float4 m = mr[cc];
            y[2 * cc] = fma2(xk, lo2(m), y[2 * cc]);
            y[2 * cc + 1] = fma2(xk, hi2(m), y[2 * cc + 1]);
        }
    }
}

// dS_start = dS_end Phi_c + Psi_c and dn_start = dn_end + dn_sum_c; dS0, dn0.
template <int D>
__global__ void __launch_bounds__(Bc<D>::NT) bc_chain_s_kernel(BcArgs a) {
    using K = Bc<D>;
    constexpr int NT = K::NT, LDC = K::LDC;
    extern __shared__ __align__(16) float s_dyn[];
    float *sx = s_dyn, *sm = s_dyn + D * LDC;
    const BwdParams &p = a.p;
    const int NC = a.L.NC, bh = (int)blockIdx.x;
    const int tid = threadIdx.x, row = tid / K::TPR, part = tid % K::TPR, c0 = part * 32;
    const size_t moff = (size_t)row * D + c0;
    float2 x[16];
    if (p.dS_T) ld_row(x, p.dS_T + (size_t)bh * D * D + moff);
    else set_diag(x, row, c0, 0.f);
    float dn = (tid < D && p.dn_T) ? p.dn_T[(size_t)bh * D + tid] : 0.f;
    for (int c = NC - 1; c >= 0; --c) {
        st_row(a.dS_end + ((size_t)bh * NC + c) * D * D + moff, x);
        if (tid < D) a.dn_end[((size_t)bh * NC + c) * D + tid] = dn;
        const float *mp = a.maps + ((size_t)bh * NC + c) * 3 * D * D;
        st_row(sx + row * LDC + c0, x);
        for (int i = tid; i < D * D / 4; i += NT)
            reinterpret_cast<float4 *>(sm)[i] = reinterpret_cast<const float4 *>(mp)[i];  // Phi
        __syncthreads();
        ld_row(x, mp + (size_t)D * D + moff);  // Psi
        row_times<D>(x, sx, sm, row, c0);
        if (tid < D) dn += a.dnsum[((size_t)bh * NC + c) * D + tid];
        __syncthreads();
    }
    if (p.dS0) st_row(p.dS0 + (size_t)bh * D * D + moff, x);
    if (tid < D && p.dn0) p.dn0[(size_t)bh * D + tid] = dn;
}

// X_start = Q_c X_end Q_c^T + Omega_c for the symmetric part X of dA, from
// sym(dA_T); xs_end per chunk and xs0.
template <int D>
__global__ void __launch_bounds__(Bc<D>::NT) bc_chain_x_kernel(BcArgs a) {
    using K = Bc<D>;
    constexpr int NT = K::NT, LDC = K::LDC;
    extern __shared__ __align__(16) float s_dyn[];
    float *sx = s_dyn, *sm = s_dyn + D * LDC;
    const BwdParams &p = a.p;
    const int NC = a.L.NC, bh = (int)blockIdx.x;
    const int tid = threadIdx.x, row = tid / K::TPR, part = tid % K::TPR, c0 = part * 32;
    const size_t moff = (size_t)row * D + c0;
    float2 x[16];
    set_diag(x, row, c0, 0.f);
    if (p.dA_T) {
        const float *g = p.dA_T + (size_t)bh * D * D;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int c = c0 + 2 * j;
            x[j] = make_float2(0.5f * (g[row * D + c] + g[c * D + row]), 0.5f * (g[row * D + c + 1] + g[(c + 1) * D + row]));
        }
    }
    for (int c = NC - 1; c >= 0; --c) {
        st_row(a.xs_end + ((size_t)bh * NC + c) * D * D + moff, x);
        const float *qt = a.maps + ((size_t)bh * NC + c) * 3 * D * D + 2 * (size_t)D * D;  // Q^T
        st_row(sx + row * LDC + c0, x);
        for (int i = tid; i < D * D / 4; i += NT)
            reinterpret_cast<float4 *>(sm)[i] = reinterpret_cast<const float4 *>(qt)[i];
        __syncthreads();
        float2 y[16];  // Y = X Q^T
        set_diag(y, row, c0, 0.f);
        row_times<D>(y, sx, sm, row, c0);
        __syncthreads();
        st_row(sx + row * LDC + c0, y);
        __syncthreads();
        // Z = Q Y: row i = sum_k Q^T[k][i] Y[k]
        ld_row(x, a.om + ((size_t)bh * NC + c) * D * D + moff);  // + Omega
#pragma unroll 4
        for (int k = 0; k < D; ++k) {
            const float2 qk = f2(sm[k * D + row]);
            const float4 *yr = reinterpret_cast<const float4 *>(sx + k * LDC + c0);
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const float4 m = yr[cc];
                x[2 * cc] = fma2(qk, lo2(m), x[2 * cc]);
                x[2 * cc + 1] = fma2(qk, hi2(m), x[2 * cc + 1]);
            }
        }
        __syncthreads();
    }
    st_row(a.xs0 + (size_t)bh * D * D + moff, x);
}

// ---------------------------------------------------------------------------
// reverse sweep of one chunk, A part, from the exact symmetric dA at its end:
// du, dk (with the stored S and n parts of dk_hat), the antisymmetric sum
// ---------------------------------------------------------------------------
template <int D, typename IO>
__global__ void __launch_bounds__(Bc<D>::NT, Bc<D>::MINB) bc_final_kernel(BcArgs a) {
    using K = Bc<D>;
    constexpr int TPR = K::TPR, VLEN = K::VLEN, NW = K::NW, REC = K::REC, CKF = K::CKF;
    __shared__ __align__(16) float v_kh[VLEN], v_z[VLEN], v_u[VLEN], v_dg[VLEN], v_dz[VLEN];
    __shared__ __align__(16) float s_w[D], s_dkh[D];
    __shared__ __align__(16) float4 s_red[2][NW];
    __shared__ float s_sc[4];
    const BwdParams &p = a.p;
    const int NC = a.L.NC, C = a.L.C, T = p.T;
    const int c = (int)(blockIdx.x % (unsigned)NC), bh = (int)(blockIdx.x / (unsigned)NC);
    const int tid = threadIdx.x, row = tid / TPR, part = tid % TPR, c0 = part * 32, vo = part * kPart;
    const int t0 = c * C, t1 = min(T, t0 + C);
    const size_t moff = (size_t)row * D + c0;
    const float *rec = a.rec + (size_t)bh * T * REC;
    const float *ckp = a.ckp + (size_t)bh * (a.NCK + 1) * CKF;
    const float *tokv = a.tokv + (size_t)bh * T * 2 * D;

    float2 am[16], X[16], as[16];
    ld_row(am, end_slot<D>(a, ckp, t1) + (size_t)D * D + moff);
    ld_row(X, a.xs_end + ((size_t)bh * NC + c) * D * D + moff);
    set_diag(as, row, c0, 0.f);

    // the token's record, u and gate terms are loaded one token ahead, so their
    // latency overlaps a token's work
    float nkh = 0.f, nz = 0.f, nu = 0.f, ndg = 0.f, ndk = 0.f, nsc = 0.f;
    auto fetch = [&](int t) {
        if (t < t0) return;
        const size_t tok = ((size_t)bh * T + t) * D;
        const float *rt = rec + (size_t)t * REC;
        if (tid < D) {
            nkh = rt[tid];
            nz = rt[D + tid];
            nu = io_to_f32(static_cast<const IO *>(p.u)[tok + tid]);
            ndg = tokv[(size_t)t * 2 * D + tid];
            ndk = tokv[(size_t)t * 2 * D + D + tid];
        }
        if (tid < 4) nsc = rt[4 * D + tid];
    };
    fetch(t1 - 1);
    for (int t = t1 - 1; t >= t0; --t) {
        if ((t + 1) % kCkB == 0 && t + 1 < t1)  // re-anchor: A after token t
            ld_row(am, ckp + (size_t)((t + 1) / kCkB) * CKF + (size_t)D * D + moff);
        const size_t tok = ((size_t)bh * T + t) * D;
        const float khj = nkh;
        if (tid < D) {
            v_kh[vidx(tid)] = khj;
            v_z[vidx(tid)] = nz;
            v_u[vidx(tid)] = nu;
            v_dg[vidx(tid)] = ndg;
            s_dkh[tid] = ndk;
        }
        if (tid < 4) s_sc[tid] = nsc;
        fetch(t - 1);
        __syncthreads();
        const float knorm = s_sc[0], beta = s_sc[1];
        const float dgi = v_dg[vidx(row)], khi = v_kh[vidx(row)], zi = v_z[vidx(row)], ui = v_u[vidx(row)];
        // X' = X + sym(dg k_hat^T); w = X' z; A_t dg
        axpy_row(X, 0.5f * dgi, v_kh + vo);
        axpy_row(X, 0.5f * khi, v_dg + vo);
        const float w = dot_row<TPR>(X, v_z + vo);
        const float adg = dot_row<TPR>(am, v_dg + vo);
        if (part == 0) {
            s_w[row] = w;
            s_dkh[row] += adg;
        }
        const float4 R = block_sum4<NW>(part == 0 ? zi * w : 0.f, 0.f, 0.f, 0.f, s_red[0]);
        const float ds1 = beta * beta * R.x;  // beta^2 z^T X' z
        const float dzi = -2.f * beta * w + ds1 * ui;
        if (part == 0) v_dz[vidx(row)] = dzi;
        __syncthreads();
        // undo the penalty update (A_{t-1} = A_t + beta z z^T), then du = ds1 z + A_{t-1} dz
        axpy_row(am, beta * zi, v_z + vo);
        const float adz = dot_row<TPR>(am, v_dz + vo);
        if (part == 0 && p.du) p.du[tok + row] = ds1 * zi + adz;
        // antisymmetric part: asym(dg k_hat^T + dz u^T), row i
        axpy_row(as, 0.5f * dgi, v_kh + vo);
        axpy_row(as, -0.5f * khi, v_dg + vo);
        axpy_row(as, 0.5f * dzi, v_u + vo);
        axpy_row(as, -0.5f * ui, v_dz + vo);
        // X <- X' - beta u w^T - beta w u^T + beta^2 (z.w) u u^T (s_w in plain layout)
        axpy_row(X, -beta * ui, s_w + c0);
        axpy_row(X, -beta * w + beta * beta * R.x * ui, v_u + vo);
        // dk = (dk_hat - k_hat (k_hat . dk_hat)) / |k|
        const float dkh = tid < D ? s_dkh[tid] : 0.f;
        const float4 R4 = block_sum4<NW>(tid < D ? khj * dkh : 0.f, 0.f, 0.f, 0.f, s_red[1]);
        if (tid < D && p.dk) p.dk[tok + tid] = knorm > kEps ? (dkh - khj * R4.x) / knorm : dkh / kEps;
        __syncthreads();
    }
    st_row(a.asum + ((size_t)bh * NC + c) * D * D + moff, as);
}

// dA0 = X_start + asym(dA_T) + the chunks' antisymmetric sums (CTA = unit).
template <int D>
__global__ void __launch_bounds__(Bc<D>::NT) bc_reduce_kernel(BcArgs a) {
    using K = Bc<D>;
    const BwdParams &p = a.p;
    const int NC = a.L.NC, bh = (int)blockIdx.x;
    const int tid = threadIdx.x, row = tid / K::TPR, part = tid % K::TPR, c0 = part * 32;
    const size_t moff = (size_t)row * D + c0;
    float2 x[16], y[16];
    ld_row(x, a.xs0 + (size_t)bh * D * D + moff);
    if (p.dA_T) {
        const float *g = p.dA_T + (size_t)bh * D * D;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int cc = c0 + 2 * j;
            x[j].x += 0.5f * (g[row * D + cc] - g[cc * D + row]);
            x[j].y += 0.5f * (g[row * D + cc + 1] - g[(cc + 1) * D + row]);
        }
    }
    for (int c = 0; c < NC; ++c) {
        ld_row(y, a.asum + ((size_t)bh * NC + c) * D * D + moff);
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = add2(x[j], y[j]);
    }
    st_row(p.dA0 + (size_t)bh * D * D + moff, x);
}

template <typename Kern>
cudaError_t smem_attr(Kern k, size_t bytes) {
    return bytes > 48 * 1024 ? cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes)
                             : cudaSuccess;
}

template <int D, typename IO>
cudaError_t launch_bc_t(const BcArgs &a, cudaStream_t st) {
    using K = Bc<D>;
    const long long BH = a.p.BH, grid = BH * a.L.NC;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const size_t chain_smem = ((size_t)D * K::LDC + (size_t)D * D) * sizeof(float);
    const size_t col_smem = 3 * (size_t)D * K::LDC * sizeof(float);
    cudaError_t e;
    if ((e = smem_attr(bc_chain_s_kernel<D>, chain_smem)) != cudaSuccess) return e;
    if ((e = smem_attr(bc_chain_x_kernel<D>, chain_smem)) != cudaSuccess) return e;
    if ((e = smem_attr(bc_spart_kernel<D, IO>, col_smem)) != cudaSuccess) return e;
    bc_starts_kernel<D><<<(unsigned)grid, K::NT, 0, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bc_fwd_maps_kernel<D, IO><<<(unsigned)grid, K::NT, 0, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bc_chain_s_kernel<D><<<(unsigned)BH, K::NT, chain_smem, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bc_spart_kernel<D, IO><<<(unsigned)grid, K::NT, col_smem, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bc_chain_x_kernel<D><<<(unsigned)BH, K::NT, chain_smem, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bc_final_kernel<D, IO><<<(unsigned)grid, K::NT, 0, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (a.p.dA0) {
        bc_reduce_kernel<D><<<(unsigned)BH, K::NT, 0, st>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace of the chunked backward: the forward's layout and workspace
// first, then its scratch outputs, the records and checkpoints, the chunk
// maps and chains, and the per-token dg and dk_hat parts (byte offsets).
struct BcLayout {
    ChunkLayout L{};
    int NCK = 0;
    bool ok = false;
    size_t sT = 0, aT = 0, nT = 0, rec = 0, ckp = 0, maps = 0, dnsum = 0, dn_end = 0, dS_end = 0, om = 0,
           xs_end = 0, xs0 = 0, asum = 0, tokv = 0, total = 0;
};

// The backward's chunk length.  Each of its three sweeps runs one C-token
// chain per CTA, three CTAs per SM at d = 64 (about eight at d = 32), on 152
// SMs: the fewest waves of the shortest chains, plus the chains along the
// chunks (about six token steps a chunk).  For 16 units of 65536 tokens that
// is 28 chunks of 2368 tokens, one wave, where the forward's 38 chunks of 1728
// take two.
int bc_chunk(int BH, int T, int d) {
    const long long slots = 152LL * (d == 64 ? 3 : 8);
    int best = 64;
    long long best_cost = -1;
    for (int m = 1; m <= (T + 63) / 64; ++m) {
        const long long C = 64LL * m, NC = (T + C - 1) / C;
        const long long cost = ((long long)BH * NC + slots - 1) / slots * C + 6 * NC;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = (int)C;
        }
    }
    return best;
}

BcLayout bc_layout(int BH, int T, int d, bool bf16) {
    BcLayout b;
    if (BH <= 0 || T <= 0 || (d != 32 && d != 64)) return b;
    b.L = chunk_layout(BH, T, d, bc_chunk(BH, T, d), bf16 && d == 64);
    if (b.L.NC < 2 || b.L.C % kCkB != 0 || b.L.C % b.L.CA != 0) return b;
    const size_t bh = (size_t)BH, t = (size_t)T, dd = (size_t)d * d, nc = (size_t)b.L.NC;
    b.NCK = (T + kCkB - 1) / kCkB;
    size_t off = al256(b.L.total);
    b.sT = off; off = al256(off + bh * dd * 4);
    b.aT = off; off = al256(off + bh * dd * 4);
    b.nT = off; off = al256(off + bh * d * 4);
    b.rec = off; off = al256(off + bh * t * (4 * (size_t)d + 4) * 4);
    b.ckp = off; off = al256(off + bh * ((size_t)b.NCK + 1) * (2 * dd + d) * 4);
    b.maps = off; off = al256(off + bh * nc * 3 * dd * 4);
    b.dnsum = off; off = al256(off + bh * nc * d * 4);
    b.dn_end = off; off = al256(off + bh * nc * d * 4);
    b.dS_end = off; off = al256(off + bh * nc * dd * 4);
    b.om = off; off = al256(off + bh * nc * dd * 4);
    b.xs_end = off; off = al256(off + bh * nc * dd * 4);
    b.xs0 = off; off = al256(off + bh * dd * 4);
    b.asum = off; off = al256(off + bh * nc * dd * 4);
    b.tokv = off; off = al256(off + bh * t * 2 * d * 4);
    b.total = off;
    b.ok = true;
    return b;
}

}  // namespace

size_t backward_chunk_bytes(int BH, int T, int d) {
    const BcLayout a = bc_layout(BH, T, d, true), b = bc_layout(BH, T, d, false);
    const size_t x = a.ok ? a.total : 0, y = b.ok ? b.total : 0;
    return x > y ? x : y;
}

cudaError_t launch_backward_chunk(const BwdParams &p, cudaStream_t st, bool *used) {
    *used = false;
    const BcLayout b = bc_layout(p.BH, p.T, p.d, p.io_bf16 != 0);
    if (!b.ok) return cudaSuccess;
    int *err = api_device_err_word();
    if (!err) return cudaGetLastError();
    unsigned char *ws = reinterpret_cast<unsigned char *>(p.ws);
    // the chunked forward: chunk-start states S^(c), M^(c), n^(c) in its workspace
    FwdParams f{};
    f.q = p.q; f.k = p.k; f.v = p.v; f.u = p.u;
    f.o = nullptr;  // the output pass is skipped
    f.S0 = p.S0; f.A0 = p.A0; f.n0 = p.n0;
    f.S_T = reinterpret_cast<float *>(ws + b.sT);
    f.A_T = reinterpret_cast<float *>(ws + b.aT);
    f.n_T = reinterpret_cast<float *>(ws + b.nT);
    f.BH = p.BH; f.T = p.T; f.d = p.d; f.io_bf16 = p.io_bf16; f.lambda0 = p.lambda0;
    f.err = err;
    f.wait_limit_ns = api_wait_limit_ns();
    f.ws = ws;
    f.ws_bytes = b.L.total;
    f.chunk = b.L.C;
    // the SIMT passes: their fp32 gates keep the chunk-start states, from which the
    // sweeps below rebuild every token's state, at fp32 accuracy (the tensor-core
    // passes hand fp16 gates on, which is within the forward's bf16 bar but shows
    // in the gradients)
    f.rows_tc = 0;
    f.skip_out = 1;  // the sweeps recompute what they need of the readout
    int nf = 0;
    f.launches = &nf;
    cudaError_t e = launch_chunk(f, b.L, st);
    if (e != cudaSuccess) return e;
    if (p.launches) *p.launches = nf + (p.dA0 ? 7 : 6);
    BcArgs a{};
    a.p = p;
    a.L = b.L;
    a.fws = ws;
    a.NCK = b.NCK;
    a.rec = reinterpret_cast<float *>(ws + b.rec);
    a.ckp = reinterpret_cast<float *>(ws + b.ckp);
    a.maps = reinterpret_cast<float *>(ws + b.maps);
    a.dnsum = reinterpret_cast<float *>(ws + b.dnsum);
    a.dn_end = reinterpret_cast<float *>(ws + b.dn_end);
    a.dS_end = reinterpret_cast<float *>(ws + b.dS_end);
    a.om = reinterpret_cast<float *>(ws + b.om);
    a.xs_end = reinterpret_cast<float *>(ws + b.xs_end);
    a.xs0 = reinterpret_cast<float *>(ws + b.xs0);
    a.asum = reinterpret_cast<float *>(ws + b.asum);
    a.tokv = reinterpret_cast<float *>(ws + b.tokv);
    *used = true;
    if (p.io_bf16) {
        if (p.d == 32) return launch_bc_t<32, __nv_bfloat16>(a, st);
        return launch_bc_t<64, __nv_bfloat16>(a, st);
    }
    if (p.d == 32) return launch_bc_t<32, float>(a, st);
    return launch_bc_t<64, float>(a, st);
}

}  // namespace vla
