// vla_decode.cu -- streaming decode step: a few tokens (typically one) per
// call for many (batch, head) units, with the state (S, A, n) read from and
// written back to HBM, usually in place ("Variational Linear Attention:
// Stable Associative Memory for Long-Context Transformers", section 5:
// streaming inference with a fixed-size state).
//
// Per token the recurrence is the same as in the sequential kernel
// (sections 2.2-2.3).  What differs is the data movement: there is no
// input-tile pipeline; the state slices are loaded once with coalesced
// 16-byte loads, each token's q, k, v, u are read directly, and the whole
// step is three block reductions:
//   1. |k|^2                                  -> k_hat, phi(k_hat), phi(q)
//   2. u.z, k_hat.z, phi(q).n_t               -> beta, z^T k_hat, denominator
//   3. |g|^2, g.phi(q)                         -> alpha, readout
// The cost is the 2 (2 d^2 + d) fp32 state words read and written per head.
// Thread (row, part) of the TPR = d / 32 threads of a row holds the 16-byte
// chunks c TPR + part (c < 8) of its rows of A and S: a row's threads read
// adjacent chunks, so each warp-wide 16-byte load or store covers whole
// 32-byte sectors (with the 32 columns of a thread in one piece, every
// instruction touched 32 lines for 16 bytes each).
#include "vla_internal.cuh"

namespace vla {
namespace {

template <int D>
struct DecCfg {
    static constexpr int TPR = D / 32;
    static constexpr int NT = D * TPR;
    static constexpr int NW = NT / 32;
};

template <int D, typename IO>
__global__ void __launch_bounds__(DecCfg<D>::NT) decode_kernel(FwdParams p) {
    using C = DecCfg<D>;
    constexpr int TPR = C::TPR, NW = C::NW;
    __shared__ __align__(16) float s_k[D], s_u[D], s_f[D], s_z[D], s_g[D];
    __shared__ __align__(16) float s_v[D];
    __shared__ __align__(16) float4 s_red[3][NW];

    const int tid = threadIdx.x;
    const int row = tid / TPR, part = tid % TPR;
    const int bh = blockIdx.x;
    const int T = p.T;
    const size_t moff = (size_t)bh * D * D + (size_t)row * D;  // row `row`; this thread's chunks c TPR + part
    auto q4 = [&](int c) { return c * TPR + part; };              // 16-byte chunk index within a row

    // state slices (row i, chunks c TPR + part) of A and S; column tid of n
    float2 a[16], s[16];
    if (p.A0) {
        const float4 *src = reinterpret_cast<const float4 *>(p.A0 + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 x = src[q4(c)];
            a[2 * c] = lo2(x);
            a[2 * c + 1] = hi2(x);
        }
    } else {
        const float il = 1.f / p.lambda0;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int j0 = 4 * q4(c);
            a[2 * c] = make_float2(j0 == row ? il : 0.f, j0 + 1 == row ? il : 0.f);
            a[2 * c + 1] = make_float2(j0 + 2 == row ? il : 0.f, j0 + 3 == row ? il : 0.f);
        }
    }
    if (p.S0) {
        const float4 *src = reinterpret_cast<const float4 *>(p.S0 + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 x = src[q4(c)];
            s[2 * c] = lo2(x);
            s[2 * c + 1] = hi2(x);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) s[j] = f2(0.f);
    }
    float nj = 0.f;
    if (tid < D && p.n0) nj = p.n0[(size_t)bh * D + tid];

    for (int t = 0; t < T; ++t) {
        const size_t tok = ((size_t)bh * T + t) * D;
        // ---- 1: token inputs, key norm ----
        float qj = 0.f, kj = 0.f, vj = 0.f, uj = 0.f;
        if (tid < D) {
            qj = io_to_f32(static_cast<const IO *>(p.q)[tok + tid]);
            kj = io_to_f32(static_cast<const IO *>(p.k)[tok + tid]);
            vj = io_to_f32(static_cast<const IO *>(p.v)[tok + tid]);
            uj = io_to_f32(static_cast<const IO *>(p.u)[tok + tid]);
        }
        const float4 r1 = block_sum4<NW>(kj * kj, 0.f, 0.f, 0.f, s_red[0]);
        const float ks = 1.f / fmaxf(sqrtf(r1.x), kEps);
        float fq = 0.f, khj = 0.f;
        if (tid < D) {
            khj = kj * ks;
            fq = phi_elu1(qj);
            nj += phi_elu1(khj);
            s_k[tid] = khj;
            s_u[tid] = uj;
            s_f[tid] = fq;
            s_v[tid] = vj;
        }
        __syncthreads();
        // ---- 2: z = A u, y = A k_hat, S k_hat, S phi(q) ----
        const float4 *up = reinterpret_cast<const float4 *>(s_u);
        const float4 *kp = reinterpret_cast<const float4 *>(s_k);
        const float4 *fp = reinterpret_cast<const float4 *>(s_f);
        float2 za = f2(0.f), ya = f2(0.f), ka = f2(0.f), qa = f2(0.f);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 u4 = up[q4(c)], k4 = kp[q4(c)], f4 = fp[q4(c)];
            za = fma2(a[2 * c], lo2(u4), za);
            za = fma2(a[2 * c + 1], hi2(u4), za);
            ya = fma2(a[2 * c], lo2(k4), ya);
            ya = fma2(a[2 * c + 1], hi2(k4), ya);
            ka = fma2(s[2 * c], lo2(k4), ka);
            ka = fma2(s[2 * c + 1], hi2(k4), ka);
            qa = fma2(s[2 * c], lo2(f4), qa);
            qa = fma2(s[2 * c + 1], hi2(f4), qa);
        }
        float z = hsum2(za), y = hsum2(ya), sk = hsum2(ka), sq = hsum2(qa);
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) {
            z += __shfl_xor_sync(0xffffffffu, z, o);
            y += __shfl_xor_sync(0xffffffffu, y, o);
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
        }
        float p1 = 0.f, p2 = 0.f;
        if (part == 0) {
            p1 = s_u[row] * z;
            p2 = s_k[row] * z;
            s_z[row] = z;
        }
        const float4 r2 = block_sum4<NW>(p1, p2, tid < D ? fq * nj : 0.f, 0.f, s_red[1]);
        const float beta = 1.f / (1.f + r2.x);
        const float rden = 1.f / (r2.z + kEps);
        // ---- 3: gate g = A_t k_hat = y - beta (z.k_hat) z; |g|, g.phi(q) ----
        const float g = y - beta * r2.y * z;
        float p3 = 0.f, p4 = 0.f;
        if (part == 0) {
            p3 = g * g;
            p4 = g * s_f[row];
            s_g[row] = g;
        }
        const float4 r3 = block_sum4<NW>(p3, p4, 0.f, 0.f, s_red[2]);
        const float inv = fminf(rsqrtf(r3.x), 1.f / kEps);
        // ---- updates: A -= beta z z^T (symmetric rounding), S += r alpha^T ----
        const float r = s_v[row] - sk;
        const float2 mb = f2(-beta), zi = f2(z), ri = f2(r * inv);
        const float4 *zp = reinterpret_cast<const float4 *>(s_z);
        const float4 *gp = reinterpret_cast<const float4 *>(s_g);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 zz = zp[q4(c)], gg = gp[q4(c)];
            a[2 * c] = fma2(mb, mul2(zi, lo2(zz)), a[2 * c]);
            a[2 * c + 1] = fma2(mb, mul2(zi, hi2(zz)), a[2 * c + 1]);
            s[2 * c] = fma2(ri, lo2(gg), s[2 * c]);
            s[2 * c + 1] = fma2(ri, hi2(gg), s[2 * c + 1]);
        }
        if (part == 0)
            static_cast<IO *>(p.o)[tok + row] = f32_to_io<IO>(fmaf(r * inv, r3.y, sq) * rden);
        __syncthreads();  // the next token overwrites the shared vectors
    }
    float4 *dA = reinterpret_cast<float4 *>(p.A_T + moff);
    float4 *dS = reinterpret_cast<float4 *>(p.S_T + moff);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        dA[q4(c)] = make_float4(a[2 * c].x, a[2 * c].y, a[2 * c + 1].x, a[2 * c + 1].y);
        dS[q4(c)] = make_float4(s[2 * c].x, s[2 * c].y, s[2 * c + 1].x, s[2 * c + 1].y);
    }
    if (tid < D && p.n_T) p.n_T[(size_t)bh * D + tid] = nj;
}

template <int D, typename IO>
cudaError_t launch_decode_t(const FwdParams &p, cudaStream_t st) {
    mark_launch(p, 0, st);
    decode_kernel<D, IO><<<p.BH, DecCfg<D>::NT, 0, st>>>(p);
    const cudaError_t e = cudaGetLastError();
    mark_launch(p, 1, st);
    return e;
}

}  // namespace

cudaError_t launch_decode(const FwdParams &p, cudaStream_t stream) {
    if (p.BH == 0) return cudaSuccess;
    if (p.io_bf16) {
        switch (p.d) {
            case 32: return launch_decode_t<32, __nv_bfloat16>(p, stream);
            case 64: return launch_decode_t<64, __nv_bfloat16>(p, stream);
            case 128: return launch_decode_t<128, __nv_bfloat16>(p, stream);
        }
    } else {
        switch (p.d) {
            case 32: return launch_decode_t<32, float>(p, stream);
            case 64: return launch_decode_t<64, float>(p, stream);
            case 128: return launch_decode_t<128, float>(p, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace vla
