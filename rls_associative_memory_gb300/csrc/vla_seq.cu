// vla_seq.cu -- token-sequential VLA forward kernel: one CTA per (batch, head)
// (d_h = 64 and 128; d_h = 32 has its own kernel in vla_seq32.cu).
//
// Recurrence ("Variational Linear Attention: Stable Associative Memory for
// Long-Context Transformers", sections 2.2-2.3), per token t:
//   z = A_{t-1} u,  beta = 1 / (1 + u^T z),  A_t = A_{t-1} - beta z z^T
//   g = A_t k_hat = A_{t-1} k_hat - beta z (z^T k_hat),  alpha = g / |g|
//   r = v - S_{t-1} k_hat,  S_t = S_{t-1} + r alpha^T
//   o = S_t phi(q) / (phi(q)^T n_t + eps),  S_t phi(q) = S_{t-1} phi(q) + r (alpha^T phi(q))
//
// Layout of the CTA: thread (row i, part p) owns columns [32p, 32p+32) of row
// i of both A and S in registers (64 fp32), so every matrix-vector product is
// a register dot product plus a shuffle across the d/32 parts of a row, and
// the rank-1 updates need only broadcast reads of z and g from shared memory.
//
// One block-wide reduction per token.  The A chain (z, y of token t) and the
// S chain (gate norm of token t-1) share it: iteration t reduces
// {u_t.z_t, z_t.k_hat_t, |g_{t-1}|^2, g_{t-1}.phi(q_{t-1})}, then applies the
// state write and readout of token t-1.  The S chain therefore lags the A
// chain by one token; it needs no reduction of its own because rows of S
// evolve independently given alpha.
//
// A is updated as A -= beta * (z_i z_j): the product z_i z_j is symmetric in
// (i, j), so A stays exactly symmetric in fp32 (an fma(-beta z_i, z_j, A)
// form drifts ~100x further from the fp64 recursion over 64k tokens).
//
// Inputs stream through shared memory in tiles of TT tokens with 1-D bulk
// async copies (cp.async.bulk, mbarrier completion), double-buffered.  Each
// tile is preprocessed once (k_hat, phi(q), fp32 u, v, the readout
// denominator phi(q_t)^T n_t + eps with n a running sum of phi(k_hat)).
#include "vla_internal.cuh"

namespace vla {
namespace {

template <int D>
struct SeqCfg {
    static constexpr int TPR = D / 32;             // threads per row
    static constexpr int NT = D * TPR;             // threads per CTA
    static constexpr int NW = NT / 32;             // warps per CTA
    static constexpr int VLEN = TPR * kPart;       // floats per skewed vector
    static constexpr int TT = (D == 32) ? 8 : 16;  // tokens per tile
};

template <int D, typename IO>
struct SeqSmem {
    using C = SeqCfg<D>;
    static constexpr size_t bars = 0;                                          // 2 x u64 + abort flag
    static constexpr size_t raw = 128;                                         // [2][4][TT*D] IO
    static constexpr size_t raw_tensor = (size_t)C::TT * D * sizeof(IO);       // bytes of one tensor tile
    static constexpr size_t khat = raw + 2 * 4 * raw_tensor;                   // [2][TT][VLEN]
    static constexpr size_t phiq = khat + 2 * C::TT * C::VLEN * 4;             // [2][TT][VLEN]
    static constexpr size_t uu = phiq + 2 * C::TT * C::VLEN * 4;               // [2][TT][VLEN]
    static constexpr size_t vv = uu + 2 * C::TT * C::VLEN * 4;                 // [2][TT][D]
    static constexpr size_t den = vv + 2 * C::TT * D * 4;                      // [2][TT]
    static constexpr size_t work = den + 2 * C::TT * 4;                        // [TT][D]
    static constexpr size_t zbuf = work + C::TT * D * 4;                       // [2][VLEN]
    static constexpr size_t gbuf = zbuf + 2 * C::VLEN * 4;                     // [2][VLEN]
    static constexpr size_t red = gbuf + 2 * C::VLEN * 4;                      // [2][NW] float4
    static constexpr size_t total = red + 2 * C::NW * 16;
    static_assert(raw_tensor % 16 == 0, "tile rows must be 16-byte multiples");
    static_assert(khat % 16 == 0 && phiq % 16 == 0 && uu % 16 == 0 && zbuf % 16 == 0 &&
                      gbuf % 16 == 0 && red % 16 == 0,
                  "16-byte aligned regions");
};

// Per-tile preprocessing (all threads).  raw: the four tensor tiles of ntok
// tokens; writes k_hat, phi(q), u (skewed fp32 vectors), v, and the
// reciprocals of the readout denominators.  nbase/ncomp (threads tid < D): Kahan-compensated running
// sum of phi(k_hat) over previous tiles, column tid.
template <int D, typename IO>
__device__ __forceinline__ void preprocess_tile(const IO *raw, size_t raw_stride, int ntok, float *khat,
                                                float *phiq, float *uu, float *vv, float *den,
                                                float *work, float &nbase, float &ncomp) {
    using C = SeqCfg<D>;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const IO *rq = raw, *rk = raw + raw_stride, *rv = raw + 2 * raw_stride, *ru = raw + 3 * raw_stride;
    constexpr int M = D / 32;
    for (int tt = warp; tt < ntok; tt += C::NW) {
        float kk[M];
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < M; ++m) {
            kk[m] = io_to_f32(rk[tt * D + lane + 32 * m]);
            ss = fmaf(kk[m], kk[m], ss);
        }
        ss = warp_sum(ss);
        const float ks = 1.f / fmaxf(sqrtf(ss), kEps);
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const int j = lane + 32 * m;
            const float kh = kk[m] * ks;
            khat[tt * C::VLEN + vidx(j)] = kh;
            work[tt * D + j] = phi_elu1(kh);
            phiq[tt * C::VLEN + vidx(j)] = phi_elu1(io_to_f32(rq[tt * D + j]));
            uu[tt * C::VLEN + vidx(j)] = io_to_f32(ru[tt * D + j]);
            vv[tt * D + j] = io_to_f32(rv[tt * D + j]);
        }
    }
    __syncthreads();
    if (tid < D) {
        // n_t = n_base + (phi(k_hat) summed over this tile up to t); work <- phi(q_t)_j n_t,j
        float run = 0.f;
        for (int tt = 0; tt < ntok; ++tt) {
            run += work[tt * D + tid];
            work[tt * D + tid] = phiq[tt * C::VLEN + vidx(tid)] * (nbase + run);
        }
        const float yk = run - ncomp;  // Kahan step for the running base
        const float tk = nbase + yk;
        ncomp = (tk - nbase) - yk;
        nbase = tk;
    }
    __syncthreads();
    for (int tt = warp; tt < ntok; tt += C::NW) {
        float sacc = 0.f;
#pragma unroll
        for (int m = 0; m < M; ++m) sacc += work[tt * D + lane + 32 * m];
        sacc = warp_sum(sacc);
        if (lane == 0) den[tt] = 1.f / (sacc + kEps);  // stored as the reciprocal
    }
}

template <int D, typename IO>
__global__ void __launch_bounds__(SeqCfg<D>::NT, (D == 128) ? 1 : 2) seq_kernel(FwdParams p) {
    using C = SeqCfg<D>;
    using L = SeqSmem<D, IO>;
    constexpr int TT = C::TT, VLEN = C::VLEN, TPR = C::TPR, NW = C::NW;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::bars + 16);
    IO *raw = reinterpret_cast<IO *>(smem + L::raw);
    float *s_khat = reinterpret_cast<float *>(smem + L::khat);
    float *s_phiq = reinterpret_cast<float *>(smem + L::phiq);
    float *s_u = reinterpret_cast<float *>(smem + L::uu);
    float *s_v = reinterpret_cast<float *>(smem + L::vv);
    float *s_den = reinterpret_cast<float *>(smem + L::den);
    float *s_work = reinterpret_cast<float *>(smem + L::work);
    float *s_z = reinterpret_cast<float *>(smem + L::zbuf);
    float *s_g = reinterpret_cast<float *>(smem + L::gbuf);
    float4 *s_red = reinterpret_cast<float4 *>(smem + L::red);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = tid / TPR, part = tid % TPR;
    const int c0 = part * 32, vo = part * kPart;
    const int bh = blockIdx.x;
    const int T = p.T;
    const int ntiles = (T + TT - 1) / TT;
    const size_t tok0 = (size_t)bh * T * D;
    const IO *gsrc[4] = {static_cast<const IO *>(p.q) + tok0, static_cast<const IO *>(p.k) + tok0,
                         static_cast<const IO *>(p.v) + tok0, static_cast<const IO *>(p.u) + tok0};
    IO *gout = static_cast<IO *>(p.o) + tok0;

    // ---- initial state (thread-owned slices) ----
    float2 a[16], s[16];  // columns 2j, 2j+1 of this thread's 32
    const size_t moff = (size_t)bh * D * D + (size_t)row * D + c0;
    if (p.A0) {
        const float4 *src = reinterpret_cast<const float4 *>(p.A0 + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 x = src[c];
            a[2 * c] = lo2(x);
            a[2 * c + 1] = hi2(x);
        }
    } else {
        const float inv_l = 1.f / p.lambda0;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            a[j] = make_float2((c0 + 2 * j == row) ? inv_l : 0.f, (c0 + 2 * j + 1 == row) ? inv_l : 0.f);
    }
    if (p.S0) {
        const float4 *src = reinterpret_cast<const float4 *>(p.S0 + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 x = src[c];
            s[2 * c] = lo2(x);
            s[2 * c + 1] = hi2(x);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) s[j] = f2(0.f);
    }
    float nbase = 0.f, ncomp = 0.f;
    if (tid < D && p.n0) nbase = p.n0[(size_t)bh * D + tid];

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    for (int i = tid; i < 2 * VLEN; i += C::NT) s_z[i] = 0.f;  // z_{-1} = 0
    __syncthreads();

    // tile m -> raw buffer (m & 1); issued by thread 0 only
    auto issue = [&](int m) {
        const int buf = m & 1;
        const int t0 = m * TT;
        const int ntok = min(TT, T - t0);
        const uint32_t bytes = (uint32_t)(ntok * D * sizeof(IO));
        mbar_arrive_expect_tx(&bars[buf], 4 * bytes);
#pragma unroll
        for (int x = 0; x < 4; ++x)
            bulk_g2s(raw + ((size_t)buf * 4 + x) * TT * D, gsrc[x] + (size_t)t0 * D, bytes, &bars[buf]);
    };
    int issued_upto = 0;  // tiles [0, issued_upto) requested (thread 0's view)
    if (tid == 0 && !p.inject) {
        if (ntiles > 0) issue(0);
        if (ntiles > 1) issue(1);
        issued_upto = min(ntiles, 2);
    }

    float beta_prev = 0.f, s2_prev = 0.f, z_prev = 0.f, y_prev = 0.f;
    int failed_tile = -1;

    for (int t = 0; t <= T; ++t) {
        const int tt = t % TT;
        const int m = t / TT;
        if (tt == 0 && t < T) {
            const int buf = m & 1;
            if (!mbar_wait_bounded(&bars[buf], (m >> 1) & 1, p.wait_limit_ns, p.err)) *abort_flag = 1;
            __syncthreads();
            if (*abort_flag) {
                failed_tile = m;
                break;
            }
            preprocess_tile<D, IO>(raw + (size_t)buf * 4 * TT * D, (size_t)TT * D, min(TT, T - t),
                                   s_khat + buf * TT * VLEN, s_phiq + buf * TT * VLEN,
                                   s_u + buf * TT * VLEN, s_v + buf * TT * D, s_den + buf * TT, s_work,
                                   nbase, ncomp);
            __syncthreads();
            if (tid == 0 && m + 2 < ntiles) {
                issue(m + 2);
                issued_upto = m + 3;
            }
        }
        const bool hasA = t < T;
        const bool hasS = t > 0;
        const int bufA = m & 1;
        const int tS = hasS ? t - 1 : 0;
        const int bufS = (tS / TT) & 1, ttS = tS % TT;
        const float *uA = s_u + (bufA * TT + tt) * VLEN;
        const float *kA = s_khat + (bufA * TT + tt) * VLEN;
        const float *kS = s_khat + (bufS * TT + ttS) * VLEN;
        const float *fS = s_phiq + (bufS * TT + ttS) * VLEN;

        // ---- A chain: rank-1 update of token t-1, then z_t = A u_t, y_t = A k_hat_t ----
        const float4 *zp = reinterpret_cast<const float4 *>(s_z + ((t - 1) & 1) * VLEN + vo);
        const float2 mb = f2(-beta_prev), zi = f2(z_prev);
        float2 za = f2(0.f), zb = f2(0.f), ya = f2(0.f), yb = f2(0.f);
        if (hasA) {
            const float4 *up = reinterpret_cast<const float4 *>(uA + vo);
            const float4 *kp = reinterpret_cast<const float4 *>(kA + vo);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 zz = zp[c], uu4 = up[c], kk = kp[c];
                a[2 * c] = fma2(mb, mul2(zi, lo2(zz)), a[2 * c]);
                a[2 * c + 1] = fma2(mb, mul2(zi, hi2(zz)), a[2 * c + 1]);
                za = fma2(a[2 * c], lo2(uu4), za);
                zb = fma2(a[2 * c + 1], hi2(uu4), zb);
                ya = fma2(a[2 * c], lo2(kk), ya);
                yb = fma2(a[2 * c + 1], hi2(kk), yb);
            }
        } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 zz = zp[c];
                a[2 * c] = fma2(mb, mul2(zi, lo2(zz)), a[2 * c]);
                a[2 * c + 1] = fma2(mb, mul2(zi, hi2(zz)), a[2 * c + 1]);
            }
        }
        // ---- S chain reads: S_{t-2} k_hat_{t-1}, S_{t-2} phi(q_{t-1}) ----
        float2 ka = f2(0.f), kb = f2(0.f), qa = f2(0.f), qb = f2(0.f);
        if (hasS) {
            const float4 *kp = reinterpret_cast<const float4 *>(kS + vo);
            const float4 *fp = reinterpret_cast<const float4 *>(fS + vo);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 kk = kp[c], ff = fp[c];
                ka = fma2(s[2 * c], lo2(kk), ka);
                kb = fma2(s[2 * c + 1], hi2(kk), kb);
                qa = fma2(s[2 * c], lo2(ff), qa);
                qb = fma2(s[2 * c + 1], hi2(ff), qb);
            }
        }
        float z = hsum2(add2(za, zb)), y = hsum2(add2(ya, yb));
        float skv = hsum2(add2(ka, kb)), sqv = hsum2(add2(qa, qb));
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) {
            z += __shfl_xor_sync(0xffffffffu, z, o);
            y += __shfl_xor_sync(0xffffffffu, y, o);
            skv += __shfl_xor_sync(0xffffffffu, skv, o);
            sqv += __shfl_xor_sync(0xffffffffu, sqv, o);
        }
        // gate row i of token t-1: g = y - beta (z^T k_hat) z
        const float g = y_prev - beta_prev * s2_prev * z_prev;
        float p1 = 0.f, p2 = 0.f, p3 = 0.f, p4 = 0.f;
        if (part == 0) {
            if (hasA) {
                p1 = uA[vidx(row)] * z;
                p2 = kA[vidx(row)] * z;
                s_z[(t & 1) * VLEN + vidx(row)] = z;
            }
            if (hasS) {
                p3 = g * g;
                p4 = g * fS[vidx(row)];
                s_g[((t - 1) & 1) * VLEN + vidx(row)] = g;
            }
        }
        const float red = warp_reduce4(p1, p2, p3, p4);  // lanes 0/8/16/24: sums of p1..p4
        if constexpr (NW > 1) {
            if ((lane & 7) == 0) reinterpret_cast<float *>(s_red)[((t & 1) * NW + warp) * 4 + (lane >> 3)] = red;
            __syncthreads();
            float4 acc = s_red[(t & 1) * NW];
#pragma unroll
            for (int w = 1; w < NW; ++w) {
                const float4 x = s_red[(t & 1) * NW + w];
                acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
            }
            p1 = acc.x; p2 = acc.y; p3 = acc.z; p4 = acc.w;
        } else {
            p1 = __shfl_sync(0xffffffffu, red, 0);
            p2 = __shfl_sync(0xffffffffu, red, 8);
            p3 = __shfl_sync(0xffffffffu, red, 16);
            p4 = __shfl_sync(0xffffffffu, red, 24);
            __syncwarp();
        }
        const float beta = 1.f / (1.f + p1);
        if (hasS) {
            // ---- state write and readout of token t-1 ----
            const float inv = fminf(rsqrtf(p3), 1.f / kEps);  // 1 / max(|g|, eps)
            const float r = s_v[(bufS * TT + ttS) * D + row] - skv;
            const float ri = r * inv;
            const float2 ri2 = f2(ri);
            const float4 *gp = reinterpret_cast<const float4 *>(s_g + ((t - 1) & 1) * VLEN + vo);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 gg = gp[c];
                s[2 * c] = fma2(ri2, lo2(gg), s[2 * c]);
                s[2 * c + 1] = fma2(ri2, hi2(gg), s[2 * c + 1]);
            }
            if (part == 0) {
                const float num = fmaf(ri, p4, sqv);
                gout[(size_t)tS * D + row] = f32_to_io<IO>(num * s_den[bufS * TT + ttS]);
            }
        }
        beta_prev = beta;
        s2_prev = p2;
        z_prev = z;
        y_prev = y;
    }

    if (failed_tile >= 0) {
        // Let tiles that were requested but not consumed land (bounded wait)
        // before the CTA's shared memory is released; no output is written.
        if (tid == 0)
            for (int m = failed_tile; m < issued_upto; ++m)
                (void)mbar_wait_bounded(&bars[m & 1], (m >> 1) & 1, p.wait_limit_ns, p.err);
        return;
    }

    // ---- final state ----
    {
        float4 *dA = reinterpret_cast<float4 *>(p.A_T + moff);
        float4 *dS = reinterpret_cast<float4 *>(p.S_T + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            dA[c] = make_float4(a[2 * c].x, a[2 * c].y, a[2 * c + 1].x, a[2 * c + 1].y);
            dS[c] = make_float4(s[2 * c].x, s[2 * c].y, s[2 * c + 1].x, s[2 * c + 1].y);
        }
        if (tid < D && p.n_T) p.n_T[(size_t)bh * D + tid] = nbase;
    }
}

template <int D, typename IO>
cudaError_t launch_seq_t(const FwdParams &p, cudaStream_t stream) {
    using C = SeqCfg<D>;
    const size_t smem = SeqSmem<D, IO>::total;
    cudaError_t e = cudaFuncSetAttribute(seq_kernel<D, IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    mark_launch(p, 0, stream);
    seq_kernel<D, IO><<<p.BH, C::NT, smem, stream>>>(p);
    e = cudaGetLastError();
    mark_launch(p, 1, stream);
    return e;
}

}  // namespace

cudaError_t launch_seq(const FwdParams &p, cudaStream_t stream) {
    if (p.BH == 0) return cudaSuccess;
    if (p.d == 32) return launch_seq32(p, stream);  // three warps a (b, h): vla_seq32.cu
    if (p.io_bf16) {
        switch (p.d) {
            case 64: return launch_seq_t<64, __nv_bfloat16>(p, stream);
            case 128: return launch_seq_t<128, __nv_bfloat16>(p, stream);
        }
    } else {
        switch (p.d) {
            case 64: return launch_seq_t<64, float>(p, stream);
            case 128: return launch_seq_t<128, float>(p, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace vla
