// vla_seq32.cu -- token-sequential VLA forward at d_h = 32: one CTA of three
// warps per (batch, head), each warp one stage of the recurrence.
//
// Recurrence ("Variational Linear Attention: Stable Associative Memory for
// Long-Context Transformers", sections 2.2-2.3), per token t:
//   z = A_{t-1} u,  beta = 1 / (1 + u^T z),  A_t = A_{t-1} - beta z z^T
//   g = A_t k_hat = A_{t-1} k_hat - beta z (z^T k_hat),  alpha = g / max(|g|, eps)
//   r = v - S_{t-1} k_hat,  S_t = S_{t-1} + r alpha^T
//   o = S_t phi(q) / (phi(q)^T n_t + eps),  n_t = n_{t-1} + phi(k_hat)
//
// At d = 32 a warp holds a whole 32 x 32 matrix, one row per lane, so the
// matrix-vector products are lane-local dot products over vectors that every
// lane reads from shared memory.  The three parts of the recurrence run in
// their own warps and hand tokens on through a ring of shared-memory slots
// (8 tokens a slot, four slots):
//   warp 2 (inputs): q, k, v, u of a slot's tokens from global memory (the
//     slot two ahead prefetched into L2), k_hat, phi(q), the running n_t and
//     the readout denominators;
//   warp 0 (A chain): the Sherman-Morrison step and the gate rows g_t;
//   warp 1 (S chain): the state write and the readout of o_t.
// The A chain is the longest serial chain; the other two run beside it.
// Each slot has three mbarriers: inputs ready (warp 2 -> 0, 1), gates ready
// (warp 0 -> 1), slot free (warp 1 -> 2); every wait is bounded.
//
// A is updated as A -= w w^T with w = sqrt(beta) z, one FMA per entry: the
// product inside an FMA is exact, so A stays exactly symmetric in fp32.
#include "vla_internal.cuh"

namespace vla {
namespace {

constexpr int kTT = 8;      // tokens per slot
constexpr int kNB = 4;      // slots in the ring
constexpr int kNT32 = 96;   // three warps

// Slot (fp32): k_hat, u, phi(q), v and the gate rows g as [kTT][32] each, then
// the kTT readout factors 1 / (phi(q_t) . n_t + eps).
struct S32Layout {
    static constexpr int kKh = 0, kU = kTT * 32, kF = 2 * kTT * 32, kV = 3 * kTT * 32, kG = 4 * kTT * 32,
                         kDen = 5 * kTT * 32;
    static constexpr int slot = 5 * kTT * 32 + kTT;  // floats
    static constexpr size_t bars = 0;                // full_in[kNB], full_g[kNB], empty[kNB]
    static constexpr size_t flag = 3 * kNB * 8;      // abort flag
    static constexpr size_t zbuf = 128;              // [2][32]: w of the A chain, by token parity
    static constexpr size_t slots = zbuf + 2 * 32 * 4;
    static constexpr size_t total = slots + (size_t)kNB * slot * 4;
};
static_assert(S32Layout::flag + 4 <= S32Layout::zbuf, "control block");
static_assert(S32Layout::slot % 4 == 0 && S32Layout::slots % 16 == 0, "16-byte aligned vectors");

__device__ __forceinline__ void prefetch_l2(const void *ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// try_wait with a suspend-time hint: a waiting thread sleeps until the phase
// completes or about `hint_ns` pass, instead of spinning on the issue slots
// that the chain warps of the SM need.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// All 32 lanes wait for phase `parity` of `bar`.  A lane gives up once another
// warp has aborted, or after limit_ns (then it sets the device error word and
// the abort flag).  The warp goes on only if every lane saw the phase.
__device__ __forceinline__ bool wait_warp(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          const FwdParams &p) {
    constexpr uint32_t kHintNs = 20000;
    bool ok = mbar_try_wait(bar, parity);
    if (!ok) {
        const unsigned long long t0 = globaltimer_ns();
        for (;;) {
            if (mbar_try_wait_sleep(bar, parity, kHintNs)) {
                ok = true;
                break;
            }
            if (*abort_flag) break;
            if ((long long)(globaltimer_ns() - t0) > p.wait_limit_ns) {
                atomicExch(p.err, kDevErrTimeout);
                *abort_flag = 1;
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// Sums of two values over the warp, returned to every lane.
__device__ __forceinline__ float2 warp_sum2(float x, float y) {
    const bool hi = threadIdx.x & 16;
    float a = hi ? y : x;
    a += __shfl_xor_sync(0xffffffffu, hi ? x : y, 16);  // lanes < 16: x, lanes >= 16: y
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    return make_float2(__shfl_sync(0xffffffffu, a, 0), __shfl_sync(0xffffffffu, a, 16));
}

// The four sums over the warp of (x0, x1, x2, x3), returned to every lane: the
// first two exchanges halve the values each lane carries (6 shuffles, then 4
// broadcasts).
__device__ __forceinline__ float4 warp_sum4(float x0, float x1, float x2, float x3) {
    const int lane = threadIdx.x & 31;
    const bool b4 = lane & 16, b3 = lane & 8;
    const float a0 = (b4 ? x2 : x0) + __shfl_xor_sync(0xffffffffu, b4 ? x0 : x2, 16);
    const float a1 = (b4 ? x3 : x1) + __shfl_xor_sync(0xffffffffu, b4 ? x1 : x3, 16);
    float c = (b3 ? a1 : a0) + __shfl_xor_sync(0xffffffffu, b3 ? a0 : a1, 8);  // sum 2 b4 + b3
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    return make_float4(__shfl_sync(0xffffffffu, c, 0), __shfl_sync(0xffffffffu, c, 8),
                       __shfl_sync(0xffffffffu, c, 16), __shfl_sync(0xffffffffu, c, 24));
}

// The eight sums over the warp of v[0..7]; lane l ends with the sum of
// v[l / 4] (the first three exchanges halve the values each lane carries:
// 4 + 2 + 1 + 2 shuffles for the eight).
__device__ __forceinline__ float warp_sum8(const float (&v)[8]) {
    const int lane = threadIdx.x & 31;
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float a[4], b[2];
#pragma unroll
    for (int j = 0; j < 4; ++j) a[j] = (b4 ? v[4 + j] : v[j]) + __shfl_xor_sync(0xffffffffu, b4 ? v[j] : v[4 + j], 16);
#pragma unroll
    for (int j = 0; j < 2; ++j) b[j] = (b3 ? a[2 + j] : a[j]) + __shfl_xor_sync(0xffffffffu, b3 ? a[j] : a[2 + j], 8);
    float c = (b2 ? b[1] : b[0]) + __shfl_xor_sync(0xffffffffu, b2 ? b[0] : b[1], 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    return c;
}

// Row `lane` of a matrix (16 fp32 pairs) times two vectors in shared memory.
__device__ __forceinline__ void row_dot2(const float2 (&a)[16], const float *x, const float *y, float &ax,
                                        float &ay) {
    const float4 *xp = reinterpret_cast<const float4 *>(x), *yp = reinterpret_cast<const float4 *>(y);
    float2 xa = f2(0.f), xb = f2(0.f), ya = f2(0.f), yb = f2(0.f);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float4 xx = xp[c], yy = yp[c];
        xa = fma2(a[2 * c], lo2(xx), xa);
        xb = fma2(a[2 * c + 1], hi2(xx), xb);
        ya = fma2(a[2 * c], lo2(yy), ya);
        yb = fma2(a[2 * c + 1], hi2(yy), yb);
    }
    ax = hsum2(add2(xa, xb));
    ay = hsum2(add2(ya, yb));
}

static_assert(kTT == 8, "the input warp reduces a slot's eight tokens at once");

template <typename IO>
__global__ void __launch_bounds__(kNT32, 7) seq32_kernel(FwdParams p) {
    using L = S32Layout;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full_in = reinterpret_cast<uint64_t *>(smem + L::bars);
    uint64_t *full_g = full_in + kNB, *empty = full_in + 2 * kNB;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::flag);
    float *zbuf = reinterpret_cast<float *>(smem + L::zbuf);
    float *slots = reinterpret_cast<float *>(smem + L::slots);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int bh = blockIdx.x, T = p.T;
    const int ntiles = (T + kTT - 1) / kTT;
    const size_t tok0 = (size_t)bh * T * 32;
    const size_t moff = (size_t)bh * 32 * 32 + (size_t)lane * 32;  // row `lane` of a state matrix

    if (threadIdx.x == 0) {
        for (int b = 0; b < kNB; ++b) {
            mbar_init(&full_in[b], 32);
            mbar_init(&full_g[b], 32);
            mbar_init(&empty[b], 32);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (threadIdx.x < 64) zbuf[threadIdx.x] = 0.f;
    __syncthreads();

    if (warp == 2) {
        // ---------------- inputs ----------------
        const IO *gq = static_cast<const IO *>(p.q) + tok0, *gk = static_cast<const IO *>(p.k) + tok0;
        const IO *gv = static_cast<const IO *>(p.v) + tok0, *gu = static_cast<const IO *>(p.u) + tok0;
        float nrun = p.n0 ? p.n0[(size_t)bh * 32 + lane] : 0.f, ncomp = 0.f;  // n_t (Kahan-compensated)
        if (p.inject) return;  // test hook: the first slot never fills
        // L2 prefetch of a slot's rows: lane l takes token l / 4 of tensor l % 4
        auto prefetch = [&](int m) {
            const int t = m * kTT + (lane >> 2);
            if (m < ntiles && t < T) {
                const IO *src = (lane & 3) == 0 ? gq : (lane & 3) == 1 ? gk : (lane & 3) == 2 ? gv : gu;
                prefetch_l2(src + (size_t)t * 32);
            }
        };
        prefetch(0);
        prefetch(1);
        for (int m = 0; m < ntiles; ++m) {
            const int s = m % kNB;
            if (m >= kNB && !wait_warp(&empty[s], (uint32_t)((m / kNB - 1) & 1), abort_flag, p)) return;
            prefetch(m + 2);
            const int t0 = m * kTT, nt = min(kTT, T - t0);
            float q[kTT], k[kTT], v[kTT], u[kTT];
#pragma unroll
            for (int tt = 0; tt < kTT; ++tt) {  // (clamped: always a valid token)
                const size_t off = (size_t)min(t0 + tt, T - 1) * 32 + lane;
                q[tt] = io_to_f32(gq[off]);
                k[tt] = io_to_f32(gk[off]);
                v[tt] = io_to_f32(gv[off]);
                u[tt] = io_to_f32(gu[off]);
            }
            float *sl = slots + (size_t)s * L::slot;
            // |k_t|^2 of the slot's tokens in one reduction; lane 4 tt holds token tt's
            float e[kTT];
#pragma unroll
            for (int tt = 0; tt < kTT; ++tt) e[tt] = k[tt] * k[tt];
            const float ksl = 1.f / fmaxf(sqrtf(warp_sum8(e)), kEps);
#pragma unroll
            for (int tt = 0; tt < kTT; ++tt) {
                const float kh = k[tt] * __shfl_sync(0xffffffffu, ksl, 4 * tt);
                if (tt < nt) {  // n_t includes token t
                    const float y = phi_elu1(kh) - ncomp;
                    const float tk = nrun + y;
                    ncomp = (tk - nrun) - y;
                    nrun = tk;
                }
                const float fq = phi_elu1(q[tt]);
                e[tt] = fq * nrun;
                sl[L::kKh + tt * 32 + lane] = kh;
                sl[L::kU + tt * 32 + lane] = u[tt];
                sl[L::kF + tt * 32 + lane] = fq;
                sl[L::kV + tt * 32 + lane] = v[tt];
            }
            // phi(q_t) . n_t of the slot's tokens, likewise
            const float dl = warp_sum8(e);
            if ((lane & 3) == 0) sl[L::kDen + (lane >> 2)] = 1.f / (dl + kEps);
            __syncwarp();
            mbar_arrive(&full_in[s]);
        }
        if (!*abort_flag && p.n_T) p.n_T[(size_t)bh * 32 + lane] = nrun;
        return;
    }

    if (warp == 0) {
        // ---------------- A chain: row `lane` of A ----------------
        float2 a[16];  // columns 2j, 2j + 1
        if (p.A0) {
            const float4 *src = reinterpret_cast<const float4 *>(p.A0 + moff);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 x = src[c];
                a[2 * c] = lo2(x);
                a[2 * c + 1] = hi2(x);
            }
        } else {
            const float il = 1.f / p.lambda0;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                a[j] = make_float2(2 * j == lane ? il : 0.f, 2 * j + 1 == lane ? il : 0.f);
        }
        // One token of lookahead keeps the products with A off the serial chain:
        // with z_t = A_{t-1} u_t and y_t = A_{t-1} k_hat_t known,
        //   z_{t+1} = A_{t-1} u_{t+1} - beta_t z_t (z_t . u_{t+1}),
        //   y_{t+1} = A_{t-1} k_hat_{t+1} - beta_t z_t (z_t . k_hat_{t+1}),
        // so the products with A_{t-1} run beside token t's one reduction (of
        // u_t . z_t, k_hat_t . z_t, z_t . u_{t+1}, z_t . k_hat_{t+1}), and the chain
        // per token is that reduction, a reciprocal square root and an FMA.
        // A_t = A_{t-1} - w w^T with w = sqrt(beta_t) z_t: the product inside an
        // FMA is exact, so w_i w_j = w_j w_i and A stays exactly symmetric.
        float z = 0.f, y = 0.f;
        if (ntiles > 0) {
            if (!wait_warp(&full_in[0], 0u, abort_flag, p)) return;
            row_dot2(a, slots + L::kU, slots + L::kKh, z, y);
        }
        int t = 0;
        for (int m = 0; m < ntiles; ++m) {
            const int s = m % kNB;
            float *sl = slots + (size_t)s * L::slot;
            const int nt = min(kTT, T - m * kTT);
            for (int tt = 0; tt < nt; ++tt, ++t) {
                // token t + 1: in this slot, or first in the next one
                const bool more = t + 1 < T;
                const float *sn = sl;
                int tn = tt + 1;
                if (tn == kTT) {
                    const int mn = m + 1;
                    sn = slots + (size_t)(mn % kNB) * L::slot;
                    tn = 0;
                    if (more && !wait_warp(&full_in[mn % kNB], (uint32_t)((mn / kNB) & 1), abort_flag, p)) return;
                }
                // (past the stream's end: this token's vectors, the results unused; no
                // branch, so that these products and the reduction below interleave)
                sn = more ? sn : sl;
                tn = more ? tn : tt;
                float zn, yn;
                row_dot2(a, sn + L::kU + tn * 32, sn + L::kKh + tn * 32, zn, yn);  // with A_{t-1}
                const float un = sn[L::kU + tn * 32 + lane], kn = sn[L::kKh + tn * 32 + lane];
                const float4 pr = warp_sum4(sl[L::kU + tt * 32 + lane] * z, sl[L::kKh + tt * 32 + lane] * z,
                                            un * z, kn * z);
                const float sb = rsqrtf(1.f + pr.x);  // sqrt(beta_t)
                const float beta = sb * sb;
                sl[L::kG + tt * 32 + lane] = fmaf(-beta * pr.y, z, y);  // (A_t k_hat_t)_i
                const float w = sb * z;
                zbuf[(t & 1) * 32 + lane] = w;
                __syncwarp();
                const float4 *wp = reinterpret_cast<const float4 *>(zbuf + (t & 1) * 32);
                const float2 mw = f2(-w);
#pragma unroll
                for (int c = 0; c < 8; ++c) {  // A_t = A_{t-1} - w w^T
                    const float4 ww = wp[c];
                    a[2 * c] = fma2(mw, lo2(ww), a[2 * c]);
                    a[2 * c + 1] = fma2(mw, hi2(ww), a[2 * c + 1]);
                }
                const float zt = z;
                z = fmaf(-beta * pr.z, zt, zn);
                y = fmaf(-beta * pr.w, zt, yn);
            }
            __syncwarp();
            mbar_arrive(&full_g[s]);
        }
        float4 *dst = reinterpret_cast<float4 *>(p.A_T + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) dst[c] = make_float4(a[2 * c].x, a[2 * c].y, a[2 * c + 1].x, a[2 * c + 1].y);
        return;
    }

    // ---------------- S chain (warp 1): row `lane` of S ----------------
    float2 sr[16];
    if (p.S0) {
        const float4 *src = reinterpret_cast<const float4 *>(p.S0 + moff);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 x = src[c];
            sr[2 * c] = lo2(x);
            sr[2 * c + 1] = hi2(x);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) sr[j] = f2(0.f);
    }
    IO *gout = static_cast<IO *>(p.o) + tok0;
    int t = 0;
    for (int m = 0; m < ntiles; ++m) {
        const int s = m % kNB;
        const uint32_t par = (uint32_t)((m / kNB) & 1);
        if (!wait_warp(&full_in[s], par, abort_flag, p) || !wait_warp(&full_g[s], par, abort_flag, p)) return;
        const float *sl = slots + (size_t)s * L::slot;
        const int nt = min(kTT, T - m * kTT);
        for (int tt = 0; tt < nt; ++tt, ++t) {
            const float4 *kp = reinterpret_cast<const float4 *>(sl + L::kKh + tt * 32);
            const float4 *fp = reinterpret_cast<const float4 *>(sl + L::kF + tt * 32);
            const float4 *gp = reinterpret_cast<const float4 *>(sl + L::kG + tt * 32);
            float2 ka = f2(0.f), kb = f2(0.f), qa = f2(0.f), qb = f2(0.f);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 kk = kp[c], ff = fp[c];
                ka = fma2(sr[2 * c], lo2(kk), ka);
                kb = fma2(sr[2 * c + 1], hi2(kk), kb);
                qa = fma2(sr[2 * c], lo2(ff), qa);
                qb = fma2(sr[2 * c + 1], hi2(ff), qb);
            }
            // |g|^2 and g . phi(q)
            const float gi = sl[L::kG + tt * 32 + lane];
            const float2 pr = warp_sum2(gi * gi, gi * sl[L::kF + tt * 32 + lane]);
            const float inv = fminf(rsqrtf(pr.x), 1.f / kEps);  // 1 / max(|g|, eps)
            const float ri = (sl[L::kV + tt * 32 + lane] - hsum2(add2(ka, kb))) * inv;
            const float2 r2 = f2(ri);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 gg = gp[c];
                sr[2 * c] = fma2(r2, lo2(gg), sr[2 * c]);
                sr[2 * c + 1] = fma2(r2, hi2(gg), sr[2 * c + 1]);
            }
            // S_t phi(q) = S_{t-1} phi(q) + r (alpha . phi(q))
            const float num = fmaf(ri, pr.y, hsum2(add2(qa, qb)));
            gout[(size_t)t * 32 + lane] = f32_to_io<IO>(num * sl[L::kDen + tt]);
        }
        __syncwarp();
        mbar_arrive(&empty[s]);
    }
    float4 *dst = reinterpret_cast<float4 *>(p.S_T + moff);
#pragma unroll
    for (int c = 0; c < 8; ++c) dst[c] = make_float4(sr[2 * c].x, sr[2 * c].y, sr[2 * c + 1].x, sr[2 * c + 1].y);
}

template <typename IO>
cudaError_t launch_seq32_t(const FwdParams &p, cudaStream_t stream) {
    constexpr size_t smem = S32Layout::total;
    cudaError_t e = cudaFuncSetAttribute(seq32_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    mark_launch(p, 0, stream);
    seq32_kernel<IO><<<p.BH, kNT32, smem, stream>>>(p);
    e = cudaGetLastError();
    mark_launch(p, 1, stream);
    return e;
}

}  // namespace

cudaError_t launch_seq32(const FwdParams &p, cudaStream_t stream) {
    if (p.BH == 0) return cudaSuccess;
    return p.io_bf16 ? launch_seq32_t<__nv_bfloat16>(p, stream) : launch_seq32_t<float>(p, stream);
}

}  // namespace vla
