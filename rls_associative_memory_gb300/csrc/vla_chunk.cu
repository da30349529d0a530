// vla_chunk.cu -- chunk-parallel VLA forward path (few (b, h) units, long T).
//
// The token axis is cut into chunks of C tokens.  Everything that does not
// need the state at the chunk start runs for all chunks at once; only two
// cheap chains run along the chunks.
//
//  gram     per chunk: G_c = sum_t u_t u_t^T and m_c = sum_t phi(k_hat_t)
//  prefix   per (b, h): exclusive prefix M^(c) = M_0 + sum_{c'<c} G_c',
//           n^(c) = n_0 + sum_{c'<c} m_c'  (M_0 = lambda0 I, or A0^{-1})
//  gates    per chunk: A^(c) = (M^(c))^{-1} (Gauss-Jordan), then the exact
//           Sherman-Morrison recursion over the chunk's tokens from A^(c):
//           this is section 2.2's A_t = M_t^{-1} with M_t = M_{t-1} + u u^T,
//           restarted at every chunk boundary from its definition.  Emits
//           the unit gates alpha_t (and A_T from the last chunk).
//  summary  per chunk: the chunk's affine map S_end = S_start P_c + H_c.
//           Rows of [H; P] follow the state write of section 2.3 step 3
//           (row x <- x + (value - x.k_hat) alpha^T) with values [v; 0] and
//           initial rows [0; I].
//  chain    per (b, h, block of rows): S^(c+1) = S^(c) P_c + H_c, storing
//           every chunk-start state; writes S_T.
//  output   per chunk: the state write and ELU+1 readout of every token,
//           from S^(c), with the gates of the gates pass.
//
// Rows of S (and of [H; P]) evolve independently once the gates are known,
// so the summary and output passes need no block-wide reduction per token.
//
// With VLA_KERNEL_CHUNK_TC at d = 64 and bf16 I/O every pass but the prefix
// and the chain runs its products on the tensor cores: the Grams from TMA
// tensor copies (vla_gram_tc.cu), the gates in block-Woodbury form
// (vla_gates_tc.cu), and the summary pass in UT form (vla_chunk_tc.cu), which
// also writes, per token, the readout of its [H; P] rows (y_t = P_t phi(q_t) /
// den_t, h_t = H_t phi(q_t) / den_t; the state is affine in S^(c) within a
// chunk), so that the output pass is the product o_t = S^(c) y_t + h_t, with
// no recurrence.
#include <algorithm>

#include "vla_internal.cuh"

namespace vla {

// Whether the driver's tensor-map encoder could be found (vla_gram_tc.cu): the
// tensor-core passes stage their inputs by tiled tensor copies.
bool tile_maps_available();
// The gates and the state pass of the tensor-core path at d = 64 in one
// persistent launch fed by a job queue (vla_tc64_queue.cu).
cudaError_t launch_tc64_queue(const ChunkArgs &a, cudaStream_t stream);
// Wave model of one tensor-core pass of `ctas` CTAs of `len` sub-blocks each.
static double tc_pass_cost(long long ctas, double len);
// Whether G gates jobs and R state-pass jobs take less time as one queue launch
// than as two.  Two launches pay each pass's part-full last wave (tc_pass_cost,
// a gates job taken as long as a state-pass job).  The queue packs both
// passes' jobs into (G + R) / 304 job times, but a gates job and a state-pass
// job on one SM run slower than two of a kind: taken as 8 % (6 % measured with
// every SM holding one of each).  The long stream's two full waves a pass stay
// two launches; 32 units of 4096 tokens (1.68 waves a pass) take the queue.
static bool tc_queue_pays_jobs(long long G, long long R) {
    return 1.08 * (double)(G + R) / (2.0 * 152) < tc_pass_cost(G, 1.0) + tc_pass_cost(R, 1.0) - 1e-9;
}
namespace {

constexpr int kTT = 16;  // tokens per staged tile

// VLA_KERNEL_CHUNK_TC takes the block-Woodbury gates of vla_gates_tc.cu
// (measured 0.90 ms against 1.26 ms for the Sherman-Morrison gates here on the
// long stream, B = 1, H = 16, T = 65536, d = 64).
constexpr bool kGatesOnTensorCores = true;

// Kahan-compensated accumulation.
__device__ __forceinline__ void kahan_add(float &sum, float &comp, float x) {
    const float y = x - comp;
    const float t = sum + y;
    comp = (t - sum) - y;
    sum = t;
}

// The exclusive Kahan prefix of x[c * stride], c < n, in place, starting from
// run; returns the total.  The loads go eight chunks at a time, ahead of the
// stores, so that a thread waits on one latency per eight chunks.
__device__ __forceinline__ float kahan_prefix_inplace(float *x, size_t stride, int n, float run) {
    float comp = 0.f;
    for (int c0 = 0; c0 < n; c0 += 8) {
        float g[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = (c0 + j < n) ? x[(size_t)(c0 + j) * stride] : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (c0 + j < n) {
                x[(size_t)(c0 + j) * stride] = run;
                kahan_add(run, comp, g[j]);
            }
        }
    }
    return run;
}

// ---------------------------------------------------------------------------
// gram: chunk Gram matrices of u and chunk sums of phi(k_hat)
// ---------------------------------------------------------------------------
template <int D, typename IO>
__global__ void __launch_bounds__(256) gram_kernel(ChunkArgs a) {
    constexpr int MT = D / 16;  // microtile edge on a 16 x 16 thread grid
    __shared__ __align__(16) float su[kTT][D];
    __shared__ __align__(16) float sf[kTT][D];
    const int c = (int)(blockIdx.x % (unsigned)a.L.NCA), bh = (int)(blockIdx.x / (unsigned)a.L.NCA);
    const int T = a.p.T, C = a.L.CA;
    const int t0 = c * C, t1 = min(T, t0 + C);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ty = tid >> 4, tx = tid & 15;
    const IO *gu = static_cast<const IO *>(a.p.u) + (size_t)bh * T * D;
    const IO *gk = static_cast<const IO *>(a.p.k) + (size_t)bh * T * D;
    float acc[MT][MT];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int n = 0; n < MT; ++n) acc[m][n] = 0.f;
    float nacc = 0.f;
    for (int tb = t0; tb < t1; tb += kTT) {
        const int ntok = min(kTT, t1 - tb);
        for (int e = tid; e < ntok * D; e += 256) {
            su[e / D][e % D] = io_to_f32(gu[(size_t)tb * D + e]);
            sf[e / D][e % D] = io_to_f32(gk[(size_t)tb * D + e]);
        }
        __syncthreads();
        for (int tt = warp; tt < ntok; tt += 8) {
            float kk[D / 32], ss = 0.f;
#pragma unroll
            for (int m = 0; m < D / 32; ++m) {
                kk[m] = sf[tt][lane + 32 * m];
                ss = fmaf(kk[m], kk[m], ss);
            }
            ss = warp_sum(ss);
            const float ks = 1.f / fmaxf(sqrtf(ss), kEps);
#pragma unroll
            for (int m = 0; m < D / 32; ++m) sf[tt][lane + 32 * m] = phi_elu1(kk[m] * ks);
        }
        __syncthreads();
        if (tid < D)
            for (int tt = 0; tt < ntok; ++tt) nacc += sf[tt][tid];
        for (int tt = 0; tt < ntok; ++tt) {
            float ui[MT], uj[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                ui[m] = su[tt][ty * MT + m];
                uj[m] = su[tt][tx * MT + m];
            }
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int n = 0; n < MT; ++n) acc[m][n] = fmaf(ui[m], uj[n], acc[m][n]);
        }
        __syncthreads();
    }
    float *G = ws_f(a, a.L.off_M) + ((size_t)bh * a.L.NCA + c) * D * D;
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int n = 0; n < MT; ++n) G[(ty * MT + m) * D + tx * MT + n] = acc[m][n];
    if (tid < D) ws_f(a, a.L.off_n)[((size_t)bh * (a.L.NCA + 1) + c) * D + tid] = nacc;
}

// ---------------------------------------------------------------------------
// gram on the tensor cores (bf16 I/O, d in {64, 128}): G_c = U_c^T U_c as
// tcgen05.mma kind::f16 with fp32 accumulation in TMEM.  bf16 x bf16
// products are exact in fp32, so only the accumulation rounds.
//   - u and k tiles of KS tokens arrive by 1-D bulk copies (double-buffered);
//   - all threads repack the u tile feature-major (rows = features, K =
//     tokens) into the K-major, unswizzled core-matrix layout; tokens past
//     the end of the chunk are written as zeros;
//   - one thread issues KS/16 MMAs with A = B = that tile (M = N = d) and
//     commits them to an mbarrier that frees the tile for reuse;
//   - the sums of phi(k_hat) are accumulated on the CUDA cores meanwhile;
//   - the accumulator is read back with tcgen05.ld (for M = 64, row r sits in
//     TMEM lane 32 (r / 16) + r % 16).
// ---------------------------------------------------------------------------
template <int D>
struct GramTc {
    static constexpr int KS = 64;                               // tokens per stage
    static constexpr int NT = 128;                              // 4 warps: all TMEM lane quarters
    static constexpr uint32_t NCOL = D;                         // TMEM columns (64 or 128)
    static constexpr size_t ctrl = 0;                           // raw_bar[2], mma_bar[2], tmem slot, abort
    static constexpr size_t raw = 128;                          // [2][2][KS*D] bf16 (u, k)
    static constexpr size_t raw_t = (size_t)KS * D * 2;
    static constexpr size_t abuf = raw + 4 * raw_t;             // [2][D x KS] bf16, K-major core matrices
    static constexpr size_t abuf_t = (size_t)D * KS * 2;
    static constexpr size_t nred = abuf + 2 * abuf_t;           // [4][D] fp32
    static constexpr size_t total = nred + 4 * D * 4;
    static_assert(abuf % 1024 == 0 || true, "");
};

template <int D>
__global__ void __launch_bounds__(GramTc<D>::NT) gram_tc_kernel(ChunkArgs a) {
    using G = GramTc<D>;
    constexpr int KS = G::KS, NT = G::NT;
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t *raw_bar = reinterpret_cast<uint64_t *>(smem + G::ctrl);
    uint64_t *mma_bar = raw_bar + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + G::ctrl + 32);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + G::ctrl + 36);
    __nv_bfloat16 *raw = reinterpret_cast<__nv_bfloat16 *>(smem + G::raw);
    unsigned char *abuf = smem + G::abuf;
    float *nred = reinterpret_cast<float *>(smem + G::nred);

    const int c = (int)(blockIdx.x % (unsigned)a.L.NCA), bh = (int)(blockIdx.x / (unsigned)a.L.NCA);
    const int T = a.p.T, C = a.L.CA;
    const int t0 = c * C, ntok = min(C, T - t0);
    const int nst = (ntok + KS - 1) / KS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t tok0 = ((size_t)bh * T + t0) * D;
    const __nv_bfloat16 *gu = static_cast<const __nv_bfloat16 *>(a.p.u) + tok0;
    const __nv_bfloat16 *gk = static_cast<const __nv_bfloat16 *>(a.p.k) + tok0;

    if (tid == 0) {
        mbar_init(&raw_bar[0], 1);
        mbar_init(&raw_bar[1], 1);
        mbar_init(&mma_bar[0], 1);
        mbar_init(&mma_bar[1], 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0) tmem_alloc(tslot, G::NCOL);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;

    auto issue = [&](int st) {
        const int buf = st & 1;
        const int nt = min(KS, ntok - st * KS);
        const uint32_t bytes = (uint32_t)(nt * D * 2);
        mbar_arrive_expect_tx(&raw_bar[buf], 2 * bytes);
        bulk_g2s(raw + ((size_t)buf * 2 + 0) * KS * D, gu + (size_t)st * KS * D, bytes, &raw_bar[buf]);
        bulk_g2s(raw + ((size_t)buf * 2 + 1) * KS * D, gk + (size_t)st * KS * D, bytes, &raw_bar[buf]);
    };
    int issued = 0, committed = 0;
    if (tid == 0) {
        if (nst > 0) issue(0);
        if (nst > 1) issue(1);
        issued = min(nst, 2);
    }
    constexpr int M32 = D / 32;
    float nk[M32];
#pragma unroll
    for (int m = 0; m < M32; ++m) nk[m] = 0.f;
    constexpr uint32_t idesc = idesc_bf16_f32(D, D);
    constexpr uint32_t sbo = KS * 16, lbo = 128;

    int failed = 0;
    for (int st = 0; st < nst; ++st) {
        const int buf = st & 1;
        const int nt = min(KS, ntok - st * KS);
        bool ok = mbar_wait_bounded(&raw_bar[buf], (st >> 1) & 1, a.p.wait_limit_ns, a.p.err);
        if (ok && st >= 2) ok = mbar_wait_bounded(&mma_bar[buf], ((st - 2) >> 1) & 1, a.p.wait_limit_ns, a.p.err);
        if (!ok) *abort_flag = 1;
        tc_fence_after();
        __syncthreads();
        if (*abort_flag) {
            failed = 1;
            break;
        }
        const __nv_bfloat16 *ru = raw + ((size_t)buf * 2 + 0) * KS * D;
        const __nv_bfloat16 *rk = raw + ((size_t)buf * 2 + 1) * KS * D;
        unsigned char *A = abuf + (size_t)buf * G::abuf_t;
        // repack u: item = (feature f, group of 8 tokens) -> one 16-byte core-matrix row
        for (int it = tid; it < D * (KS / 8); it += NT) {
            const int f = it % D, g8 = it / D;
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int ta = g8 * 8 + 2 * h, tb = ta + 1;
                const unsigned short lo = ta < nt ? __bfloat16_as_ushort(ru[ta * D + f]) : (unsigned short)0;
                const unsigned short hi = tb < nt ? __bfloat16_as_ushort(ru[tb * D + f]) : (unsigned short)0;
                w[h] = (uint32_t)lo | ((uint32_t)hi << 16);
            }
            *reinterpret_cast<uint4 *>(A + kmajor_off_bf16(f, g8 * 8, KS)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        // phi(k_hat) sums on the CUDA cores
        for (int tt = warp; tt < nt; tt += NT / 32) {
            float kk[M32], ss = 0.f;
#pragma unroll
            for (int m = 0; m < M32; ++m) {
                kk[m] = __bfloat162float(rk[tt * D + lane + 32 * m]);
                ss = fmaf(kk[m], kk[m], ss);
            }
            ss = warp_sum(ss);
            const float ks = 1.f / fmaxf(sqrtf(ss), kEps);
#pragma unroll
            for (int m = 0; m < M32; ++m) nk[m] += phi_elu1(kk[m] * ks);
        }
        fence_proxy_async_smem();  // the repacked tile is read by the tensor core (async proxy)
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t abase = smem_u32(A);
#pragma unroll
            for (int ks = 0; ks < KS / 16; ++ks) {
                const uint64_t dsc = umma_desc_kmajor(abase + ks * 256, lbo, sbo);
                umma_bf16(tbase, dsc, dsc, idesc, (st > 0 || ks > 0) ? 1u : 0u);
            }
            umma_commit(&mma_bar[buf]);
            committed = st + 1;
            if (st + 2 < nst) {
                issue(st + 2);
                issued = st + 3;
            }
        }
    }
    // wait for the last MMAs (thread 0 knows what it committed; everyone waits on the same phase)
    if (!failed && nst > 0) {
        const int last = nst - 1;
        if (!mbar_wait_bounded(&mma_bar[last & 1], (last >> 1) & 1, a.p.wait_limit_ns, a.p.err)) *abort_flag = 1;
    }
    tc_fence_after();
    __syncthreads();
    if (failed || *abort_flag) {
        if (tid == 0) {
            if (committed > 0)
                (void)mbar_wait_bounded(&mma_bar[(committed - 1) & 1], ((committed - 1) >> 1) & 1, a.p.wait_limit_ns,
                                        a.p.err);
            for (int st = committed; st < issued; ++st)
                (void)mbar_wait_bounded(&raw_bar[st & 1], (st >> 1) & 1, a.p.wait_limit_ns, a.p.err);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tbase, G::NCOL);
        return;
    }
    // ---- G out: accumulator rows from TMEM ----
    float *Gout = ws_f(a, a.L.off_M) + ((size_t)bh * a.L.NCA + c) * D * D;
    const bool has_row = (D == 128) || (lane < 16);
    const int grow = (D == 128) ? (32 * warp + lane) : (16 * warp + lane);
#pragma unroll
    for (int cb = 0; cb < D; cb += 16) {
        float v[16];
        tmem_ld16(tbase + ((uint32_t)(32 * warp) << 16) + (uint32_t)cb, v);
        if (has_row) {
            float4 *dst = reinterpret_cast<float4 *>(Gout + (size_t)grow * D + cb);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
    }
    // ---- sums of phi(k_hat) ----
#pragma unroll
    for (int m = 0; m < M32; ++m) nred[warp * D + lane + 32 * m] = nk[m];
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, G::NCOL);
    if (tid < D) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) sum += nred[w * D + tid];
        ws_f(a, a.L.off_n)[((size_t)bh * (a.L.NCA + 1) + c) * D + tid] = sum;
    }
}

// ---------------------------------------------------------------------------
// prefix: exclusive prefix sums of G and m along the chunks (Kahan, fp32)
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) prefix_kernel(ChunkArgs a) {
    constexpr int NB = (D * D + D + 255) / 256;  // blocks per (b, h)
    const int bh = a.bh_lo + (int)(blockIdx.x / NB);
    const int e = (int)(blockIdx.x % NB) * 256 + threadIdx.x;
    const int NC = a.L.NCA;  // A-chunks
    if (e < D * D) {
        const int i = e / D, j = e % D;
        const float run = a.p.A0 ? ws_f(a, a.L.off_M0)[(size_t)bh * D * D + e] : (i == j ? a.p.lambda0 : 0.f);
        (void)kahan_prefix_inplace(ws_f(a, a.L.off_M) + (size_t)bh * NC * D * D + e, (size_t)D * D, NC, run);
    } else if (e < D * D + D) {
        const int j = e - D * D;
        float *n = ws_f(a, a.L.off_n) + (size_t)bh * (NC + 1) * D + j;
        const float run = kahan_prefix_inplace(n, D, NC, a.p.n0 ? a.p.n0[(size_t)bh * D + j] : 0.f);
        n[(size_t)NC * D] = run;
        if (a.p.n_T) a.p.n_T[(size_t)bh * D + j] = run;
    }
}

// Same elimination with RPT rows per thread: rows row0 + r * rstride.
template <int D, int CPT, int RPT>
__device__ __forceinline__ void gj_inverse_rows(float (&x)[RPT][CPT], float *piv, int row0, int rstride, int part) {
    constexpr int TPR = D / CPT;
    constexpr int VLEN = (D / 32) * kPart;
    const int c0 = part * CPT;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < RPT; ++r)
        if (row0 + r * rstride == 0) {
#pragma unroll
            for (int j = 0; j < CPT; ++j) piv[vidx(c0 + j)] = x[r][j];
        }
    __syncthreads();
#pragma unroll 1
    for (int k = 0; k < D; ++k) {
        const float *pr = piv + (k & 1) * VLEN;
        const float rp = 1.f / pr[vidx(k)];
        const int kp = k / CPT, kr = k % CPT;
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            float mk = 0.f;
#pragma unroll
            for (int j = 0; j < CPT; ++j)
                if (j == kr) mk = x[r][j];
            if (TPR > 1) mk = __shfl_sync(0xffffffffu, mk, (lane & ~(TPR - 1)) | kp);
            if (row0 + r * rstride == k) {
#pragma unroll
                for (int j = 0; j < CPT; ++j) x[r][j] = (c0 + j == k) ? rp : x[r][j] * rp;
            } else {
                const float f = mk * rp;
#pragma unroll
                for (int c4 = 0; c4 < CPT / 4; ++c4) {
                    const float4 pv = *reinterpret_cast<const float4 *>(pr + vidx(c0 + 4 * c4));
                    const float pj[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int j = 4 * c4 + q;
                        x[r][j] = (c0 + j == k) ? -f : fmaf(-f, pj[q], x[r][j]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RPT; ++r)
            if (k + 1 < D && row0 + r * rstride == k + 1) {
                float *nx = piv + ((k + 1) & 1) * VLEN;
#pragma unroll
                for (int j = 0; j < CPT; ++j) nx[vidx(c0 + j)] = x[r][j];
            }
        __syncthreads();
    }
}

template <int D>
struct RowCfg {
    static constexpr int TPR = D / 32;
    static constexpr int NT = D * TPR;
    static constexpr int VLEN = TPR * kPart;
};

// Issue the bulk copies of one tile: ntens tensors of ntok tokens each.
__device__ __forceinline__ void issue_tile(uint64_t *bar, void *const *dst, const void *const *src,
                                           const uint32_t *bytes_per_tok, int ntens, int ntok) {
    uint32_t total = 0;
    for (int x = 0; x < ntens; ++x) total += bytes_per_tok[x] * ntok;
    mbar_arrive_expect_tx(bar, total);
    for (int x = 0; x < ntens; ++x) bulk_g2s(dst[x], src[x], bytes_per_tok[x] * ntok, bar);
}

// ---------------------------------------------------------------------------
// gates: A^(c) by Gauss-Jordan, then Sherman-Morrison over the chunk
// ---------------------------------------------------------------------------
// Thread layout: thread (rows row0 + r * RSTRIDE, part p) owns CPT columns of
// RPT rows of A.  d = 64: two warps per chunk, a whole row per thread;
// d = 128: 256 threads, half a row each; d = 32: one warp, a row each.  (Two
// rows per lane was measured slower at d = 64, both with one warp per chunk
// (1.20 -> 1.49 ms) and with 32 columns x two rows per thread (-> 1.55 ms):
// fewer A-chains fit per SM and the pass is bound by chains in flight.)
template <int D>
struct GatesCfg {
    static constexpr int CPT = (D >= 64) ? 64 : 32;
    static constexpr int TPR = D / CPT;
    static constexpr int RPT = 1;
    static constexpr int NT = D * TPR / RPT;
    static constexpr int NW = NT / 32;
    static constexpr int RSTRIDE = NT / TPR;  // distance between a thread's rows
    static constexpr int VLEN = (D / 32) * kPart;
};

template <int D, typename IO>
struct GatesSmem {
    using R = GatesCfg<D>;
    static constexpr size_t bars = 0;
    static constexpr size_t raw = 128;                                        // [2][2][TT*D] IO (u, k)
    static constexpr size_t raw_t = (size_t)kTT * D * sizeof(IO);
    static constexpr size_t khat = raw + 4 * raw_t;                           // [TT][VLEN]
    static constexpr size_t uu = khat + kTT * R::VLEN * 4;                    // [TT][VLEN]
    static constexpr size_t zbuf = uu + kTT * R::VLEN * 4;                    // [2][VLEN]
    static constexpr size_t piv = zbuf + 2 * R::VLEN * 4;                     // [2][VLEN]
    static constexpr size_t red = piv + 2 * R::VLEN * 4;                      // [2][NW] float4
    static constexpr size_t total = red + 2 * R::NW * 16;
};

// Within a chunk A starts from its exact definition (M^(c))^{-1} and takes at
// most C rank-1 steps, so the update is the single-FMA form
// A_ij -= (beta z_i) z_j; the sequential kernel, which runs all T steps from
// one start, uses the symmetric-rounding form instead.
template <int D, typename IO>
__global__ void __launch_bounds__(GatesCfg<D>::NT) gates_kernel(ChunkArgs a) {
    using R = GatesCfg<D>;
    using Lo = GatesSmem<D, IO>;
    constexpr int TPR = R::TPR, VLEN = R::VLEN, NW = R::NW, CPT = R::CPT, RPT = R::RPT, RS = R::RSTRIDE;
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lo::bars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Lo::bars + 16);
    IO *raw = reinterpret_cast<IO *>(smem + Lo::raw);
    float *s_khat = reinterpret_cast<float *>(smem + Lo::khat);
    float *s_u = reinterpret_cast<float *>(smem + Lo::uu);
    float *s_z = reinterpret_cast<float *>(smem + Lo::zbuf);
    float *s_piv = reinterpret_cast<float *>(smem + Lo::piv);
    float4 *s_red = reinterpret_cast<float4 *>(smem + Lo::red);

    const int c = (int)(blockIdx.x % (unsigned)a.L.NCA), bh = (int)(blockIdx.x / (unsigned)a.L.NCA);
    const int T = a.p.T, C = a.L.CA, NC = a.L.NCA;  // A-chunks
    const int t0 = c * C, ntok = min(C, T - t0);
    const int ntiles = (ntok + kTT - 1) / kTT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row0 = tid / TPR, part = tid % TPR;
    const int c0 = part * CPT;
    const size_t tok0 = ((size_t)bh * T + t0) * D;
    const IO *gu = static_cast<const IO *>(a.p.u) + tok0;
    const IO *gk = static_cast<const IO *>(a.p.k) + tok0;
    float *galpha = ws_f(a, a.L.off_alpha) + tok0;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    for (int i = tid; i < 2 * VLEN; i += R::NT) s_z[i] = 0.f;
    __syncthreads();
    const uint32_t bpt[2] = {(uint32_t)(D * sizeof(IO)), (uint32_t)(D * sizeof(IO))};
    auto issue = [&](int m) {
        const int buf = m & 1;
        const int nt = min(kTT, ntok - m * kTT);
        void *dst[2] = {raw + ((size_t)buf * 2 + 0) * kTT * D, raw + ((size_t)buf * 2 + 1) * kTT * D};
        const void *src[2] = {gu + (size_t)m * kTT * D, gk + (size_t)m * kTT * D};
        issue_tile(&bars[buf], dst, src, bpt, 2, nt);
    };
    int issued = 0;
    if (tid == 0) {
        if (ntiles > 0) issue(0);
        if (ntiles > 1) issue(1);
        issued = min(ntiles, 2);
    }

    // ---- A at the chunk start ----
    float2 am[RPT][CPT / 2];
    {
        float x[RPT][CPT];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int row = row0 + r * RS;
            const float *src = nullptr;
            if (c > 0) src = ws_f(a, a.L.off_M) + ((size_t)bh * NC + c) * D * D + row * D + c0;
            else if (a.p.A0) src = a.p.A0 + (size_t)bh * D * D + row * D + c0;
            if (src) {
#pragma unroll
                for (int q = 0; q < CPT / 4; ++q) {
                    const float4 v = reinterpret_cast<const float4 *>(src)[q];
                    x[r][4 * q] = v.x; x[r][4 * q + 1] = v.y; x[r][4 * q + 2] = v.z; x[r][4 * q + 3] = v.w;
                }
            } else {
                const float il = 1.f / a.p.lambda0;
#pragma unroll
                for (int j = 0; j < CPT; ++j) x[r][j] = (c0 + j == row) ? il : 0.f;
            }
        }
        if (c > 0) gj_inverse_rows<D, CPT, RPT>(x, s_piv, row0, RS, part);
#pragma unroll
        for (int r = 0; r < RPT; ++r)
#pragma unroll
            for (int j = 0; j < CPT / 2; ++j) am[r][j] = make_float2(x[r][2 * j], x[r][2 * j + 1]);
    }

    float bz_prev[RPT], z_prev[RPT], y_prev[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) bz_prev[r] = z_prev[r] = y_prev[r] = 0.f;
    float bs2_prev = 0.f;
    int failed = -1;
    for (int t = 0; t <= ntok; ++t) {
        const int tt = t % kTT, m = t / kTT;
        if (tt == 0 && t < ntok) {
            const int buf = m & 1;
            if (!mbar_wait_bounded(&bars[buf], (m >> 1) & 1, a.p.wait_limit_ns, a.p.err)) *abort_flag = 1;
            __syncthreads();
            if (*abort_flag) {
                failed = m;
                break;
            }
            const IO *ru = raw + ((size_t)buf * 2 + 0) * kTT * D;
            const IO *rk = raw + ((size_t)buf * 2 + 1) * kTT * D;
            const int nt = min(kTT, ntok - t);
            for (int q = warp; q < nt; q += NW) {
                float kk[D / 32], ss = 0.f;
#pragma unroll
                for (int mm = 0; mm < D / 32; ++mm) {
                    kk[mm] = io_to_f32(rk[q * D + lane + 32 * mm]);
                    ss = fmaf(kk[mm], kk[mm], ss);
                }
                ss = warp_sum(ss);
                const float ks = 1.f / fmaxf(sqrtf(ss), kEps);
#pragma unroll
                for (int mm = 0; mm < D / 32; ++mm) {
                    const int j = lane + 32 * mm;
                    s_khat[q * VLEN + vidx(j)] = kk[mm] * ks;
                    s_u[q * VLEN + vidx(j)] = io_to_f32(ru[q * D + j]);
                }
            }
            __syncthreads();
            if (tid == 0 && m + 2 < ntiles) {
                issue(m + 2);
                issued = m + 3;
            }
        }
        const bool hasA = t < ntok, hasG = t > 0;
        const float *uA = s_u + tt * VLEN;
        const float *kA = s_khat + tt * VLEN;
        const float *zv = s_z + ((t - 1) & 1) * VLEN;
        float2 za[RPT], zb[RPT], ya[RPT], yb[RPT];
#pragma unroll
        for (int r = 0; r < RPT; ++r) za[r] = zb[r] = ya[r] = yb[r] = f2(0.f);
#pragma unroll
        for (int q = 0; q < CPT / 4; ++q) {
            const int j = c0 + 4 * q;
            const float4 zz = *reinterpret_cast<const float4 *>(zv + vidx(j));
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const float2 mbz = f2(-bz_prev[r]);  // -beta_{t-1} z_{t-1,i}
                am[r][2 * q] = fma2(mbz, lo2(zz), am[r][2 * q]);
                am[r][2 * q + 1] = fma2(mbz, hi2(zz), am[r][2 * q + 1]);
            }
            if (hasA) {
                const float4 u4 = *reinterpret_cast<const float4 *>(uA + vidx(j));
                const float4 k4 = *reinterpret_cast<const float4 *>(kA + vidx(j));
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    za[r] = fma2(am[r][2 * q], lo2(u4), za[r]);
                    zb[r] = fma2(am[r][2 * q + 1], hi2(u4), zb[r]);
                    ya[r] = fma2(am[r][2 * q], lo2(k4), ya[r]);
                    yb[r] = fma2(am[r][2 * q + 1], hi2(k4), yb[r]);
                }
            }
        }
        float z[RPT], y[RPT], g[RPT];
        float p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            z[r] = hsum2(add2(za[r], zb[r]));
            y[r] = hsum2(add2(ya[r], yb[r]));
#pragma unroll
            for (int o = 1; o < TPR; o <<= 1) {
                z[r] += __shfl_xor_sync(0xffffffffu, z[r], o);
                y[r] += __shfl_xor_sync(0xffffffffu, y[r], o);
            }
            g[r] = y_prev[r] - bs2_prev * z_prev[r];  // gate of token t-1: y - beta (z.k_hat) z
            const int row = row0 + r * RS;
            if (part == 0) {
                if (hasA) {
                    p1 += uA[vidx(row)] * z[r];
                    p2 += kA[vidx(row)] * z[r];
                    s_z[(t & 1) * VLEN + vidx(row)] = z[r];
                }
                if (hasG) p3 += g[r] * g[r];
            }
        }
        const float red = warp_reduce4(p1, p2, p3, 0.f);
        if constexpr (NW > 1) {
            if ((lane & 7) == 0) reinterpret_cast<float *>(s_red)[((t & 1) * NW + warp) * 4 + (lane >> 3)] = red;
            __syncthreads();
            float4 acc = s_red[(t & 1) * NW];
#pragma unroll
            for (int w = 1; w < NW; ++w) {
                const float4 v = s_red[(t & 1) * NW + w];
                acc.x += v.x; acc.y += v.y; acc.z += v.z;
            }
            p1 = acc.x; p2 = acc.y; p3 = acc.z;
        } else {
            p1 = __shfl_sync(0xffffffffu, red, 0);
            p2 = __shfl_sync(0xffffffffu, red, 8);
            p3 = __shfl_sync(0xffffffffu, red, 16);
            __syncwarp();
        }
        const float inv = fminf(rsqrtf(p3), 1.f / kEps);
        const float beta = 1.f / (1.f + p1);
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            if (hasG && part == 0) galpha[(size_t)(t - 1) * D + row0 + r * RS] = g[r] * inv;
            bz_prev[r] = beta * z[r];
            z_prev[r] = z[r];
            y_prev[r] = y[r];
        }
        bs2_prev = beta * p2;
    }
    if (failed >= 0) {
        if (tid == 0)
            for (int m = failed; m < issued; ++m)
                (void)mbar_wait_bounded(&bars[m & 1], (m >> 1) & 1, a.p.wait_limit_ns, a.p.err);
        return;
    }
    if (c == NC - 1) {
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            float *dA = a.p.A_T + (size_t)bh * D * D + (row0 + r * RS) * D + c0;
#pragma unroll
            for (int q = 0; q < CPT / 4; ++q)
                reinterpret_cast<float4 *>(dA)[q] =
                    make_float4(am[r][2 * q].x, am[r][2 * q].y, am[r][2 * q + 1].x, am[r][2 * q + 1].y);
        }
    }
}

// ---------------------------------------------------------------------------
// Row recurrences given the gates (summary and output passes)
// ---------------------------------------------------------------------------
// Shared tile for both passes: raw IO tiles of up to three tensors plus the
// fp32 gate tile, and processed skewed vectors.
template <int D, typename IO>
struct RowsSmem {
    using R = RowCfg<D>;
    static constexpr size_t bars = 0;
    static constexpr size_t raw = 128;                                   // [2][3][TT*D] IO (q, k, v)
    static constexpr size_t raw_t = (size_t)kTT * D * sizeof(IO);
    static constexpr size_t ral = raw + 6 * raw_t;                       // [2][TT*D] fp32 gates
    static constexpr size_t khat = ral + 2 * (size_t)kTT * D * 4;        // [TT][VLEN]
    static constexpr size_t alp = khat + kTT * R::VLEN * 4;              // [TT][VLEN]
    static constexpr size_t phiq = alp + kTT * R::VLEN * 4;              // [TT][VLEN]
    static constexpr size_t vv = phiq + kTT * R::VLEN * 4;               // [TT][D]
    static constexpr size_t den = vv + (size_t)kTT * D * 4;              // [TT] reciprocal denominators
    static constexpr size_t ga = den + kTT * 4;                          // [TT]
    static constexpr size_t work = ga + kTT * 4;                         // [TT][D]
    static constexpr size_t total = work + (size_t)kTT * D * 4;
};

// MODE 0 (summary): per thread, rows h_i (values v, start 0) and p_i (values
//                   0, start I) of one row index i; writes P_c, H_c.
// MODE 1 (output):  rows s (values v, start S^(c)); writes o.  For d = 128
//                   each thread owns two rows, i and i + d/2, so that every
//                   vector loaded from shared memory feeds two independent
//                   dot products (measured 1.6x faster at d = 128; at d = 64
//                   the halved thread count costs more latency hiding than
//                   it saves, 1.09 -> 1.24 ms, so d = 64 keeps one row).
template <int D, int MODE>
struct RowsCfg {
    static constexpr int TPR = D / 32;
    static constexpr int RPT = (MODE == 1 && D >= 128) ? 2 : 1;
    static constexpr int NT = D * TPR / RPT;
    static constexpr int NW = NT / 32;
    static constexpr int VLEN = TPR * kPart;
};

template <int D, typename IO, int MODE>
__global__ void __launch_bounds__(RowsCfg<D, MODE>::NT) rows_kernel(ChunkArgs a) {
    using R = RowsCfg<D, MODE>;
    using Lo = RowsSmem<D, IO>;
    constexpr int TPR = R::TPR, VLEN = R::VLEN, NW = R::NW, RPT = R::RPT;
    constexpr int ROW2 = D / 2;  // second row of a thread in MODE 1 with RPT = 2
    constexpr int NIO = (MODE == 0) ? 2 : 3;  // k, v (+ q)
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lo::bars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Lo::bars + 16);
    IO *raw = reinterpret_cast<IO *>(smem + Lo::raw);
    float *s_ral = reinterpret_cast<float *>(smem + Lo::ral);
    float *s_khat = reinterpret_cast<float *>(smem + Lo::khat);
    float *s_alp = reinterpret_cast<float *>(smem + Lo::alp);
    float *s_phiq = reinterpret_cast<float *>(smem + Lo::phiq);
    float *s_v = reinterpret_cast<float *>(smem + Lo::vv);
    float *s_den = reinterpret_cast<float *>(smem + Lo::den);
    float *s_ga = reinterpret_cast<float *>(smem + Lo::ga);
    float *s_work = reinterpret_cast<float *>(smem + Lo::work);

    const int c = (int)(blockIdx.x % (unsigned)a.L.NC), bh = (int)(blockIdx.x / (unsigned)a.L.NC);
    const int T = a.p.T, C = a.L.C, NC = a.L.NC;
    const int t0 = c * C, ntok = min(C, T - t0);
    const int ntiles = (ntok + kTT - 1) / kTT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = tid / TPR, part = tid % TPR;
    const int c0 = part * 32, vo = part * kPart;
    const size_t tok0 = ((size_t)bh * T + t0) * D;
    const IO *gk = static_cast<const IO *>(a.p.k) + tok0;
    const IO *gv = static_cast<const IO *>(a.p.v) + tok0;
    const IO *gq = static_cast<const IO *>(a.p.q) + tok0;
    const float *galpha = ws_f(a, a.L.off_alpha) + tok0;
    IO *gout = static_cast<IO *>(a.p.o) + tok0;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    const uint32_t bio = (uint32_t)(D * sizeof(IO));
    const uint32_t bpt[4] = {bio, bio, bio, (uint32_t)(D * 4)};
    auto issue = [&](int m) {
        const int buf = m & 1;
        const int nt = min(kTT, ntok - m * kTT);
        const size_t off = (size_t)m * kTT * D;
        void *dst[4];
        const void *src[4];
        dst[0] = raw + ((size_t)buf * 3 + 0) * kTT * D; src[0] = gk + off;
        dst[1] = raw + ((size_t)buf * 3 + 1) * kTT * D; src[1] = gv + off;
        if (MODE == 1) {
            dst[2] = raw + ((size_t)buf * 3 + 2) * kTT * D;
            src[2] = gq + off;
        }
        dst[NIO] = s_ral + (size_t)buf * kTT * D;
        src[NIO] = galpha + off;
        uint32_t b[4] = {bpt[0], bpt[1], MODE == 1 ? bpt[2] : bpt[3], bpt[3]};
        issue_tile(&bars[buf], dst, src, b, NIO + 1, nt);
    };
    int issued = 0;
    if (tid == 0) {
        if (ntiles > 0) issue(0);
        if (ntiles > 1) issue(1);
        issued = min(ntiles, 2);
    }

    // row state
    float2 h[16], p[16];  // columns 2j, 2j+1 of this thread's 32
    const size_t moff = (size_t)row * D + c0;
    if (MODE == 0) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            h[j] = f2(0.f);
            p[j] = make_float2((c0 + 2 * j == row) ? 1.f : 0.f, (c0 + 2 * j + 1 == row) ? 1.f : 0.f);
        }
    } else {
        const float *sbase = ws_f(a, a.L.off_S) + ((size_t)bh * NC + c) * D * D;
        const float4 *src = reinterpret_cast<const float4 *>(sbase + moff);
        const float4 *src2 = reinterpret_cast<const float4 *>(sbase + moff + (size_t)ROW2 * D);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 v = src[q];
            h[2 * q] = lo2(v);
            h[2 * q + 1] = hi2(v);
            if (RPT == 2) {
                const float4 w = src2[q];
                p[2 * q] = lo2(w);
                p[2 * q + 1] = hi2(w);
            }
        }
    }
    float nbase = 0.f;
    if (MODE == 1 && tid < D)  // n^(c) at this S-chunk's start = at A-chunk c * C / CA
        nbase = ws_f(a, a.L.off_n)[((size_t)bh * (a.L.NCA + 1) + (size_t)c * (C / a.L.CA)) * D + tid];

    int failed = -1;
    for (int m = 0; m < ntiles; ++m) {
        const int buf = m & 1;
        const int nt = min(kTT, ntok - m * kTT);
        if (!mbar_wait_bounded(&bars[buf], (m >> 1) & 1, a.p.wait_limit_ns, a.p.err)) *abort_flag = 1;
        __syncthreads();
        if (*abort_flag) {
            failed = m;
            break;
        }
        // ---- preprocess the tile ----
        const IO *rk = raw + ((size_t)buf * 3 + 0) * kTT * D;
        const IO *rv = raw + ((size_t)buf * 3 + 1) * kTT * D;
        const IO *rq = raw + ((size_t)buf * 3 + 2) * kTT * D;
        const float *ra = s_ral + (size_t)buf * kTT * D;
        float *khat = s_khat;
        float *alp = s_alp;
        float *phiq = s_phiq;
        float *vv = s_v;
        for (int q = warp; q < nt; q += NW) {
            float kk[D / 32], ss = 0.f;
#pragma unroll
            for (int mm = 0; mm < D / 32; ++mm) {
                kk[mm] = io_to_f32(rk[q * D + lane + 32 * mm]);
                ss = fmaf(kk[mm], kk[mm], ss);
            }
            ss = warp_sum(ss);
            const float ks = 1.f / fmaxf(sqrtf(ss), kEps);
            float gdot = 0.f;
#pragma unroll
            for (int mm = 0; mm < D / 32; ++mm) {
                const int j = lane + 32 * mm;
                const float kh = kk[mm] * ks;
                const float al = ra[q * D + j];
                khat[q * VLEN + vidx(j)] = kh;
                alp[q * VLEN + vidx(j)] = al;
                vv[q * D + j] = io_to_f32(rv[q * D + j]);
                if (MODE == 1) {
                    const float fq = phi_elu1(io_to_f32(rq[q * D + j]));
                    phiq[q * VLEN + vidx(j)] = fq;
                    s_work[q * D + j] = phi_elu1(kh);
                    gdot = fmaf(al, fq, gdot);
                }
            }
            if (MODE == 1) {
                gdot = warp_sum(gdot);
                if (lane == 0) s_ga[q] = gdot;
            }
        }
        __syncthreads();
        if (MODE == 1) {
            if (tid < D) {
                float run = 0.f;
                for (int q = 0; q < nt; ++q) {
                    run += s_work[q * D + tid];
                    s_work[q * D + tid] = phiq[q * VLEN + vidx(tid)] * (nbase + run);
                }
                nbase += run;
            }
            __syncthreads();
            for (int q = warp; q < nt; q += NW) {
                float sacc = 0.f;
#pragma unroll
                for (int mm = 0; mm < D / 32; ++mm) sacc += s_work[q * D + lane + 32 * mm];
                sacc = warp_sum(sacc);
                if (lane == 0) s_den[q] = 1.f / (sacc + kEps);
            }
            __syncthreads();
        }
        if (tid == 0 && m + 2 < ntiles) {
            issue(m + 2);
            issued = m + 3;
        }
        // ---- token recurrences (row-local, no barrier) ----
        for (int q = 0; q < nt; ++q) {
            const float4 *kp = reinterpret_cast<const float4 *>(khat + q * VLEN + vo);
            const float4 *ap = reinterpret_cast<const float4 *>(alp + q * VLEN + vo);
            const float vi = vv[q * D + row];
            if (MODE == 0) {
                float2 ha = f2(0.f), hb = f2(0.f), pa = f2(0.f), pb = f2(0.f);
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    const float4 k4 = kp[w];
                    ha = fma2(h[2 * w], lo2(k4), ha);
                    hb = fma2(h[2 * w + 1], hi2(k4), hb);
                    pa = fma2(p[2 * w], lo2(k4), pa);
                    pb = fma2(p[2 * w + 1], hi2(k4), pb);
                }
                float hk = hsum2(add2(ha, hb)), pk = hsum2(add2(pa, pb));
#pragma unroll
                for (int o = 1; o < TPR; o <<= 1) {
                    hk += __shfl_xor_sync(0xffffffffu, hk, o);
                    pk += __shfl_xor_sync(0xffffffffu, pk, o);
                }
                const float2 rh = f2(vi - hk), rp = f2(-pk);
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    const float4 a4 = ap[w];
                    h[2 * w] = fma2(rh, lo2(a4), h[2 * w]);
                    h[2 * w + 1] = fma2(rh, hi2(a4), h[2 * w + 1]);
                    p[2 * w] = fma2(rp, lo2(a4), p[2 * w]);
                    p[2 * w + 1] = fma2(rp, hi2(a4), p[2 * w + 1]);
                }
            } else {
                const float4 *fp = reinterpret_cast<const float4 *>(phiq + q * VLEN + vo);
                float2 ka = f2(0.f), kb = f2(0.f), fa = f2(0.f), fb = f2(0.f);
                float2 kc = f2(0.f), kd = f2(0.f), fc = f2(0.f), fd = f2(0.f);
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    const float4 k4 = kp[w], f4 = fp[w];
                    ka = fma2(h[2 * w], lo2(k4), ka);
                    kb = fma2(h[2 * w + 1], hi2(k4), kb);
                    fa = fma2(h[2 * w], lo2(f4), fa);
                    fb = fma2(h[2 * w + 1], hi2(f4), fb);
                    if (RPT == 2) {
                        kc = fma2(p[2 * w], lo2(k4), kc);
                        kd = fma2(p[2 * w + 1], hi2(k4), kd);
                        fc = fma2(p[2 * w], lo2(f4), fc);
                        fd = fma2(p[2 * w + 1], hi2(f4), fd);
                    }
                }
                float sk = hsum2(add2(ka, kb)), sq = hsum2(add2(fa, fb));
                float sk2 = hsum2(add2(kc, kd)), sq2 = hsum2(add2(fc, fd));
#pragma unroll
                for (int o = 1; o < TPR; o <<= 1) {
                    sk += __shfl_xor_sync(0xffffffffu, sk, o);
                    sq += __shfl_xor_sync(0xffffffffu, sq, o);
                    if (RPT == 2) {
                        sk2 += __shfl_xor_sync(0xffffffffu, sk2, o);
                        sq2 += __shfl_xor_sync(0xffffffffu, sq2, o);
                    }
                }
                const float r = vi - sk;
                const float r2s = (RPT == 2) ? vv[q * D + row + ROW2] - sk2 : 0.f;
                const float2 r2 = f2(r), rr2 = f2(r2s);
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    const float4 a4 = ap[w];
                    h[2 * w] = fma2(r2, lo2(a4), h[2 * w]);
                    h[2 * w + 1] = fma2(r2, hi2(a4), h[2 * w + 1]);
                    if (RPT == 2) {
                        p[2 * w] = fma2(rr2, lo2(a4), p[2 * w]);
                        p[2 * w + 1] = fma2(rr2, hi2(a4), p[2 * w + 1]);
                    }
                }
                if (part == 0) {
                    const float ga = s_ga[q], rd = s_den[q];
                    gout[(size_t)(m * kTT + q) * D + row] = f32_to_io<IO>(fmaf(r, ga, sq) * rd);
                    if (RPT == 2)
                        gout[(size_t)(m * kTT + q) * D + row + ROW2] = f32_to_io<IO>(fmaf(r2s, ga, sq2) * rd);
                }
            }
        }
        __syncthreads();  // the next tile's preprocessing overwrites the processed arrays
    }
    if (failed >= 0) {
        if (tid == 0)
            for (int m = failed; m < issued; ++m)
                (void)mbar_wait_bounded(&bars[m & 1], (m >> 1) & 1, a.p.wait_limit_ns, a.p.err);
        return;
    }
    if (MODE == 0) {
        float4 *dP = reinterpret_cast<float4 *>(ws_f(a, a.L.off_P) + ((size_t)bh * NC + c) * D * D + moff);
        float4 *dH = reinterpret_cast<float4 *>(ws_f(a, a.L.off_H) + ((size_t)bh * NC + c) * D * D + moff);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            dP[q] = make_float4(p[2 * q].x, p[2 * q].y, p[2 * q + 1].x, p[2 * q + 1].y);
            dH[q] = make_float4(h[2 * q].x, h[2 * q].y, h[2 * q + 1].x, h[2 * q + 1].y);
        }
    }
}

// ---------------------------------------------------------------------------
// chain: S^(c+1) = S^(c) P_c + H_c for a block of RB rows of S
// ---------------------------------------------------------------------------
// Rows of S per chain CTA: few rows per CTA keep each step a single short dot
// product per thread (one or two outputs), with many CTAs walking the chain
// side by side; every CTA of a (b, h) reads the same chunk maps (L2 hits).
// At d = 64 a thread instead applies one column of P_c to all 4 rows over a
// quarter of the sum (each P element is read once, the rows of S broadcast),
// and the four partial sums meet in shared memory.
template <int D>
constexpr int chain_rows() { return D == 32 ? 8 : 4; }

template <int D>
struct ChainSmem {
    static constexpr int RB = chain_rows<D>();
    static constexpr int NS = (D == 128) ? 2 : 4;                    // prefetch depth (chunk maps in flight)
    static constexpr size_t bars = 0;                                // NS mbarriers + abort flag
    static constexpr size_t P = 128;                                 // [NS][D][D]
    static constexpr size_t H = P + NS * (size_t)D * D * 4;          // [NS][RB][D]
    static constexpr size_t S = H + NS * (size_t)RB * D * 4;         // [RB][D]
    static constexpr size_t red = S + (size_t)RB * D * 4;            // (d = 64) [4 quarters][RB][D] partial sums
    static constexpr size_t total = red + (D == 64 ? 4 * (size_t)RB * D * 4 : 0);
};

template <int D>
__global__ void __launch_bounds__(256) chain_kernel(ChunkArgs a) {
    using Lo = ChainSmem<D>;
    constexpr int NS = Lo::NS, kRB = Lo::RB;
    constexpr int OPT = kRB * D / 256;  // outputs per thread: one row, OPT consecutive columns
    static_assert(OPT >= 1, "at least one output per thread");
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lo::bars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Lo::bars + 8 * NS);
    float *sP = reinterpret_cast<float *>(smem + Lo::P);
    float *sH = reinterpret_cast<float *>(smem + Lo::H);
    float *sS = reinterpret_cast<float *>(smem + Lo::S);
    const int rb = (int)(blockIdx.x % (D / kRB)), bh = a.bh_lo + (int)(blockIdx.x / (D / kRB));  // row block, unit
    const int NC = a.L.NC;
    const int tid = threadIdx.x;
    const int r = tid / (D / OPT), j0 = (tid % (D / OPT)) * OPT;
    const int grow = rb * kRB + r;  // row of S
    const float *gP = ws_f(a, a.L.off_P) + (size_t)bh * NC * D * D;
    const float *gH = ws_f(a, a.L.off_H) + (size_t)bh * NC * D * D + (size_t)rb * kRB * D;
    float *gS = ws_f(a, a.L.off_S) + (size_t)bh * NC * D * D + (size_t)rb * kRB * D;

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    float s[OPT];
#pragma unroll
    for (int q = 0; q < OPT; ++q)
        s[q] = a.p.S0 ? a.p.S0[((size_t)bh * D + grow) * D + j0 + q] : 0.f;
#pragma unroll
    for (int q = 0; q < OPT; ++q) sS[r * D + j0 + q] = s[q];
    __syncthreads();
    auto issue = [&](int cc) {
        const int buf = cc % NS;
        mbar_arrive_expect_tx(&bars[buf], (uint32_t)((D * D + kRB * D) * 4));
        bulk_g2s(sP + (size_t)buf * D * D, gP + (size_t)cc * D * D, (uint32_t)(D * D * 4), &bars[buf]);
        bulk_g2s(sH + (size_t)buf * kRB * D, gH + (size_t)cc * D * D, (uint32_t)(kRB * D * 4), &bars[buf]);
    };
    int issued = 0;
    if (tid == 0) {
        for (int cc = 0; cc < NS && cc < NC; ++cc) issue(cc);
        issued = min(NC, NS);
    }
    int failed = -1;
    for (int cc = 0; cc < NC; ++cc) {
        // chunk-start state S^(cc)
#pragma unroll
        for (int q = 0; q < OPT; ++q) gS[(size_t)cc * D * D + r * D + j0 + q] = s[q];
        const int buf = cc % NS;
        if (!mbar_wait_bounded(&bars[buf], (cc / NS) & 1, a.p.wait_limit_ns, a.p.err)) *abort_flag = 1;
        __syncthreads();
        if (*abort_flag) {
            failed = cc;
            break;
        }
        const float *P = sP + (size_t)buf * D * D;
        const float *Hh = sH + (size_t)buf * kRB * D;
        float acc[OPT];
        if constexpr (D == 64) {
            // column jj of P_c on all 4 rows, over the quarter k in [16 kq, 16 kq + 16)
            float *red = reinterpret_cast<float *>(smem + Lo::red);
            const int kq = tid >> 6, jj = tid & 63;
            float part[kRB];
#pragma unroll
            for (int q = 0; q < kRB; ++q) part[q] = 0.f;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int k0 = 16 * kq + 4 * g;
                float4 sv[kRB];
#pragma unroll
                for (int q = 0; q < kRB; ++q) sv[q] = *reinterpret_cast<const float4 *>(sS + q * D + k0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const float pv = P[(k0 + kk) * D + jj];
#pragma unroll
                    for (int q = 0; q < kRB; ++q) {
                        const float sk = kk == 0 ? sv[q].x : kk == 1 ? sv[q].y : kk == 2 ? sv[q].z : sv[q].w;
                        part[q] = fmaf(sk, pv, part[q]);
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < kRB; ++q) red[(kq * kRB + q) * D + jj] = part[q];
            __syncthreads();
            acc[0] = Hh[r * D + j0];
#pragma unroll
            for (int h = 0; h < 4; ++h) acc[0] += red[(h * kRB + r) * D + j0];
        } else {
#pragma unroll
            for (int q = 0; q < OPT; ++q) acc[q] = Hh[r * D + j0 + q];
            const float *srow = sS + r * D;
#pragma unroll 8
            for (int k = 0; k < D; ++k) {
                const float sk = srow[k];
#pragma unroll
                for (int q = 0; q < OPT; ++q) acc[q] = fmaf(sk, P[k * D + j0 + q], acc[q]);
            }
        }
        __syncthreads();  // everyone done reading sS and this buffer
#pragma unroll
        for (int q = 0; q < OPT; ++q) {
            s[q] = acc[q];
            sS[r * D + j0 + q] = acc[q];
        }
        if (tid == 0 && cc + NS < NC) {
            issue(cc + NS);
            issued = cc + NS + 1;
        }
        __syncthreads();
    }
    if (failed >= 0) {
        if (tid == 0)
            for (int m = failed; m < issued; ++m)
                (void)mbar_wait_bounded(&bars[m % NS], (m / NS) & 1, a.p.wait_limit_ns, a.p.err);
        return;
    }
#pragma unroll
    for (int q = 0; q < OPT; ++q) a.p.S_T[((size_t)bh * D + grow) * D + j0 + q] = s[q];
}

// ---------------------------------------------------------------------------
// M_0 = A0^{-1} (only when A0 is given)
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(RowCfg<D>::NT) invert_a0_kernel(ChunkArgs a) {
    using R = RowCfg<D>;
    __shared__ __align__(16) float piv[2 * R::VLEN];
    const int bh = a.bh_lo + (int)blockIdx.x;
    const int tid = threadIdx.x, row = tid / R::TPR, part = tid % R::TPR, c0 = part * 32;
    float x[32];
    const float *src = a.p.A0 + (size_t)bh * D * D + row * D + c0;
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = src[j];
    gj_inverse<D, 32>(x, piv, row, part);
    float *dst = ws_f(a, a.L.off_M0) + (size_t)bh * D * D + row * D + c0;
#pragma unroll
    for (int j = 0; j < 32; ++j) dst[j] = x[j];
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// The tensor-core path (d = 64, bf16 I/O) in two parts per range of units:
// the front (the initial-A inverse when A0 is given, the Grams, their prefix
// and the gates: reads u and k) and the back (the state pass, the chain and
// the output pass: reads q, k, v and the gates). Launch boundaries are
// numbered on from *p.launches.
bool tc_parts_ok(const FwdParams &p, const ChunkLayout &L) {
    return p.d == 64 && p.io_bf16 && p.rows_tc && kGatesOnTensorCores && gram_tma_supported(p, L) &&
           gates_tc_supported(p, L) && rows_tc_supported(p, L);
}

cudaError_t tc_front(const ChunkArgs &a, cudaStream_t st) {
    constexpr int D = 64;
    using R = RowCfg<D>;
    const long long n_units = a.bh_n > 0 ? a.bh_n : a.p.BH;
    int n = a.p.launches ? *a.p.launches : 0;
    if (n == 0) mark_launch(a.p, 0, st);
    cudaError_t e;
    if (a.p.A0) {
        invert_a0_kernel<D><<<(unsigned)n_units, R::NT, 0, st>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        mark_launch(a.p, ++n, st);
    }
    if ((e = launch_gram_tma(a, st)) != cudaSuccess) return e;
    mark_launch(a.p, ++n, st);
    prefix_kernel<D><<<(unsigned)(((D * D + D + 255) / 256) * n_units), 256, 0, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mark_launch(a.p, ++n, st);
    if ((e = launch_gates_tc(a, st)) != cudaSuccess) return e;
    mark_launch(a.p, ++n, st);
    return cudaSuccess;
}

// Both passes over resident inputs: the Grams, their prefix, the gates and the
// state pass as one queue launch, the chain, the output pass.
cudaError_t tc_fused(const ChunkArgs &a, cudaStream_t st) {
    constexpr int D = 64;
    using R = RowCfg<D>;
    const long long n_units = a.bh_n > 0 ? a.bh_n : a.p.BH;
    int n = a.p.launches ? *a.p.launches : 0;
    if (n == 0) mark_launch(a.p, 0, st);
    cudaError_t e;
    if (a.p.A0) {
        invert_a0_kernel<D><<<(unsigned)n_units, R::NT, 0, st>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        mark_launch(a.p, ++n, st);
    }
    if ((e = launch_gram_tma(a, st)) != cudaSuccess) return e;
    mark_launch(a.p, ++n, st);
    prefix_kernel<D><<<(unsigned)(((D * D + D + 255) / 256) * n_units), 256, 0, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mark_launch(a.p, ++n, st);
    if ((e = launch_tc64_queue(a, st)) != cudaSuccess) return e;
    mark_launch(a.p, ++n, st);
    if ((e = set_smem(chain_kernel<D>, ChainSmem<D>::total)) != cudaSuccess) return e;
    chain_kernel<D><<<(unsigned)((D / chain_rows<D>()) * n_units), 256, ChainSmem<D>::total, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mark_launch(a.p, ++n, st);
    if ((e = launch_rows_tc(a, 1, st)) != cudaSuccess) return e;
    mark_launch(a.p, ++n, st);
    return cudaSuccess;
}

// The device entry's choice between one queue launch and two (tc_queue_pays_jobs).
bool tc_queue_pays(const ChunkArgs &a) {
    const long long n = a.bh_n > 0 ? a.bh_n : a.p.BH;
    return tc_queue_pays_jobs(n * a.L.NCA, n * a.L.NC);
}

cudaError_t tc_back(const ChunkArgs &a, cudaStream_t st) {
    constexpr int D = 64;
    const long long n_units = a.bh_n > 0 ? a.bh_n : a.p.BH;
    int n = a.p.launches ? *a.p.launches : 0;
    cudaError_t e;
    if ((e = set_smem(chain_kernel<D>, ChainSmem<D>::total)) != cudaSuccess) return e;
    if ((e = launch_rows_tc(a, 0, st)) != cudaSuccess) return e;
    mark_launch(a.p, ++n, st);
    chain_kernel<D><<<(unsigned)((D / chain_rows<D>()) * n_units), 256, ChainSmem<D>::total, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mark_launch(a.p, ++n, st);
    if ((e = launch_rows_tc(a, 1, st)) != cudaSuccess) return e;
    mark_launch(a.p, ++n, st);
    return cudaSuccess;
}

template <int D, typename IO>
cudaError_t launch_chunk_t(const ChunkArgs &a, cudaStream_t st) {
    using R = RowCfg<D>;
    const long long BH = a.p.BH, NC = a.L.NC, NCA = a.L.NCA;
    if (NCA * BH > 0x7fffffffLL || BH * ((D * D + D + 255) / 256) > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    cudaError_t e;
    if constexpr (D == 128 && sizeof(IO) == 2) {
        if (a.p.rows_tc && a.L.NC == 1 && a.L.NCA == 1 && tile_maps_available()) {
            // one chunk per unit: the gates from A0, then the state pass on S itself
            // (writes o); both in one queue launch unless q and v are still arriving
            mark_launch(a.p, 0, st);
            if (!a.p.wait_qv) {
                if ((e = launch_tc128_queue(a, st)) != cudaSuccess) return e;
                mark_launch(a.p, 1, st);
                return cudaSuccess;
            }
            if ((e = launch_gates_tc128(a, st)) != cudaSuccess) return e;
            mark_launch(a.p, 1, st);
            if (a.p.wait_qv && (e = cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(a.p.wait_qv), 0)) != cudaSuccess)
                return e;
            if ((e = launch_rows_tc128(a, st)) != cudaSuccess) return e;
            mark_launch(a.p, 2, st);
            return cudaSuccess;
        }
    }
    if constexpr (D == 64 && sizeof(IO) == 2) {
        if (tc_parts_ok(a.p, a.L)) {
            if (!a.p.wait_qv && tc_queue_pays(a)) return tc_fused(a, st);
            if ((e = tc_front(a, st)) != cudaSuccess) return e;
            // the front reads u and k only; q and v may still be arriving
            if (a.p.wait_qv && (e = cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(a.p.wait_qv), 0)) != cudaSuccess)
                return e;
            return tc_back(a, st);
        }
    }
    if ((e = set_smem(gates_kernel<D, IO>, GatesSmem<D, IO>::total)) != cudaSuccess) return e;
    using G = GatesCfg<D>;
    if ((e = set_smem(rows_kernel<D, IO, 0>, RowsSmem<D, IO>::total)) != cudaSuccess) return e;
    if ((e = set_smem(chain_kernel<D>, ChainSmem<D>::total)) != cudaSuccess) return e;
    if constexpr (sizeof(IO) == 2 && D >= 64)
        if ((e = set_smem(gram_tc_kernel<D>, GramTc<D>::total)) != cudaSuccess) return e;
    if ((e = set_smem(rows_kernel<D, IO, 1>, RowsSmem<D, IO>::total)) != cudaSuccess) return e;
    int n = 0;
    mark_launch(a.p, n, st);
    if (a.p.A0) {
        invert_a0_kernel<D><<<(unsigned)BH, R::NT, 0, st>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        mark_launch(a.p, ++n, st);
    }
    if (a.p.rows_tc && gram_tma_supported(a.p, a.L)) {
        if ((e = launch_gram_tma(a, st)) != cudaSuccess) return e;
    } else if constexpr (sizeof(IO) == 2 && D >= 64) {
        gram_tc_kernel<D><<<(unsigned)(NCA * BH), GramTc<D>::NT, GramTc<D>::total, st>>>(a);
    } else {
        gram_kernel<D, IO><<<(unsigned)(NCA * BH), 256, 0, st>>>(a);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mark_launch(a.p, ++n, st);
    prefix_kernel<D><<<(unsigned)(((D * D + D + 255) / 256) * BH), 256, 0, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mark_launch(a.p, ++n, st);
    const bool gtc = kGatesOnTensorCores && a.p.rows_tc && gates_tc_supported(a.p, a.L);
    if (gtc) {
        if ((e = launch_gates_tc(a, st)) != cudaSuccess) return e;
    } else {
        gates_kernel<D, IO><<<(unsigned)(NCA * BH), G::NT, GatesSmem<D, IO>::total, st>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    mark_launch(a.p, ++n, st);
    // the tensor-core state pass reads the gates in the fp16 form that only the
    // tensor-core gates write
    const bool tc = gtc && rows_tc_supported(a.p, a.L);
    // the passes so far read u and k only; q and v may still be arriving
    if (a.p.wait_qv && (e = cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(a.p.wait_qv), 0)) != cudaSuccess)
        return e;
    if (tc) {
        if ((e = launch_rows_tc(a, 0, st)) != cudaSuccess) return e;
    } else {
        rows_kernel<D, IO, 0><<<(unsigned)(NC * BH), RowsCfg<D, 0>::NT, RowsSmem<D, IO>::total, st>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    mark_launch(a.p, ++n, st);
    chain_kernel<D><<<(unsigned)((D / chain_rows<D>()) * BH), 256, ChainSmem<D>::total, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mark_launch(a.p, ++n, st);
    if (tc) {
        if ((e = launch_rows_tc(a, 1, st)) != cudaSuccess) return e;
    } else if (!a.p.skip_out) {
        rows_kernel<D, IO, 1><<<(unsigned)(NC * BH), RowsCfg<D, 1>::NT, RowsSmem<D, IO>::total, st>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    } else {
        return cudaSuccess;
    }
    mark_launch(a.p, ++n, st);
    return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

// S-chunk length: long chunks keep the chain along the chunks short.
int chunk_default(int BH, int T) {
    int C = T >= 16384 ? 512 : (T >= 4096 ? 256 : (T >= 1024 ? 128 : 64));
    while (C > 64 && (long long)BH * ((T + C - 1) / C) < 2 * 152) C /= 2;
    return C;
}

// A-chunk length (divides C): the gates pass is a latency-bound recurrence,
// one CTA per A-chunk, so pick the length that minimises
// waves x (chunk length + Gauss-Jordan restart), with the resident CTAs per
// SM of each d on the 152 SMs of a GB300.
int chunk_default_a(int BH, int T, int d, int C) {
    const long long resident = 152LL * (d == 32 ? 32 : (d == 64 ? 10 : 1));
    const int restart = 20;  // Gauss-Jordan inverse, in token-steps
    int best = C;
    long long best_cost = -1;
    for (int CA = C; CA >= 64; CA /= 2) {
        if (C % CA) continue;
        const long long chunks = (long long)BH * ((T + CA - 1) / CA);
        const long long waves = (chunks + resident - 1) / resident;
        const long long cost = waves * (CA + restart);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = CA;
        }
    }
    return best;
}

// Wave model of the tensor-core passes (d = 64): each CTA walks its chunk one
// 64-token sub-block after another, two CTAs resident per SM. The time of a
// pass of `ctas` CTAs, each `len` sub-block times long: its full waves on the
// 2 x 152 slots, then a partial one, which costs a whole CTA time if some SM
// holds two of its CTAs and about 0.72 of one if none does (a CTA alone on an
// SM runs that much faster, measured on the state pass).
static double tc_pass_cost(long long ctas, double len) {
    const long long slots = 2LL * 152;
    const long long full = ctas / slots, rem = ctas % slots;
    return len * ((double)full + (rem == 0 ? 0.0 : (rem <= 152 ? 0.72 : 1.0)));
}

// S-chunk length of the tensor-core path, a multiple of 64 (the long stream,
// 16 units of 65536 tokens: 1728, two full waves of 27 sub-blocks, where 512
// took seven waves of 8 with the last one part full). It minimises, in
// sub-block times, the passes of vla_forward over all units plus the same pass
// over each half of the units (the host entry runs the halves one after the
// other, to overlap the copies), plus the chain along the chunks, about 0.045
// of a sub-block per chunk (measured), counted for both.  A CTA costs its
// sub-blocks plus kTcCtaCost for its start and end (the chunk start in, the
// chunk maps out).  Where vla_forward takes the queue launch (tc_queue_pays)
// its passes cost their packed jobs plus half a job of ragged end.
constexpr double kTcCtaCost = 0.6;  // fitted: 0.4 .. 1.0 give the same lengths on the
                                    // five shapes timed (8 x 16 x 1024 tokens: 0.446 ms at
                                    // C = 64, 0.295 ms at C = 256)
int chunk_default_tc(int BH, int T) {
    static thread_local int last_BH = -1, last_T = -1, last_C = 64;
    if (BH == last_BH && T == last_T) return last_C;
    const int maxm = std::min((T + 63) / 64, 1024);
    const long long h1 = BH / 2, h2 = BH - BH / 2;
    int best = 64;
    double best_cost = -1;
    for (int m = 1; m <= maxm; ++m) {
        const long long NC = (T + 64LL * m - 1) / (64LL * m);
        const double len = m + kTcCtaCost;
        double full = tc_pass_cost(BH * NC, len);
        if (tc_queue_pays_jobs(BH * NC, BH * NC))  // per pass: half the packed jobs and of the ragged end
            full = 1.08 * (double)(BH * NC) * len / (2.0 * 152) + 0.25 * len;
        const double halves = h1 > 0 ? tc_pass_cost(h1 * NC, len) + tc_pass_cost(h2 * NC, len) : full;
        const double cost = full + halves + 2 * 0.045 * (double)NC;
        if (best_cost < 0 || cost < best_cost - 1e-9) {
            best_cost = cost;
            best = 64 * m;
        }
    }
    last_BH = BH, last_T = T, last_C = best;
    return best;
}

// A-chunk length of the tensor-core gates: a multiple of 64 that divides C
// (each S-chunk starts on an A-chunk boundary), by the same wave model, each
// A-chunk its sub-blocks plus the restart (the inverse of the prefix), about
// 0.4 of a sub-block.
int chunk_default_a_tc(int BH, int T, int C) {
    const int m = C / 64;
    int best = C;
    double best_cost = -1;
    for (int j = m; j >= 1; --j) {
        if (m % j) continue;
        const long long NCA = (T + 64LL * j - 1) / (64LL * j);
        const double cost = tc_pass_cost(BH * NCA, j + 0.4);
        if (best_cost < 0 || cost < best_cost - 1e-9) {
            best_cost = cost;
            best = 64 * j;
        }
    }
    return best;
}

// The tensor-core path at d = 128 runs one chunk per unit, one CTA per unit
// and pass at one CTA per SM: the default when the units alone fill the GPU.
constexpr int kTc128MinUnits = 128;

// S-chunk length of the tensor-core path for one range of the host entry, a
// problem of `units` units on its own: the wave model of tc_pass_cost for one
// pass, plus the chain along the chunks (chunk_default_tc also weighs the pass
// over each half of the units, which a range does not run).
static int chunk_default_tc_range(int units, int T) {
    const int maxm = std::min((T + 63) / 64, 1024);
    int best = 64;
    double best_cost = -1;
    for (int m = 1; m <= maxm; ++m) {
        const long long NC = (T + 64LL * m - 1) / (64LL * m);
        const double cost = tc_pass_cost((long long)units * NC, m) + 0.045 * (double)NC;
        if (best_cost < 0 || cost < best_cost - 1e-9) {
            best_cost = cost;
            best = 64 * m;
        }
    }
    return best;
}

static ChunkLayout layout_for(int BH, int T, int d, int C, int CA, bool tc);

ChunkLayout chunk_layout(int BH, int T, int d, int chunk, bool tc_path) {
    const bool single = chunk == 0 && tc_path && d == 128 && BH >= kTc128MinUnits;
    const int C = chunk > 0 ? chunk
                            : (single ? (T + 63) / 64 * 64
                                      : (tc_path && d == 64 ? chunk_default_tc(BH, T) : chunk_default(BH, T)));
    const bool tc = tc_path && d == 64 && C % 64 == 0;
    const int CA = chunk > 0 || single ? C : (tc ? chunk_default_a_tc(BH, T, C) : chunk_default_a(BH, T, d, C));
    return layout_for(BH, T, d, C, CA, tc);
}

TcHostPlan tc_host_plan(int BH, int T, int chunk) {
    TcHostPlan P{};
    if (BH < 2 || T <= 0) return P;
    const int h = BH / 2;
    P.sub_lo[0] = 0;
    P.sub_lo[1] = h;
    P.sub_lo[2] = BH;
    P.n = (BH - h >= 2) ? 3 : 2;
    P.lo[0] = 0;
    P.lo[1] = h;
    if (P.n == 3) P.lo[2] = h + (BH - h) / 2;
    P.lo[P.n] = BH;
    for (int r = 0; r < P.n; ++r) P.part[r] = r == 0 ? 0 : 1;
    // The first half keeps the whole problem's chunk length.  The second half's
    // last back range is what runs after the last upload: it takes the chunk
    // length of a lone pass over that range (its passes then fill the GPU for
    // fewer sub-blocks) when that is at least 512 tokens; below that the longer
    // chain along the chunks and the fixed cost of each launch outweigh what the
    // shorter chunks save (measured: 4 x 8 x 4096 end to end 0.551 -> 0.568 ms
    // with 128-token chunks there, 16 units x 65536 tokens 3.141 -> 3.118 ms
    // with 896).
    const int whole = chunk_default_tc(BH, T);
    const int last = chunk_default_tc_range(P.lo[P.n] - P.lo[P.n - 1], T);
    size_t off = 0;
    for (int s = 0; s < 2; ++s) {
        // A-chunks as long as the S-chunks, as with an explicit chunk length: a
        // range is then exactly vla_forward on its units with chunk = C
        const int C = chunk > 0 ? chunk : (s == 1 && last >= 512 ? last : whole);
        P.L[s] = layout_for(P.sub_lo[s + 1] - P.sub_lo[s], T, 64, C, C, C % 64 == 0);
        P.off[s] = off;
        off = align256(off + P.L[s].total);
    }
    P.total = off;
    return P;
}

static ChunkLayout layout_for(int BH, int T, int d, int C, int CA, bool tc) {
    ChunkLayout L{};
    L.C = C;
    L.CA = CA;
    L.NC = (T + L.C - 1) / L.C;
    L.NCA = (T + L.CA - 1) / L.CA;
    const size_t bh = (size_t)BH, nc = (size_t)L.NC, nca = (size_t)L.NCA, dd = (size_t)d * d;
    size_t off = 0;
    L.off_M = off; off = align256(off + bh * nca * dd * 4);
    L.off_n = off; off = align256(off + bh * (nca + 1) * d * 4);
    L.off_M0 = off; off = align256(off + bh * dd * 4);
    L.off_alpha = off; off = align256(off + bh * (size_t)T * d * 4);
    L.off_P = off; off = align256(off + bh * nc * dd * 4);
    L.off_H = off; off = align256(off + bh * nc * dd * 4);
    L.off_S = off; off = align256(off + bh * nc * dd * 4);
    L.off_yh = off;
    L.yh = tc ? 1 : 0;
    if (L.yh) off = align256(off + bh * nc * (size_t)(L.C / 64) * 16384);
    L.off_q = off; off = align256(off + (bh * nca + 1) * 4);  // job counter and flags of the queue launches
    L.total = off;
    return L;
}

bool chunk_tc_parts_supported(const FwdParams &p, const ChunkLayout &L) { return tc_parts_ok(p, L); }

bool chunk_tc128_parts_supported(const FwdParams &p, const ChunkLayout &L) {
    return p.d == 128 && p.io_bf16 && p.rows_tc && L.NC == 1 && L.NCA == 1 && tile_maps_available();
}

cudaError_t launch_chunk_tc128_part(const FwdParams &p, const ChunkLayout &L, int part, int bh_lo, int bh_n,
                                    cudaStream_t stream) {
    if (!chunk_tc128_parts_supported(p, L) || bh_lo < 0 || bh_n <= 0 || bh_lo + bh_n > p.BH)
        return cudaErrorInvalidValue;
    ChunkArgs a{p, L};
    a.bh_lo = bh_lo;
    a.bh_n = bh_n;
    int n = p.launches ? *p.launches : 0;
    if (n == 0) mark_launch(p, 0, stream);
    const cudaError_t e = part == 0 ? launch_gates_tc128(a, stream) : launch_rows_tc128(a, stream);
    if (e != cudaSuccess) return e;
    mark_launch(p, ++n, stream);
    return cudaSuccess;
}

cudaError_t launch_chunk_tc_part(const FwdParams &p, const ChunkLayout &L, int part, int bh_lo, int bh_n,
                                 cudaStream_t stream) {
    if (!tc_parts_ok(p, L) || bh_lo < 0 || bh_n <= 0 || bh_lo + bh_n > p.BH) return cudaErrorInvalidValue;
    if ((long long)L.NCA * bh_n > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    ChunkArgs a{p, L};
    a.bh_lo = bh_lo;
    a.bh_n = bh_n;
    return part == 0 ? tc_front(a, stream) : tc_back(a, stream);
}

cudaError_t launch_chunk(const FwdParams &p, const ChunkLayout &L, cudaStream_t stream) {
    if (p.BH == 0) return cudaSuccess;
    ChunkArgs a{p, L};
    if (p.io_bf16) {
        switch (p.d) {
            case 32: return launch_chunk_t<32, __nv_bfloat16>(a, stream);
            case 64: return launch_chunk_t<64, __nv_bfloat16>(a, stream);
            case 128: return launch_chunk_t<128, __nv_bfloat16>(a, stream);
        }
    } else {
        switch (p.d) {
            case 32: return launch_chunk_t<32, float>(a, stream);
            case 64: return launch_chunk_t<64, float>(a, stream);
            case 128: return launch_chunk_t<128, float>(a, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace vla
