// vla_internal.cuh -- shared declarations of libvla's translation units:
// launch parameter block, launcher prototypes and the sm_100-family PTX
// helpers (mbarrier, bulk async copy, bounded waits) the kernels use.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace vla {

constexpr float kEps = 1e-6f;  // key norm, gate norm and readout denominator guard

// Shared-memory vectors are stored in 32-float parts with a stride of 36
// floats, so that the d/32 threads of a row, which read different parts in
// the same instruction, hit different banks.
constexpr int kPart = 36;
__host__ __device__ __forceinline__ int vidx(int j) { return (j >> 5) * kPart + (j & 31); }

// Device error word values (written with atomicExch, read by vla_device_status).
constexpr int kDevErrTimeout = 1;

struct FwdParams {
    const void *q, *k, *v, *u;  // [BH, T, d] io dtype
    void *o;                    // [BH, T, d] io dtype
    const float *S0, *A0, *n0;  // optional initial state
    float *S_T, *A_T, *n_T;     // final state (n_T optional)
    int BH, T, d;
    int io_bf16;                // 1: bf16 I/O, 0: fp32 I/O
    float lambda0;
    int *err;                   // device error word
    long long wait_limit_ns;    // bound on every device-side wait
    int inject;                 // test hook: 1 = never request the first input tile
    void *ws;                   // workspace (chunked kernel)
    size_t ws_bytes;
    int chunk;                  // chunk length (chunked kernel)
    int rows_tc;                // chunked kernel: state passes on the tensor cores where supported
    int skip_out;               // chunked kernel, SIMT passes: no output pass (o not written); the
                                // backward's forward, which needs only the chunk-start states
    void *wait_qv;              // optional cudaEvent_t: the stream waits for it before the first pass
                                // that reads q or v (the chunked path's state pass)
    void *const *events;        // measurement hook: cudaEvent_t handles, or null
    int n_events;
    int *launches;              // out: number of kernels launched
};

// Records the measurement event for launch boundary i (0 = before the first
// kernel) and counts launches.
inline void mark_launch(const FwdParams &p, int i, cudaStream_t st) {
    if (p.events && i < p.n_events && p.events[i])
        cudaEventRecord(static_cast<cudaEvent_t>(p.events[i]), st);
    if (p.launches && i > *p.launches) *p.launches = i;
}

// Sequential kernel: one CTA per (b, h).  Returns a cudaError_t.
cudaError_t launch_seq(const FwdParams &p, cudaStream_t stream);
// Its d = 32 form: three warps per (b, h) (inputs, A chain, S chain).
cudaError_t launch_seq32(const FwdParams &p, cudaStream_t stream);

// Backward pass (gradients of the recurrence); one CTA per (b, h).
struct BwdParams {
    const void *q, *k, *v, *u, *dO;                  // [BH, T, d] io dtype
    const float *S0, *A0, *n0, *dS_T, *dA_T, *dn_T;  // optional
    float *dq, *dk, *dv, *du;                        // [BH, T, d] fp32 (each optional)
    float *dS0, *dA0, *dn0;                          // optional
    int BH, T, d, io_bf16;
    float lambda0;
    float *ws;                                       // backward_workspace_floats(BH, T, d) floats
    int *launches;                                   // out (optional): kernels launched
};
size_t backward_workspace_floats(int BH, int T, int d);
// Tokens between the state checkpoints of the sequential backward (its
// workspace holds, per (b, h), T records of 4 d + 4 floats, then one (S, A,
// n) checkpoint of 2 d^2 + d floats per kBwdCk tokens).
constexpr int kBwdCk = 64;
// The sequential backward at d = 128 (vla_backward128.cu): S and dS in shared memory.
cudaError_t launch_backward128(const BwdParams &p, cudaStream_t stream);
cudaError_t launch_backward(const BwdParams &p, cudaStream_t stream);
// The backward in parallel over the chunked forward's S-chunks (vla_backward_chunk.cu):
// its workspace bytes (the larger of the bf16 and fp32 layouts; 0 when fewer
// than two chunks), and its launches (*used = false, nothing launched, when it
// does not apply to the shape).
size_t backward_chunk_bytes(int BH, int T, int d);
cudaError_t launch_backward_chunk(const BwdParams &p, cudaStream_t stream, bool *used);

// Decode step: one CTA per (b, h), state streamed from HBM.  Returns a cudaError_t.
cudaError_t launch_decode(const FwdParams &p, cudaStream_t stream);

// Workspace of the chunk-parallel path (byte offsets, 256-byte aligned).
// Two chunkings of the token axis: A-chunks of CA tokens (Grams, prefix,
// gates) and S-chunks of C tokens (transitions, chain, readout); CA divides C.
struct ChunkLayout {
    int C;               // S-chunk length (multiple of 16)
    int NC;              // S-chunks per (b, h) = ceil(T / C)
    int CA;              // A-chunk length (multiple of 16, divides C)
    int NCA;             // A-chunks per (b, h) = ceil(T / CA)
    size_t off_M;        // [BH][NCA][d][d]  A-chunk Grams, then exclusive prefix M^(c)
    size_t off_n;        // [BH][NCA+1][d]   A-chunk sums of phi(k_hat), then exclusive prefix n^(c)
    size_t off_M0;       // [BH][d][d]      inverse of A0 (only when A0 is given)
    size_t off_alpha;    // [BH][T][d]      unit gates alpha_t (fp32; fp16 on the tensor-core passes)
    size_t off_P;        // [BH][NC][d][d]  chunk transition P_c
    size_t off_H;        // [BH][NC][d][d]  chunk offset H_c
    size_t off_S;        // [BH][NC][d][d]  chunk-start states S^(c)
    size_t off_yh;       // [BH][NC][C/64][2][64][64] bf16: readout coefficients y_t, h_t (operand
                         // tiles) of every 64-token sub-block, written by the tensor-core
                         // state pass for the output pass
    int yh;              // 1 when the off_yh region is reserved
    size_t off_q;        // [BH NCA + 1] u32: job counter and flags of the queue launches
    size_t total;
};

// C-ABI helpers defined in vla_api.cu, shared by the other entry points.
int api_check_common(int io_dtype, float lambda0, int B, int H, int T, int d_h, int kernel);
int *api_device_err_word();
long long api_wait_limit_ns();
int api_cuda_fail(cudaError_t e);

// Layout for a shape; chunk > 0 (a multiple of 16) sets both chunk lengths,
// chunk == 0 picks the defaults.  tc reserves the readout coefficients of
// the tensor-core state pass (d = 64, chunks a multiple of 64 tokens).
ChunkLayout chunk_layout(int BH, int T, int d, int chunk, bool tc = false);
// The host entry's plan on the tensor-core path at d = 64 with bf16 I/O: two
// problems of their own, the first half of the units and the rest (sub_lo),
// each with its layout at byte offset off[s] of the workspace (total bytes in
// all) and S- and A-chunks of one length (`chunk` when given; else the whole
// problem's default, and for the second half that of a lone pass over its last
// back range when that is at least 512 tokens).  The fronts run
// per half; the backs per range r (n of them: the first half, then the rest in
// one or two), range r from unit lo[r] in half part[r].  n = 0 when BH < 2.
struct TcHostPlan {
    int n;
    int lo[4];          // first unit of back range r; lo[n] = BH
    int part[3];        // the half back range r lies in
    int sub_lo[3];      // first unit of half s; sub_lo[2] = BH
    ChunkLayout L[2];
    size_t off[2];
    size_t total;
};
TcHostPlan tc_host_plan(int BH, int T, int chunk);
// Chunk-parallel path (six launches).  Returns a cudaError_t.
cudaError_t launch_chunk(const FwdParams &p, const ChunkLayout &L, cudaStream_t stream);
// The tensor-core path (d = 64, bf16 I/O, every pass on its tensor-core
// kernel) for a range of units [bh_lo, bh_lo + bh_n), in two parts: part 0,
// the front (the initial-A inverse when A0 is given, the Grams, their prefix
// and the gates; reads u and k), and part 1, the back (the state pass, the
// chain and the output pass; reads q, k, v and the front's gates). A caller
// that overlaps the input uploads runs the fronts and the backs of its
// ranges as the data lands; each back after its range's front. Launch
// boundaries are numbered on from *p.launches.
bool chunk_tc_parts_supported(const FwdParams &p, const ChunkLayout &L);
cudaError_t launch_chunk_tc_part(const FwdParams &p, const ChunkLayout &L, int part, int bh_lo, int bh_n,
                                 cudaStream_t stream);

// Kernel argument of the chunk-parallel kernels.
struct ChunkArgs {
    FwdParams p;
    ChunkLayout L;
    int bh_lo = 0, bh_n = 0;  // (b, h) units of a state-pass launch (bh_n = 0: all)
};
__device__ __forceinline__ float *ws_f(const ChunkArgs &a, size_t off) {
    return reinterpret_cast<float *>(static_cast<unsigned char *>(a.p.ws) + off);
}

// Tensor-core state passes (UT transform over 64-token sub-blocks) for d = 64
// with bf16 I/O and S-chunks a multiple of 64 tokens; mode 0 = the state
// pass (chunk transitions P_c, H_c and the readout coefficients y_t, h_t),
// mode 1 = the output pass o_t = S^(c) y_t + h_t.  Defined in vla_chunk_tc.cu.
bool rows_tc_supported(const FwdParams &p, const ChunkLayout &L);
cudaError_t launch_rows_tc(const ChunkArgs &a, int mode, cudaStream_t stream);
// Tensor-core gates (block Woodbury over 64-token sub-blocks), same shapes;
// A-chunks a multiple of 64 tokens.  Defined in vla_gates_tc.cu.
bool gates_tc_supported(const FwdParams &p, const ChunkLayout &L);
cudaError_t launch_gates_tc(const ChunkArgs &a, cudaStream_t stream);
// d = 128 with bf16 I/O and one chunk per (b, h) unit (L.NC == L.NCA == 1):
// the gates (block Woodbury from A0, vla_gates_tc128.cu) and the state pass
// that runs S itself and writes o (vla_rows_tc128.cu), one CTA per unit each.
cudaError_t launch_gates_tc128(const ChunkArgs &a, cudaStream_t stream);
cudaError_t launch_rows_tc128(const ChunkArgs &a, cudaStream_t stream);
// Both in one persistent launch over all units, a CTA per SM taking the units'
// passes from a queue in the workspace (vla_tc128.cu).
cudaError_t launch_tc128_queue(const ChunkArgs &a, cudaStream_t stream);
// The same for a range of units [bh_lo, bh_lo + bh_n): part 0 the gates (reads u
// and k), part 1 the state pass (reads q, k, v and the gates; writes o, S_T,
// n_T).  Launch boundaries are numbered on from *p.launches.
bool chunk_tc128_parts_supported(const FwdParams &p, const ChunkLayout &L);
cudaError_t launch_chunk_tc128_part(const FwdParams &p, const ChunkLayout &L, int part, int bh_lo, int bh_n,
                                    cudaStream_t stream);
// Chunk Grams with TMA tensor loads (vla_gram_tc.cu), same shapes.
bool gram_tma_supported(const FwdParams &p, const ChunkLayout &L);
cudaError_t launch_gram_tma(const ChunkArgs &a, cudaStream_t stream);

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

// Ends an mbarrier's life, so that its bytes may serve another purpose.
__device__ __forceinline__ void mbar_inval(uint64_t *bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One arrival (release semantics at CTA scope: this thread's earlier writes are
// visible to whoever observes the phase complete).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Waits for phase `parity` of `bar`, giving up after limit_ns.  Returns true
// on success; on expiry sets the device error word and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, long long limit_ns,
                                                  int *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((long long)(globaltimer_ns() - t0) > limit_ns) {
            atomicExch(err, kDevErrTimeout);
            return false;
        }
    }
}

// 1-D bulk async copy global -> shared, completion counted on `bar` in bytes.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core) helpers, cta_group::1
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor, K-major operand without swizzle: 8-row x
// 16-byte core matrices; lbo = byte distance between core matrices adjacent
// along K, sbo = between core matrices adjacent along M/N.
__device__ __forceinline__ uint64_t umma_desc_kmajor(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for the sm_100 family
    return d;                // base offset 0, no swizzle
}
// Byte offset of element (r, k) of a bf16 tile of K columns in that layout
// (core matrices adjacent along K are contiguous: lbo = 128, sbo = K * 16).
__host__ __device__ __forceinline__ uint32_t kmajor_off_bf16(int r, int k, int K) {
    return (uint32_t)((r >> 3) * K * 16 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}
// Instruction descriptor of kind::f16 with bf16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// (relinquish: the CTA gives up its permit to allocate again, which lets other
// CTAs on the SM allocate sooner; a CTA that allocates once per job of a
// persistent loop keeps it)
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols, bool relinquish = true) {  // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    if (relinquish) asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// Arrive on `bar` once every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
// 16 consecutive 32-bit TMEM columns of this thread's lane (shape 32x32b).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// Packed fp32 pairs (sm_100 family FFMA2/FMUL2: one instruction, two IEEE
// single-precision results).
__device__ __forceinline__ float2 f2(float x) { return make_float2(x, x); }
__device__ __forceinline__ float2 lo2(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(float4 v) { return make_float2(v.z, v.w); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float hsum2(float2 a) { return a.x + a.y; }

// Warp reduction of four values at once with six shuffles (transpose
// reduction): afterwards lane L holds the warp-wide sum of value number
// 2 * bit4(L) + bit3(L); lanes 0, 8, 16 and 24 hold the sums of v0..v3.
__device__ __forceinline__ float warp_reduce4(float v0, float v1, float v2, float v3) {
    const int lane = threadIdx.x & 31;
    const bool hi16 = lane & 16;
    float a0 = hi16 ? v2 : v0, a1 = hi16 ? v3 : v1;
    const float s0 = hi16 ? v0 : v2, s1 = hi16 ? v1 : v3;
    a0 += __shfl_xor_sync(0xffffffffu, s0, 16);
    a1 += __shfl_xor_sync(0xffffffffu, s1, 16);
    const bool hi8 = lane & 8;
    float b = hi8 ? a1 : a0;
    const float sb = hi8 ? a0 : a1;
    b += __shfl_xor_sync(0xffffffffu, sb, 8);
    b += __shfl_xor_sync(0xffffffffu, b, 4);
    b += __shfl_xor_sync(0xffffffffu, b, 2);
    b += __shfl_xor_sync(0xffffffffu, b, 1);
    return b;
}

// Block-wide sum of four values over NW warps; every thread gets the four
// totals.  red: NW float4 of shared memory, not reused before the next
// block barrier.
template <int NW>
__device__ __forceinline__ float4 block_sum4(float v0, float v1, float v2, float v3, float4 *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float r = warp_reduce4(v0, v1, v2, v3);
    if ((lane & 7) == 0) reinterpret_cast<float *>(red)[warp * 4 + (lane >> 3)] = r;
    __syncthreads();
    float4 acc = red[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) {
        const float4 x = red[w];
        acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
    }
    return acc;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// phi(x) = ELU(x) + 1: x + 1 for x > 0, exp(x) otherwise.
__device__ __forceinline__ float phi_elu1(float x) { return x > 0.f ? x + 1.f : expf(x); }

template <typename IO>
__device__ __forceinline__ float io_to_f32(IO x);
template <>
__device__ __forceinline__ float io_to_f32<float>(float x) {
    return x;
}
template <>
__device__ __forceinline__ float io_to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}

template <typename IO>
__device__ __forceinline__ IO f32_to_io(float x);
template <>
__device__ __forceinline__ float f32_to_io<float>(float x) {
    return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 f32_to_io<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// ---------------------------------------------------------------------------
// Register-resident inverse of an SPD matrix by Gauss-Jordan elimination
// (no pivoting: the pivots of an SPD matrix are positive).  Thread (row i,
// part) holds x[CPT] = row i, columns [CPT part, CPT part + CPT).  piv: two
// skewed shared vectors for the pivot row (double-buffered).  All threads of
// the block must call it.
// ---------------------------------------------------------------------------
template <int D, int CPT>
__device__ __forceinline__ void gj_inverse(float (&x)[CPT], float *piv, int row, int part) {
    constexpr int TPR = D / CPT;
    constexpr int VLEN = (D / 32) * kPart;
    const int c0 = part * CPT;
    const int lane = threadIdx.x & 31;
    if (row == 0) {
#pragma unroll
        for (int j = 0; j < CPT; ++j) piv[vidx(c0 + j)] = x[j];
    }
    __syncthreads();
#pragma unroll 1
    for (int k = 0; k < D; ++k) {
        const float *pr = piv + (k & 1) * VLEN;
        const float p = pr[vidx(k)];
        const float rp = 1.f / p;
        // m = x[i][k]: held by part k / CPT of this row, register k % CPT
        float mk = 0.f;
        const int kp = k / CPT, kr = k % CPT;
#pragma unroll
        for (int j = 0; j < CPT; ++j)
            if (j == kr) mk = x[j];
        if (TPR > 1) mk = __shfl_sync(0xffffffffu, mk, (lane & ~(TPR - 1)) | kp);
        if (row == k) {
#pragma unroll
            for (int j = 0; j < CPT; ++j) x[j] = (c0 + j == k) ? rp : x[j] * rp;
        } else {
            const float f = mk * rp;
#pragma unroll
            for (int c4 = 0; c4 < CPT / 4; ++c4) {
                const float4 pv = *reinterpret_cast<const float4 *>(pr + vidx(c0 + 4 * c4));
                const float pj[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j = 4 * c4 + q;
                    x[j] = (c0 + j == k) ? -f : fmaf(-f, pj[q], x[j]);
                }
            }
        }
        if (k + 1 < D && row == k + 1) {
            float *nx = piv + ((k + 1) & 1) * VLEN;
#pragma unroll
            for (int j = 0; j < CPT; ++j) nx[vidx(c0 + j)] = x[j];
        }
        __syncthreads();
    }
}

}  // namespace vla
