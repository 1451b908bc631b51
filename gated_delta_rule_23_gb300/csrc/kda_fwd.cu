// KDA chunked forward pass for sm_103a (GB300).
//
// One CTA (16 warps) owns one (sequence, head) pair and walks its tokens in
// 32-token chunks.  Per chunk it runs the token-parallel intra-chunk stage (gate,
// L2 norm, decay factors, the strictly-lower beta*K*K^T and causal Q*K^T matrices,
// the (I + A)^-1 inverse and the WY transform) on CUDA cores and mma.sync, and the
// chunk recurrence on the 5th-generation tensor cores with the state resident in
// tensor memory.  This follows the split into an intra-chunk stage (gate
// activation -> L2 norm -> decay -> L / Mqk construction -> inversion) and a
// chunk-wise delta-rule recurrence described in the guancyxx.cn FlashKDA article,
// section 2.2, fused into one launch so the intermediates never leave the SM.
//
// Notation (per chunk, rows i = 0..31, channel c, state S in R^{K x V}):
//   a_i    = lower_bound * sigmoid(exp(A_log) * (g_i + dt_bias))   (natural-log decay)
//   alpha  = exp(a); G_i = sum_{s <= i} a_s; Gamma_i = exp(G_i)
//   Akk[i][j] = b_i sum_c k^_ic k^_jc exp(G_ic - G_jc)  (j < i),  Aqk likewise with q^ (j <= i)
//   Tm = (I + Akk)^-1, T' = Tm diag(b), W = T' (K^ . Gamma), U = T' V - W S
//   O = scale (Q~ S + Aqk U), Q~ = Q^ . Gamma;  S <- Diag(Gamma_31) S + K~^T U,
//   K~_j = k^_j . Gamma_31 / Gamma_j.
// The decay factors are formed per 16-row sub-block so that no factor leaves
// [2^-115.5, 2^115.5] when lower_bound >= -5 (at most 7.22 binary orders of
// magnitude per token, 16 tokens per sub-block): the numerical-range argument for
// CHUNK = 16 in the FlashKDA article, section 2.1, applied per sub-block.  With
// P_i / E_i the within-sub-block prefix (inclusive) / suffix (exclusive) products
// of alpha and D_b the product over sub-block b:
//   exp(G_i - G_j) = P_i E_j / D_b          (i, j in sub-block b, j <= i)
//   exp(G_i - G_j) = P_i E_j                (i in sub-block 1, j in sub-block 0)
//   Gamma_i = P_i (b(i) = 0) or D_0 P_i;    Gamma_31 / Gamma_j = E_j D_1 (b(j) = 0) or E_j.
//
// The recurrence is computed transposed, M = 128 value rows on the tensor-memory
// lanes: S^T (fp32, 128 columns) is the A operand of kind::tf32 MMAs straight from
// tensor memory, as are Y^T and U^T; B operands are tf32-rounded fp32 tiles in
// shared memory (no-swizzle K-major core-matrix layout).  Per chunk, using
// U = T' (V - (K^ . Gamma) S):
//   [O^T | X^T] = S^T [Q~ ; K^.Gamma]^T        (issued right after the gate pass;
//                                               overlaps the Akk/Aqk products and the inverse)
//   Y^T = V^T - X^T (threads);  U^T = Y^T T'^T;  S^T *= Gamma_31 (threads);
//   [S^T | O^T] += U^T [K~^T ; Aqk]^T.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "kda.h"

// Set when a bounded wait on the tensor cores expires (read by kda_device_status).
__device__ unsigned int g_kda_device_error;

namespace {

constexpr int D = 128;        // K = V = 128
constexpr int CH = 32;        // tokens per chunk
constexpr int SB = 16;        // tokens per decay sub-block
constexpr int NTHREADS = 512;
constexpr int TMEM_COLS = 256;
// tensor-memory columns: S^T | O^T | X^T | Y^T | U^T (O^T follows S^T and X^T follows O^T so
// that the merged MMAs write one contiguous accumulator)
constexpr int TM_S = 0, TM_O = 128, TM_X = 160, TM_Y = 192, TM_U = 224;
constexpr int MMA_TID = 384;                     // issuing thread: warp 12 has no Akk/Aqk item
// An issuing thread blocks while the tensor-core queue drains, so between the early MMA group and
// the end of the inverse the other warps synchronise on a named barrier without warp 12.
constexpr int BAR_NO_MMA = 1, NO_MMA_THREADS = NTHREADS - 32;
constexpr float LOG2E = 1.4426950408889634f;
constexpr uint32_t WAIT_LIMIT = 1u << 24;        // try_wait polls before a wait is declared hung
constexpr int LPT_MAX_SEQS = 256;                // longest-first ordering of varlen sequences up to this count

// ---------------------------------------------------------------- shared memory map
// Half-precision [32][136] tiles (272-byte rows).  The q, k, g tiles and K^.Gamma swizzle
// their 16-byte chunks by (row >> 3) & 3, which makes the gate pass (lanes spread over
// eight 4-row segments) and ldmatrix free of bank conflicts.
constexpr int PH = 136;
constexpr int PF = 132;                          // fp32 pitch of 128-wide tf32 mma.sync operands (conflict-free fragment loads)
constexpr int PA = 36;                           // fp32 pitch of 32-wide matrices
constexpr int HT = CH * PH * 2;                  // 8704 B
// tcgen05 operand tiles: element (row r, k) of a K-major tile sits at
// (r / 8) * SBO + (k / 4) * LBO + (r % 8) * 16 + (k % 4) * 4 (fp32, 8x16-byte core matrices).
constexpr int QX_LBO = 144, QX_SBO = 4640;       // [Q~ ; K^.Gamma] [64 t][128 k]  (padded: conflict-free stores)
constexpr int SO_LBO = 144, SO_SBO = 1152;       // [K~^T ; Aqk]    [160][32 t]
constexpr int TP_LBO = 128, TP_SBO = 1024;       // T'              [32 t][32 t']

constexpr int OFF_RAW_Q = 0;
constexpr int OFF_RAW_K = OFF_RAW_Q + HT;
constexpr int OFF_RAW_G = OFF_RAW_K + HT;
constexpr int OFF_RAW_V = OFF_RAW_G + HT;
constexpr int OFF_RAW_B = OFF_RAW_V + HT;        // beta logits, 32 bf16 (128 B reserved)
constexpr int OFF_INTRA = OFF_RAW_B + 128;
constexpr int F32H = SB * PF * 4;                // 8448 B: 16 rows of 128 fp32
constexpr int OFF_LQ = OFF_INTRA;                // fp32 [16][132]  q^ P, rows 16..31 (sub-block 1)
constexpr int OFF_LK = OFF_LQ + F32H;            // fp32 [16][132]  k^ P, rows 16..31
constexpr int OFF_ED = OFF_LK + F32H;            // fp32 [32][132]  k^ E / D_b
constexpr int INTRA_BYTES = 4 * F32H;
// after the Akk / Aqk products the same region holds:
constexpr int OFF_AKK = OFF_INTRA;               // fp32 [32][36]
constexpr int OFF_TMD = OFF_AKK + CH * PA * 4;   // fp32 [32][36]  diagonal blocks of Tm
constexpr int OFF_MT = OFF_TMD + CH * PA * 4;    // fp32 [16][16]  inverse scratch
constexpr int INTRA_END = OFF_MT + 16 * 16 * 4;
constexpr int OFF_QX = OFF_INTRA + INTRA_BYTES;  // tcgen05 B tiles from here on
constexpr int SO_BYTES = 20 * SO_SBO;
constexpr int OFF_SO = OFF_QX + 8 * QX_SBO;      // two buffers: the update of chunk c reads one while
constexpr int OFF_TP = OFF_SO + 2 * SO_BYTES;    // the gate pass of chunk c+1 writes the other
constexpr int OFF_RED = OFF_TP + 4 * TP_SBO;     // fp32 [3 pairs][2 kinds][32 lanes][8] K-half partials
constexpr int OFF_OST = OFF_RED + 3 * 2 * 32 * 8 * 4;   // bf16 [32][136] output staging
constexpr int OFF_MISC = OFF_OST + HT;
constexpr int OFF_RQ = OFF_MISC;                 // fp32 [32] 1/|q|
constexpr int OFF_RK = OFF_RQ + 128;             // fp32 [32] 1/|k|
constexpr int OFF_BT = OFF_RK + 128;             // fp32 [32] b = sigmoid(beta), 0 past the end
constexpr int OFF_GC = OFF_BT + 128;             // fp32 [128] chunk decay Gamma_31
constexpr int OFF_BAR = OFF_GC + D * 4;          // 3 mbarriers, tensor-memory base address, hang flag
constexpr int SMEM_BYTES = OFF_BAR + 32;
static_assert(INTRA_END <= OFF_QX, "post-product overlay exceeds the intra region");
static_assert((LPT_MAX_SEQS + 1) * 8 + LPT_MAX_SEQS * 4 <= OFF_INTRA, "varlen scheduler scratch");
static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
static_assert(OFF_INTRA % 128 == 0 && OFF_QX % 16 == 0 && OFF_SO % 16 == 0 && OFF_TP % 16 == 0 &&
              OFF_MISC % 16 == 0 && OFF_RED % 16 == 0 && OFF_OST % 16 == 0 && OFF_BAR % 8 == 0, "alignment");

// byte offset of element (row, col) in a swizzled [32][136] half tile
__host__ __device__ constexpr int swz(int row, int col)
{
    return row * PH * 2 + (((col >> 3) ^ ((row >> 3) & 3)) << 4) + ((col & 7) << 1);
}
// byte offset of fp32 element (r, k) in a K-major tcgen05 tile
__host__ __device__ constexpr int kmaj(int r, int k, int lbo, int sbo)
{
    return (r >> 3) * sbo + (k >> 2) * lbo + ((r & 7) << 4) + ((k & 3) << 2);
}

// ---------------------------------------------------------------- small device helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float sigmoidf_fast(float z)
{
    return rcp_approx(1.0f + ex2_approx(-z * LOG2E));
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t to_tf32(float x)
{
    uint32_t y;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(y) : "f"(x));
    return y;
}

// D += A * B, m16n8k8, tf32 operands, fp32 accumulators
__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- tcgen05 helpers
// Shared-memory matrix descriptor: start address, leading (K-direction) and stride
// (M/N-direction) byte offsets between 8x16-byte core matrices, no swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}
// Instruction descriptor: fp32 accumulator, tf32 A and B, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_tf32_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, int acc)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}"
                 ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void umma_commit(uint32_t mbar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar));
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&u)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
                   "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]),
                   "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]),
                   "=r"(u[22]), "=r"(u[23]), "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]),
                   "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&u)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 ::"r"(taddr), "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]),
                   "r"(u[7]), "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]), "r"(u[13]), "r"(u[14]),
                   "r"(u[15]), "r"(u[16]), "r"(u[17]), "r"(u[18]), "r"(u[19]), "r"(u[20]), "r"(u[21]), "r"(u[22]),
                   "r"(u[23]), "r"(u[24]), "r"(u[25]), "r"(u[26]), "r"(u[27]), "r"(u[28]), "r"(u[29]), "r"(u[30]),
                   "r"(u[31]));
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&u)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&u)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 ::"r"(taddr), "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7]));
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Bounded wait for an mbarrier phase; returns false if the wait gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity)
{
    uint32_t done = 0;
    for (uint32_t it = 0; it < WAIT_LIMIT; ++it) {
        asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                     : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
        if (done)
            return true;
    }
    return false;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid)
{
    const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N> __device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

// Stage rows [tok0, tok0 + len) of one [rows, H, 128] bf16 tensor (head h) into a
// [32][136] tile (swizzled or plain); rows past len are zero-filled.  len >= 1.
template <bool SWZ>
__device__ __forceinline__ void load_tile_async(unsigned char *smem, int off, const __nv_bfloat16 *base,
                                                int64_t tok0, int len, int H, int h)
{
    static_assert((CH * 16) % NTHREADS == 0, "tile load split");
    const int tid = threadIdx.x;
#pragma unroll
    for (int m = 0; m < CH * 16 / NTHREADS; ++m) {
        const int idx = tid + m * NTHREADS;   // 32 rows x 16 chunks of 16 bytes
        const int r = idx >> 4, c16 = idx & 15;
        const bool valid = r < len;
        const int64_t row = tok0 + (valid ? r : 0);
        const __nv_bfloat16 *src = base + (row * H + h) * D + c16 * 8;
        const int dst = SWZ ? swz(r, c16 * 8) : r * PH * 2 + c16 * 16;
        cp_async16(smem_u32(smem + off + dst), src, valid);
    }
}

__device__ __forceinline__ void named_bar(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

struct Params {
    const __nv_bfloat16 *q, *k, *v, *g, *beta;
    __nv_bfloat16 *out;
    const float *A_log, *dt_bias;
    const void *init;
    void *fin;
    const int64_t *cu;
    float scale, lb_log2e;
    int N, H;
    int64_t T;
};

__device__ __forceinline__ float tf32r(float x) { return __uint_as_float(to_tf32(x)); }

// ---------------------------------------------------------------- the kernel
template <int STATE, bool VARLEN>  // STATE: 0 none, 1 bf16, 2 fp32
__global__ void __launch_bounds__(NTHREADS, 1) kda_fwd_kernel(const Params p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;             // mma.sync fragment coordinates
    const int H = p.H;
    const int h = blockIdx.x % H;
    int n = blockIdx.x / H;
    if (VARLEN && p.N > 1 && p.N <= LPT_MAX_SEQS) {
        // Varlen scheduler: blocks are dispatched in index order, so block b takes the (b / H)-th
        // longest sequence (ties by index) and the longest sequences start first.
        int64_t *cu_s = reinterpret_cast<int64_t *>(smem + OFF_RAW_Q);   // scratch before the first tile load
        int *order = reinterpret_cast<int *>(smem + OFF_RAW_Q + (LPT_MAX_SEQS + 1) * 8);
        for (int s = tid; s <= p.N; s += NTHREADS)
            cu_s[s] = p.cu[s];
        __syncthreads();
        for (int s = tid; s < p.N; s += NTHREADS) {
            const int64_t ls = cu_s[s + 1] - cu_s[s];
            int rank = 0;
            for (int m = 0; m < p.N; ++m) {
                const int64_t lm = cu_s[m + 1] - cu_s[m];
                rank += (lm > ls) || (lm == ls && m < s);
            }
            order[rank] = s;
        }
        __syncthreads();
        n = order[blockIdx.x / H];
        __syncthreads();   // the scratch is overwritten by the first tile loads
    }

    int64_t bos, len;
    if (VARLEN) {
        bos = p.cu[n];
        len = p.cu[n + 1] - bos;
    } else {
        bos = (int64_t)n * p.T;
        len = p.T;
    }

    float *rq = reinterpret_cast<float *>(smem + OFF_RQ);
    float *rk = reinterpret_cast<float *>(smem + OFF_RK);
    float *bt = reinterpret_cast<float *>(smem + OFF_BT);
    float *Gc = reinterpret_cast<float *>(smem + OFF_GC);
    __nv_bfloat16 *rawb = reinterpret_cast<__nv_bfloat16 *>(smem + OFF_RAW_B);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + OFF_BAR + 24);
    volatile uint32_t *hang_flag = reinterpret_cast<volatile uint32_t *>(smem + OFF_BAR + 28);
    const uint32_t mbarX = smem_u32(smem + OFF_BAR), mbarU = smem_u32(smem + OFF_BAR + 8);
    const uint32_t mbarB = smem_u32(smem + OFF_BAR + 16);
    const uint32_t s_qx = smem_u32(smem + OFF_QX), s_so = smem_u32(smem + OFF_SO), s_tp = smem_u32(smem + OFF_TP);

    // -------- tensor memory, barriers, constant-zero tile parts
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        tc_fence_before();
    }
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbarX));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbarU));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbarB));
        *hang_flag = 0u;
    }
    // Aqk (rows 128..159 of both [K~^T ; Aqk] tiles) and T' are written block-lower-triangular
    // only; their upper blocks stay zero.
    for (int e = tid; e < 2 * 4 * SO_SBO / 16; e += NTHREADS) {
        const int b = e / (4 * SO_SBO / 16), o = e % (4 * SO_SBO / 16);
        reinterpret_cast<uint4 *>(smem + OFF_SO + b * SO_BYTES + 16 * SO_SBO)[o] = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int e = tid; e < 4 * TP_SBO / 16; e += NTHREADS)
        reinterpret_cast<uint4 *>(smem + OFF_TP)[e] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    // tensor-memory lanes a warp may touch: quarter q4; this thread's value row and column group
    const int q4 = warp & 3, cg = warp >> 2;
    const int vrow = q4 * 32 + lane;
    const uint32_t trow = tbase + ((uint32_t)(q4 * 32) << 16);
    const size_t srow = ((size_t)n * H + h) * D * D + (size_t)vrow * D + cg * 32;

    // -------- initial state -> S^T in tensor memory (row v, columns k)
    {
        uint32_t u[32];
        if (STATE == 2 && p.init) {
            const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(p.init) + srow);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float4 x = src[e];
                u[4 * e] = __float_as_uint(x.x);
                u[4 * e + 1] = __float_as_uint(x.y);
                u[4 * e + 2] = __float_as_uint(x.z);
                u[4 * e + 3] = __float_as_uint(x.w);
            }
        } else if (STATE == 1 && p.init) {
            const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.init) + srow);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint4 x = src[e];
                const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int f = 0; f < 4; ++f) {
                    u[8 * e + 2 * f] = w4[f] << 16;
                    u[8 * e + 2 * f + 1] = w4[f] & 0xffff0000u;
                }
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
                u[e] = 0u;
        }
        tmem_st32(trow + TM_S + cg * 32, u);
    }
    tc_fence_before();

    // gate-pass lane roles: channel pair cp of this warp's 8 channels, 4-row segment sg
    const int cp = lane & 3, sg = lane >> 2, blk = sg >> 2, si = sg & 3;
    const int c0 = warp * 8 + 2 * cp;
    const float eA = expf(p.A_log[h]);
    const float2 dtb = *reinterpret_cast<const float2 *>(p.dt_bias + h * D + c0);
    const int nchunks = (int)((len + CH - 1) / CH);
    bool hung = false;

    // prologue: stage chunk 0 (q, k, g as one group, v as a second group)
    if (nchunks > 0) {
        const int L0 = (int)(len < CH ? len : CH);
        load_tile_async<true>(smem, OFF_RAW_Q, p.q, bos, L0, H, h);
        load_tile_async<true>(smem, OFF_RAW_K, p.k, bos, L0, H, h);
        load_tile_async<true>(smem, OFF_RAW_G, p.g, bos, L0, H, h);
        cp_async_commit();
        load_tile_async<false>(smem, OFF_RAW_V, p.v, bos, L0, H, h);
        cp_async_commit();
        if (tid < CH)
            rawb[tid] = tid < L0 ? p.beta[(bos + tid) * H + h] : __float2bfloat16(0.f);
    }

    // Output of the previous chunk: wait for its last update and move O^T from tensor memory to the
    // bf16 staging tile [t][v] (this thread: its value row, tokens 8cg..8cg+7); after the next
    // barrier store_previous writes it to HBM with 16-byte coalesced stores.
    auto read_out_previous = [&](uint32_t prev_parity) -> bool {
        const bool ok = mbar_wait(mbarB, prev_parity) && *hang_flag == 0u;
        if (__syncthreads_or(!ok))
            return false;
        tc_fence_after();
        uint32_t o[8];
        tmem_ld8(trow + TM_O + cg * 8, o);
        __nv_bfloat16 *Ost = reinterpret_cast<__nv_bfloat16 *>(smem + OFF_OST);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
            Ost[(cg * 8 + jj) * PH + vrow] = __float2bfloat16_rn(__uint_as_float(o[jj]) * p.scale);
        tc_fence_before();
        return true;
    };
    auto store_previous = [&](int64_t ptok0, int pL) {
        const int r = tid >> 4, c16 = tid & 15;
        if (r < pL)
            *reinterpret_cast<uint4 *>(p.out + ((ptok0 + r) * H + h) * D + c16 * 8) =
                *reinterpret_cast<const uint4 *>(smem + OFF_OST + r * PH * 2 + c16 * 16);
    };

    // [S^T | O^T] += U^T [K~^T ; Aqk]^T for chunk c, issued once U^T of that chunk is done; the issuing
    // thread calls this one stage later (after the next chunk's norms) so that it never blocks a barrier.
    auto issue_update = [&](int c) {
        if (mbar_wait(mbarU, c & 1) && *hang_flag == 0u) {
            tc_fence_after();
            const uint32_t s_sob = s_so + (c & 1) * SO_BYTES;
#pragma unroll
            for (int s = 0; s < CH / 8; ++s)
                mma_tf32_ts(tbase + TM_S, tbase + TM_U + 8 * s, umma_desc(s_sob + s * 2 * SO_LBO, SO_LBO, SO_SBO),
                            idesc_tf32(128, D + CH), 1);
            umma_commit(mbarB);
        } else {
            *hang_flag = 1u;
        }
    };

    int64_t prev_tok0 = 0;
    int prev_L = 0;
    for (int ci = 0; ci < nchunks; ++ci) {
        const int64_t tok0 = bos + (int64_t)ci * CH;
        const int64_t rem = len - (int64_t)ci * CH;
        const int L = (int)(rem < CH ? rem : CH);
        const bool has_next = ci + 1 < nchunks;
        const int64_t ntok0 = tok0 + CH;
        const int Ln = has_next ? (int)((rem - CH) < CH ? (rem - CH) : CH) : 0;
        const uint32_t parity = ci & 1;
        const int sob = ci & 1;                                 // [K~^T ; Aqk] buffer of this chunk
        unsigned char *so = smem + OFF_SO + sob * SO_BYTES;

        cp_async_wait<1>();   // q, k, g of this chunk have landed (v may still be in flight)
        __syncthreads();

        // ---- S1a: row norms (16 lanes per row, 8 channels per lane) and beta
        {
            const int half = lane >> 4, l16 = lane & 15;
            const int r = warp * 2 + half;
            const uint4 qa = *reinterpret_cast<const uint4 *>(smem + OFF_RAW_Q + swz(r, l16 * 8));
            const uint4 ka = *reinterpret_cast<const uint4 *>(smem + OFF_RAW_K + swz(r, l16 * 8));
            const uint32_t qw[4] = {qa.x, qa.y, qa.z, qa.w}, kw[4] = {ka.x, ka.y, ka.z, ka.w};
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float q0 = bf16_lo(qw[e]), q1 = bf16_hi(qw[e]), k0 = bf16_lo(kw[e]), k1 = bf16_hi(kw[e]);
                sq = fmaf(q0, q0, fmaf(q1, q1, sq));
                sk = fmaf(k0, k0, fmaf(k1, k1, sk));
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            if (l16 == 0) {
                rq[r] = rsqrtf(sq + 1e-6f);
                rk[r] = rsqrtf(sk + 1e-6f);
            }
            if (tid < CH)
                bt[tid] = tid < L ? sigmoidf_fast(__bfloat162float(rawb[tid])) : 0.f;
        }
        if (ci > 0 && tid == MMA_TID)
            issue_update(ci - 1);
        __syncthreads();

        // ---- S1b: gate, sub-block decay products and every operand of this chunk (one pass)
        {
            uint32_t gqv[4], gkv[4];
            float al0[4], al1[4], qn[4], kn[4];
            float tot0 = 1.f, tot1 = 1.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = sg * 4 + i;
                const uint32_t gg = *reinterpret_cast<const uint32_t *>(smem + OFF_RAW_G + swz(r, c0));
                gqv[i] = *reinterpret_cast<const uint32_t *>(smem + OFF_RAW_Q + swz(r, c0));
                gkv[i] = *reinterpret_cast<const uint32_t *>(smem + OFF_RAW_K + swz(r, c0));
                qn[i] = rq[r];
                kn[i] = rk[r];
                const float z0 = eA * (bf16_lo(gg) + dtb.x), z1 = eA * (bf16_hi(gg) + dtb.y);
                const bool live = r < L;
                al0[i] = live ? ex2_approx(p.lb_log2e * sigmoidf_fast(z0)) : 1.f;
                al1[i] = live ? ex2_approx(p.lb_log2e * sigmoidf_fast(z1)) : 1.f;
                tot0 *= al0[i];
                tot1 *= al1[i];
            }
            // scans over the four 4-row segments of this sub-block (lane bits 2-3), per channel
            const unsigned FULL = 0xffffffffu;
            float x0 = tot0, x1 = tot1, y0, y1;
            y0 = __shfl_up_sync(FULL, x0, 4);
            y1 = __shfl_up_sync(FULL, x1, 4);
            if (si >= 1) { x0 *= y0; x1 *= y1; }
            y0 = __shfl_up_sync(FULL, x0, 8);
            y1 = __shfl_up_sync(FULL, x1, 8);
            if (si >= 2) { x0 *= y0; x1 *= y1; }                         // inclusive prefix
            float ex0 = __shfl_up_sync(FULL, x0, 4), ex1 = __shfl_up_sync(FULL, x1, 4);
            if (si == 0) { ex0 = 1.f; ex1 = 1.f; }                       // exclusive prefix
            const float D0 = __shfl_sync(FULL, x0, lane | 12), D1 = __shfl_sync(FULL, x1, lane | 12);
            float z0 = tot0, z1 = tot1, w0, w1;
            w0 = __shfl_down_sync(FULL, z0, 4);
            w1 = __shfl_down_sync(FULL, z1, 4);
            if (si <= 2) { z0 *= w0; z1 *= w1; }
            w0 = __shfl_down_sync(FULL, z0, 8);
            w1 = __shfl_down_sync(FULL, z1, 8);
            if (si <= 1) { z0 *= w0; z1 *= w1; }                         // inclusive suffix
            float es0 = __shfl_down_sync(FULL, z0, 4), es1 = __shfl_down_sync(FULL, z1, 4);
            if (si == 3) { es0 = 1.f; es1 = 1.f; }                       // exclusive suffix
            const float Do0 = __shfl_xor_sync(FULL, D0, 16), Do1 = __shfl_xor_sync(FULL, D1, 16);
            const float pre0 = blk ? Do0 : 1.f, pre1 = blk ? Do1 : 1.f;       // Gamma at sub-block start
            const float post0 = blk ? 1.f : Do0, post1 = blk ? 1.f : Do1;     // decay after sub-block end
            const float iD0 = rcp_approx(D0), iD1 = rcp_approx(D1);
            float *Lq = reinterpret_cast<float *>(smem + OFF_LQ);
            float *Lk = reinterpret_cast<float *>(smem + OFF_LK);
            float *Ed = reinterpret_cast<float *>(smem + OFF_ED);
            float P0 = ex0, P1 = ex1;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = sg * 4 + i;
                const float q0 = bf16_lo(gqv[i]) * qn[i], q1 = bf16_hi(gqv[i]) * qn[i];
                const float k0 = bf16_lo(gkv[i]) * kn[i], k1 = bf16_hi(gkv[i]) * kn[i];
                P0 *= al0[i];
                P1 *= al1[i];
                const float qp0 = q0 * P0, qp1 = q1 * P1, kp0 = k0 * P0, kp1 = k1 * P1;
                // chunk-start reference: Q~ = q^ Gamma and K^.Gamma (also the sub-block-0 product operands)
                *reinterpret_cast<float2 *>(smem + OFF_QX + kmaj(r, c0, QX_LBO, QX_SBO)) =
                    make_float2(tf32r(qp0 * pre0), tf32r(qp1 * pre1));
                *reinterpret_cast<float2 *>(smem + OFF_QX + kmaj(CH + r, c0, QX_LBO, QX_SBO)) =
                    make_float2(tf32r(kp0 * pre0), tf32r(kp1 * pre1));
                if (blk) {   // sub-block-1 reference for the (1,1) products
                    *reinterpret_cast<float2 *>(Lq + (r - SB) * PF + c0) = make_float2(tf32r(qp0), tf32r(qp1));
                    *reinterpret_cast<float2 *>(Lk + (r - SB) * PF + c0) = make_float2(tf32r(kp0), tf32r(kp1));
                }
            }
            float E0 = es0, E1 = es1;
            float kt0[4], kt1[4];
#pragma unroll
            for (int i = 3; i >= 0; --i) {
                const int r = sg * 4 + i;
                const float ke0 = bf16_lo(gkv[i]) * kn[i] * E0, ke1 = bf16_hi(gkv[i]) * kn[i] * E1;
                *reinterpret_cast<float2 *>(Ed + r * PF + c0) = make_float2(tf32r(ke0 * iD0), tf32r(ke1 * iD1));
                kt0[i] = tf32r(ke0 * post0);
                kt1[i] = tf32r(ke1 * post1);
                E0 *= al0[i];
                E1 *= al1[i];
            }
            *reinterpret_cast<float4 *>(so + kmaj(c0, sg * 4, SO_LBO, SO_SBO)) = make_float4(kt0[0], kt0[1], kt0[2], kt0[3]);
            *reinterpret_cast<float4 *>(so + kmaj(c0 + 1, sg * 4, SO_LBO, SO_SBO)) = make_float4(kt1[0], kt1[1], kt1[2], kt1[3]);
            if (sg == 0)
                *reinterpret_cast<float2 *>(Gc + c0) = make_float2(D0 * Do0, D1 * Do1);
        }
        fence_async_smem();
        // ---- the previous chunk's output (its final update ran during this gate pass)
        if (ci > 0 && !read_out_previous((ci - 1) & 1)) {
            hung = true;
            break;
        }
        __syncthreads();

        // ---- the previous chunk's output to HBM; raw q, k, g, beta are consumed: stage the next chunk's
        if (ci > 0)
            store_previous(prev_tok0, prev_L);
        if (has_next) {
            load_tile_async<true>(smem, OFF_RAW_Q, p.q, ntok0, Ln, H, h);
            load_tile_async<true>(smem, OFF_RAW_K, p.k, ntok0, Ln, H, h);
            load_tile_async<true>(smem, OFF_RAW_G, p.g, ntok0, Ln, H, h);
        }
        cp_async_commit();
        __nv_bfloat16 next_beta = __float2bfloat16(0.f);
        if (has_next && tid < Ln)
            next_beta = p.beta[(ntok0 + tid) * H + h];

        // ---- tensor cores: [O^T | X^T] = S^T [Q~ ; K^.Gamma]^T (overlaps the products and the inverse)
        if (tid == MMA_TID) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < D / 8; ++s)
                mma_tf32_ts(tbase + TM_O, tbase + TM_S + 8 * s, umma_desc(s_qx + s * 2 * QX_LBO, QX_LBO, QX_SBO),
                            idesc_tf32(128, 2 * CH), s > 0);
            umma_commit(mbarX);
        }

        // ---- S2: Akk and Aqk on tf32 mma.sync; warp = (pair, K half, kind), both n-tiles of the pair.
        // pair 0 = (0,0), 1 = (1,0): left factor from the chunk-start tile, right factor k^ E / D_0;
        // pair 2 = (1,1): left factor q^ P / k^ P of sub-block 1, right factor k^ E / D_1.
        const int pair = warp >> 2, khalf = (warp >> 1) & 1, qk = warp & 1;
        const int rb1 = pair == 0 ? 0 : 16, cb0 = pair == 2 ? 16 : 0;
        float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if (warp < 12) {
            const float *Y = reinterpret_cast<const float *>(smem + OFF_ED) + (cb0 + gq) * PF + tq;
            const int ks0 = khalf * 8;
            if (pair < 2) {
                const unsigned char *X = smem + OFF_QX + kmaj((qk ? 0 : CH) + rb1 + gq, tq, QX_LBO, QX_SBO);
#pragma unroll
                for (int ks = ks0; ks < ks0 + 8; ++ks) {
                    const unsigned char *x0 = X + ks * 2 * QX_LBO;
                    const uint32_t a0 = *reinterpret_cast<const uint32_t *>(x0);
                    const uint32_t a1 = *reinterpret_cast<const uint32_t *>(x0 + QX_SBO);
                    const uint32_t a2 = *reinterpret_cast<const uint32_t *>(x0 + QX_LBO);
                    const uint32_t a3 = *reinterpret_cast<const uint32_t *>(x0 + QX_SBO + QX_LBO);
                    const int k0 = ks * 8;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
                        mma_tf32(acc2[nt], a0, a1, a2, a3, __float_as_uint(Y[nt * 8 * PF + k0]),
                                 __float_as_uint(Y[nt * 8 * PF + k0 + 4]));
                }
            } else {
                const float *X = reinterpret_cast<const float *>(smem + (qk ? OFF_LQ : OFF_LK)) + gq * PF + tq;
#pragma unroll
                for (int ks = ks0; ks < ks0 + 8; ++ks) {
                    const int k0 = ks * 8;
                    const uint32_t a0 = __float_as_uint(X[k0]), a1 = __float_as_uint(X[8 * PF + k0]);
                    const uint32_t a2 = __float_as_uint(X[k0 + 4]), a3 = __float_as_uint(X[8 * PF + k0 + 4]);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
                        mma_tf32(acc2[nt], a0, a1, a2, a3, __float_as_uint(Y[nt * 8 * PF + k0]),
                                 __float_as_uint(Y[nt * 8 * PF + k0 + 4]));
                }
            }
            if (khalf) {
                float4 *red = reinterpret_cast<float4 *>(smem + OFF_RED) + ((pair * 2 + qk) * 32 + lane) * 2;
                red[0] = make_float4(acc2[0][0], acc2[0][1], acc2[0][2], acc2[0][3]);
                red[1] = make_float4(acc2[1][0], acc2[1][1], acc2[1][2], acc2[1][3]);
            }
        }
        if (warp != MMA_TID / 32)
            named_bar(BAR_NO_MMA, NO_MMA_THREADS);   // the intra operands are dead; the region is reused below
        if (warp < 12 && !khalf) {
            const float4 *red = reinterpret_cast<const float4 *>(smem + OFF_RED) + ((pair * 2 + qk) * 32 + lane) * 2;
            const float4 r0 = red[0], r1 = red[1];
            acc2[0][0] += r0.x; acc2[0][1] += r0.y; acc2[0][2] += r0.z; acc2[0][3] += r0.w;
            acc2[1][0] += r1.x; acc2[1][1] += r1.y; acc2[1][2] += r1.z; acc2[1][3] += r1.w;
            float *Akk = reinterpret_cast<float *>(smem + OFF_AKK);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int i = rb1 + gq + 8 * hh, j = cb0 + nt * 8 + 2 * tq;
                    const float x0 = acc2[nt][2 * hh], x1 = acc2[nt][2 * hh + 1];
                    if (qk) {
                        *reinterpret_cast<float2 *>(so + kmaj(D + i, j, SO_LBO, SO_SBO)) =
                            make_float2(tf32r(j <= i ? x0 : 0.f), tf32r(j + 1 <= i ? x1 : 0.f));
                    } else {
                        const float bi = bt[i];
                        *reinterpret_cast<float2 *>(Akk + i * PA + j) =
                            make_float2(j < i ? bi * x0 : 0.f, j + 1 < i ? bi * x1 : 0.f);
                    }
                }
        }
        if (warp != MMA_TID / 32)
            named_bar(BAR_NO_MMA, NO_MMA_THREADS);

        // ---- S3: Tm = (I + Akk)^-1 (fp32) and the tf32 tile of T' = Tm diag(b)
        float *Akk = reinterpret_cast<float *>(smem + OFF_AKK);
        float *Tmd = reinterpret_cast<float *>(smem + OFF_TMD);
        if (warp < 2 && lane < 16) {
            // diagonal 16x16 blocks, column j per lane, right-looking forward substitution
            const int b = warp, j = lane;
            float x[SB], acc[SB];
#pragma unroll
            for (int i = 0; i < SB; ++i)
                acc[i] = 0.f;
#pragma unroll
            for (int l = 0; l < SB; ++l) {
                x[l] = l == j ? 1.f : (l < j ? 0.f : -acc[l]);
#pragma unroll
                for (int i = l + 1; i < SB; ++i)
                    acc[i] = fmaf(Akk[(b * SB + i) * PA + b * SB + l], x[l], acc[i]);
            }
            const float bj = bt[b * SB + j];
#pragma unroll
            for (int i = 0; i < SB; ++i) {
                const int r = b * SB + i, c = b * SB + j;
                Tmd[r * PA + c] = x[i];
                *reinterpret_cast<float *>(smem + OFF_TP + kmaj(r, c, TP_LBO, TP_SBO)) = tf32r(x[i] * bj);
            }
        }
        if (warp != MMA_TID / 32)
            named_bar(BAR_NO_MMA, NO_MMA_THREADS);
        {
            // off-diagonal block: Tm_10 = -Tm_11 (A_10 Tm_00);  threads 0..255 = (i, j)
            const int i = (tid >> 4) & 15, j = tid & 15;
            float *Mt = reinterpret_cast<float *>(smem + OFF_MT);
            if (tid < 256) {
                float s = 0.f, s2 = 0.f;
#pragma unroll
                for (int l = 0; l < SB; l += 2) {
                    s = fmaf(Akk[(SB + i) * PA + l], Tmd[l * PA + j], s);
                    s2 = fmaf(Akk[(SB + i) * PA + l + 1], Tmd[(l + 1) * PA + j], s2);
                }
                Mt[i * 16 + j] = s + s2;
            }
            if (warp != MMA_TID / 32)
                named_bar(BAR_NO_MMA, NO_MMA_THREADS);
            if (tid < 256) {
                float s = 0.f, s2 = 0.f;
#pragma unroll
                for (int l = 0; l < SB; l += 2) {
                    s = fmaf(Tmd[(SB + i) * PA + SB + l], Mt[l * 16 + j], s);
                    s2 = fmaf(Tmd[(SB + i) * PA + SB + l + 1], Mt[(l + 1) * 16 + j], s2);
                }
                *reinterpret_cast<float *>(smem + OFF_TP + kmaj(SB + i, j, TP_LBO, TP_SBO)) = tf32r(-(s + s2) * bt[j]);
            }
        }
        fence_async_smem();
        cp_async_wait<1>();   // v of this chunk (the next chunk's q, k, g may stay in flight)
        __syncthreads();

        // ---- Y^T = V^T - X^T into tensor memory, and S^T <- S^T Diag(Gamma_31)
        hung = !mbar_wait(mbarX, parity);
        if (__syncthreads_or(hung)) {
            hung = true;
            break;
        }
        tc_fence_after();
        {
            uint32_t xv[8];
            tmem_ld8(trow + TM_X + cg * 8, xv);
            const __nv_bfloat16 *rv = reinterpret_cast<const __nv_bfloat16 *>(smem + OFF_RAW_V);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                xv[jj] = __float_as_uint(__bfloat162float(rv[(cg * 8 + jj) * PH + vrow]) - __uint_as_float(xv[jj]));
            tmem_st8(trow + TM_Y + cg * 8, xv);
            uint32_t u[32];
            tmem_ld32(trow + TM_S + cg * 32, u);
            const float4 *g4 = reinterpret_cast<const float4 *>(Gc + cg * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float4 gm = g4[e];
                u[4 * e] = __float_as_uint(__uint_as_float(u[4 * e]) * gm.x);
                u[4 * e + 1] = __float_as_uint(__uint_as_float(u[4 * e + 1]) * gm.y);
                u[4 * e + 2] = __float_as_uint(__uint_as_float(u[4 * e + 2]) * gm.z);
                u[4 * e + 3] = __float_as_uint(__uint_as_float(u[4 * e + 3]) * gm.w);
            }
            tmem_st32(trow + TM_S + cg * 32, u);
        }
        tc_fence_before();
        __syncthreads();
        // ---- tensor cores: U^T = Y^T T'^T, then [S^T | O^T] += U^T [K~^T ; Aqk]^T (completes while the
        //      next chunk's gate pass runs; its output is read out there)
        if (tid == MMA_TID) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < CH / 8; ++s)
                mma_tf32_ts(tbase + TM_U, tbase + TM_Y + 8 * s, umma_desc(s_tp + s * 2 * TP_LBO, TP_LBO, TP_SBO),
                            idesc_tf32(128, CH), s > 0);
            umma_commit(mbarU);
        }

        // ---- stage the next chunk's v and beta
        if (has_next)
            load_tile_async<false>(smem, OFF_RAW_V, p.v, ntok0, Ln, H, h);
        cp_async_commit();
        if (tid < CH)
            rawb[tid] = next_beta;
        prev_tok0 = tok0;
        prev_L = L;
    }
    if (!hung && nchunks > 0 && tid == MMA_TID)
        issue_update(nchunks - 1);
    cp_async_wait<0>();
    __syncthreads();
    // the last chunk's output
    if (!hung && nchunks > 0) {
        if (read_out_previous((nchunks - 1) & 1)) {
            __syncthreads();
            store_previous(prev_tok0, prev_L);
        } else {
            hung = true;
        }
    }

    // -------- final state, tensor memory release
    if (hung) {
        // give any tensor-core work still in flight a bounded chance to finish before releasing
        mbar_wait(mbarX, 0);
        mbar_wait(mbarU, 0);
        mbar_wait(mbarB, 0);
        if (tid == 0)
            atomicOr(&g_kda_device_error, 1u);
    } else if (STATE != 0 && p.fin) {
        tc_fence_after();
        uint32_t u[32];
        tmem_ld32(trow + TM_S + cg * 32, u);
        if (STATE == 2) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.fin) + srow);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(__uint_as_float(u[4 * e]), __uint_as_float(u[4 * e + 1]),
                                     __uint_as_float(u[4 * e + 2]), __uint_as_float(u[4 * e + 3]));
        } else {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.fin) + srow);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                uint32_t w4[4];
#pragma unroll
                for (int f = 0; f < 4; ++f) {
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(u[8 * e + 2 * f]),
                                                              __uint_as_float(u[8 * e + 2 * f + 1]));
                    w4[f] = *reinterpret_cast<uint32_t *>(&b2);
                }
                dst[e] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(TMEM_COLS));
    }
}

// ---------------------------------------------------------------- host side
template <int STATE, bool VARLEN>
cudaError_t launch(const Params &p, int grid, cudaStream_t stream)
{
    static std::atomic<uint64_t> configured{0};   // bit d: attribute set on device d
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        err = cudaFuncSetAttribute(kda_fwd_kernel<STATE, VARLEN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   SMEM_BYTES);
        if (err != cudaSuccess)
            return err;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    kda_fwd_kernel<STATE, VARLEN><<<grid, NTHREADS, SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

bool aligned(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

}  // namespace

extern "C" kda_status_t kda_fwd(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                float scale, void *out, const float *A_log, const float *dt_bias,
                                float lower_bound, const void *initial_state, void *final_state,
                                kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H,
                                kda_stream_t stream)
{
    if (N < 1 || H < 1 || T < 0)
        return KDA_ERR_INVALID_ARGUMENT;
    // with no tokens at all the token tensors may be empty (NULL)
    const bool no_tokens = T == 0;
    if (!no_tokens && (!q || !k || !v || !g || !beta || !out))
        return KDA_ERR_INVALID_ARGUMENT;
    if (!A_log || !dt_bias)
        return KDA_ERR_INVALID_ARGUMENT;
    if ((int64_t)N * H > INT32_MAX)
        return KDA_ERR_INVALID_ARGUMENT;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(g, 16) || !aligned(out, 16) ||
        !aligned(beta, 2) || !aligned(A_log, 4) || !aligned(dt_bias, 4) || !aligned(cu_seqlens, 8))
        return KDA_ERR_INVALID_ARGUMENT;
    const bool has_state = initial_state || final_state;
    if (has_state) {
        if (state_dtype != KDA_DTYPE_BF16 && state_dtype != KDA_DTYPE_FP32)
            return KDA_ERR_INVALID_ARGUMENT;
        if (!aligned(initial_state, 16) || !aligned(final_state, 16))
            return KDA_ERR_INVALID_ARGUMENT;
    }
    if (!(lower_bound >= -5.0f && lower_bound <= 0.0f))
        return KDA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale))
        return KDA_ERR_UNSUPPORTED;

    Params p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.g = static_cast<const __nv_bfloat16 *>(g);
    p.beta = static_cast<const __nv_bfloat16 *>(beta);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.A_log = A_log;
    p.dt_bias = dt_bias;
    p.init = initial_state;
    p.fin = final_state;
    p.cu = cu_seqlens;
    p.scale = scale;
    p.lb_log2e = lower_bound * LOG2E;
    p.N = N;
    p.H = H;
    p.T = T;
    const int grid = N * H;
    const int st = has_state ? (state_dtype == KDA_DTYPE_FP32 ? 2 : 1) : 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err;
    if (cu_seqlens) {
        err = st == 2 ? launch<2, true>(p, grid, s) : st == 1 ? launch<1, true>(p, grid, s) : launch<0, true>(p, grid, s);
    } else {
        err = st == 2 ? launch<2, false>(p, grid, s) : st == 1 ? launch<1, false>(p, grid, s) : launch<0, false>(p, grid, s);
    }
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

extern "C" kda_status_t kda_check_cu_seqlens(const int64_t *cu, int N, int64_t T)
{
    if (!cu || N < 1 || T < 0 || cu[0] != 0 || cu[N] != T)
        return KDA_ERR_INVALID_ARGUMENT;
    for (int i = 0; i < N; ++i)
        if (cu[i + 1] < cu[i])
            return KDA_ERR_INVALID_ARGUMENT;
    return KDA_OK;
}

extern "C" const char *kda_status_string(kda_status_t s)
{
    switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported argument value";
    case KDA_ERR_CUDA: return "CUDA error";
    case KDA_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

extern "C" size_t kda_fwd_smem_bytes(void) { return SMEM_BYTES; }

extern "C" kda_status_t kda_device_status(kda_stream_t stream)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KDA_ERR_CUDA;
    unsigned int flag = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&flag, g_kda_device_error, sizeof flag) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (flag && cudaMemcpyToSymbol(g_kda_device_error, &zero, sizeof zero) != cudaSuccess)
        return KDA_ERR_CUDA;
    return flag ? KDA_ERR_TIMEOUT : KDA_OK;
}
