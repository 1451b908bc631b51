// Device-side helpers shared by the KDA kernels (sm_103a): PTX wrappers for the
// special-function unit, mma.sync, ldmatrix, cp.async, bulk copies, mbarriers and the
// 5th-generation tensor cores (tcgen05), plus the problem description both kernels read.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kda_plan.h"

namespace kda {

constexpr int D = 128;                     // K = V = 128
constexpr int CH = 64;                     // tokens per chunk
constexpr int SB = 16;                     // tokens per decay sub-block
constexpr int NSB = CH / SB;               // sub-blocks per chunk
constexpr float LOG2E = 1.4426950408889634f;
constexpr uint32_t WAIT_LIMIT = 1u << 24;  // mbarrier polls before a wait is declared hung
// Bits of the kernels' device-side error words (read and cleared by kda_device_status).
constexpr unsigned int DEVERR_TIMEOUT = 1u;     // a bounded wait gave up; the call's results are not valid
constexpr unsigned int DEVERR_NONFINITE = 2u;   // a state ended non-finite (fp16 operand overflow or inf/NaN inputs)
constexpr unsigned int DEVERR_CU_SEQLENS = 4u;  // cu_seqlens broke its contract; it was clamped into range

// ---------------------------------------------------------------- per-chunk operand slot
// The prep kernel writes, for every (chunk, head), one slot of fp16 operands in exactly the
// shared-memory image the recurrence kernel's tensor-core descriptors expect, so the
// recurrence kernel stages a chunk with a single bulk copy.
//   QW  [128 rows n][128 k]: rows 0..63 W = T'(K^.Gamma), rows 64..127 Q~ = Q^.Gamma
//   KA  [192 rows n][64 j] : rows 0..63 Aqk (row i), rows 64..191 K~^T (row = key channel)
//   U0T [128 v][64 t]      : (T' V)^T, 16-byte chunks XOR-swizzled by (v & 7)
//   GC  [128] fp32         : Gamma_C, the decay of the whole chunk per key channel
// QW and KA use the no-swizzle K-major core-matrix layout: element (n, k) at
//   (n / 8) * SBO + (k / 8) * 128 + (n % 8) * 16 + (k % 8) * 2.
constexpr int QW_SBO = 2048, KA_SBO = 1024, CORE_LBO = 128;
constexpr int SLOT_QW = 0;
constexpr int SLOT_KA = SLOT_QW + 128 * D * 2;        // 32768
constexpr int SLOT_U0 = SLOT_KA + 192 * CH * 2;       // 57344
constexpr int SLOT_GC = SLOT_U0 + D * CH * 2;         // 73728
constexpr int SLOT_BYTES = SLOT_GC + D * 4;           // 74240
static_assert(SLOT_BYTES % 256 == 0, "slot alignment");

__host__ __device__ constexpr int qw_off(int n, int k)
{
    return (n >> 3) * QW_SBO + (k >> 3) * CORE_LBO + ((n & 7) << 4) + ((k & 7) << 1);
}
__host__ __device__ constexpr int ka_off(int n, int j)
{
    return SLOT_KA + (n >> 3) * KA_SBO + (j >> 3) * CORE_LBO + ((n & 7) << 4) + ((j & 7) << 1);
}
__host__ __device__ constexpr int u0_off(int v, int t)
{
    return SLOT_U0 + v * (CH * 2) + ((((t >> 3) ^ (v & 7))) << 4) + ((t & 7) << 1);
}

// ---------------------------------------------------------------- problem description
struct Problem {
    const __nv_bfloat16 *q, *k, *v, *g, *beta;
    __nv_bfloat16 *out;
    const float *A_log, *dt_bias;
    const void *init;
    void *fin;
    const int64_t *cu;        // cu_seqlens (device) or nullptr
    const int64_t *chunk_off; // varlen: first chunk of each sequence, [N + 1] (workspace)
    const longlong2 *chunk_info; // varlen: (first token, tokens left in its sequence) per chunk (workspace)
    const int *order;         // varlen: sequences longest first, [N] (workspace), or nullptr
    unsigned char *slots;     // operand slots (workspace)
    float scale, lb_log2e;    // lb_log2e = lower_bound * log2(e)
    int N, H;
    int64_t T;
    int64_t nch_fixed;        // without cu_seqlens: chunks of each sequence in this launch
    int64_t ch_base;          // without cu_seqlens: first chunk of this launch within each sequence
    // chunk-transition scan (fixed length): the recurrence kernel runs `groups` groups of group_len chunks
    // of every sequence side by side (group_len = nch_fixed and groups = 1 otherwise)
    int groups;
    int64_t group_len;
    float *sc_a, *sc_b;       // compose launches: each group's transition, [groups - 1][N][H][128][128] fp32
    const float *sc_s;        // grouped launches: start states of groups 1 .. groups - 1, same layout
    int prep_pf;              // prep: each CTA prefetches its next item's rows into L2 (0: off)
    int64_t chunk_cap;        // varlen: entries of the per-chunk table (every sequence's chunks are clamped to it)
    uint32_t wait_polls;      // chunked kernels: polls of a wait before it gives up (kda_set_wait_limit)
    uint32_t variant;         // VARIANT_* bits (kda_fwd_ws_variant); 0 for the library's own design
};
// Measurement variants of the chunked path after the FlashKDA pages' own choices (kda_fwd_ws_variant).
constexpr uint32_t VARIANT_BF16_STATE = 1u;        // the state rounded to bf16 between chunks
constexpr uint32_t VARIANT_NEUMANN_INVERSE = 2u;   // (I + A)^-1 by the fp16 Neumann-series product

// ---------------------------------------------------------------- small helpers
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
__device__ __forceinline__ float sigmoid_fast(float z) { return rcp_approx(1.0f + ex2_approx(-z * LOG2E)); }
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
// Round to tf32 (10 explicit mantissa bits), to nearest with ties away from zero, on the integer
// pipe: adding half a tf32 ulp to the magnitude bits and truncating is that rounding for finite
// values (a carry into the exponent is the correct round-up).
// fp32 value prepared for a kind::tf32 tensor-core operand: the tensor cores use the top 19 bits of an
// fp32 operand and drop the low 13, so adding half a tf32 unit to the bit pattern makes that drop a
// round-to-nearest (ties away from zero, as cvt.rna.tf32.f32 rounds finite values)
__device__ __forceinline__ float tf32r(float x) { return __uint_as_float(__float_as_uint(x) + 0x1000u); }

// ---------------------------------------------------------------- packed fp32 pairs (f32x2)
typedef unsigned long long f2;
__device__ __forceinline__ f2 f2_pack(float lo, float hi)
{
    return ((f2)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float f2_lo(f2 a) { return __uint_as_float((uint32_t)a); }
__device__ __forceinline__ float f2_hi(f2 a) { return __uint_as_float((uint32_t)(a >> 32)); }
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b)
{
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c)
{
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// bf16x2 word (low half = the even element) -> packed fp32 pair, exactly
__device__ __forceinline__ f2 f2_bf16x2(uint32_t w) { return f2_pack(bf16_lo(w), bf16_hi(w)); }
__device__ __forceinline__ f2 f2_tf32r(f2 a) { return f2_pack(tf32r(f2_lo(a)), tf32r(f2_hi(a))); }
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}
// bf16x2 word -> fp16x2 word (both halves through fp32)
__device__ __forceinline__ uint32_t bf16x2_to_half2(uint32_t u) { return pack_half2(bf16_lo(u), bf16_hi(u)); }


// D += A * B, m16n8k16, fp16 operands, fp32 accumulators
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid)
{
    const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------- mbarriers and bulk copies
__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t mbar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}
// Bounded wait for an mbarrier phase: at most `polls` try_wait polls (0: give up at once); returns false if
// the wait gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, uint32_t polls = WAIT_LIMIT)
{
    uint32_t done = 0;
    for (uint32_t it = 0; it < polls; ++it) {
        asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                     : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
        if (done)
            return true;
    }
    return false;
}
// global -> shared bulk copy completing on an mbarrier (addresses 16-byte aligned, size % 16 == 0)
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t mbar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(mbar) : "memory");
}
// shared -> global bulk copy in the thread's bulk async-group (addresses 16-byte aligned, size % 16 == 0)
__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// waits until every bulk copy this thread committed has finished reading its shared-memory source
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }


// ---------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor: start address, leading (K-direction) and stride
// (M/N-direction) byte offsets between 8x16-byte core matrices, no swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}
// Instruction descriptor: fp32 accumulator, fp16 A and B, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N)
{
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// Instruction descriptor: fp32 accumulator, tf32 A and B, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::tf32, one CTA
__device__ __forceinline__ void mma_tf32_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, int acc)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}"
                 ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16, one CTA
__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, int acc)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
                 ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void umma_commit(uint32_t mbar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar));
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

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
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&u)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
                   "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]),
                   "=r"(u[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&u)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16};"
                 ::"r"(taddr), "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]),
                   "r"(u[7]), "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]), "r"(u[13]), "r"(u[14]),
                   "r"(u[15]));
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace kda
