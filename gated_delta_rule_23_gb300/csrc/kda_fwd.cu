// KDA chunked forward pass for sm_103a (GB300).
//
// One CTA owns one (sequence, head) pair and walks its tokens in 32-token
// chunks.  Per chunk it runs the token-parallel intra-chunk stage (gate, L2 norm,
// decay factors, the strictly-lower beta*K*K^T and causal Q*K^T matrices, the
// (I + A)^-1 inverse and the WY transform) and then the chunk recurrence on the
// state; this follows the split into an intra-chunk stage (gate activation -> L2
// norm -> decay -> L / Mqk construction -> inversion) and a chunk-wise delta-rule
// recurrence described in the guancyxx.cn FlashKDA article, section 2.2, but
// fuses both into one launch so the intermediates never leave shared memory.
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
// The inter-chunk stage is computed transposed: each warp owns 16 value columns of
// the state (rows of S^T) and keeps S^T (fp32 master), U^T and O^T for them in
// registers, since the recurrence never mixes value columns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "kda.h"

namespace {

constexpr int D = 128;        // K = V = 128
constexpr int CH = 32;        // tokens per chunk
constexpr int SB = 16;        // tokens per decay sub-block
constexpr int NTHREADS = 256;
constexpr float LOG2E = 1.4426950408889634f;

// ---------------------------------------------------------------- shared memory map
// Half-precision [32][136] tiles (272-byte rows) hold q, k, g, v and the fp16 operands.
// The q, k, g tiles and the fp16 operands written by the gate pass swizzle their
// 16-byte chunks by ((row >> 3) & 3) << 1, which makes the gate pass (lanes spread
// over four 8-row segments) and ldmatrix both free of bank conflicts.  fp32 tf32
// operands use a 132-float pitch, conflict-free for the mma fragment loads.
constexpr int PH = 136;                          // half row pitch (elements)
constexpr int PF = 132;                          // fp32 pitch of 128-wide tf32 operands
constexpr int PA = 36;                           // fp32 pitch of 32-wide matrices
constexpr int PS = 40;                           // half pitch of 32-wide matrices
constexpr int HT = CH * PH * 2;                  // 8704 B: one [32][136] half tile

constexpr int OFF_RAW_Q = 0;
constexpr int OFF_RAW_K = OFF_RAW_Q + HT;
constexpr int OFF_RAW_G = OFF_RAW_K + HT;
constexpr int OFF_RAW_V = OFF_RAW_G + HT;
constexpr int OFF_RAW_B = OFF_RAW_V + HT;        // beta logits, 32 bf16 (128 B reserved)
constexpr int OFF_INTRA = OFF_RAW_B + 128;
constexpr int F32T = CH * PF * 4;                // 16896 B
constexpr int OFF_LQ = OFF_INTRA;                // fp32 [32][132]  q^ P          (tf32-rounded)
constexpr int OFF_LK = OFF_LQ + F32T;            // fp32 [32][132]  k^ P
constexpr int OFF_ED = OFF_LK + F32T;            // fp32 [32][132]  k^ E / D_b
constexpr int OFF_EK = OFF_ED + F32T;            // fp32 [16][132]  k^ E  (sub-block 0 only)
constexpr int INTRA_BYTES = 3 * F32T + F32T / 2;
// after the Akk / Aqk products the same region holds:
constexpr int OFF_AKK = OFF_INTRA;               // fp32 [32][36]
constexpr int OFF_TM = OFF_AKK + CH * PA * 4;    // fp32 [32][36]  diagonal blocks of Tm
constexpr int OFF_AQK = OFF_TM + CH * PA * 4;    // fp16 [32][40]
constexpr int OFF_TP = OFF_AQK + CH * PS * 2;    // fp16 [32][40]  T' = Tm diag(b)
constexpr int OFF_MT = OFF_TP + CH * PS * 2;     // fp32 [16][16]  inverse scratch
constexpr int OFF_WN = OFF_MT + 16 * 16 * 4;     // fp16 [32][136] -W
constexpr int OFF_OST = OFF_WN + HT;             // bf16 [32][136] output staging
constexpr int INTRA_END = OFF_OST + HT;
constexpr int OFF_INTER = OFF_INTRA + INTRA_BYTES;
constexpr int OFF_QT = OFF_INTER;                // fp16 [32][136] Q~          (swizzled)
constexpr int OFF_KT = OFF_QT + HT;              // fp16 [32][136] K~          (swizzled)
constexpr int OFF_KG = OFF_KT + HT;              // fp16 [32][136] K^ . Gamma  (swizzled)
constexpr int OFF_MISC = OFF_KG + HT;
constexpr int OFF_RQ = OFF_MISC;                 // fp32 [32] 1/|q|
constexpr int OFF_RK = OFF_RQ + 128;             // fp32 [32] 1/|k|
constexpr int OFF_BT = OFF_RK + 128;             // fp32 [32] b = sigmoid(beta), 0 past the end
constexpr int OFF_GC = OFF_BT + 128;             // fp32 [128] chunk decay Gamma_31
constexpr int SMEM_BYTES = OFF_GC + D * 4;
static_assert(INTRA_END <= OFF_INTER, "post-product overlay exceeds the intra region");
static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
static_assert(OFF_INTRA % 128 == 0 && OFF_INTER % 16 == 0 && OFF_MISC % 16 == 0 && OFF_WN % 16 == 0 &&
              OFF_OST % 16 == 0 && OFF_TP % 16 == 0 && OFF_AQK % 16 == 0, "alignment");

// byte offset of element (row, col) in a swizzled [32][136] half tile
__host__ __device__ constexpr int swz(int row, int col)
{
    return row * PH * 2 + ((((col >> 3) ^ (((row >> 3) & 3) << 1))) << 4) + ((col & 7) << 1);
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

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t bf16x2_to_half2(uint32_t u) { return pack_half2(bf16_lo(u), bf16_hi(u)); }

__device__ __forceinline__ uint32_t to_tf32(float x)
{
    uint32_t y;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// D += A * B, m16n8k16, fp16 operands, fp32 accumulators
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                       uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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
    const int tid = threadIdx.x;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const int idx = tid + m * NTHREADS;   // 0..511: 32 rows x 16 chunks of 16 bytes
        const int r = idx >> 4, c16 = idx & 15;
        const bool valid = r < len;
        const int64_t row = tok0 + (valid ? r : 0);
        const __nv_bfloat16 *src = base + (row * H + h) * D + c16 * 8;
        const int dst = SWZ ? swz(r, c16 * 8) : r * PH * 2 + c16 * 16;
        cp_async16(smem_u32(smem + off + dst), src, valid);
    }
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
    const int gq = lane >> 2, tq = lane & 3;             // mma fragment coordinates
    const int mi = lane >> 3, lr = lane & 7;             // ldmatrix lane roles
    const int n = blockIdx.x / p.H, h = blockIdx.x % p.H;
    const int H = p.H;

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

    // -------- state: each warp owns value rows vr0..vr0+15 of S^T, all 128 key columns
    const int vr0 = warp * 16;
    float accS[16][4];
    {
        const size_t sbase = ((size_t)n * H + h) * D * D;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int kc = nt * 8 + 2 * tq;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int vv = vr0 + gq + 8 * hh;
                float x0 = 0.f, x1 = 0.f;
                if (STATE == 2 && p.init) {
                    const float2 s = *reinterpret_cast<const float2 *>(
                        static_cast<const float *>(p.init) + sbase + (size_t)vv * D + kc);
                    x0 = s.x;
                    x1 = s.y;
                } else if (STATE == 1 && p.init) {
                    const uint32_t s = *reinterpret_cast<const uint32_t *>(
                        static_cast<const __nv_bfloat16 *>(p.init) + sbase + (size_t)vv * D + kc);
                    x0 = bf16_lo(s);
                    x1 = bf16_hi(s);
                }
                accS[nt][2 * hh] = x0;
                accS[nt][2 * hh + 1] = x1;
            }
        }
    }

    // gate-pass lane roles: channel pair cp of this warp's 16 channels, 8-row segment sg
    const int cp = lane & 7, sg = lane >> 3, blk = sg >> 1;
    const int c0 = warp * 16 + 2 * cp;
    const float eA = expf(p.A_log[h]);
    const float2 dtb = *reinterpret_cast<const float2 *>(p.dt_bias + h * D + c0);
    const int nchunks = (int)((len + CH - 1) / CH);

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

    for (int ci = 0; ci < nchunks; ++ci) {
        const int64_t tok0 = bos + (int64_t)ci * CH;
        const int64_t rem = len - (int64_t)ci * CH;
        const int L = (int)(rem < CH ? rem : CH);
        const bool has_next = ci + 1 < nchunks;
        const int64_t ntok0 = tok0 + CH;
        const int Ln = has_next ? (int)((rem - CH) < CH ? (rem - CH) : CH) : 0;

        cp_async_wait<1>();   // q, k, g of this chunk have landed (v may still be in flight)
        __syncthreads();

        // ---- S1a: row norms (16 lanes per row, 8 channels per lane) and beta
        {
            const int half = lane >> 4, l16 = lane & 15;
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const int r = warp * 4 + it * 2 + half;
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
            }
            if (tid < CH)
                bt[tid] = tid < L ? sigmoidf_fast(__bfloat162float(rawb[tid])) : 0.f;
        }
        __syncthreads();

        // ---- S1b: gate, sub-block decay products, all operands of this chunk (one pass)
        {
            uint32_t gqv[8], gkv[8];
            float al0[8], al1[8];
            float tot0 = 1.f, tot1 = 1.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = sg * 8 + i;
                const uint32_t gg = *reinterpret_cast<const uint32_t *>(smem + OFF_RAW_G + swz(r, c0));
                gqv[i] = *reinterpret_cast<const uint32_t *>(smem + OFF_RAW_Q + swz(r, c0));
                gkv[i] = *reinterpret_cast<const uint32_t *>(smem + OFF_RAW_K + swz(r, c0));
                const float z0 = eA * (bf16_lo(gg) + dtb.x), z1 = eA * (bf16_hi(gg) + dtb.y);
                const bool live = r < L;
                al0[i] = live ? ex2_approx(p.lb_log2e * sigmoidf_fast(z0)) : 1.f;
                al1[i] = live ? ex2_approx(p.lb_log2e * sigmoidf_fast(z1)) : 1.f;
                tot0 *= al0[i];
                tot1 *= al1[i];
            }
            // the other 8-row segment of this sub-block (lane ^ 8) and the other sub-block (lane ^ 16)
            const float ot0 = __shfl_xor_sync(0xffffffffu, tot0, 8), ot1 = __shfl_xor_sync(0xffffffffu, tot1, 8);
            const float D0 = tot0 * ot0, D1 = tot1 * ot1;                     // this sub-block's decay
            const float Do0 = __shfl_xor_sync(0xffffffffu, D0, 16), Do1 = __shfl_xor_sync(0xffffffffu, D1, 16);
            const float pre0 = blk ? Do0 : 1.f, pre1 = blk ? Do1 : 1.f;       // Gamma at sub-block start
            const float post0 = blk ? 1.f : Do0, post1 = blk ? 1.f : Do1;     // decay after sub-block end
            const float iD0 = rcp_approx(D0), iD1 = rcp_approx(D1);
            const bool odd = sg & 1;
            float P0 = odd ? ot0 : 1.f, P1 = odd ? ot1 : 1.f;
            float E0 = odd ? 1.f : ot0, E1 = odd ? 1.f : ot1;
            float *Lq = reinterpret_cast<float *>(smem + OFF_LQ);
            float *Lk = reinterpret_cast<float *>(smem + OFF_LK);
            float *Ed = reinterpret_cast<float *>(smem + OFF_ED);
            float *Ek = reinterpret_cast<float *>(smem + OFF_EK);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = sg * 8 + i;
                const float qn = rq[r], kn = rk[r];
                const float q0 = bf16_lo(gqv[i]) * qn, q1 = bf16_hi(gqv[i]) * qn;
                const float k0 = bf16_lo(gkv[i]) * kn, k1 = bf16_hi(gkv[i]) * kn;
                P0 *= al0[i];
                P1 *= al1[i];
                *reinterpret_cast<float2 *>(Lq + r * PF + c0) = make_float2(tf32r(q0 * P0), tf32r(q1 * P1));
                *reinterpret_cast<float2 *>(Lk + r * PF + c0) = make_float2(tf32r(k0 * P0), tf32r(k1 * P1));
                *reinterpret_cast<uint32_t *>(smem + OFF_QT + swz(r, c0)) = pack_half2(q0 * P0 * pre0, q1 * P1 * pre1);
                *reinterpret_cast<uint32_t *>(smem + OFF_KG + swz(r, c0)) = pack_half2(k0 * P0 * pre0, k1 * P1 * pre1);
            }
#pragma unroll
            for (int i = 7; i >= 0; --i) {
                const int r = sg * 8 + i;
                const float kn = rk[r];
                const float k0 = bf16_lo(gkv[i]) * kn, k1 = bf16_hi(gkv[i]) * kn;
                *reinterpret_cast<float2 *>(Ed + r * PF + c0) = make_float2(tf32r(k0 * E0 * iD0), tf32r(k1 * E1 * iD1));
                if (blk == 0)
                    *reinterpret_cast<float2 *>(Ek + r * PF + c0) = make_float2(tf32r(k0 * E0), tf32r(k1 * E1));
                *reinterpret_cast<uint32_t *>(smem + OFF_KT + swz(r, c0)) = pack_half2(k0 * E0 * post0, k1 * E1 * post1);
                E0 *= al0[i];
                E1 *= al1[i];
            }
            if (sg == 0)
                *reinterpret_cast<float2 *>(Gc + c0) = make_float2(D0 * Do0, D1 * Do1);
        }
        __syncthreads();

        // ---- raw q, k, g, beta are consumed: start staging the next chunk's
        if (has_next) {
            load_tile_async<true>(smem, OFF_RAW_Q, p.q, ntok0, Ln, H, h);
            load_tile_async<true>(smem, OFF_RAW_K, p.k, ntok0, Ln, H, h);
            load_tile_async<true>(smem, OFF_RAW_G, p.g, ntok0, Ln, H, h);
        }
        cp_async_commit();
        __nv_bfloat16 next_beta = __float2bfloat16(0.f);
        if (has_next && tid < Ln)
            next_beta = p.beta[(ntok0 + tid) * H + h];

        // ---- S2: Akk and Aqk on tf32 tensor cores; items (pair, kind), pairs (0,0), (1,0), (1,1)
        float acc2[2][4] = {};
        const int item = warp;           // warps 0..5
        const int pair = item >> 1, qk = item & 1;
        const int rb1 = pair == 0 ? 0 : 16;                  // row block of the left factor
        if (item < 6) {
            const float *X = reinterpret_cast<const float *>(smem + (qk ? OFF_LQ : OFF_LK)) + (rb1 + gq) * PF + tq;
            const float *Y = reinterpret_cast<const float *>(smem + (pair == 1 ? OFF_EK : OFF_ED)) +
                             ((pair == 2 ? 16 : 0) + gq) * PF + tq;
#pragma unroll 8
            for (int ks = 0; ks < D / 8; ++ks) {
                const int k0 = ks * 8;
                const uint32_t a0 = __float_as_uint(X[k0]), a1 = __float_as_uint(X[8 * PF + k0]);
                const uint32_t a2 = __float_as_uint(X[k0 + 4]), a3 = __float_as_uint(X[8 * PF + k0 + 4]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    mma_tf32(acc2[nt], a0, a1, a2, a3, __float_as_uint(Y[nt * 8 * PF + k0]),
                             __float_as_uint(Y[nt * 8 * PF + k0 + 4]));
            }
        }
        __syncthreads();   // the intra operands are dead; the region is reused below
        if (item < 6) {
            float *Akk = reinterpret_cast<float *>(smem + OFF_AKK);
            __half *Aqk = reinterpret_cast<__half *>(smem + OFF_AQK);
            const int cb0 = pair == 2 ? 16 : 0;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int i = rb1 + gq + 8 * hh, j = cb0 + nt * 8 + 2 * tq;
                    const float x0 = acc2[nt][2 * hh], x1 = acc2[nt][2 * hh + 1];
                    if (qk) {
                        *reinterpret_cast<uint32_t *>(Aqk + i * PS + j) =
                            pack_half2(j <= i ? x0 : 0.f, j + 1 <= i ? x1 : 0.f);
                    } else {
                        const float bi = bt[i];
                        *reinterpret_cast<float2 *>(Akk + i * PA + j) =
                            make_float2(j < i ? bi * x0 : 0.f, j + 1 < i ? bi * x1 : 0.f);
                    }
                }
        }
        __syncthreads();

        // ---- S3: Tm = (I + Akk)^-1 (fp32) and T' = Tm diag(b) (fp16)
        float *Akk = reinterpret_cast<float *>(smem + OFF_AKK);
        float *Tm = reinterpret_cast<float *>(smem + OFF_TM);
        __half *Tp = reinterpret_cast<__half *>(smem + OFF_TP);
        if (warp < 2 && lane < 16) {
            // diagonal 16x16 blocks by forward substitution; lane = column
            const int b = warp, j = lane;
            float x[SB];
#pragma unroll
            for (int i = 0; i < SB; ++i) {
                float s = 0.f;
#pragma unroll
                for (int l = 0; l < i; ++l)
                    s = fmaf(Akk[(b * SB + i) * PA + b * SB + l], x[l], s);
                x[i] = i == j ? 1.f : (i < j ? 0.f : -s);
            }
            const float bj = bt[b * SB + j];
#pragma unroll
            for (int i = 0; i < SB; ++i) {
                Tm[(b * SB + i) * PA + b * SB + j] = x[i];
                Tp[(b * SB + i) * PS + b * SB + j] = __float2half_rn(x[i] * bj);
            }
        } else if (warp >= 2 && warp < 4) {
            // upper off-diagonal block of T' is zero
            const int e = (warp - 2) * 32 + lane;            // 0..63: 16 rows x 4 groups of 4 columns
            const int i = e >> 2, j4 = (e & 3) * 4;
            *reinterpret_cast<uint2 *>(Tp + i * PS + 16 + j4) = make_uint2(0u, 0u);
        }
        __syncthreads();
        {
            // off-diagonal block: Tm_10 = -Tm_11 (A_10 Tm_00);  thread = (i, j)
            const int i = tid >> 4, j = tid & 15;
            float *Mt = reinterpret_cast<float *>(smem + OFF_MT);
            float s = 0.f;
#pragma unroll
            for (int l = 0; l < SB; ++l)
                s = fmaf(Akk[(SB + i) * PA + l], Tm[l * PA + j], s);
            Mt[i * 16 + j] = s;
            __syncthreads();
            s = 0.f;
#pragma unroll
            for (int l = 0; l < SB; ++l)
                s = fmaf(Tm[(SB + i) * PA + SB + l], Mt[l * 16 + j], s);
            Tp[(SB + i) * PS + j] = __float2half_rn(-s * bt[j]);
        }
        __syncthreads();

        // ---- S4: -W = -T' (K^ . Gamma); warp: key columns 16w..16w+15
        {
            const uint32_t tp_base = smem_u32(smem + OFF_TP);
            const uint32_t kg_base = smem_u32(smem + OFF_KG);
            __half *Wn = reinterpret_cast<__half *>(smem + OFF_WN);
#pragma unroll
            for (int rb = 0; rb < 2; ++rb) {
                float acc[2][4] = {};
#pragma unroll
                for (int ks = 0; ks <= rb; ++ks) {
                    uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                    ldsm_x4(tp_base + ((rb * 16 + lr + (mi & 1) * 8) * PS + ks * 16 + (mi >> 1) * 8) * 2, a0, a1, a2, a3);
                    ldsm_x4_t(kg_base + swz(ks * 16 + lr + (mi & 1) * 8, warp * 16 + (mi >> 1) * 8), b0, b1, b2, b3);
                    mma_f16(acc[0], a0, a1, a2, a3, b0, b1);
                    mma_f16(acc[1], a0, a1, a2, a3, b2, b3);
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int i = rb * 16 + gq + 8 * hh, j = warp * 16 + nt * 8 + 2 * tq;
                        *reinterpret_cast<uint32_t *>(Wn + i * PH + j) = pack_half2(-acc[nt][2 * hh], -acc[nt][2 * hh + 1]);
                    }
            }
        }
        cp_async_wait<1>();   // v of this chunk (the next chunk's q, k, g may stay in flight)
        __syncthreads();

        // ---- S5: chunk recurrence, transposed, per warp: value rows vr0..vr0+15
        {
            const uint32_t v_base = smem_u32(smem + OFF_RAW_V);
            const uint32_t tp_base = smem_u32(smem + OFF_TP);
            const uint32_t wn_base = smem_u32(smem + OFF_WN);
            const uint32_t qt_base = smem_u32(smem + OFF_QT);
            const uint32_t aq_base = smem_u32(smem + OFF_AQK);
            const uint32_t kt_base = smem_u32(smem + OFF_KT);
            float accU[4][4], accO[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    accU[nt][e] = accO[nt][e] = 0.f;

            // U^T = V^T T'^T  (k = t', token blocks t' <= t only)
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(v_base + ((ks * 16 + lr + (mi >> 1) * 8) * PH + vr0 + (mi & 1) * 8) * 2, a0, a1, a2, a3);
                a0 = bf16x2_to_half2(a0);
                a1 = bf16x2_to_half2(a1);
                a2 = bf16x2_to_half2(a2);
                a3 = bf16x2_to_half2(a3);
#pragma unroll
                for (int np = ks; np < 2; ++np) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(tp_base + ((np * 16 + lr + (mi >> 1) * 8) * PS + ks * 16 + (mi & 1) * 8) * 2, b0, b1, b2, b3);
                    mma_f16(accU[2 * np], a0, a1, a2, a3, b0, b1);
                    mma_f16(accU[2 * np + 1], a0, a1, a2, a3, b2, b3);
                }
            }
            // U^T += S^T (-W)^T,  O^T = S^T Q~^T   (k = key channel)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t a0 = pack_half2(accS[2 * ks][0], accS[2 * ks][1]);
                const uint32_t a1 = pack_half2(accS[2 * ks][2], accS[2 * ks][3]);
                const uint32_t a2 = pack_half2(accS[2 * ks + 1][0], accS[2 * ks + 1][1]);
                const uint32_t a3 = pack_half2(accS[2 * ks + 1][2], accS[2 * ks + 1][3]);
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    uint32_t b0, b1, b2, b3;
                    const int row = np * 16 + lr + (mi >> 1) * 8, col = ks * 16 + (mi & 1) * 8;
                    ldsm_x4(wn_base + (row * PH + col) * 2, b0, b1, b2, b3);
                    mma_f16(accU[2 * np], a0, a1, a2, a3, b0, b1);
                    mma_f16(accU[2 * np + 1], a0, a1, a2, a3, b2, b3);
                    ldsm_x4(qt_base + swz(row, col), b0, b1, b2, b3);
                    mma_f16(accO[2 * np], a0, a1, a2, a3, b0, b1);
                    mma_f16(accO[2 * np + 1], a0, a1, a2, a3, b2, b3);
                }
            }
            // U^T as fp16 A fragments (k = token)
            uint32_t ua[2][4];
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                ua[ks][0] = pack_half2(accU[2 * ks][0], accU[2 * ks][1]);
                ua[ks][1] = pack_half2(accU[2 * ks][2], accU[2 * ks][3]);
                ua[ks][2] = pack_half2(accU[2 * ks + 1][0], accU[2 * ks + 1][1]);
                ua[ks][3] = pack_half2(accU[2 * ks + 1][2], accU[2 * ks + 1][3]);
            }
            // O^T += U^T Aqk^T  (token blocks t' <= t only)
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
                for (int np = ks; np < 2; ++np) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(aq_base + ((np * 16 + lr + (mi >> 1) * 8) * PS + ks * 16 + (mi & 1) * 8) * 2, b0, b1, b2, b3);
                    mma_f16(accO[2 * np], ua[ks][0], ua[ks][1], ua[ks][2], ua[ks][3], b0, b1);
                    mma_f16(accO[2 * np + 1], ua[ks][0], ua[ks][1], ua[ks][2], ua[ks][3], b2, b3);
                }
            }
            // S^T <- S^T Diag(Gamma_31) + U^T K~
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                const float2 gm = *reinterpret_cast<const float2 *>(Gc + nt * 8 + 2 * tq);
                accS[nt][0] *= gm.x;
                accS[nt][1] *= gm.y;
                accS[nt][2] *= gm.x;
                accS[nt][3] *= gm.y;
            }
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
                for (int np = 0; np < 8; ++np) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(kt_base + swz(ks * 16 + lr + (mi & 1) * 8, np * 16 + (mi >> 1) * 8), b0, b1, b2, b3);
                    mma_f16(accS[2 * np], ua[ks][0], ua[ks][1], ua[ks][2], ua[ks][3], b0, b1);
                    mma_f16(accS[2 * np + 1], ua[ks][0], ua[ks][1], ua[ks][2], ua[ks][3], b2, b3);
                }
            }
            // O^T * scale -> bf16 staging tile [t][v]
            __nv_bfloat16 *Ost = reinterpret_cast<__nv_bfloat16 *>(smem + OFF_OST);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int vv = vr0 + gq + 8 * hh, t = nt * 8 + 2 * tq;
                    Ost[t * PH + vv] = __float2bfloat16_rn(accO[nt][2 * hh] * p.scale);
                    Ost[(t + 1) * PH + vv] = __float2bfloat16_rn(accO[nt][2 * hh + 1] * p.scale);
                }
        }
        __syncthreads();

        // ---- write this chunk's outputs; stage the next chunk's v and beta
        {
            const unsigned char *Ost = smem + OFF_OST;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int idx = tid + m * NTHREADS, r = idx >> 4, c16 = idx & 15;
                if (r < L)
                    *reinterpret_cast<uint4 *>(p.out + ((tok0 + r) * H + h) * D + c16 * 8) =
                        *reinterpret_cast<const uint4 *>(Ost + r * PH * 2 + c16 * 16);
            }
        }
        if (has_next)
            load_tile_async<false>(smem, OFF_RAW_V, p.v, ntok0, Ln, H, h);
        cp_async_commit();
        if (tid < CH)
            rawb[tid] = next_beta;
    }
    cp_async_wait<0>();

    // -------- final state
    if (STATE != 0 && p.fin) {
        const size_t sbase = ((size_t)n * H + h) * D * D;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int kc = nt * 8 + 2 * tq;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int vv = vr0 + gq + 8 * hh;
                if (STATE == 2) {
                    *reinterpret_cast<float2 *>(static_cast<float *>(p.fin) + sbase + (size_t)vv * D + kc) =
                        make_float2(accS[nt][2 * hh], accS[nt][2 * hh + 1]);
                } else {
                    __nv_bfloat162 s = __floats2bfloat162_rn(accS[nt][2 * hh], accS[nt][2 * hh + 1]);
                    *reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(p.fin) + sbase +
                                                        (size_t)vv * D + kc) = s;
                }
            }
        }
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
