// KDA prep kernel: the token-parallel intra-chunk stage, one CTA per (64-token chunk, head).
//
// This is the first of the two stages the guancyxx.cn FlashKDA article (section 2.2) splits
// the forward pass into: gate activation -> L2 norm -> cumulative decay -> the L / Mqk
// matrices -> their inversion, run for every chunk at once, independent of the state.  The
// CTA writes the chunk's state-free operands of the recurrence into its workspace slot
// (layout in kda_device.cuh), in fp16, ready for the tensor cores of the recurrence kernel:
//   W = T' (K^ . Gamma),  Q~ = Q^ . Gamma,  Aqk,  K~ = K^ . Gamma_C / Gamma,  U0 = T' V,  Gamma_C
// with T' = (I + Akk)^-1 diag(b).  The recurrence kernel then only evaluates
//   U = U0 - W S,   O = scale (Q~ S + Aqk U),   S <- Diag(Gamma_C) S + K~^T U.
//
// Decay factors.  Per key channel c, a_t = lower_bound * sigmoid(exp(A_log) (g_t + dt_bias)),
// alpha_t = exp(a_t) and Gamma_t = prod_{s <= t} alpha_s (chunk-relative).  The chunk is cut
// into four 16-token sub-blocks b with inclusive prefix P_t, exclusive suffix E_t and total D_b
// of alpha inside the sub-block; pre_b / post_b are the products of D over the earlier / later
// sub-blocks, so Gamma_t = pre_b P_t and Gamma_C / Gamma_t = E_t post_b.
// The intra-chunk products need Gamma_i / Gamma_j (j <= i).  Each 32-token half h is anchored
// at the end of its first sub-block (token m_0 = 15, m_1 = 47): row i of half h uses
//   left  factor Gamma_i / Gamma_{m_h}   (1 / E_i on sub-blocks 0 and 2, P_i on 1 and 3)
//   right factor Gamma_{m_h} / Gamma_j   (E_j, E_j D_1 D_2, E_j D_2 or 1 / P_j by sub-block)
// and Gamma_i / Gamma_j is their product.  Inside a half every factor lies within 16 tokens of
// its anchor, so it stays in [2^-115.5, 2^115.5] when lower_bound >= -5 (at most 7.22 binary
// orders of decay per token): the CHUNK = 16 range argument of the article (section 2.1),
// applied around each anchor.  Right factors of the second half's anchor for columns in the
// first half only shrink (a value below fp32 range stands for a contribution below 2^-41).
// With both halves' rows stacked, Akk and Aqk of the whole chunk are ONE tf32 tensor-core
// product: [k^ L ; q^ L] (128 rows) times [k^ R] (96 columns), K = 128.
#include "kda_device.cuh"
#include "kda_internal.h"

// Set when a bounded wait on the tensor cores expires in the prep kernel.
__device__ unsigned int g_kda_prep_error;

namespace kda {
namespace {

constexpr int PREP_THREADS = 256;
#ifndef KDA_PREP_PF_BETA
#define KDA_PREP_PF_BETA 1
#endif
#ifndef KDA_PREP_PREFETCH
#define KDA_PREP_PREFETCH 1
#endif
constexpr int TMEM_COLS = 128;          // Akk / Aqk accumulators: 128 lanes x 96 columns
// tf32 operand tiles of the Akk / Aqk product for one half of the channels (the gate pass runs in
// two passes of 64 channels; the tensor cores accumulate both).  No-swizzle K-major core-matrix
// layout, element (row r, pass channel kk) at (r / 8) * OPS_SBO + (kk / 4) * OPS_LBO
// + (r % 8) * 16 + (kk % 4) * 4.  The strides (LBO = 16 mod 128, SBO = 32 mod 128) make the gate
// pass's 8-byte stores (8 row groups x 4 channel pairs per warp) conflict-free.  Rows of A:
// [k^ L_0 (tokens 0..31) ; q^ L_0 ; k^ L_1 (tokens 32..63) ; q^ L_1]; rows of B: [k^ R_0 (tokens 0..31) ;
// k^ R_1 (tokens 0..63)].
constexpr int OPS_LBO = 144, OPS_SBO = 2336;
constexpr int OPS_A = 0;
constexpr int OPS_B = 16 * OPS_SBO;                 // 37376
constexpr int OPS_BYTES = OPS_B + 12 * OPS_SBO;     // 65408
// shared memory map (bytes)
constexpr int OFF_OPS = 0;
constexpr int OFF_PART = OFF_OPS;                   // fp32 [8 warps][2][64] sums of squares (before the gate pass)
// q, k, g of the chunk as loaded (bf16 [64 t][128 c] each, 16-byte chunks XOR-swizzled by t / 8), read into
// registers before the gate pass overwrites the region
constexpr int OFF_STG = OFF_PART + 8 * 2 * CH * 4;   // 4096
static_assert(OFF_STG + 3 * CH * D * 2 <= OPS_BYTES, "staging inside the operand tiles");
// reused once the Akk / Aqk product has completed:
constexpr int PA = 68;                              // fp32 pitch of 64-wide matrices
constexpr int OFF_AKK = OFF_OPS;                    // fp32 [64][68] b_i Akk (strictly lower)
constexpr int OFF_TM = OFF_AKK + CH * PA * 4;       // fp32 [64][68] (I + Akk)^-1
constexpr int OFF_TP = OFF_TM + CH * PA * 4;        // fp16 [64 t][64 j] T' (swizzled)
constexpr int OFF_ZW = OFF_TP + CH * CH * 2;        // fp32 [8 warps][16][8] off-diagonal partial products
constexpr int OFF_AQS = OFF_ZW + 8 * 16 * 8 * 4;  // Aqk rows of the slot (KA rows 0..63), staged for a bulk copy
static_assert(OFF_AQS + 64 * CH * 2 <= OPS_BYTES, "post-product overlay");
constexpr int OFF_KG = 65536;                       // fp16 [64 j][128 c] K^ . Gamma (kg_off swizzle)
constexpr int OFF_V = OFF_KG + CH * D * 2;          // bf16 [64 j][128 v] (swizzled)
// once the WY products have read K^.Gamma and V, the W and U0^T parts of the slot are staged over them for bulk
// copies, which may still be reading while the next item stages its q, k, g (the next item's first write to
// these tiles is in its gate pass, after a wait for those copies)
constexpr int OFF_WS = OFF_KG, OFF_US = OFF_V;
static_assert(64 * D * 2 <= CH * D * 2 && D * CH * 2 <= CH * D * 2, "W / U0 staging fits K^.Gamma / V");
constexpr int OFF_RQ = OFF_V + CH * D * 2;          // fp32 pairs [68][2] 1 / |q| (both halves; norm_slot order)
constexpr int OFF_RK = OFF_RQ + 544;                // fp32 pairs [68][2] 1 / |k|
constexpr int OFF_BT = OFF_RK + 544;                // fp32 [64] b = sigmoid(beta), 0 past the end
constexpr int OFF_MISC = OFF_BT + 256;              // mbarriers (+0 products, +16 drain), tensor-memory base (+8)
constexpr int PREP_SMEM = OFF_MISC + 24;
static_assert(OFF_KG >= OPS_BYTES && OFF_KG % 128 == 0, "shared memory map");
static_assert(2 * (PREP_SMEM + 1024) <= 233472, "two CTAs per SM");

// byte offset of a 16-bit element in a [64][128] / [64][64] tile; 16-byte chunks XOR-swizzled
// by row (conflict-free ldmatrix)
__device__ __forceinline__ int h128(int r, int c) { return r * 256 + ((((c >> 3) ^ (r & 7))) << 4) + ((c & 7) << 1); }
__device__ __forceinline__ int h64(int r, int c) { return r * 128 + ((((c >> 3) ^ (r & 7))) << 4) + ((c & 7) << 1); }
// byte offset of 16-byte chunk c16 of token row t in the q / k / g staging tiles: swizzled by t / 8, so
// that the 8 token runs a warp reads at once (rows 8 m + j) fall on 8 different bank groups
__device__ __forceinline__ int stg_off(int t, int c16) { return t * 256 + ((c16 ^ ((t >> 3) & 7)) << 4); }
// byte offset of element (token t, channel c) in the K^.Gamma tile: 16-byte chunks XOR-swizzled by t % 8 and
// t / 8, so that both the gate pass's stores (tokens 8 m + j of one channel group) and ldmatrix (8
// consecutive tokens) spread over the banks
__device__ __forceinline__ int kg_off(int t, int c) { return t * 256 + ((((c >> 3) ^ (t & 7) ^ ((t >> 3) & 7))) << 4) + ((c & 7) << 1); }

// slot of token t in the pair tables of the norms: one 8-byte pad every 16 tokens, so that the eight token runs a
// warp reads at once (tokens 16 sb + 8 hh + j) fall on eight different bank pairs
__host__ __device__ constexpr int norm_slot(int t) { return t + (t >> 4); }

__device__ __forceinline__ void st_global_v8(void *ptr, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4,
                                             uint32_t a5, uint32_t a6, uint32_t a7)
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(a0), "r"(a1), "r"(a2),
                 "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
                 : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void *ptr) { asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr)); }
// all but the most recently committed bulk group have read their shared-memory source
__device__ __forceinline__ void bulk_wait_read_but_last() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

__device__ __forceinline__ f2 f2_add(f2 a, f2 b)
{
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 f2_sub(f2 a, f2 b)
{
    f2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 f2_ex2(f2 a) { return f2_pack(ex2_approx(f2_lo(a)), ex2_approx(f2_hi(a))); }
__device__ __forceinline__ uint2 u2_tf32r(f2 a) { return make_uint2(__float_as_uint(tf32r(f2_lo(a))), __float_as_uint(tf32r(f2_hi(a)))); }
__device__ __forceinline__ uint32_t half2_of(f2 a) { return pack_half2(f2_lo(a), f2_hi(a)); }

// C = X Y (+ Z) for fp16 [64][64] matrices in the h64 layout (row-major, 16-byte chunks XOR-swizzled by row), fp32
// accumulation on mma.sync, result rounded to fp16; warp w computes rows 16 (w / 2) .. + 15, columns 32 (w % 2) .. + 31.
__device__ __forceinline__ void mm64_f16(uint32_t sx, uint32_t sy, const unsigned char *z, unsigned char *c, int warp, int lane)
{
    const int mt = warp >> 1, nh = warp & 1, gq = lane >> 2, t4 = lane & 3, lr = lane & 7, lsel = lane >> 3;
    float acc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float2 v = make_float2(0.f, 0.f);
            if (z)
                v = __half22float2(*reinterpret_cast<const __half2 *>(z + h64(16 * mt + gq + 8 * hh, 32 * nh + 8 * nt + 2 * t4)));
            acc[nt][2 * hh] = v.x;
            acc[nt][2 * hh + 1] = v.y;
        }
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        uint32_t af[4];
        ldsm_x4(sx + h64(16 * mt + (lsel & 1) * 8 + lr, 16 * ks + (lsel >> 1) * 8), af);
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
            uint32_t bf[4];
            ldsm_x4_t(sy + h64(16 * ks + (lsel & 1) * 8 + lr, 32 * nh + 16 * pr + (lsel >> 1) * 8), bf);
            mma_f16(acc[2 * pr], af, bf[0], bf[1]);
            mma_f16(acc[2 * pr + 1], af, bf[2], bf[3]);
        }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
            *reinterpret_cast<uint32_t *>(c + h64(16 * mt + gq + 8 * hh, 32 * nh + 8 * nt + 2 * t4)) =
                pack_half2(acc[nt][2 * hh], acc[nt][2 * hh + 1]);
}

// first token and tokens left of chunk gc (a chunk index over all sequences of the launch; the launch keeps
// every item index, and so gc, below 2^31, so the divisions are 32-bit); fixed-length launches cover
// chunks ch_base .. ch_base + nch_fixed - 1 of every sequence; varlen chunks come from the
// plan's per-chunk table, which has an entry for every launched chunk index (0 tokens left past the
// last chunk)
template <bool VARLEN>
__device__ __forceinline__ void chunk_tokens(const Problem &p, uint32_t gc, int64_t &tok0, int64_t &rem)
{
    if (VARLEN) {
        const longlong2 ci = p.chunk_info[gc];
        tok0 = ci.x;
        rem = ci.y;
    } else {
        const uint32_t nch = (uint32_t)p.nch_fixed, n = gc / nch;
        const int64_t c = p.ch_base + (int64_t)(gc - n * nch);   // chunk index within sequence n
        tok0 = (int64_t)n * p.T + c * CH;
        rem = p.T - c * CH;
    }
}

// NEUMANN: the measurement variant that forms (I + A)^-1 as the fp16 Neumann-series product (the guancyxx.cn
// FlashKDA article, section 2.3) instead of the blocked fp32 substitution.
template <bool VARLEN, bool NEUMANN>
__global__ void __launch_bounds__(PREP_THREADS, 2) kda_prep_kernel(const Problem p, uint32_t n_items)
{
    extern __shared__ __align__(128) unsigned char sm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.H;
    float *rq = reinterpret_cast<float *>(sm + OFF_RQ);
    float *rk = reinterpret_cast<float *>(sm + OFF_RK);
    float *bt = reinterpret_cast<float *>(sm + OFF_BT);
    const uint32_t mbarA = smem_u32(sm + OFF_MISC), mbarD = smem_u32(sm + OFF_MISC + 16);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_MISC + 8);
    bool hung = false;

    // -------- once per CTA: the Akk / Aqk accumulator columns and the tensor-core mbarrier (two phases per item)
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        tc_fence_before();
    }
    if (tid == 32) {
        mbar_init(mbarA, 1);
        mbar_init(mbarD, 1);
        mbar_fence_init();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t s_ops = smem_u32(sm + OFF_OPS);

    // -------- the items of this CTA: blockIdx.x, + gridDim.x, ... (every item's work is the same)
#pragma unroll 1
    for (uint32_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    const uint32_t gc = item / (uint32_t)H;
    const int h = (int)(item - gc * (uint32_t)H);

    // -------- this item's chunk: first token tok0 and L valid tokens
    int64_t tok0, rem;
    chunk_tokens<VARLEN>(p, gc, tok0, rem);   // the table has an entry for every launched item
    if (VARLEN && rem <= 0)
        continue;   // past the last chunk (the same for every thread)
    const int L = (int)(rem < CH ? rem : CH);
    unsigned char *slot = p.slots + (size_t)item * SLOT_BYTES;

    // -------- phase 0: the chunk's q, k, g rows into the staging tiles (cp.async, 512 contiguous bytes per
    // warp instruction; rows past the end zero-filled), the beta and gate parameters into registers
#pragma unroll
    for (int m = 0; m < (3 * CH * 16) / PREP_THREADS; ++m) {
        const int idx = tid + m * PREP_THREADS, which = idx >> 10, t = (idx >> 4) & (CH - 1), c16 = idx & 15;
        const __nv_bfloat16 *base = which == 0 ? p.q : which == 1 ? p.k : p.g;
        const bool valid = t < L;
        cp_async16(smem_u32(sm + OFF_STG + which * (CH * D * 2) + stg_off(t, c16)),
                   base + ((size_t)(tok0 + (valid ? t : 0)) * H + h) * D + c16 * 8, valid);
    }
    cp_async_commit();
    // lane roles in the gate pass: sub-block sb (16 tokens), run half hh (8 tokens of it), channel pair cpl of
    // the warp's 8 channels in each pass; the thread's tokens are t0 .. t0 + 7
    const int sb = lane >> 3, hh = (lane >> 2) & 1, cpl = lane & 3;
    const int t0 = 16 * sb + 8 * hh;
    const __nv_bfloat16 bval = tid < L ? p.beta[(tok0 + (tid < L ? tid : 0)) * H + h] : __float2bfloat16(0.f);
    const float alog = p.A_log[h];
    const float2 dtb0 = *reinterpret_cast<const float2 *>(p.dt_bias + (size_t)h * D + 8 * warp + 2 * cpl);
    const float2 dtb1 = *reinterpret_cast<const float2 *>(p.dt_bias + (size_t)h * D + 64 + 8 * warp + 2 * cpl);

    // rows of this CTA's next item: q, k, g and v into L2 (two 128-byte lines per token and tensor), so that its
    // first loads hit L2
    if (p.prep_pf > 0 && item + gridDim.x < n_items) {
        const uint32_t pit = item + gridDim.x, pgc = pit / (uint32_t)H;
        const int ph = (int)(pit - pgc * (uint32_t)H);
        int64_t ptok0, prem;
        chunk_tokens<VARLEN>(p, pgc, ptok0, prem);
        {   // (varlen: 0 tokens left past the last chunk)
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int li = tid + m * PREP_THREADS, which = li >> 7, t = (li >> 1) & (CH - 1);
                if (t < prem) {
                    const __nv_bfloat16 *base = which == 0 ? p.q : which == 1 ? p.k : which == 2 ? p.g : p.v;
                    prefetch_l2(base + ((size_t)(ptok0 + t) * H + ph) * D + (li & 1) * 64);
                }
            }
#if KDA_PREP_PF_BETA
            // beta of the chunk for every head (contiguous, shared by the chunk's CTAs): by its first head
            if (ph == 0) {
                const int64_t nb = (prem < CH ? prem : CH) * H * 2;   // bytes
                for (int64_t o = (int64_t)tid * 128; o < nb; o += (int64_t)PREP_THREADS * 128)
                    prefetch_l2(reinterpret_cast<const unsigned char *>(p.beta + (size_t)ptok0 * H) + o);
            }
#endif
        }
    }
    if (tid < CH)
        bt[tid] = tid < L ? sigmoid_fast(__bfloat162float(bval)) : 0.f;
    const float eA = expf(alog);
    cp_async_wait_all();
    if (tid == 0)
        bulk_wait_read_all();   // the previous item's W / U0^T copies have read K^.Gamma / V
    __syncthreads();
    // this thread's q, k, g words: tokens t0 + j, channels 64 ps + 8 warp + 2 cpl + {0, 1} (bf16 pairs)
    uint32_t qw[2][8], kw[2][8], gw[2][8];
#pragma unroll
    for (int ps = 0; ps < 2; ++ps)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int o = OFF_STG + stg_off(t0 + j, 8 * ps + warp) + 4 * cpl;
            qw[ps][j] = *reinterpret_cast<const uint32_t *>(sm + o);
            kw[ps][j] = *reinterpret_cast<const uint32_t *>(sm + o + CH * D * 2);
            gw[ps][j] = *reinterpret_cast<const uint32_t *>(sm + o + 2 * CH * D * 2);
        }

    // -------- phase 1: row norms of q and k (partial sums over the thread's 4 channels, then over the
    //          warp's 4 channel pairs by shuffles, then over the 8 warps in shared memory)
    {
        float *part = reinterpret_cast<float *>(sm + OFF_PART);   // below the staging tiles
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int ps = 0; ps < 2; ++ps) {
                const float q0 = bf16_lo(qw[ps][j]), q1 = bf16_hi(qw[ps][j]);
                const float k0 = bf16_lo(kw[ps][j]), k1 = bf16_hi(kw[ps][j]);
                sq = fmaf(q0, q0, fmaf(q1, q1, sq));
                sk = fmaf(k0, k0, fmaf(k1, k1, sk));
            }
            sq += __shfl_xor_sync(0xffffffffu, sq, 1);
            sk += __shfl_xor_sync(0xffffffffu, sk, 1);
            sq += __shfl_xor_sync(0xffffffffu, sq, 2);
            sk += __shfl_xor_sync(0xffffffffu, sk, 2);
            if (cpl == 0) {
                part[(warp * 2) * CH + t0 + j] = sq;
                part[(warp * 2 + 1) * CH + t0 + j] = sk;
            }
        }
        __syncthreads();
        if (tid < 2 * CH) {
            const int t = tid & (CH - 1), which = tid >> 6;
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w)
                s += part[(w * 2 + which) * CH + t];
            const float r = rsqrtf(s + 1e-6f);
            reinterpret_cast<float2 *>(which ? rk : rq)[norm_slot(t)] = make_float2(r, r);
        }
        __syncthreads();
    }
    tc_fence_after();

    // -------- phase 2: gate, decay factors and every per-token operand, in two passes of 64 channels; each
    //          pass fills the Akk / Aqk operand tiles for its channels, then the tensor cores accumulate them.
    //          Per channel the thread walks its 8 tokens in order: the log2-decay a = lb log2(e) sigmoid(.)
    //          is summed serially (G, inclusive, from the start of the run), then shuffles give the run and
    //          sub-block offsets.  Every factor below is an exponential of a difference of these sums.
    {
        // sigmoid(eA (g + dt)) = 1 / (1 + 2^(g gz + gz dt))
        const float gz = -eA * LOG2E;
        const f2 gz2 = f2_pack(gz, gz), lb2 = f2_pack(p.lb_log2e, p.lb_log2e);
        // 1 / |q_t|, 1 / |k_t| of the thread's tokens, stored twice over (as the pair multiplier)
        const f2 *rq2 = reinterpret_cast<const f2 *>(rq) + norm_slot(t0), *rk2 = reinterpret_cast<const f2 *>(rk) + norm_slot(t0);
        const bool first_half = sb < 2, anchor_sb = (sb & 1) == 0;
#pragma unroll
        for (int ps = 0; ps < 2; ++ps) {
            const int c0 = 64 * ps + 8 * warp + 2 * cpl;     // this thread's channels c0, c0 + 1
            const int kk = 8 * warp + 2 * cpl;               // their index in the pass's operand tiles
            const float2 dtb = ps ? dtb1 : dtb0;
            const f2 gd2 = f2_pack(gz * dtb.x, gz * dtb.y);
            // log2-decay per token, summed along the run (past the end of a partial chunk: no decay)
            f2 G[8];
            f2 acc = f2_pack(0.f, 0.f);
            if (L == CH) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const f2 e = f2_add(f2_ex2(f2_fma(f2_bf16x2(gw[ps][j]), gz2, gd2)), f2_pack(1.f, 1.f));
                    acc = f2_add(acc, f2_mul(f2_pack(rcp_approx(f2_lo(e)), rcp_approx(f2_hi(e))), lb2));
                    G[j] = acc;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const f2 e = f2_add(f2_ex2(f2_fma(f2_bf16x2(gw[ps][j]), gz2, gd2)), f2_pack(1.f, 1.f));
                    const f2 a = f2_mul(f2_pack(rcp_approx(f2_lo(e)), rcp_approx(f2_hi(e))), lb2);
                    if (t0 + j < L)
                        acc = f2_add(acc, a);
                    G[j] = acc;
                }
            }
            // the second run of each sub-block adds the first run's total; Tot = the sub-block's total
            const f2 prev = f2_pack(__shfl_xor_sync(0xffffffffu, f2_lo(acc), 4), __shfl_xor_sync(0xffffffffu, f2_hi(acc), 4));
            const f2 tot = hh ? f2_add(prev, acc) : f2_add(acc, prev);   // the same sum, in the same order, in both lanes
            if (hh) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    G[j] = f2_add(prev, G[j]);
            }
            // the four sub-block totals of these channels
            f2 T[4];
#pragma unroll
            for (int b = 0; b < 4; ++b)
                T[b] = f2_pack(__shfl_sync(0xffffffffu, f2_lo(tot), 8 * b + (lane & 7)),
                               __shfl_sync(0xffffffffu, f2_hi(tot), 8 * b + (lane & 7)));
            // Anchors: the end of sub-block 0 (token 15) for the first half, of sub-block 2 (token 47) for the
            // second.  Every factor formed below is either at most 1 (and may underflow only where its true value
            // is below fp32 range) or lies within 16 tokens of an anchor (within 2^+-115.5 for lower_bound >= -5).
            const f2 e2 = f2_add(f2_add(T[0], T[1]), T[2]);
            const f2 e3 = f2_add(e2, T[3]);
            const f2 zero2 = f2_pack(0.f, 0.f), one2 = f2_pack(1.f, 1.f);
            const f2 cq = f2_ex2(first_half ? T[0] : e2);  // Gamma_anchor: Q~ = q^ L cq, K^.Gamma = k^ L cq
            // per-lane constants of the sub-block's role (one per pass, so the token loop has no selects):
            //   gr = G - toff = log2 (Gamma_t / Gamma_anchor);  Rs = 2^(rbase - gr) = Gamma_end(sb) / Gamma_t <= 1;
            //   R = Gamma_anchor / Gamma_t = Rs rmul;  K~ = k^ Rs ks;  the B rows of the second anchor: k^ Rs r1m
            const f2 toff = anchor_sb ? tot : zero2, rbase = anchor_sb ? zero2 : tot;
            const f2 rmul = anchor_sb ? one2 : f2_ex2(f2_sub(zero2, tot));
            const f2 ks = f2_ex2(sb == 0 ? f2_add(f2_add(T[1], T[2]), T[3]) : sb == 1 ? f2_add(T[2], T[3])
                                 : sb == 2 ? T[3] : zero2);
            const f2 r1m = first_half ? f2_ex2(sb == 0 ? f2_add(T[1], T[2]) : T[2]) : rmul;
            if (sb == 3 && hh == 1)
                *reinterpret_cast<float2 *>(slot + SLOT_GC + c0 * 4) = make_float2(ex2_approx(f2_lo(e3)), ex2_approx(f2_hi(e3)));
            // the previous pass's tensor-core product has read the operand tiles
            if (ps == 1 && !mbar_wait(mbarA, 0, p.wait_polls))
                hung = true;
            const int co = (kk >> 2) * OPS_LBO + (kk & 3) * 4;
            unsigned char *const opsA = sm + OFF_OPS + OPS_A + co, *const opsB = sm + OFF_OPS + OPS_B + co;
            uint32_t qt[8], ktp[8];   // Q~ and K~ of tokens t0 + j (fp16 pairs of the two channels)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int t = t0 + j;
                const f2 gr = f2_sub(G[j], toff);
                const f2 Lf = f2_ex2(gr), Rs = f2_ex2(f2_sub(rbase, gr));
                const f2 qh = f2_mul(f2_bf16x2(qw[ps][j]), rq2[j]);
                const f2 kh = f2_mul(f2_bf16x2(kw[ps][j]), rk2[j]);
                const f2 kL = f2_mul(kh, Lf), qL = f2_mul(qh, Lf), kS = f2_mul(kh, Rs);
                const f2 kR = f2_mul(kS, rmul);
                const int ra = (t >> 5) * 64 + (t & 31);
                *reinterpret_cast<uint2 *>(opsA + ((ra >> 3) * OPS_SBO) + ((ra & 7) << 4)) = u2_tf32r(kL);
                *reinterpret_cast<uint2 *>(opsA + (((ra + 32) >> 3) * OPS_SBO) + ((ra & 7) << 4)) = u2_tf32r(qL);
                *reinterpret_cast<uint2 *>(opsB + (((32 + t) >> 3) * OPS_SBO) + ((t & 7) << 4)) = u2_tf32r(f2_mul(kS, r1m));
                if (first_half)
                    *reinterpret_cast<uint2 *>(opsB + ((t >> 3) * OPS_SBO) + ((t & 7) << 4)) = u2_tf32r(kR);
                *reinterpret_cast<uint32_t *>(sm + OFF_KG + kg_off(t, c0)) = half2_of(f2_mul(kL, cq));
                qt[j] = half2_of(f2_mul(qL, cq));
                ktp[j] = half2_of(f2_mul(kS, ks));
            }
            // K~ (slot rows = key channels c0, c0 + 1; 8 tokens per 16-byte core row): rows c0 and c0 + 1 of
            // tokens t0 .. t0 + 7 are 32 contiguous bytes
            {
                uint32_t r0[4], r1[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    r0[m] = __byte_perm(ktp[2 * m], ktp[2 * m + 1], 0x5410);
                    r1[m] = __byte_perm(ktp[2 * m], ktp[2 * m + 1], 0x7632);
                }
                st_global_v8(slot + ka_off(CH + c0, t0), r0[0], r0[1], r0[2], r0[3], r1[0], r1[1], r1[2], r1[3]);
            }
            // Q~ (slot rows = tokens, 8 channels per 16-byte core row): the four lanes of a run hold the four
            // channel pairs of rows t0 .. t0 + 7; a two-step butterfly over lanes ^2 and ^1 leaves rows
            // t0 + 2 cpl and t0 + 2 cpl + 1 (all four pairs, 32 contiguous bytes) in lane cpl
            {
                const bool b = (cpl >> 1) & 1, a = cpl & 1;
                uint32_t kp[4], rv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t snd = b ? qt[i] : qt[4 + i];
                    kp[i] = b ? qt[4 + i] : qt[i];
                    rv[i] = __shfl_xor_sync(0xffffffffu, snd, 2);
                }
                // rows 4 b + i now: own pair (kp[i]) and pair cpl ^ 2 (rv[i])
                uint32_t own[2][2], got[2][2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const uint32_t s0 = a ? kp[e] : kp[2 + e], s1 = a ? rv[e] : rv[2 + e];
                    own[e][0] = a ? kp[2 + e] : kp[e];
                    own[e][1] = a ? rv[2 + e] : rv[e];
                    got[e][0] = __shfl_xor_sync(0xffffffffu, s0, 1);
                    got[e][1] = __shfl_xor_sync(0xffffffffu, s1, 1);
                }
                // row t0 + 2 cpl + e, pair p: p ^ cpl = 0 own, 1 partner's own, 2 own's ^2, 3 partner's ^2
                uint32_t y[2][4];
#pragma unroll
                for (int e = 0; e < 2; ++e)
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp) {
                        const int d = pp ^ cpl;
                        y[e][pp] = (d & 2) ? ((d & 1) ? got[e][1] : own[e][1]) : ((d & 1) ? got[e][0] : own[e][0]);
                    }
                st_global_v8(slot + qw_off(CH + t0 + 2 * cpl, 64 * ps + 8 * warp), y[0][0], y[0][1], y[0][2], y[0][3],
                             y[1][0], y[1][1], y[1][2], y[1][3]);
            }
            // this half of the channels: [Akk | Aqk] (+)= A B^T on the tensor cores
            fence_async_smem();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_tf32_ss(tbase, umma_desc(s_ops + OPS_A + s * 2 * OPS_LBO, OPS_LBO, OPS_SBO),
                                umma_desc(s_ops + OPS_B + s * 2 * OPS_LBO, OPS_LBO, OPS_SBO), idesc_tf32(128, 96),
                                ps > 0 || s > 0);
                umma_commit(mbarA);
            }
        }
    }

    // v rows (bf16) for the WY products: requested after the gate pass so that they do not compete
    // with q, k, g; the readout and the inverse hide their latency
#pragma unroll
    for (int m = 0; m < (CH * 16) / PREP_THREADS; ++m) {
        const int idx = tid + m * PREP_THREADS, r = idx >> 4, c16 = idx & 15;
        const bool valid = r < L;
        const __nv_bfloat16 *src = p.v + ((size_t)(tok0 + (valid ? r : 0)) * H + h) * D + c16 * 8;
        cp_async16(smem_u32(sm + OFF_V + h128(r, c16 * 8)), src, valid);
    }
    cp_async_commit();
    // -------- phase 3: Akk / Aqk out of tensor memory.  Lanes 0..31 / 32..63: Akk / Aqk rows 0..31
    //          (columns 0..31 = tokens 0..31); lanes 64..95 / 96..127: rows 32..63 (columns 32..95 =
    //          tokens 0..63).  Aqk (causal) goes to the slot, b_i Akk (strictly lower) to shared memory.
    if (!mbar_wait(mbarA, 1, p.wait_polls))
        hung = true;
    tc_fence_after();
    {
        const int q4 = warp & 3, hw = warp >> 2;
        const uint32_t tl = tbase + ((uint32_t)(q4 * 32) << 16);
        float *Akk = reinterpret_cast<float *>(sm + OFF_AKK);
        if (q4 < 2) {
            const int i = lane, j0 = 16 * hw;
            uint32_t u[16];
            tmem_ld16(tl + j0, u);
            if (q4 == 0) {
                const float bi = bt[i];
#pragma unroll
                for (int e = 0; e < 16; e += 4) {
                    float x[4];
#pragma unroll
                    for (int f = 0; f < 4; ++f)
                        x[f] = j0 + e + f < i ? bi * __uint_as_float(u[e + f]) : 0.f;
                    *reinterpret_cast<float4 *>(Akk + i * PA + j0 + e) = make_float4(x[0], x[1], x[2], x[3]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; e += 8) {
                    uint32_t w[4];
#pragma unroll
                    for (int f = 0; f < 4; ++f) {
                        const int j = j0 + e + 2 * f;
                        w[f] = pack_half2(j <= i ? __uint_as_float(u[e + 2 * f]) : 0.f,
                                          j + 1 <= i ? __uint_as_float(u[e + 2 * f + 1]) : 0.f);
                    }
                    *reinterpret_cast<uint4 *>(sm + OFF_AQS + ka_off(i, j0 + e) - SLOT_KA) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                // columns 32..63 of rows 0..31 are zero
                *reinterpret_cast<uint4 *>(sm + OFF_AQS + ka_off(i, 32 + j0) - SLOT_KA) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(sm + OFF_AQS + ka_off(i, 40 + j0) - SLOT_KA) = make_uint4(0u, 0u, 0u, 0u);
            }
        } else {
            const int i = 32 + lane, j0 = 32 * hw;
            uint32_t u[32];
            tmem_ld32(tl + 32 + j0, u);
            if (q4 == 2) {
                const float bi = bt[i];
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    float x[4];
#pragma unroll
                    for (int f = 0; f < 4; ++f)
                        x[f] = j0 + e + f < i ? bi * __uint_as_float(u[e + f]) : 0.f;
                    *reinterpret_cast<float4 *>(Akk + i * PA + j0 + e) = make_float4(x[0], x[1], x[2], x[3]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    uint32_t w[4];
#pragma unroll
                    for (int f = 0; f < 4; ++f) {
                        const int j = j0 + e + 2 * f;
                        w[f] = pack_half2(j <= i ? __uint_as_float(u[e + 2 * f]) : 0.f,
                                          j + 1 <= i ? __uint_as_float(u[e + 2 * f + 1]) : 0.f);
                    }
                    *reinterpret_cast<uint4 *>(sm + OFF_AQS + ka_off(i, j0 + e) - SLOT_KA) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
    }
    tc_fence_before();
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {   // Aqk rows of the slot: one bulk copy
        bulk_s2g(slot + SLOT_KA, smem_u32(sm + OFF_AQS), 64 * CH * 2);
        bulk_commit();
    }

    if (NEUMANN) {
        // -------- phase 4 (variant): T = (I + A)^-1 = (I + B)(I + B^2)(I + B^4)(I + B^8)(I + B^16)(I + B^32) with
        //          B = -A (strictly lower, so B^64 = 0): five squarings and five products P += P B^(2^k), fp16
        //          operands and fp32 accumulation, then T' = T diag(b) in fp16
        const float *Akk = reinterpret_cast<const float *>(sm + OFF_AKK);
        unsigned char *bufs[4] = {sm + OFF_TM, sm + OFF_TM + CH * CH * 2, sm, sm + CH * CH * 2};
        {
            const int i = tid >> 2, j0 = (tid & 3) * 16;
            uint32_t bw[8], pw[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                // the strictly lower part only: the readout leaves the block above rows 0..31 unwritten
                const int j = j0 + 2 * e;
                const float a0 = j < i ? -Akk[i * PA + j] : 0.f, a1 = j + 1 < i ? -Akk[i * PA + j + 1] : 0.f;
                bw[e] = pack_half2(a0, a1);
                pw[e] = pack_half2(a0 + (i == j0 + 2 * e ? 1.f : 0.f), a1 + (i == j0 + 2 * e + 1 ? 1.f : 0.f));
            }
            __syncthreads();   // every thread has read its part of Akk: buffers 2 and 3 may overwrite it
#pragma unroll
            for (int e = 0; e < 8; e += 4) {
                *reinterpret_cast<uint4 *>(bufs[0] + h64(i, j0 + 2 * e)) = make_uint4(bw[e], bw[e + 1], bw[e + 2], bw[e + 3]);
                *reinterpret_cast<uint4 *>(bufs[1] + h64(i, j0 + 2 * e)) = make_uint4(pw[e], pw[e + 1], pw[e + 2], pw[e + 3]);
            }
        }
        __syncthreads();
        int ib = 0, ip = 1, in_ = 2, ip2 = 3;   // B^(2^(k-1)), P, B^(2^k), next P
#pragma unroll 1
        for (int k = 0; k < 5; ++k) {
            mm64_f16(smem_u32(bufs[ib]), smem_u32(bufs[ib]), nullptr, bufs[in_], warp, lane);
            __syncthreads();
            mm64_f16(smem_u32(bufs[ip]), smem_u32(bufs[in_]), bufs[ip], bufs[ip2], warp, lane);
            __syncthreads();
            const int ob = ib, op = ip;
            ib = in_;
            ip = ip2;
            in_ = ob;
            ip2 = op;
        }
        {
            const int i = tid >> 2, j0 = (tid & 3) * 16;
            unsigned char *tp = sm + OFF_TP;
#pragma unroll
            for (int e = 0; e < 16; e += 8) {
                const uint4 w = *reinterpret_cast<const uint4 *>(bufs[ip] + h64(i, j0 + e));
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                uint32_t o[4];
#pragma unroll
                for (int f = 0; f < 4; ++f) {
                    const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&ww[f]));
                    o[f] = pack_half2(v.x * bt[j0 + e + 2 * f], v.y * bt[j0 + e + 2 * f + 1]);
                }
                *reinterpret_cast<uint4 *>(tp + h64(i, j0 + e)) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    } else
    // -------- phase 4: Tm = (I + Akk)^-1 by 16-token blocks: fp32 forward substitution on the
    //          diagonal blocks, then the two 32-token halves' off-diagonal blocks
    //          t_{1,0} = -t_{1,1} A_{1,0} t_{0,0}, t_{3,2} = -t_{3,3} A_{3,2} t_{2,2}, then the lower-left
    //          32 x 32 block T21 = -T2 A21 T1 of the whole chunk (T1, T2 the halves' inverses), on fp16
    //          mma.sync with fp32 accumulation.  Every block writer also stores its part of
    //          T' = Tm diag(b) in fp16 for the WY products (blocks above the diagonal are never read).
    {
        const float *Akk = reinterpret_cast<const float *>(sm + OFF_AKK);
        float *Tm = reinterpret_cast<float *>(sm + OFF_TM);
        unsigned char *tp = sm + OFF_TP;
        if (warp < NSB && lane < SB) {
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
                Tm[(b * SB + i) * PA + b * SB + j] = x[i];
                *reinterpret_cast<__half *>(tp + h64(b * SB + i, b * SB + j)) = __float2half_rn(x[i] * bj);
            }
        }
        __syncthreads();
        const int gq = lane >> 2, t4 = lane & 3;
        float *Zw = reinterpret_cast<float *>(sm + OFF_ZW) + warp * 128;   // [16][8]
        // A operand (16 x 16 block at rows r0, columns k0) of an fp32 [64][PA] matrix, as fp16
        auto frag_a = [&](const float *M, int r0, int k0, uint32_t (&f)[4]) {
            const float2 a0 = *reinterpret_cast<const float2 *>(M + (r0 + gq) * PA + k0 + 2 * t4);
            const float2 a1 = *reinterpret_cast<const float2 *>(M + (r0 + gq + 8) * PA + k0 + 2 * t4);
            const float2 a2 = *reinterpret_cast<const float2 *>(M + (r0 + gq) * PA + k0 + 2 * t4 + 8);
            const float2 a3 = *reinterpret_cast<const float2 *>(M + (r0 + gq + 8) * PA + k0 + 2 * t4 + 8);
            f[0] = pack_half2(a0.x, a0.y);
            f[1] = pack_half2(a1.x, a1.y);
            f[2] = pack_half2(a2.x, a2.y);
            f[3] = pack_half2(a3.x, a3.y);
        };
        // z += A_{m, k} Tm_{k, n-tile}: rows m0 .. + 15, Tm rows k0 .. + 15, column cn of this lane
        auto acc_az = [&](float (&z)[4], int m0, int k0, int cn) {
            uint32_t af[4];
            frag_a(Akk, m0, k0, af);
            const uint32_t b0 = pack_half2(Tm[(k0 + 2 * t4) * PA + cn], Tm[(k0 + 2 * t4 + 1) * PA + cn]);
            const uint32_t b1 = pack_half2(Tm[(k0 + 2 * t4 + 8) * PA + cn], Tm[(k0 + 2 * t4 + 9) * PA + cn]);
            mma_f16(z, af, b0, b1);
        };
        // tt += Tm_{r0.., c0..} Z, with Z (16 x 8, this warp's fragment z) through the warp's scratch
        auto acc_tz = [&](float (&tt)[4], int r0, int c0t, const float (&z)[4]) {
            Zw[gq * 8 + 2 * t4] = z[0];
            Zw[gq * 8 + 2 * t4 + 1] = z[1];
            Zw[(gq + 8) * 8 + 2 * t4] = z[2];
            Zw[(gq + 8) * 8 + 2 * t4 + 1] = z[3];
            __syncwarp();
            uint32_t df[4];
            frag_a(Tm, r0, c0t, df);
            const uint32_t zb0 = pack_half2(Zw[(2 * t4) * 8 + gq], Zw[(2 * t4 + 1) * 8 + gq]);
            const uint32_t zb1 = pack_half2(Zw[(2 * t4 + 8) * 8 + gq], Zw[(2 * t4 + 9) * 8 + gq]);
            mma_f16(tt, df, zb0, zb1);
            __syncwarp();   // the scratch is free again
        };
        // -tt -> Tm block (rows r0.., columns cc = n-tile column base + 2 t4) and T'
        auto put = [&](int r0, int cc, const float (&tt)[4]) {
            *reinterpret_cast<float2 *>(Tm + (r0 + gq) * PA + cc) = make_float2(-tt[0], -tt[1]);
            *reinterpret_cast<float2 *>(Tm + (r0 + gq + 8) * PA + cc) = make_float2(-tt[2], -tt[3]);
            const float b0 = bt[cc], b1 = bt[cc + 1];
            *reinterpret_cast<uint32_t *>(tp + h64(r0 + gq, cc)) = pack_half2(-tt[0] * b0, -tt[1] * b1);
            *reinterpret_cast<uint32_t *>(tp + h64(r0 + gq + 8, cc)) = pack_half2(-tt[2] * b0, -tt[3] * b1);
        };
        // level A: t_{1,0} and t_{3,2} (warps 0..3: block, n-tile)
        if (warp < 4) {
            const int bj = (warp >> 1) * 2, bi = bj + 1, nt = warp & 1;
            float z[4] = {0.f, 0.f, 0.f, 0.f}, tt[4] = {0.f, 0.f, 0.f, 0.f};
            acc_az(z, bi * SB, bj * SB, bj * SB + nt * 8 + gq);
            acc_tz(tt, bi * SB, bi * SB, z);
            put(bi * SB, bj * SB + nt * 8 + 2 * t4, tt);
        }
        __syncthreads();
        // level B: T21 blocks (bi, bj), bi in {2, 3}, bj in {0, 1} (warps: bi, bj, n-tile):
        //   Z_{m,bj} = sum_{k=bj..1} A_{m,k} t_{k,bj},  t_{bi,bj} = -sum_{m=2..bi} t_{bi,m} Z_{m,bj}
        {
            const int bi = 2 + (warp >> 2), bj = (warp >> 1) & 1, nt = warp & 1;
            const int cn = bj * SB + nt * 8 + gq;
            float tt[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m = 2; m < 4; ++m) {
                if (m > bi)
                    break;
                float z[4] = {0.f, 0.f, 0.f, 0.f};
                for (int k = bj; k < 2; ++k)
                    acc_az(z, m * SB, k * SB, cn);
                acc_tz(tt, bi * SB, m * SB, z);
            }
            put(bi * SB, bj * SB + nt * 8 + 2 * t4, tt);
        }
    }
    cp_async_wait_all();
    __syncthreads();

    // -------- phase 5: W = T' (K^.Gamma) and U0^T = V^T T'^T (fp16 mma.sync), to the slot
    {
        const uint32_t s_tp = smem_u32(sm + OFF_TP), s_kg = smem_u32(sm + OFF_KG), s_v = smem_u32(sm + OFF_V);
        const int gq = lane >> 2, t4 = lane & 3;
        const int lr = lane & 7, lsel = lane >> 3;   // ldmatrix: row within a matrix, matrix index
        // W (channels of n-tiles 2 warp, 2 warp + 1, all rows t) and U0^T (value rows 16 warp .. + 15, all tokens)
        // together: T' is block lower triangular, so k-step ks needs its blocks (mt, ks), mt >= ks, only, and each
        // block's A fragment of W's product is also the B fragment of U0^T's (T'^T) for the tokens of m-tile mt
        float accw[4][2][4], accu[8][4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int a = 0; a < 2; ++a)
                accw[m][a][0] = accw[m][a][1] = accw[m][a][2] = accw[m][a][3] = 0.f;
#pragma unroll
        for (int a = 0; a < 8; ++a)
            accu[a][0] = accu[a][1] = accu[a][2] = accu[a][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < CH / 16; ++ks) {
            uint32_t bf[4];   // K^.Gamma rows j of k-step ks, the warp's two n-tiles
            ldsm_x4_t(s_kg + kg_off(ks * 16 + (lsel & 1) * 8 + lr, (2 * warp + (lsel >> 1)) * 8), bf);
            uint32_t vf[4];   // A = V^T: matrices (v 0-7, j 0-7), (v 8-15, j 0-7), (v 0-7, j 8-15), (v 8-15, j 8-15)
            ldsm_x4_t(s_v + h128(ks * 16 + (lsel >> 1) * 8 + lr, warp * 16 + (lsel & 1) * 8), vf);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                vf[e] = bf16x2_to_half2(vf[e]);
#pragma unroll
            for (int mt = ks; mt < 4; ++mt) {
                uint32_t af[4];   // T' block (mt, ks): (t 0-7, j 0-7), (t 8-15, j 0-7), (t 0-7, j 8-15), (t 8-15, j 8-15)
                ldsm_x4(s_tp + h64(mt * 16 + (lsel & 1) * 8 + lr, ks * 16 + (lsel >> 1) * 8), af);
                mma_f16(accw[mt][0], af, bf[0], bf[1]);
                mma_f16(accw[mt][1], af, bf[2], bf[3]);
                mma_f16(accu[2 * mt], vf, af[0], af[2]);       // tokens 16 mt .. + 7
                mma_f16(accu[2 * mt + 1], vf, af[1], af[3]);   // tokens 16 mt + 8 .. + 15
            }
        }
        __syncthreads();   // every warp has read K^.Gamma and V: their tiles take the staging
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int t = mt * 16 + gq + 8 * hh, c = (2 * warp + a) * 8 + 2 * t4;
                    *reinterpret_cast<uint32_t *>(sm + OFF_WS + qw_off(t, c)) =
                        pack_half2(accw[mt][a][2 * hh], accw[mt][a][2 * hh + 1]);
                }
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int vr = warp * 16 + gq + 8 * hh, t = a * 8 + 2 * t4;
                *reinterpret_cast<uint32_t *>(sm + OFF_US + u0_off(vr, t) - SLOT_U0) =
                    pack_half2(accu[a][2 * hh], accu[a][2 * hh + 1]);
            }
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
        // W rows (QW rows 0..63) and U0^T of the slot: bulk copies, left reading while the next item starts.
        // The Aqk copy (this item's older group) has read its staging before the next item's q, k, g land
        // over it; the writes complete before the kernel does.
        bulk_s2g(slot + SLOT_QW, smem_u32(sm + OFF_WS), 64 * D * 2);
        bulk_s2g(slot + SLOT_U0, smem_u32(sm + OFF_US), D * CH * 2);
        bulk_commit();
        bulk_wait_read_but_last();
    }
    // the next item's tensor-core product reuses the accumulator columns this item read out
    tc_fence_before();
    if (__syncthreads_or(hung))
        break;   // a wait gave up: stop, and drain below
    tc_fence_after();
    }

    // -------- release tensor memory; report a bounded wait that gave up.  A wait that gave up may have left
    //          tensor-core work in flight, and the product mbarrier's phase is then no longer known: the thread
    //          that issued every product commits once more to a fresh mbarrier, whose single phase completes
    //          after all of them (awaited with the long limit), before the columns are freed.
    if (hung && tid == 0) {
        umma_commit(mbarD);
        mbar_wait(mbarD, 0);
        atomicOr(&g_kda_prep_error, DEVERR_TIMEOUT);
    }
    if (tid == 0)
        bulk_wait_read_all();   // the last item's copies have read their staging
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(TMEM_COLS));
    }
    // launched early beside a recurrence (a programmatic dependent of it): the grid's last CTA exits only
    // after that recurrence has completed, so work ordered after this kernel is ordered after both (a
    // no-op for a normal launch)
    if (blockIdx.x == gridDim.x - 1)
        asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <bool VARLEN, bool NEUMANN>
cudaError_t launch_prep_t(const Problem &p, int64_t items, bool persistent, bool early, cudaStream_t stream)
{
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev >= 64 || !configured[dev]) {
        err = cudaFuncSetAttribute(kda_prep_kernel<VARLEN, NEUMANN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   PREP_SMEM);
        if (err != cudaSuccess)
            return err;
        if (dev < 64)
            configured[dev] = true;
    }
    static int sms[64] = {};
    int nsm = dev < 64 ? sms[dev] : 0;
    if (nsm == 0) {
        err = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess)
            return err;
        if (dev < 64)
            sms[dev] = nsm;
    }
    Problem q = p;
    q.prep_pf = KDA_PREP_PREFETCH;   // each CTA prefetches its next item's rows into L2
    // persistent: two CTAs per SM (their shared memory), each walking the items blockIdx.x + k gridDim.x;
    // otherwise one CTA per item, so that the SMs come free item by item for a kernel running beside it
    const int64_t cap = persistent ? 2 * (int64_t)nsm : items;
    const int64_t grid = items < cap ? items : cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(PREP_THREADS);
    cfg.dynamicSmemBytes = PREP_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kda_prep_kernel<VARLEN, NEUMANN>, q, (uint32_t)items);
}

}  // namespace

cudaError_t launch_prep(const Problem &p, int64_t max_chunks, cudaStream_t stream, bool persistent, bool early)
{
    const int64_t items = max_chunks * p.H;
    if (items <= 0)
        return cudaSuccess;
    if (items > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    if (p.variant & VARIANT_NEUMANN_INVERSE)
        return p.cu ? launch_prep_t<true, true>(p, items, persistent, early, stream)
                    : launch_prep_t<false, true>(p, items, persistent, early, stream);
    return p.cu ? launch_prep_t<true, false>(p, items, persistent, early, stream)
                : launch_prep_t<false, false>(p, items, persistent, early, stream);
}

size_t prep_smem_bytes() { return PREP_SMEM; }

cudaError_t prep_read_and_clear_error(unsigned int *flag)
{
    unsigned int zero = 0;
    cudaError_t err = cudaMemcpyFromSymbol(flag, g_kda_prep_error, sizeof *flag);
    if (err == cudaSuccess && *flag)
        err = cudaMemcpyToSymbol(g_kda_prep_error, &zero, sizeof zero);
    return err;
}

}  // namespace kda
