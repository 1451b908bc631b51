// KDA recurrence kernel: the head-parallel chunk-wise delta-rule recurrence (the second stage
// of the guancyxx.cn FlashKDA article, section 2.2), one CTA per (sequence, head).
//
// Per 64-token chunk, with the operands the prep kernel left in the chunk's slot:
//   U = U0 - W S,   O = scale (Q~ S + Aqk U),   S <- Diag(Gamma_C) S + K~^T U.
// Everything runs transposed on the 5th-generation tensor cores with the value dimension on the
// 128 tensor-memory lanes (M = 128) and fp32 accumulators:
//   [X^T | O'^T] = S^T [W ; Q~]^T               (A = S^T as fp16 in tensor memory, K = 128)
//   U^T = U0^T - X^T                            (threads; fp16 into tensor memory)
//   [O^T | S^T] += U^T [Aqk ; K~^T]^T           (A = U^T, K = 64; S^T decayed beforehand)
// The fp32 master state S^T never leaves tensor memory; an fp16 copy of it is the A operand of
// the first product.  The slots stream through three shared-memory buffers, each requested two
// chunks ahead; the output of a chunk is transposed (stmatrix) into its consumed slot and stored
// during the next chunk.
//
// Tensor-memory columns: X^T 0..63 | O^T 64..127 | S^T 128..255 | fp16 S^T 256..319 |
// fp16 U^T 320..351 (512 allocated).
#include "kda_device.cuh"
#include "kda_internal.h"

// Error bits of the recurrence kernel (DEVERR_*: a bounded wait expired, a non-finite final state),
// read and cleared by kda_device_status.
__device__ unsigned int g_kda_device_error;

namespace kda {
namespace {

constexpr int RT = 256;                     // threads: warp w reads lanes 32 (w % 4) .. + 31
constexpr int TMEM_COLS = 512;
constexpr int TM_X = 0, TM_O = 64, TM_S = 128, TM_S16 = 256, TM_U16 = 320;
// Three slot buffers: chunk c lives in buffer c % 3.  The slot of chunk c + 2 is requested while chunk c runs, in
// two bulk copies: QW and KA when chunk c starts (chunk c - 1's products, their only readers, are complete), U0^T
// and Gamma_C once chunk c's last product is issued, because the output of chunk c - 1 is staged in that part of
// chunk c - 1's buffer (bf16 [64 t][128 v], 16-byte pieces XOR-swizzled by t % 8) until it is stored.
constexpr int NBUF = 3;
constexpr int SLOT_HEAD = SLOT_U0;          // bytes of the first copy
constexpr int OFF_BAR = NBUF * SLOT_BYTES;
constexpr int RECUR_SMEM = OFF_BAR + 64;    // mbarriers: load 0..2, product X|O, update; tmem slot
static_assert(RECUR_SMEM <= 232448, "shared memory budget");
static_assert(SLOT_BYTES % 128 == 0 && SLOT_HEAD % 16 == 0 && OFF_BAR % 8 == 0, "alignment");
static_assert(SLOT_BYTES - SLOT_HEAD >= CH * D * 2, "output staging fits in U0^T and Gamma_C");
__device__ __forceinline__ int ost_off(int t, int v) { return t * (D * 2) + ((((v >> 3) ^ (t & 7))) << 4) + ((v & 7) << 1); }

// S^T (64 columns, one lane per thread) and O^T (32 columns of the warp's 32 lanes in the mma accumulator
// fragment layout: registers 16 h + 4 k + {0, 1} hold lane 16 h + i / 4 and 16 h + 8 + i / 4 for + {2, 3},
// columns 8 k + 2 (i % 4) + {0, 1}) in one round trip
__device__ __forceinline__ void tmem_ld_s_ofrag(uint32_t taddr_s, uint32_t (&u)[64], uint32_t taddr_o, uint32_t (&o)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
                 "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
                 "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%96];\n"
                 "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79}, [%97];\n"
                 "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%98];\n"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
                   "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]),
                   "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]),
                   "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31]),
                   "=r"(u[32]), "=r"(u[33]), "=r"(u[34]), "=r"(u[35]), "=r"(u[36]), "=r"(u[37]), "=r"(u[38]), "=r"(u[39]),
                   "=r"(u[40]), "=r"(u[41]), "=r"(u[42]), "=r"(u[43]), "=r"(u[44]), "=r"(u[45]), "=r"(u[46]), "=r"(u[47]),
                   "=r"(u[48]), "=r"(u[49]), "=r"(u[50]), "=r"(u[51]), "=r"(u[52]), "=r"(u[53]), "=r"(u[54]), "=r"(u[55]),
                   "=r"(u[56]), "=r"(u[57]), "=r"(u[58]), "=r"(u[59]), "=r"(u[60]), "=r"(u[61]), "=r"(u[62]), "=r"(u[63]),
                   "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]), "=r"(o[4]), "=r"(o[5]), "=r"(o[6]), "=r"(o[7]),
                   "=r"(o[8]), "=r"(o[9]), "=r"(o[10]), "=r"(o[11]), "=r"(o[12]), "=r"(o[13]), "=r"(o[14]), "=r"(o[15]),
                   "=r"(o[16]), "=r"(o[17]), "=r"(o[18]), "=r"(o[19]), "=r"(o[20]), "=r"(o[21]), "=r"(o[22]), "=r"(o[23]),
                   "=r"(o[24]), "=r"(o[25]), "=r"(o[26]), "=r"(o[27]), "=r"(o[28]), "=r"(o[29]), "=r"(o[30]), "=r"(o[31])
                 : "r"(taddr_s), "r"(taddr_o), "r"(taddr_o + (16u << 16)));
}
// 64 columns of this warp's 32 lanes (one value per lane and column), waited for
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&u)[64])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
                 "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
                 "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
                   "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]),
                   "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]),
                   "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31]),
                   "=r"(u[32]), "=r"(u[33]), "=r"(u[34]), "=r"(u[35]), "=r"(u[36]), "=r"(u[37]), "=r"(u[38]), "=r"(u[39]),
                   "=r"(u[40]), "=r"(u[41]), "=r"(u[42]), "=r"(u[43]), "=r"(u[44]), "=r"(u[45]), "=r"(u[46]), "=r"(u[47]),
                   "=r"(u[48]), "=r"(u[49]), "=r"(u[50]), "=r"(u[51]), "=r"(u[52]), "=r"(u[53]), "=r"(u[54]), "=r"(u[55]),
                   "=r"(u[56]), "=r"(u[57]), "=r"(u[58]), "=r"(u[59]), "=r"(u[60]), "=r"(u[61]), "=r"(u[62]), "=r"(u[63])
                 : "r"(taddr));
}
// stmatrix.trans: four 8x8 16-bit matrices from mma-fragment registers, each stored transposed (matrix m:
// rows at the addresses of lanes 8m .. 8m + 7)
__device__ __forceinline__ void stsm_x4_t(uint32_t addr, const uint32_t (&r)[4])
{
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}

// tcgen05.st without the completion wait (tmem_wait_st() before the tensor core or another thread reads the data)
__device__ __forceinline__ void tmem_st64_nw(uint32_t taddr, const uint32_t (&u)[64])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,"
                 "%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
                 "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};"
                 ::"r"(taddr), "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7]),
                    "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]), "r"(u[13]), "r"(u[14]), "r"(u[15]),
                    "r"(u[16]), "r"(u[17]), "r"(u[18]), "r"(u[19]), "r"(u[20]), "r"(u[21]), "r"(u[22]), "r"(u[23]),
                    "r"(u[24]), "r"(u[25]), "r"(u[26]), "r"(u[27]), "r"(u[28]), "r"(u[29]), "r"(u[30]), "r"(u[31]),
                    "r"(u[32]), "r"(u[33]), "r"(u[34]), "r"(u[35]), "r"(u[36]), "r"(u[37]), "r"(u[38]), "r"(u[39]),
                    "r"(u[40]), "r"(u[41]), "r"(u[42]), "r"(u[43]), "r"(u[44]), "r"(u[45]), "r"(u[46]), "r"(u[47]),
                    "r"(u[48]), "r"(u[49]), "r"(u[50]), "r"(u[51]), "r"(u[52]), "r"(u[53]), "r"(u[54]), "r"(u[55]),
                    "r"(u[56]), "r"(u[57]), "r"(u[58]), "r"(u[59]), "r"(u[60]), "r"(u[61]), "r"(u[62]), "r"(u[63]));
}
__device__ __forceinline__ void tmem_st32_nw(uint32_t taddr, const uint32_t (&u)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 ::"r"(taddr), "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7]),
                    "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]), "r"(u[13]), "r"(u[14]), "r"(u[15]),
                    "r"(u[16]), "r"(u[17]), "r"(u[18]), "r"(u[19]), "r"(u[20]), "r"(u[21]), "r"(u[22]), "r"(u[23]),
                    "r"(u[24]), "r"(u[25]), "r"(u[26]), "r"(u[27]), "r"(u[28]), "r"(u[29]), "r"(u[30]), "r"(u[31]));
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// STATE: 0 none, 1 bf16, 2 fp32.  BSTATE: the measurement variant that keeps the state in bf16 between chunks
// (rounded to nearest at each chunk boundary, as the guancyxx.cn FlashKDA article's design does, section 2.3);
// the default keeps the fp32 accumulator as the state.
//
// Fixed length, p.groups > 1 (the chunk-transition scan): CTA (group g, sequence n, head h) runs chunks
// g group_len .. of sequence n from the start state of group g (the initial state for g = 0, else sc_s) and
// stores a final state for the last group only.  COMPOSE > 0: the scan's first level, no outputs: the group's
// chunks map a start state S to M S + B (M = the product of the chunks' Diag(Gamma_C) - K~^T W, B = the state
// reached from S = 0).  Tile 0 runs from S = I with U0 taken as 0 (leaving M), tile 1 from S = 0 (leaving B),
// both stored transposed like a state (sc_a / sc_b).  COMPOSE = 1: one tile per CTA (two CTAs per (group, n,
// h), the tile in the low bit of the CTA index), tensor memory as in the recurrence.  COMPOSE = 2: one CTA per
// (group, n, h) carries both tiles; tensor memory: X^T of tile t at 64 t, S^T at 128 + 128 t, its fp16 copy at
// 384 + 64 t, where U^T (fp16) also goes once the first product has read the copy.
template <int STATE, bool VARLEN, bool BSTATE, int COMPOSE>
__global__ void __launch_bounds__(RT, 1) kda_recur_kernel(const Problem p)
{
    extern __shared__ __align__(128) unsigned char sm[];
    // a kernel launched after this one as its programmatic dependent (the next piece's prep kernel, which
    // reads nothing this kernel writes) may start once every CTA of this grid runs
    asm volatile("griddepcontrol.launch_dependents;");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.H;
    const int ctile = COMPOSE == 1 ? (int)(blockIdx.x & 1u) : 0;   // the tile of a one-tile compose CTA
    const int cta = COMPOSE == 1 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int NH = p.N * H;
    const int grp = VARLEN ? 0 : cta / NH;   // group of the scan (0 without one)
    const int pr = cta - grp * NH;
    const int h = pr % H;
    int n = pr / H;
    if (VARLEN && p.order)
        n = p.order[n];   // longest sequences first
    // the state this CTA starts from and the one it leaves (fp32 in the scan's launches)
    const void *init = p.init;
    void *fin = p.fin;
    if (!VARLEN && grp > 0)
        init = p.sc_s + (size_t)(grp - 1) * NH * D * D;
    if (!VARLEN && grp < p.groups - 1)
        fin = nullptr;
    if (COMPOSE) {
        init = nullptr;
        fin = nullptr;   // sc_a / sc_b per tile
    }
    int64_t bos, len, slot0;
    if (VARLEN) {
        seq_range(p.cu, n, p.N, p.T, bos, len);   // clamped into [0, T]; the plan flags a malformed cu_seqlens
        slot0 = p.chunk_off[n];
        const int64_t usable = usable_chunks(slot0, seq_chunks(len), p.chunk_cap);
        if (usable * CH < len)
            len = usable * CH;   // only a malformed cu_seqlens gets here: chunks past the table are skipped
    } else {
        // chunks cb .. cb + group_len - 1 of the sequence (all of them unless the call runs in pieces or groups)
        const int64_t cb = p.ch_base + (int64_t)grp * p.group_len;
        bos = (int64_t)n * p.T + cb * CH;
        len = p.T - cb * CH < p.group_len * CH ? p.T - cb * CH : p.group_len * CH;
        if (len < 0)
            len = 0;
        slot0 = (int64_t)n * p.nch_fixed + (int64_t)grp * p.group_len;
    }
    const int nch = (int)((len + CH - 1) / CH);

    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_BAR + 40);
    const uint32_t mbarL = smem_u32(sm + OFF_BAR);   // + 8 b: slot of buffer b landed
    const uint32_t mbarQ = smem_u32(sm + OFF_BAR + 24), mbarB = smem_u32(sm + OFF_BAR + 32);
    auto slot_ptr = [&](int c) -> const unsigned char * {
        return p.slots + (size_t)((slot0 + c) * H + h) * SLOT_BYTES;
    };
    auto buf_of = [&](int c) -> unsigned char * { return sm + (c % NBUF) * SLOT_BYTES; };
    // one thread: the first / second part of the slot of chunk c into buffer c % 3 (both complete one phase
    // of that buffer's mbarrier)
    // COMPOSE reads only what the state updates need: W (QW rows 0 .. 63), K~^T (KA rows 64 .. 191), U0^T and
    // Gamma_C
    constexpr int CMP_W = CH * D * 2, CMP_K = D * CH * 2, CMP_KOFF = SLOT_KA + (CH / 8) * KA_SBO;
    constexpr uint32_t tx_bytes = !COMPOSE ? (uint32_t)SLOT_BYTES : (uint32_t)(CMP_W + CMP_K + SLOT_BYTES - SLOT_U0);
    auto issue_head = [&](int c) {
        const uint32_t mb = mbarL + 8 * (c % NBUF);
        mbar_expect_tx(mb, tx_bytes);
        if (COMPOSE) {
            bulk_g2s(smem_u32(buf_of(c) + SLOT_QW), slot_ptr(c) + SLOT_QW, CMP_W, mb);
            bulk_g2s(smem_u32(buf_of(c) + CMP_KOFF), slot_ptr(c) + CMP_KOFF, CMP_K, mb);
        } else {
            bulk_g2s(smem_u32(buf_of(c)), slot_ptr(c), SLOT_HEAD, mb);
        }
    };
    auto issue_tail = [&](int c) {
        fence_async_smem();   // the buffer's generic-proxy readers and writers finished before a barrier
        bulk_g2s(smem_u32(buf_of(c) + SLOT_HEAD), slot_ptr(c) + SLOT_HEAD, SLOT_BYTES - SLOT_HEAD,
                 mbarL + 8 * (c % NBUF));
    };

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        tc_fence_before();
    }
    if (tid == 0) {
        for (int b = 0; b < NBUF; ++b)
            mbar_init(mbarL + 8 * b, 1);
        mbar_init(mbarQ, 1);
        mbar_init(mbarB, 1);
        mbar_fence_init();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    // copies requested so far (the same count in every thread): heads and tails of chunks 0 .. heads - 1 / tails - 1
    int heads = nch < 2 ? nch : 2, tails = heads;
    if (tid == 0)
        for (int k = 0; k < heads; ++k) {
            issue_head(k);
            issue_tail(k);
        }

    const int q4 = warp & 3, half = warp >> 2;
    const int vrow = q4 * 32 + lane;
    const uint32_t trow = tbase + ((uint32_t)(q4 * 32) << 16);
    const size_t srow = ((size_t)n * H + h) * D * D + (size_t)vrow * D + half * 64;

    // tensor-memory columns of tile t (COMPOSE carries two states; otherwise t = 0)
    auto col_x = [](int t) -> uint32_t { return COMPOSE == 2 ? 64u * t : (uint32_t)TM_X; };
    auto col_s = [](int t) -> uint32_t { return COMPOSE == 2 ? 128u + 128u * t : (uint32_t)TM_S; };
    auto col_s16 = [](int t) -> uint32_t { return COMPOSE == 2 ? 384u + 64u * t : (uint32_t)TM_S16; };
    auto col_u16 = [](int t) -> uint32_t { return COMPOSE == 2 ? 384u + 64u * t : (uint32_t)TM_U16; };
    constexpr int TILES = COMPOSE == 2 ? 2 : 1;
    auto tile_of = [&](int t) { return COMPOSE == 2 ? t : ctile; };   // 0: M, 1: B

    // -------- initial state -> S^T (row v, key columns 64 half .. + 63)
#pragma unroll
    for (int t = 0; t < TILES; ++t)
#pragma unroll
    for (int part = 0; part < 2; ++part) {
        uint32_t u[32];
        if (COMPOSE && tile_of(t) == 0) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
                u[e] = half * 64 + 32 * part + e == vrow ? 0x3f800000u : 0u;   // S = I
        } else if (COMPOSE) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
                u[e] = 0u;   // S = 0
        } else if (STATE == 2 && init) {
            const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(init) + srow + 32 * part);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float4 x = src[e];
                u[4 * e] = __float_as_uint(x.x);
                u[4 * e + 1] = __float_as_uint(x.y);
                u[4 * e + 2] = __float_as_uint(x.z);
                u[4 * e + 3] = __float_as_uint(x.w);
            }
        } else if (STATE == 1 && init) {
            const uint4 *src =
                reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(init) + srow + 32 * part);
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
        tmem_st32(trow + col_s(t) + half * 64 + 32 * part, u);
    }
    tc_fence_before();

    // O^T of the chunk just updated -> bf16 staging tile [t][v] (this thread: tokens 32 half .. + 31)
    // o: O^T of this warp's 32 value lanes x tokens 32 half .. + 31 in fragment form (tmem_ld_s_ofrag); each 8 x 8
    // (value, token) block goes to the staging tile transposed by stmatrix
    const int lr = lane & 7, mi = lane >> 3;
    auto write_out = [&](unsigned char *ost, const uint32_t (&o)[32]) {
#pragma unroll
        for (int sh = 0; sh < 2; ++sh)
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                uint32_t f[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(o[16 * sh + 8 * kk + 2 * m]) * p.scale,
                                                                    __uint_as_float(o[16 * sh + 8 * kk + 2 * m + 1]) * p.scale);
                    f[m] = *reinterpret_cast<const uint32_t *>(&b2);
                }
                // matrix m: values q4 32 + 16 sh + 8 (m & 1) .., tokens of column group 2 kk + (m >> 1)
                const int t = half * 32 + 8 * (2 * kk + (mi >> 1)) + lr, v = q4 * 32 + 16 * sh + 8 * (mi & 1);
                stsm_x4_t(smem_u32(ost + ost_off(t, v)), f);
            }
    };
    auto read_out = [&](unsigned char *ost) {
        uint32_t u[64], o[32];
        tmem_ld_s_ofrag(trow + TM_S, u, trow + TM_O + half * 32, o);
        write_out(ost, o);
    };
    auto store_out = [&](const unsigned char *ost, int64_t ptok0, int pL) {
#pragma unroll
        for (int m = 0; m < (CH * 16) / RT; ++m) {
            const int idx = tid + m * RT, r = idx >> 4, c16 = idx & 15;
            if (r < pL)
                *reinterpret_cast<uint4 *>(p.out + ((ptok0 + r) * H + h) * D + c16 * 8) =
                    *reinterpret_cast<const uint4 *>(ost + r * (D * 2) + ((c16 ^ (r & 7)) << 4));
        }
    };

    bool hung = false;
    int nq = 0, nb = 0;   // commits issued on mbarQ / mbarB (same count in every thread)
    int64_t prev_tok0 = 0;
    int prev_L = 0;
    int c = 0;
    for (; c < nch; ++c) {
        const unsigned char *sb = buf_of(c);
        const uint32_t s_buf = smem_u32(sb);
        unsigned char *ost = buf_of(c + NBUF - 1) + SLOT_HEAD;   // staging of chunk c - 1's output
        const int64_t tok0 = bos + (int64_t)c * CH;
        const int64_t rem = len - (int64_t)c * CH;
        const int L = (int)(rem < CH ? rem : CH);

        // the previous update is complete and this chunk's slot has landed (each thread waits; no barrier here: a
        // wait that gave up is reduced over the CTA at P1's barrier, which every thread reaches either way)
        bool ok = true;
        if (c > 0)
            ok = mbar_wait(mbarB, (c - 1) & 1, p.wait_polls);
        ok = ok && mbar_wait(mbarL + 8 * (c % NBUF), (c / NBUF) & 1, p.wait_polls);
        __syncwarp();   // the warp's lanes leave their waits together before the warp-wide tensor-memory loads
        tc_fence_after();

        // ---- P1: fp16 copy of S^T (A operand), S^T <- S^T Diag(Gamma_C), previous output read-out (one
        //      tensor-memory load of S^T and O^T; the stores complete together before the barrier)
        {
            const float *gam = reinterpret_cast<const float *>(sb + SLOT_GC) + half * 64;
#pragma unroll 1
            for (int t = 0; t < TILES; ++t) {
                uint32_t u[64], o[32];
                if (COMPOSE)
                    tmem_ld64(trow + col_s(t) + half * 64, u);
                else
                    tmem_ld_s_ofrag(trow + TM_S + half * 64, u, trow + TM_O + half * 32, o);   // O^T unused at c = 0
                if (BSTATE) {
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        u[e] = __float_as_uint(__bfloat162float(__float2bfloat16_rn(__uint_as_float(u[e]))));
                }
                {
                    uint32_t hv[32];
#pragma unroll
                    for (int m = 0; m < 32; ++m)
                        hv[m] = pack_half2(__uint_as_float(u[2 * m]), __uint_as_float(u[2 * m + 1]));
                    tmem_st32_nw(trow + col_s16(t) + half * 32, hv);
                }
#pragma unroll
                for (int e = 0; e < 64; ++e)
                    u[e] = __float_as_uint(__uint_as_float(u[e]) * gam[e]);
                tmem_st64_nw(trow + col_s(t) + half * 64, u);
                if (!COMPOSE && c > 0)
                    write_out(ost, o);
            }
            tmem_wait_st();
        }
        tc_fence_before();
        if (__syncthreads_or(!ok)) {   // a wait above gave up in some thread
            hung = true;
            break;
        }
        // QW and KA of chunk c + 2 into chunk c - 1's buffer (only chunk c - 1's products, complete, read them), by
        // another warp while the first product is issued
        if (c + 2 < nch) {
            if (tid == 32)
                issue_head(c + 2);
            ++heads;
        }
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < TILES; ++t)
#pragma unroll
                for (int s = 0; s < D / 16; ++s)
                    mma_f16_ts(tbase + col_x(t), tbase + col_s16(t) + 8 * s,
                               umma_desc(s_buf + SLOT_QW + s * 2 * CORE_LBO, CORE_LBO, QW_SBO),
                               idesc_f16(128, COMPOSE ? CH : 128), s > 0);   // [W ; Q~] rows (W only: no outputs)
            umma_commit(mbarQ);
        }
        ++nq;
        if (!COMPOSE && c > 0)
            store_out(ost, prev_tok0, prev_L);

        // ---- P2: U^T = U0^T - X^T as fp16 into tensor memory
        // (no barrier: each thread waits for the product itself; a wait that gave up is reported through the
        // reduction of the next barrier)
        // this thread's U0^T row of the slot (landed with it), read before the wait for the first product
        uint4 u0w[4];
        {
            const unsigned char *u0row = sb + SLOT_U0 + vrow * (CH * 2);
#pragma unroll
            for (int m = 0; m < 4; ++m)
                u0w[m] = *reinterpret_cast<const uint4 *>(u0row + (((half * 4 + m) ^ (vrow & 7)) << 4));
        }
        const bool qok = mbar_wait(mbarQ, c & 1, p.wait_polls);
        tc_fence_after();
#pragma unroll 1
        for (int t = 0; t < TILES; ++t) {
            uint32_t x[32], hv[16];
            tmem_ld32(trow + col_x(t) + half * 32, x);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint4 w = u0w[m];
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&ww[e]));
                    if (COMPOSE && tile_of(t) == 0)
                        f = make_float2(0.f, 0.f);   // the linear part: U = -X
                    hv[4 * m + e] = pack_half2(f.x - __uint_as_float(x[8 * m + 2 * e]),
                                               f.y - __uint_as_float(x[8 * m + 2 * e + 1]));
                }
            }
            // (two-tile compose: over the tile's fp16 state copy, which the completed first product has read)
            tmem_st16(trow + col_u16(t) + half * 16, hv);
        }
        tc_fence_before();
        if (__syncthreads_or(!qok)) {
            hung = true;
            break;
        }
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < CH / 16; ++s)
                if (COMPOSE) {   // the state updates alone: B = the K~^T rows of KA (rows 64 ..)
#pragma unroll
                    for (int t = 0; t < TILES; ++t)
                        mma_f16_ts(tbase + col_s(t), tbase + col_u16(t) + 8 * s,
                                   umma_desc(s_buf + SLOT_KA + (CH / 8) * KA_SBO + s * 2 * CORE_LBO, CORE_LBO, KA_SBO),
                                   idesc_f16(128, D), 1);
                } else
                    mma_f16_ts(tbase + TM_O, tbase + TM_U16 + 8 * s,
                               umma_desc(s_buf + SLOT_KA + s * 2 * CORE_LBO, CORE_LBO, KA_SBO), idesc_f16(128, 64 + D), 1);
            umma_commit(mbarB);
        }
        ++nb;
        // U0^T and Gamma_C of chunk c + 2: chunk c - 1's staged output was stored before the barrier after the
        // first product, and chunk c - 1 read its U0^T and Gamma_C before the barriers of its own chunk
        if (c + 2 < nch) {
            if (tid == 32)
                issue_tail(c + 2);
            ++tails;
        }
        prev_tok0 = tok0;
        prev_L = L;
    }

    if (!hung && nch > 0) {
        const bool ok = mbar_wait(mbarB, (nch - 1) & 1, p.wait_polls);
        if (__syncthreads_or(!ok)) {
            hung = true;
        } else if (!COMPOSE) {
            tc_fence_after();
            read_out(buf_of(nch - 1) + SLOT_HEAD);
            __syncthreads();
            store_out(buf_of(nch - 1) + SLOT_HEAD, prev_tok0, prev_L);
        }
    }

    // -------- final state, release
    if (hung) {
        // let tensor-core work and bulk copies still in flight finish (bounded) before leaving
        if (tid == 0) {
            if (nq > 0)
                mbar_wait(mbarQ, (nq - 1) & 1);
            if (nb > 0)
                mbar_wait(mbarB, (nb - 1) & 1);
            for (int k = c; k < heads; ++k) {
                if (k >= tails)
                    issue_tail(k);   // completes the phase the head's expect_tx opened
                mbar_wait(mbarL + 8 * (k % NBUF), (k / NBUF) & 1);
            }
            atomicOr(&g_kda_device_error, DEVERR_TIMEOUT);
        }
    } else {
        // the final state (stored if requested) and a finiteness check of it: an fp16 tensor-core operand
        // that overflowed (or an inf / NaN input) leaves the fp32 state non-finite from that chunk on
        tc_fence_after();
        bool bad = false;
#pragma unroll 1
        for (int t = 0; t < TILES; ++t)
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            uint32_t u[32];
            tmem_ld32(trow + col_s(t) + half * 64 + 32 * part, u);
#pragma unroll
            for (int e = 0; e < 32; ++e)
                bad |= !(fabsf(__uint_as_float(u[e])) <= 3.402823466e38f);
            if (COMPOSE) {   // M (tile 0) or B (tile 1) of this group
                float4 *dst = reinterpret_cast<float4 *>((tile_of(t) ? p.sc_b : p.sc_a) + (size_t)grp * NH * D * D +
                                                         srow + 32 * part);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    dst[e] = make_float4(__uint_as_float(u[4 * e]), __uint_as_float(u[4 * e + 1]),
                                         __uint_as_float(u[4 * e + 2]), __uint_as_float(u[4 * e + 3]));
            } else if (STATE == 2 && fin) {
                float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(fin) + srow + 32 * part);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    dst[e] = make_float4(__uint_as_float(u[4 * e]), __uint_as_float(u[4 * e + 1]),
                                         __uint_as_float(u[4 * e + 2]), __uint_as_float(u[4 * e + 3]));
            } else if (STATE == 1 && fin) {
                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(fin) + srow + 32 * part);
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
        if (__any_sync(0xffffffffu, bad) && lane == 0)
            atomicOr(&g_kda_device_error, DEVERR_NONFINITE);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(TMEM_COLS));
    }
}

template <int STATE, bool VARLEN, bool BSTATE, int COMPOSE>
cudaError_t launch_recur_t(const Problem &p, int grid, cudaStream_t stream)
{
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev >= 64 || !configured[dev]) {
        err = cudaFuncSetAttribute(kda_recur_kernel<STATE, VARLEN, BSTATE, COMPOSE>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, RECUR_SMEM);
        if (err != cudaSuccess)
            return err;
        if (dev < 64)
            configured[dev] = true;
    }
    if (grid <= 0)
        return cudaSuccess;
    kda_recur_kernel<STATE, VARLEN, BSTATE, COMPOSE><<<grid, RT, RECUR_SMEM, stream>>>(p);
    return cudaGetLastError();
}

template <bool BSTATE>
cudaError_t launch_recur_b(const Problem &p, int state_kind, cudaStream_t stream)
{
    const int grid = p.N * p.H;
    if (p.cu)
        return state_kind == 2 ? launch_recur_t<2, true, BSTATE, 0>(p, grid, stream)
             : state_kind == 1 ? launch_recur_t<1, true, BSTATE, 0>(p, grid, stream)
                               : launch_recur_t<0, true, BSTATE, 0>(p, grid, stream);
    const int fgrid = grid * p.groups;
    return state_kind == 2 ? launch_recur_t<2, false, BSTATE, 0>(p, fgrid, stream)
         : state_kind == 1 ? launch_recur_t<1, false, BSTATE, 0>(p, fgrid, stream)
                           : launch_recur_t<0, false, BSTATE, 0>(p, fgrid, stream);
}

}  // namespace

cudaError_t launch_recur(const Problem &p, int state_kind, cudaStream_t stream)
{
    return (p.variant & VARIANT_BF16_STATE) ? launch_recur_b<true>(p, state_kind, stream)
                                            : launch_recur_b<false>(p, state_kind, stream);
}

cudaError_t launch_compose(const Problem &p, bool two_tiles, cudaStream_t stream)
{
    const int grid = (p.groups - 1) * p.N * p.H;
    return two_tiles ? launch_recur_t<2, false, false, 2>(p, grid, stream)
                     : launch_recur_t<2, false, false, 1>(p, 2 * grid, stream);
}

size_t recur_smem_bytes() { return RECUR_SMEM; }

cudaError_t read_and_clear_device_error(unsigned int *flag)
{
    unsigned int zero = 0;
    cudaError_t err = cudaMemcpyFromSymbol(flag, g_kda_device_error, sizeof *flag);
    if (err == cudaSuccess && *flag)
        err = cudaMemcpyToSymbol(g_kda_device_error, &zero, sizeof zero);
    return err;
}

}  // namespace kda
