// KDA token-recurrent kernel: the per-token gated delta rule (guancyxx.cn FlashKDA article,
// section 一; the argument table of the FlashKDA README mirror, "内核 API") evaluated token by token,
// for decode steps and short prefills, where the chunked path's per-chunk operands cost more than
// the state itself.  No workspace.
//
// Per token t (state S in R^{K x V}, stored transposed [V][K]):
//   S' = Diag(alpha) S,   u = b (v - S'^T k^),   S = S' + k^ u^T,   o = scale S^T q^
// with alpha = exp(lower_bound sigmoid(exp(A_log) (g + dt_bias))), b = sigmoid(beta) and
// k^ = rk k, q^ = rq q (rk, rq the inverse L2 norms); every operand is fp32.
//
// Work item = (sequence, head, half of the values): 64 columns of S, a contiguous 32 KB (fp32) or
// 16 KB (bf16) block of the state tensor.  The grid is persistent (two CTAs per SM); each CTA takes
// items round robin and streams them as a sequence of stages, one stage = up to 8 tokens of one
// item:
//   * token rows (q, k, g, the value half of v), dt_bias[h] and A_log[h] of stage s + 2 arrive by
//     cp.async while stage s runs (three raw slots);
//   * the state block of item i + 2 arrives by one bulk copy (mbarrier, bounded wait) while item i
//     runs (two state slots); at an item's first stage it moves into registers;
//   * a token-parallel pass (one warp per token) computes the inverse norms, b and log2 alpha of the
//     stage's tokens, and a channel-parallel pass accumulates, per key, A_t = the decay from the
//     stage start through token t, giving A_t k^, k^ / A_t and scale A_t q^ in fp32;
//   * the serial loop then runs without barriers on S / A (reset to S at every stage end):
//       p = (S/A)^T (A_t k^),  u = b (v - p),  S/A += (k^ / A_t) u^T,  o = (S/A)^T (scale A_t q^),
//     three packed FMAs per state pair and token.  Within a stage A_t >= 2^(8 lower_bound log2 e)
//     > 2^-58, so S / A stays far inside the fp32 range.
// Thread (value quad vq, key group kg) holds S[64 f + 4 kg + j][4 vq + c] (f < 2, j < 4, c < 4) as
// 16 packed f32x2 registers; the dot products are reduced over the 16 key groups of a value quad
// (lane bits 0..3) by a reduce-scatter of shuffles.
#include "kda_device.cuh"
#include "kda_internal.h"

__device__ unsigned int g_kda_rc_error;   // set when a bounded wait of the token-recurrent kernel gave up

namespace kda {
namespace {

constexpr int RC_THREADS = 256;
constexpr int RC_VALUES = 64;            // values per item
constexpr int RC_L = 8;                  // tokens per stage
constexpr int RC_NRAW = 3;               // raw token slots (prefetch distance 2 stages)
constexpr int RC_NST = 2;                // state slots (prefetch distance 2 items)

// raw slot: bf16 rows of up to RC_L tokens, this item's gate parameters and the stage header
struct RcHdr {
    long long tok0;    // global token index of the stage's first token
    int cnt;           // tokens in this stage (0 for an empty sequence)
    int item;          // item ordinal within this CTA
    int n, h, vhalf;   // the item: sequence, head, half of the values
    int first, last;   // first / last stage of the item
    int valid;         // 0 past the CTA's last stage
    int pad[2];
};
struct RcRaw {
    uint16_t q[RC_L][D], k[RC_L][D], g[RC_L][D], v[RC_L][RC_VALUES];
    float dtb[D];
    float alog[4];
    RcHdr hdr;
};
struct RcPrep {
    float l[RC_L][D];      // log2 of alpha per key channel
    float ka[RC_L][D];     // A_t k^      (A_t = decay from the stage start through token t)
    float kd[RC_L][D];     // k^ / A_t
    float qa[RC_L][D];     // scale A_t q^
    float aend[D];         // A of the stage's last token
    float4 sc[RC_L];       // rk, rq * scale, b, -
};
template <int STATE>
struct RcSmem {
    static constexpr int SB = (STATE == 1 ? 2 : 4) * RC_VALUES * D;   // bytes of one state block
    unsigned char st[RC_NST][STATE == 0 ? 16 : SB];                    // state slots (bulk-copy targets)
    RcRaw raw[RC_NRAW];
    RcPrep prep;
    uint16_t rawb[RC_NRAW][RC_L];
    unsigned long long mbar[RC_NST];
};

static_assert(sizeof(RcRaw) % 16 == 0, "raw slots keep 16-byte alignment");
static_assert(sizeof(RcSmem<2>) <= 113 * 1024, "two CTAs per SM");


__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Sum over the 16 key groups (lane bits 0..3) of the partial dot products a[c] of the thread's four
// values: afterwards each lane holds the full sum of value 2 b3 + b2 (b3, b2 = lane bits 3 and 2).
__device__ __forceinline__ float reduce_scatter16(const float (&a)[4], bool b3, bool b2)
{
    float k0 = b3 ? a[2] : a[0], k1 = b3 ? a[3] : a[1];
    const float s0 = b3 ? a[0] : a[2], s1 = b3 ? a[1] : a[3];
    k0 += __shfl_xor_sync(0xffffffffu, s0, 8);
    k1 += __shfl_xor_sync(0xffffffffu, s1, 8);
    float k = b2 ? k1 : k0;
    k += __shfl_xor_sync(0xffffffffu, b2 ? k0 : k1, 4);
    k += __shfl_xor_sync(0xffffffffu, k, 2);
    k += __shfl_xor_sync(0xffffffffu, k, 1);
    return k;
}
// The four full sums in every lane, from reduce_scatter16's result.
__device__ __forceinline__ void all_gather16(float mine, bool b3, bool b2, float (&out)[4])
{
    const float x = __shfl_xor_sync(0xffffffffu, mine, 4);
    const float lo = b2 ? x : mine, hi = b2 ? mine : x;   // values 2 b3, 2 b3 + 1
    const float ylo = __shfl_xor_sync(0xffffffffu, lo, 8), yhi = __shfl_xor_sync(0xffffffffu, hi, 8);
    out[0] = b3 ? ylo : lo;
    out[1] = b3 ? yhi : hi;
    out[2] = b3 ? lo : ylo;
    out[3] = b3 ? hi : yhi;
}

struct ItemId {
    int n, h, vhalf;
};
// item ordinal k of this CTA (items are taken round robin over the grid; 2 N H < 2^31)
__device__ __forceinline__ ItemId item_id(int k, int H)
{
    const unsigned it = blockIdx.x + (unsigned)k * gridDim.x;
    const unsigned nh = it >> 1;
    ItemId r;
    r.vhalf = (int)(it & 1u);
    r.n = (int)(nh / (unsigned)H);
    r.h = (int)(nh - (unsigned)r.n * (unsigned)H);
    return r;
}

template <int STATE, bool VARLEN>  // STATE: 0 none, 1 bf16, 2 fp32
__global__ void __launch_bounds__(RC_THREADS, 2) kda_recurrent_kernel(const Problem p, int n_items)
{
    extern __shared__ __align__(128) unsigned char rc_smem_raw[];
    RcSmem<STATE> &sm = *reinterpret_cast<RcSmem<STATE> *>(rc_smem_raw);
    constexpr int SB = RcSmem<STATE>::SB;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.H;
    const int my_items = (int)(((unsigned)n_items - blockIdx.x + gridDim.x - 1) / gridDim.x);
    const int kg = lane & 15;                 // key group: keys 64 f + 4 kg + j (f < 2, j < 4)
    const int vq = warp * 2 + (lane >> 4);    // value quad: values 4 vq + c (c < 4) of the item's half
    const bool b3 = (lane & 8) != 0, b2 = (lane & 4) != 0;
    const bool has_state_in = STATE != 0 && p.init != nullptr;

    auto seq_of = [&](int k, long long &bos, int &len) {
        const ItemId id = item_id(k, H);
        if (VARLEN) {   // clamped into [0, T] (the entry point keeps T below 2^31)
            int64_t b, l;
            if (seq_range(p.cu, id.n, p.N, p.T, b, l) && tid == 0)
                atomicOr(&g_kda_rc_error, DEVERR_CU_SEQLENS);
            bos = b;
            len = (int)l;
        } else {
            bos = (long long)id.n * p.T;
            len = (int)p.T;
        }
    };
    auto issue_state = [&](int k) {   // one thread: the state block of item k -> slot k & 1
        const ItemId id = item_id(k, H);
        const size_t off = ((((size_t)id.n * H + id.h) * D) + (size_t)id.vhalf * RC_VALUES) * D;
        const unsigned char *src = static_cast<const unsigned char *>(p.init) + off * (STATE == 1 ? 2 : 4);
        const uint32_t mb = smem_u32(&sm.mbar[k & 1]);
        mbar_expect_tx(mb, SB);
        bulk_g2s(smem_u32(sm.st[k & 1]), src, SB, mb);
    };

    // issue cursor: stage ij of item ik (ibos, ilen); nbos, nlen belong to item ik + 1
    int ik = 0, ij = 0, ilen = 0, nlen = 0;
    long long ibos = 0, nbos = 0;
    // raw rows, gate parameters and header of the cursor's stage -> raw slot rs; returns the bf16
    // beta bits of token tid of the stage (tid < 8)
    auto issue_stage = [&](int rs) -> uint16_t {
        RcRaw &r = sm.raw[rs];
        const bool valid = ik < my_items;
        int cnt = 0;
        long long tok0 = 0;
        ItemId id{0, 0, 0};
        if (valid) {
            id = item_id(ik, H);
            tok0 = ibos + (long long)RC_L * ij;
            cnt = min(RC_L, ilen - RC_L * ij);
        }
        const int nrow = cnt * 56;   // 16-byte pieces per token: 16 each of q, k, g and 8 of the v half
        const int nchunk = valid ? nrow + 33 : 0;
        for (int c = tid; c < nchunk; c += RC_THREADS) {
            if (c < nrow) {
                const int tt = c / 56, rr = c - tt * 56;
                const size_t row = ((size_t)(tok0 + tt) * H + id.h) * D;
                const __nv_bfloat16 *src;
                uint16_t *dst;
                if (rr < 48) {
                    const int which = rr >> 4, part = rr & 15;
                    src = (which == 0 ? p.q : which == 1 ? p.k : p.g) + row + part * 8;
                    dst = (which == 0 ? r.q[tt] : which == 1 ? r.k[tt] : r.g[tt]) + part * 8;
                } else {
                    const int part = rr - 48;
                    src = p.v + row + id.vhalf * RC_VALUES + part * 8;
                    dst = r.v[tt] + part * 8;
                }
                cp_async16(smem_u32(dst), src, true);
            } else if (c < nrow + 32) {
                const int part = c - nrow;
                cp_async16(smem_u32(r.dtb + part * 4), p.dt_bias + (size_t)id.h * D + part * 4, true);
            } else {
                cp_async4(smem_u32(r.alog), p.A_log + id.h);
            }
        }
        if (tid == 0) {
            r.hdr.tok0 = tok0;
            r.hdr.cnt = cnt;
            r.hdr.item = ik;
            r.hdr.n = id.n;
            r.hdr.h = id.h;
            r.hdr.vhalf = id.vhalf;
            r.hdr.first = ij == 0;
            r.hdr.last = valid && RC_L * (ij + 1) >= ilen;
            r.hdr.valid = valid;
        }
        cp_async_commit();
        return tid < cnt ? __bfloat16_as_ushort(p.beta[(size_t)(tok0 + tid) * H + id.h]) : (uint16_t)0;
    };
    auto advance = [&]() {
        if (ik >= my_items)
            return;
        if (RC_L * (ij + 1) < ilen) {
            ++ij;
        } else {
            ++ik;
            ij = 0;
            ibos = nbos;
            ilen = nlen;
            if (ik + 1 < my_items)
                seq_of(ik + 1, nbos, nlen);
        }
    };

    // -------- prologue: barriers, the first two state blocks and the first two stages
    if (tid == 0) {
        mbar_init(smem_u32(&sm.mbar[0]), 1);
        mbar_init(smem_u32(&sm.mbar[1]), 1);
        mbar_fence_init();
    }
    __syncthreads();
    seq_of(0, ibos, ilen);
    if (my_items > 1)
        seq_of(1, nbos, nlen);
    if (tid == 0 && has_state_in) {
        issue_state(0);
        if (my_items > 1)
            issue_state(1);
    }
    uint16_t bpend = issue_stage(0);
    advance();
    if (tid < RC_L)
        sm.rawb[0][tid] = bpend;
    bpend = issue_stage(1);
    advance();

    // -------- the stage loop
    // S2[c][2 f + jj]: keys 64 f + 4 kg + 2 jj and + 1 of value 4 vq + c; inside a stage it holds
    // S / A (A = decay since the stage start, per key), so a token costs three packed FMAs per pair
    f2 S2[4][4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            S2[c][i] = 0ull;
    bool ok = true;
    int rs = 0;   // raw slot of the current stage
    for (;;) {
        const int rs1 = rs == RC_NRAW - 1 ? 0 : rs + 1, rs2 = rs1 == RC_NRAW - 1 ? 0 : rs1 + 1;
        if (tid < RC_L)
            sm.rawb[rs1][tid] = bpend;   // beta of the next stage (its slot was last read two stages ago)
        cp_async_wait_1();
        __syncthreads();   // this stage's rows are complete; the previous stage is done with slot rs2
        const RcHdr hd = sm.raw[rs].hdr;
        bpend = issue_stage(rs2);
        advance();
        if (!hd.valid)
            break;
        const RcRaw &r = sm.raw[rs];
        const ItemId id{hd.n, hd.h, hd.vhalf};

        // item start: its state block, from the slot into registers
        if (hd.first) {
            if (has_state_in) {
                const int slot = hd.item & 1;
                const uint32_t mb = smem_u32(&sm.mbar[slot]), par = (uint32_t)(hd.item >> 1) & 1u;
                if (!mbar_wait(mb, par) && !mbar_wait(mb, par))
                    ok = false;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int f = 0; f < 2; ++f) {
                        const int e = (4 * vq + c) * D + 64 * f + 4 * kg;
                        if (STATE == 2) {
                            const float4 x = *reinterpret_cast<const float4 *>(sm.st[slot] + 4 * e);
                            S2[c][2 * f] = f2_pack(x.x, x.y);
                            S2[c][2 * f + 1] = f2_pack(x.z, x.w);
                        } else {
                            const uint2 w = *reinterpret_cast<const uint2 *>(sm.st[slot] + 2 * e);
                            S2[c][2 * f] = f2_bf16x2(w.x);
                            S2[c][2 * f + 1] = f2_bf16x2(w.y);
                        }
                    }
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        S2[c][i] = 0ull;
            }
        }

        // -------- phase A, token-parallel: warp w takes token w (channels 4 lane .. 4 lane + 3):
        // inverse norms, b and log2 alpha = lower_bound log2(e) sigmoid(exp(A_log) (g + dt_bias))
        if (warp < hd.cnt) {
            const int tt = warp;
            const float gz = -expf(r.alog[0]) * LOG2E;
            const uint2 qw = *reinterpret_cast<const uint2 *>(&r.q[tt][4 * lane]);
            const uint2 kw = *reinterpret_cast<const uint2 *>(&r.k[tt][4 * lane]);
            const uint2 gw = *reinterpret_cast<const uint2 *>(&r.g[tt][4 * lane]);
            const float4 dt = *reinterpret_cast<const float4 *>(&r.dtb[4 * lane]);
            const float q4[4] = {bf16_lo(qw.x), bf16_hi(qw.x), bf16_lo(qw.y), bf16_hi(qw.y)};
            const float k4[4] = {bf16_lo(kw.x), bf16_hi(kw.x), bf16_lo(kw.y), bf16_hi(kw.y)};
            const float g4[4] = {bf16_lo(gw.x), bf16_hi(gw.x), bf16_lo(gw.y), bf16_hi(gw.y)};
            const float d4[4] = {dt.x, dt.y, dt.z, dt.w};
            float sq = 0.f, sk = 0.f, l4[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                sq = fmaf(q4[j], q4[j], sq);
                sk = fmaf(k4[j], k4[j], sk);
                l4[j] = p.lb_log2e * rcp_approx(1.f + ex2_approx(fmaf(g4[j], gz, gz * d4[j])));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            *reinterpret_cast<float4 *>(&sm.prep.l[tt][4 * lane]) = make_float4(l4[0], l4[1], l4[2], l4[3]);
            if (lane == 0)
                sm.prep.sc[tt] = make_float4(rsqrtf(sk + 1e-6f), rsqrtf(sq + 1e-6f) * p.scale,
                                             sigmoid_fast(__uint_as_float((uint32_t)sm.rawb[rs][tt] << 16)), 0.f);
        }
        __syncthreads();   // phase A done; every thread has read the state slot

        // the state slot just read takes the block of item + 2
        if (hd.first && tid == 0 && has_state_in && hd.item + 2 < my_items) {
            fence_async_smem();
            issue_state(hd.item + 2);
        }

        // -------- phase B, channel-parallel: A_t = 2^(sum of log2 alpha from the stage start through
        // token t) folded into A_t k^, k^ / A_t (threads 0..127) and scale A_t q^ (threads 128..255)
        {
            const int c = tid & (D - 1);
            const bool qside = tid >= D;
            float L = 0.f;
            for (int tt = 0; tt < hd.cnt; ++tt) {
                L += sm.prep.l[tt][c];
                const float4 sc = sm.prep.sc[tt];
                if (!qside) {
                    const float kh = __uint_as_float((uint32_t)r.k[tt][c] << 16) * sc.x;
                    sm.prep.ka[tt][c] = kh * ex2_approx(L);
                    sm.prep.kd[tt][c] = kh * ex2_approx(-L);
                } else {
                    sm.prep.qa[tt][c] = __uint_as_float((uint32_t)r.q[tt][c] << 16) * sc.y * ex2_approx(L);
                }
            }
            if (!qside)
                sm.prep.aend[c] = ex2_approx(L);
        }
        __syncthreads();

        // -------- serial loop over the stage's tokens (no barriers):
        //   p = S^T (A k^),  u = b (v - p),  S += (k^ / A) u^T,  o = S^T (scale A q^)
        __nv_bfloat16 *outp = p.out + ((size_t)hd.tok0 * H + id.h) * D + id.vhalf * RC_VALUES + 4 * vq +
                              (b3 ? 2 : 0) + (b2 ? 1 : 0);
        const bool writer = (lane & 3) == 0;
#pragma unroll 2
        for (int tt = 0; tt < hd.cnt; ++tt) {
            f2 ka[4], kd[4], qa[4];
#pragma unroll
            for (int f = 0; f < 2; ++f) {
                const int key = 64 * f + 4 * kg;
                const float4 x = *reinterpret_cast<const float4 *>(&sm.prep.ka[tt][key]);
                ka[2 * f] = f2_pack(x.x, x.y);
                ka[2 * f + 1] = f2_pack(x.z, x.w);
            }
            float pk[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                f2 acc = f2_mul(S2[c][0], ka[0]);
                acc = f2_fma(S2[c][1], ka[1], acc);
                acc = f2_fma(S2[c][2], ka[2], acc);
                acc = f2_fma(S2[c][3], ka[3], acc);
                pk[c] = f2_lo(acc) + f2_hi(acc);
            }
            float P[4];
            all_gather16(reduce_scatter16(pk, b3, b2), b3, b2, P);
#pragma unroll
            for (int f = 0; f < 2; ++f) {
                const int key = 64 * f + 4 * kg;
                const float4 x = *reinterpret_cast<const float4 *>(&sm.prep.kd[tt][key]);
                const float4 y = *reinterpret_cast<const float4 *>(&sm.prep.qa[tt][key]);
                kd[2 * f] = f2_pack(x.x, x.y);
                kd[2 * f + 1] = f2_pack(x.z, x.w);
                qa[2 * f] = f2_pack(y.x, y.y);
                qa[2 * f + 1] = f2_pack(y.z, y.w);
            }
            const float b = sm.prep.sc[tt].z;
            const uint2 vw = *reinterpret_cast<const uint2 *>(&r.v[tt][4 * vq]);
            const float vv[4] = {bf16_lo(vw.x), bf16_hi(vw.x), bf16_lo(vw.y), bf16_hi(vw.y)};
            float oc[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float u = b * (vv[c] - P[c]);
                const f2 U = f2_pack(u, u);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    S2[c][i] = f2_fma(kd[i], U, S2[c][i]);
                f2 o = f2_mul(S2[c][0], qa[0]);
                o = f2_fma(S2[c][1], qa[1], o);
                o = f2_fma(S2[c][2], qa[2], o);
                o = f2_fma(S2[c][3], qa[3], o);
                oc[c] = f2_lo(o) + f2_hi(o);
            }
            const float om = reduce_scatter16(oc, b3, b2);
            if (writer)
                *outp = __float2bfloat16_rn(om);
            outp += (size_t)H * D;
        }

        // stage end: back from S / A to S
#pragma unroll
        for (int f = 0; f < 2; ++f) {
            const float4 x = *reinterpret_cast<const float4 *>(&sm.prep.aend[64 * f + 4 * kg]);
            const f2 a01 = f2_pack(x.x, x.y), a23 = f2_pack(x.z, x.w);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                S2[c][2 * f] = f2_mul(S2[c][2 * f], a01);
                S2[c][2 * f + 1] = f2_mul(S2[c][2 * f + 1], a23);
            }
        }

        // item end: the final state block
        if (hd.last && STATE != 0 && p.fin) {
            const size_t row0 = (((size_t)id.n * H + id.h) * D + (size_t)id.vhalf * RC_VALUES + 4 * vq) * D;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int f = 0; f < 2; ++f) {
                    const size_t e = row0 + (size_t)c * D + 64 * f + 4 * kg;
                    if (STATE == 2) {
                        *reinterpret_cast<float4 *>(static_cast<float *>(p.fin) + e) =
                            make_float4(f2_lo(S2[c][2 * f]), f2_hi(S2[c][2 * f]), f2_lo(S2[c][2 * f + 1]),
                                        f2_hi(S2[c][2 * f + 1]));
                    } else {
                        const __nv_bfloat162 h0 = __floats2bfloat162_rn(f2_lo(S2[c][2 * f]), f2_hi(S2[c][2 * f]));
                        const __nv_bfloat162 h1 =
                            __floats2bfloat162_rn(f2_lo(S2[c][2 * f + 1]), f2_hi(S2[c][2 * f + 1]));
                        *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.fin) + e) =
                            make_uint2(*reinterpret_cast<const uint32_t *>(&h0), *reinterpret_cast<const uint32_t *>(&h1));
                    }
                }
        }
        rs = rs1;
    }
    cp_async_wait_all();
    if (!ok)
        atomicOr(&g_kda_rc_error, 1u);
}

template <int S, bool V>
cudaError_t launch_one(const Problem &p, cudaStream_t stream)
{
    static bool configured[64] = {};
    static int sms[64] = {};
    const int smem = (int)sizeof(RcSmem<S>);
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    int nsm = dev < 64 ? sms[dev] : 0;
    if (nsm == 0) {
        err = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess)
            return err;
        if (dev < 64)
            sms[dev] = nsm;
    }
    if (dev >= 64 || !configured[dev]) {
        err = cudaFuncSetAttribute(kda_recurrent_kernel<S, V>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess)
            return err;
        if (dev < 64)
            configured[dev] = true;
    }
    const int n_items = 2 * p.N * p.H;   // the entry point checks 2 N H <= INT32_MAX
    const int grid = n_items < 2 * nsm ? n_items : 2 * nsm;
    kda_recurrent_kernel<S, V><<<grid, RC_THREADS, smem, stream>>>(p, n_items);
    return cudaGetLastError();
}

}  // namespace

size_t recurrent_smem_bytes() { return sizeof(RcSmem<2>); }

cudaError_t launch_recurrent(const Problem &p, int state_kind, cudaStream_t stream)
{
    if (p.cu) {
        if (state_kind == 2) return launch_one<2, true>(p, stream);
        if (state_kind == 1) return launch_one<1, true>(p, stream);
        return launch_one<0, true>(p, stream);
    }
    if (state_kind == 2) return launch_one<2, false>(p, stream);
    if (state_kind == 1) return launch_one<1, false>(p, stream);
    return launch_one<0, false>(p, stream);
}

cudaError_t recurrent_read_and_clear_error(unsigned int *flag)
{
    unsigned int zero = 0;
    cudaError_t err = cudaMemcpyFromSymbol(flag, g_kda_rc_error, sizeof *flag);
    if (err == cudaSuccess && *flag)
        err = cudaMemcpyToSymbol(g_kda_rc_error, &zero, sizeof zero);
    return err;
}

}  // namespace kda
