// KDA decode kernel: the per-token gated delta rule (guancyxx.cn FlashKDA article, section 一) for
// fixed-length problems of 1 to 8 tokens per sequence -- decode steps, and short speculative runs.
//
// Per token (state S in R^{K x V}, stored transposed [V][K]):
//   S' = Diag(alpha) S,   u = b (v - S'^T k^),   S = S' + k^ u^T,   o = scale S^T q^
// with alpha = exp(lower_bound sigmoid(exp(A_log) (g + dt_bias))), b = sigmoid(beta), k^ = rk k, q^ = rq q.
// The tokens of an item form one stage evaluated exactly as the token-recurrent kernel evaluates a stage
// (the decay folded into A k^, k^ / A and scale A q^, the same rounding and summation orders), so the two
// kernels give the same bits.
//
// Work item = (sequence, head, half of the values), a contiguous 32 KB (fp32) or 16 KB (bf16) block of the
// state.  The grid is persistent (two CTAs per SM).  In each CTA one producer warp fills a ring of shared-
// memory slots -- the state block, the item's token rows (q, k, g and the value half of v) and dt_bias[h] by
// bulk copies on the slot's "full" mbarrier, beta and A_log[h] by plain loads into the slot header (a second
// arrival on the same barrier releases it) -- and
// eight consumer warps each take every item: a consumer warp owns 8 of the 64 values and computes the gate,
// the norms (shuffle sums over the 16 key groups of its lanes), the update and the output for its values
// without any CTA barrier, writes its state columns and outputs straight to global memory and releases the
// slot on its "empty" mbarrier.  Every wait is bounded; a wait that gives up sets the kernel's error word.
#include "kda_device.cuh"
#include "kda_internal.h"

__device__ unsigned int g_kda_dc_error;   // set when a bounded wait of the decode kernel gave up

namespace kda {
namespace {

constexpr int DC_CONSUMER_WARPS = 8;
constexpr int DC_THREADS = (DC_CONSUMER_WARPS + 1) * 32;
constexpr int DC_VALUES = 64;      // values per item
constexpr int DC_RING = 3;         // slots
#ifndef KDA_DC_MAX_T
#define KDA_DC_MAX_T 8
#endif
constexpr int DC_MAX_T = KDA_DC_MAX_T;   // one stage of the token-recurrent kernel at most (same bits)

struct DcHdr {
    long long tok0;                // first token of the item's sequence
    int n, h, vhalf;
    float alog;
    uint16_t beta[DC_MAX_T];
};

// slot layout (bytes); the state block first (bulk-copy target, 128-byte aligned)
struct DcLayout {
    int sb, q, k, g, v, dtb, hdr, bytes;
    __host__ __device__ DcLayout(int state_bytes, int T)
    {
        sb = state_bytes;
        q = sb;
        k = q + T * D * 2;
        g = k + T * D * 2;
        v = g + T * D * 2;
        dtb = v + T * DC_VALUES * 2;
        hdr = dtb + D * 4;
        bytes = (hdr + (int)sizeof(DcHdr) + 127) / 128 * 128;
    }
};

struct DcItem {
    int n, h, vhalf;
};
__device__ __forceinline__ DcItem dc_item(int k, int H)
{
    const unsigned it = blockIdx.x + (unsigned)k * gridDim.x;
    const unsigned nh = it >> 1;
    DcItem r;
    r.vhalf = (int)(it & 1u);
    r.n = (int)(nh / (unsigned)H);
    r.h = (int)(nh - (unsigned)r.n * (unsigned)H);
    return r;
}

// sum over the 16 key groups (lane bits 0..3) of a value held by every lane
__device__ __forceinline__ float allsum16(float x)
{
    x += __shfl_xor_sync(0xffffffffu, x, 8);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x;
}
// reduce-scatter of four per-value partial sums over the 16 key groups: afterwards each lane holds the
// full sum of value 2 b3 + b2 (b3, b2 = lane bits 3 and 2)
__device__ __forceinline__ float rs16(const float (&a)[4], bool b3, bool b2)
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
__device__ __forceinline__ void ag16(float mine, bool b3, bool b2, float (&out)[4])
{
    const float x = __shfl_xor_sync(0xffffffffu, mine, 4);
    const float lo = b2 ? x : mine, hi = b2 ? mine : x;
    const float ylo = __shfl_xor_sync(0xffffffffu, lo, 8), yhi = __shfl_xor_sync(0xffffffffu, hi, 8);
    out[0] = b3 ? ylo : lo;
    out[1] = b3 ? yhi : hi;
    out[2] = b3 ? lo : ylo;
    out[3] = b3 ? hi : yhi;
}

template <int STATE>  // 0 none, 1 bf16, 2 fp32
__global__ void __launch_bounds__(DC_THREADS, 2) kda_decode_kernel(const Problem p, int n_items, int slot_bytes)
{
    extern __shared__ __align__(128) unsigned char dc_smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.H, T = (int)p.T;
    const int my_items = (int)(((unsigned)n_items - blockIdx.x + gridDim.x - 1) / gridDim.x);
    constexpr int SBYTES = STATE == 1 ? DC_VALUES * D * 2 : (STATE == 2 ? DC_VALUES * D * 4 : 0);
    const DcLayout lay(SBYTES, T);
    uint64_t *full = reinterpret_cast<uint64_t *>(dc_smem + DC_RING * slot_bytes);
    uint64_t *empty = full + DC_RING;
    const bool has_in = STATE != 0 && p.init != nullptr;

    if (tid == 0) {
        for (int s = 0; s < DC_RING; ++s) {
            mbar_init(smem_u32(&full[s]), 2);   // the producer's expect_tx, then its header arrival
            mbar_init(smem_u32(&empty[s]), DC_CONSUMER_WARPS);
        }
        mbar_fence_init();
    }
    __syncthreads();
    bool ok = true;

    if (warp == DC_CONSUMER_WARPS) {
        // ---------------- producer (lane 0)
        if (lane == 0) {
            const uint32_t tok_bytes = (uint32_t)T * (3 * D * 2 + DC_VALUES * 2);
            for (int i = 0; i < my_items; ++i) {
                const int slot = i % DC_RING, round = i / DC_RING;
                const DcItem it = dc_item(i, H);
                const long long tok0 = (long long)it.n * T;
                // the header's loads first: their latency overlaps the slot wait and the bulk copies
                const float alog = p.A_log[it.h];
                uint16_t bts[DC_MAX_T];
#pragma unroll
                for (int t = 0; t < DC_MAX_T; ++t)
                    bts[t] = t < T ? __bfloat16_as_ushort(p.beta[(size_t)(tok0 + t) * H + it.h]) : (uint16_t)0;
                if (i >= DC_RING && !mbar_wait(smem_u32(&empty[slot]), (uint32_t)(round - 1) & 1u) &&
                    !mbar_wait(smem_u32(&empty[slot]), (uint32_t)(round - 1) & 1u))
                    ok = false;
                unsigned char *s = dc_smem + (size_t)slot * slot_bytes;
                const uint32_t fb = smem_u32(&full[slot]);
                mbar_expect_tx(fb, (has_in ? (uint32_t)SBYTES : 0u) + tok_bytes + (uint32_t)D * 4);
                if (has_in) {
                    const size_t off = ((((size_t)it.n * H + it.h) * D) + (size_t)it.vhalf * DC_VALUES) * D;
                    bulk_g2s(smem_u32(s), static_cast<const unsigned char *>(p.init) + off * (STATE == 1 ? 2 : 4),
                             SBYTES, fb);
                }
                for (int t = 0; t < T; ++t) {
                    const size_t row = ((size_t)(tok0 + t) * H + it.h) * D;
                    bulk_g2s(smem_u32(s + lay.q + t * D * 2), p.q + row, D * 2, fb);
                    bulk_g2s(smem_u32(s + lay.k + t * D * 2), p.k + row, D * 2, fb);
                    bulk_g2s(smem_u32(s + lay.g + t * D * 2), p.g + row, D * 2, fb);
                    bulk_g2s(smem_u32(s + lay.v + t * DC_VALUES * 2), p.v + row + it.vhalf * DC_VALUES,
                             DC_VALUES * 2, fb);
                }
                bulk_g2s(smem_u32(s + lay.dtb), p.dt_bias + (size_t)it.h * D, D * 4, fb);
                DcHdr *hd = reinterpret_cast<DcHdr *>(s + lay.hdr);
                hd->tok0 = tok0;
                hd->n = it.n;
                hd->h = it.h;
                hd->vhalf = it.vhalf;
                hd->alog = alog;
#pragma unroll
                for (int t = 0; t < DC_MAX_T; ++t)
                    hd->beta[t] = bts[t];
                mbar_arrive(fb);   // releases the header
            }
        }
    } else {
        // ---------------- consumers: warp w owns values 8 w .. 8 w + 7 of the item's half
        const int kg = lane & 15;                 // keys 64 f + 4 kg + j (f < 2, j < 4)
        const int vq = warp * 2 + (lane >> 4);    // values 4 vq + c (c < 4)
        const bool b3 = (lane & 8) != 0, b2 = (lane & 4) != 0;
        const bool writer = (lane & 3) == 0;
        for (int i = 0; i < my_items; ++i) {
            const int slot = i % DC_RING, round = i / DC_RING;
            const uint32_t fb = smem_u32(&full[slot]);
            if (!mbar_wait(fb, (uint32_t)round & 1u) && !mbar_wait(fb, (uint32_t)round & 1u))
                ok = false;
            const unsigned char *s = dc_smem + (size_t)slot * slot_bytes;
            const DcHdr *hdp = reinterpret_cast<const DcHdr *>(s + lay.hdr);
            const long long htok0 = hdp->tok0;
            const int hn = hdp->n, hh = hdp->h, hvh = hdp->vhalf;
            const float halog = hdp->alog;
            const float gz = -expf(halog) * LOG2E;
            float gd[4];   // this lane's key group (see below)
            {
                const float4 d4 = *reinterpret_cast<const float4 *>(s + lay.dtb + (64 * (lane >> 4) + 4 * kg) * 4);
                gd[0] = gz * d4.x; gd[1] = gz * d4.y; gd[2] = gz * d4.z; gd[3] = gz * d4.w;
            }
            // the state columns of this thread
            f2 S2[4][4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int f = 0; f < 2; ++f) {
                    const int e = (4 * vq + c) * D + 64 * f + 4 * kg;
                    if (STATE == 2 && has_in) {
                        const float4 x = *reinterpret_cast<const float4 *>(s + 4 * e);
                        S2[c][2 * f] = f2_pack(x.x, x.y);
                        S2[c][2 * f + 1] = f2_pack(x.z, x.w);
                    } else if (STATE == 1 && has_in) {
                        const uint2 w = *reinterpret_cast<const uint2 *>(s + 2 * e);
                        S2[c][2 * f] = f2_bf16x2(w.x);
                        S2[c][2 * f + 1] = f2_bf16x2(w.y);
                    } else {
                        S2[c][2 * f] = S2[c][2 * f + 1] = 0ull;
                    }
                }
            __nv_bfloat16 *outp = p.out + ((size_t)htok0 * H + hh) * D + hvh * DC_VALUES + 4 * vq +
                                  (b3 ? 2 : 0) + (b2 ? 1 : 0);
            // the tokens as one stage from the sequence start, in the arithmetic of the token-recurrent
            // kernel's stages (same rounding, so both kernels give the same bits): per key, A_t = 2^(sum of
            // log2 alpha through token t); S holds S / A_t; p = (S/A)^T (A k^), S/A += (k^ / A) u^T,
            // o = (S/A)^T (scale A q^); at the end S = A_T (S / A)
            // The two half-warps hold the same keys (they differ in values), so each computes the per-key
            // quantities of one key group, fo = lane / 16 (keys 64 fo + 4 kg + j), with the expressions and
            // summation orders of the staged kernel, and takes the other group's from its partner lane.
            const int fo = lane >> 4;
            float Lk[4];   // log2 of A for this lane's 4 keys
#pragma unroll
            for (int j = 0; j < 4; ++j)
                Lk[j] = 0.f;
            for (int t = 0; t < T; ++t) {
                const int key = 64 * fo + 4 * kg;
                const uint2 qw = *reinterpret_cast<const uint2 *>(s + lay.q + (t * D + key) * 2);
                const uint2 kw = *reinterpret_cast<const uint2 *>(s + lay.k + (t * D + key) * 2);
                const uint2 gw = *reinterpret_cast<const uint2 *>(s + lay.g + (t * D + key) * 2);
                const float q4[4] = {bf16_lo(qw.x), bf16_hi(qw.x), bf16_lo(qw.y), bf16_hi(qw.y)};
                const float k4[4] = {bf16_lo(kw.x), bf16_hi(kw.x), bf16_lo(kw.y), bf16_hi(kw.y)};
                const float g4[4] = {bf16_lo(gw.x), bf16_hi(gw.x), bf16_lo(gw.y), bf16_hi(gw.y)};
                float sq = 0.f, sk = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    sq = fmaf(q4[j], q4[j], sq);
                    sk = fmaf(k4[j], k4[j], sk);
                    // the product is rounded before the sum (no contraction), as in the staged kernel
                    Lk[j] += __fmul_rn(p.lb_log2e, rcp_approx(1.f + ex2_approx(fmaf(g4[j], gz, gd[j]))));
                }
                // the norms: the same summation tree as a warp over 4-channel groups (groups f = 0, 1 first)
                const float sqp = __shfl_xor_sync(0xffffffffu, sq, 16), skp = __shfl_xor_sync(0xffffffffu, sk, 16);
                const float rq = rsqrtf(allsum16(fo ? sqp + sq : sq + sqp) + 1e-6f) * p.scale;
                const float rk = rsqrtf(allsum16(fo ? skp + sk : sk + skp) + 1e-6f);
                const float b = sigmoid_fast(__uint_as_float((uint32_t)hdp->beta[t] << 16));
                float a4[4], d4[4], e4[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float A = ex2_approx(Lk[j]), kh = k4[j] * rk;
                    a4[j] = kh * A;
                    d4[j] = kh * ex2_approx(-Lk[j]);
                    e4[j] = q4[j] * rq * A;
                }
                // key group f's pairs in slots 2 f, 2 f + 1: this lane's group from itself, the other from lane ^ 16
                f2 ka[4], kd[4], qa[4];
                {
                    const f2 o[6] = {f2_pack(a4[0], a4[1]), f2_pack(a4[2], a4[3]), f2_pack(d4[0], d4[1]),
                                     f2_pack(d4[2], d4[3]), f2_pack(e4[0], e4[1]), f2_pack(e4[2], e4[3])};
                    f2 x[6];
#pragma unroll
                    for (int m = 0; m < 6; ++m)
                        x[m] = __shfl_xor_sync(0xffffffffu, o[m], 16);
                    ka[0] = fo ? x[0] : o[0]; ka[1] = fo ? x[1] : o[1]; ka[2] = fo ? o[0] : x[0]; ka[3] = fo ? o[1] : x[1];
                    kd[0] = fo ? x[2] : o[2]; kd[1] = fo ? x[3] : o[3]; kd[2] = fo ? o[2] : x[2]; kd[3] = fo ? o[3] : x[3];
                    qa[0] = fo ? x[4] : o[4]; qa[1] = fo ? x[5] : o[5]; qa[2] = fo ? o[4] : x[4]; qa[3] = fo ? o[5] : x[5];
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
                ag16(rs16(pk, b3, b2), b3, b2, P);
                const uint2 vw = *reinterpret_cast<const uint2 *>(s + lay.v + (t * DC_VALUES + 4 * vq) * 2);
                const float vv[4] = {bf16_lo(vw.x), bf16_hi(vw.x), bf16_lo(vw.y), bf16_hi(vw.y)};
                float oc[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float u = b * (vv[c] - P[c]);
                    const f2 U = f2_pack(u, u);
#pragma unroll
                    for (int i2 = 0; i2 < 4; ++i2)
                        S2[c][i2] = f2_fma(kd[i2], U, S2[c][i2]);
                    f2 o = f2_mul(S2[c][0], qa[0]);
                    o = f2_fma(S2[c][1], qa[1], o);
                    o = f2_fma(S2[c][2], qa[2], o);
                    o = f2_fma(S2[c][3], qa[3], o);
                    oc[c] = f2_lo(o) + f2_hi(o);
                }
                const float om = rs16(oc, b3, b2);
                if (writer)
                    *outp = __float2bfloat16_rn(om);
                outp += (size_t)H * D;
            }
            // back from S / A to S (this lane's key group's A from itself, the other group's from lane ^ 16)
            {
                const f2 o01 = f2_pack(ex2_approx(Lk[0]), ex2_approx(Lk[1]));
                const f2 o23 = f2_pack(ex2_approx(Lk[2]), ex2_approx(Lk[3]));
                const f2 x01 = __shfl_xor_sync(0xffffffffu, o01, 16), x23 = __shfl_xor_sync(0xffffffffu, o23, 16);
                const f2 a[4] = {fo ? x01 : o01, fo ? x23 : o23, fo ? o01 : x01, fo ? o23 : x23};
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i2 = 0; i2 < 4; ++i2)
                        S2[c][i2] = f2_mul(S2[c][i2], a[i2]);
            }
            // the slot is read: release it to the producer
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&empty[slot]));
            // final state columns
            if (STATE != 0 && p.fin) {
                const size_t row0 = (((size_t)hn * H + hh) * D + (size_t)hvh * DC_VALUES + 4 * vq) * D;
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
                            *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.fin) + e) = make_uint2(
                                *reinterpret_cast<const uint32_t *>(&h0), *reinterpret_cast<const uint32_t *>(&h1));
                        }
                    }
            }
        }
    }
    if (!ok)
        atomicOr(&g_kda_dc_error, 1u);
}

template <int S>
cudaError_t launch_decode_t(const Problem &p, cudaStream_t stream)
{
    static bool configured[64] = {};
    static int sms[64] = {};
    constexpr int SBYTES = S == 1 ? DC_VALUES * D * 2 : (S == 2 ? DC_VALUES * D * 4 : 0);
    const DcLayout lay(SBYTES, (int)p.T);
    const int smem = DC_RING * lay.bytes + 2 * DC_RING * 8;
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
        const DcLayout big(SBYTES, DC_MAX_T);
        err = cudaFuncSetAttribute(kda_decode_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   DC_RING * big.bytes + 2 * DC_RING * 8);
        if (err != cudaSuccess)
            return err;
        if (dev < 64)
            configured[dev] = true;
    }
    // persistent: as many CTAs per SM as their shared memory allows (two up to 4 tokens with an fp32 state)
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_decode_kernel<S>, DC_THREADS, smem);
    if (err != cudaSuccess)
        return err;
    per_sm = per_sm < 1 ? 1 : (per_sm > 2 ? 2 : per_sm);
    const int n_items = 2 * p.N * p.H;   // the entry point checks 2 N H <= INT32_MAX
    const int grid = n_items < per_sm * nsm ? n_items : per_sm * nsm;
    kda_decode_kernel<S><<<grid, DC_THREADS, smem, stream>>>(p, n_items, lay.bytes);
    return cudaGetLastError();
}

}  // namespace

// Fixed-length problems of up to DC_MAX_T tokens.  Both kernels give the same bits; the choice is by measurement
// on GB300 (64 and 256 sequences x 96 heads, decode kernel against the staged kernel):
//   fp32 state: 1 token 0.493 against 0.494 ms (the staged kernel streams the state as fast); 2-5 tokens faster
//     (1.15x at 5); from 6 tokens slower (0.8x: the three-slot ring of 8 tokens and a 32 KB state leaves one
//     CTA per SM);
//   bf16 state: faster up to 7 tokens (1.65x at 1, 1.11x at 5, 1.03x at 7), the same at 8.
bool decode_applies(const Problem &p, int state_kind)
{
    if (p.cu != nullptr || p.T < 1)
        return false;
    return state_kind == 2 ? (p.T >= 2 && p.T <= 5) : p.T <= 7;
}

cudaError_t launch_decode(const Problem &p, int state_kind, cudaStream_t stream)
{
    if (state_kind == 2) return launch_decode_t<2>(p, stream);
    if (state_kind == 1) return launch_decode_t<1>(p, stream);
    return launch_decode_t<0>(p, stream);
}

size_t decode_smem_bytes() { return DC_RING * DcLayout(DC_VALUES * D * 4, DC_MAX_T).bytes + 2 * DC_RING * 8; }

cudaError_t decode_read_and_clear_error(unsigned int *flag)
{
    unsigned int zero = 0;
    cudaError_t err = cudaMemcpyFromSymbol(flag, g_kda_dc_error, sizeof *flag);
    if (err == cudaSuccess && *flag)
        err = cudaMemcpyToSymbol(g_kda_dc_error, &zero, sizeof zero);
    return err;
}

}  // namespace kda
