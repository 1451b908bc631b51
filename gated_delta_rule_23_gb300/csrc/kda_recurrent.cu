// KDA token-recurrent kernel: the per-token gated delta rule (guancyxx.cn FlashKDA article,
// section 一; the argument table of the FlashKDA README mirror, "内核 API") evaluated token by token,
// for decode steps and short prefills, where the chunked path's per-chunk operand slots cost more
// than the state itself.  No workspace.
//
// Per token t (state S in R^{K x V}, stored transposed [V][K]):
//   S' = Diag(alpha) S,   u = b (v - S'^T k^),   S = S' + k^ u^T,   o = scale S^T q^
// with alpha = exp(lower_bound sigmoid(exp(A_log) (g + dt_bias))), b = sigmoid(beta) and q^, k^ the
// L2-normalised q, k.
//
// One CTA per (sequence, head, half of the values): 256 threads, thread (value v, key quarter kq)
// holds 32 keys of column v of S in fp32 registers for the whole sequence, and the two dot products
// over the keys are reduced across the four key quarters (lane bits 0..1) with warp shuffles.
// Tokens are staged 16 at a time: cp.async brings the raw bf16 rows of the next tile while the
// current tile is processed; a token-parallel pass (one warp per token) turns a raw tile into
// q^ scale, k^ and alpha in fp32, after which the serial loop runs without barriers.
#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int RC_THREADS = 256;      // 64 values x 4 key quarters
constexpr int RC_VALUES = 64;        // values per CTA
constexpr int RC_L = 16;             // tokens per staged tile
constexpr int RC_WARPS = RC_THREADS / 32;
constexpr int RC_CHUNKS_PER_TOKEN = 3 * (D * 2 / 16) + RC_VALUES * 2 / 16;   // 16-byte pieces: q, k, g, v half

struct RawTile {                      // bf16 bits as loaded
    uint16_t q[RC_L][D], k[RC_L][D], g[RC_L][D], v[RC_L][RC_VALUES];
};
struct PrepTile {
    float qh[RC_L][D];                // q^ * scale
    float kh[RC_L][D];                // k^
    float al[RC_L][D];                // alpha
    float b[RC_L];
};
struct RcSmem {
    RawTile raw[2];
    PrepTile prep;
    float gd[D];                      // gz dt_bias per key channel
    uint16_t rawb[RC_L];
};

// key of register group f (4 consecutive keys) for key quarter kq: fp32 states are read as 16-byte
// pieces interleaved by quarter, bf16 states as 16-byte pieces of 8 keys interleaved by quarter
template <int STATE>
__device__ __forceinline__ int kbase(int f, int kq)
{
    return STATE == 1 ? 32 * (f >> 1) + 8 * kq + 4 * (f & 1) : 16 * f + 4 * kq;
}

__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

template <int STATE, bool VARLEN>  // STATE: 0 none, 1 bf16, 2 fp32
__global__ void __launch_bounds__(RC_THREADS, 2) kda_recurrent_kernel(const Problem p)
{
    extern __shared__ __align__(16) unsigned char rc_smem_raw[];
    RcSmem &sm = *reinterpret_cast<RcSmem *>(rc_smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.H;
    const int h = blockIdx.x % H;
    const int n = blockIdx.x / H;
    const int vhalf = blockIdx.y;
    int64_t bos;
    int len;                           // sequences of this path are shorter than 2^31 tokens
    if (VARLEN) {
        bos = p.cu[n];
        len = (int)(p.cu[n + 1] - bos);
    } else {
        bos = (int64_t)n * p.T;
        len = (int)p.T;
    }
    const int kq = lane & 3;
    const int vl = warp * 8 + (lane >> 2);            // value within this CTA's half
    const int vv = vhalf * RC_VALUES + vl;
    const size_t srow = (((size_t)n * H + h) * D + vv) * D;
    const int ntiles = (len + RC_L - 1) / RC_L;

    // raw tile t0 .. t0 + cnt - 1 -> sm.raw[buf] (cp.async, one commit group)
    auto issue_tile = [&](int tile, int buf) {
        const int t0 = tile * RC_L;
        const int cnt = min(RC_L, len - t0);
        for (int c = tid; c < cnt * RC_CHUNKS_PER_TOKEN; c += RC_THREADS) {
            const int tt = c / RC_CHUNKS_PER_TOKEN, r = c - tt * RC_CHUNKS_PER_TOKEN;
            const size_t row = ((size_t)(bos + t0 + tt) * H + h) * D;
            const __nv_bfloat16 *src;
            uint16_t *dst;
            if (r < 48) {
                const int which = r >> 4, part = r & 15;
                src = (which == 0 ? p.q : which == 1 ? p.k : p.g) + row + part * 8;
                dst = (which == 0 ? sm.raw[buf].q[tt] : which == 1 ? sm.raw[buf].k[tt] : sm.raw[buf].g[tt]) +
                      part * 8;
            } else {
                const int part = r - 48;
                src = p.v + row + vhalf * RC_VALUES + part * 8;
                dst = sm.raw[buf].v[tt] + part * 8;
            }
            cp_async16(smem_u32(dst), src, true);
        }
        cp_async_commit();
    };
    auto load_beta = [&](int tile) -> uint16_t {
        const int t = tile * RC_L + tid;
        return (tid < RC_L && t < len) ? __bfloat16_as_ushort(p.beta[(bos + t) * H + h]) : (uint16_t)0;
    };

    uint16_t bcur = 0;
    if (ntiles > 0) {
        issue_tile(0, 0);
        bcur = load_beta(0);
    }

    // -------- S[32 keys][vv] in registers
    float S[32];
    if (STATE == 2 && p.init) {
        const float *src = static_cast<const float *>(p.init) + srow;
#pragma unroll
        for (int f = 0; f < 8; ++f) {
            const float4 x = *reinterpret_cast<const float4 *>(src + kbase<2>(f, kq));
            S[4 * f] = x.x; S[4 * f + 1] = x.y; S[4 * f + 2] = x.z; S[4 * f + 3] = x.w;
        }
    } else if (STATE == 1 && p.init) {
        const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(p.init) + srow;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint4 x = *reinterpret_cast<const uint4 *>(src + 32 * e + 8 * kq);
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int f = 0; f < 4; ++f) {
                S[8 * e + 2 * f] = bf16_lo(w[f]);
                S[8 * e + 2 * f + 1] = bf16_hi(w[f]);
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < 32; ++e)
            S[e] = 0.f;
    }

    // per-channel gate constants of this lane's prep channels 4 lane .. 4 lane + 3:
    // alpha = 2^(lower_bound log2(e) / (1 + 2^(gz g + gd))), gz = -exp(A_log) log2(e), gd = gz dt_bias
    const float gz = -expf(p.A_log[h]) * LOG2E;
    if (tid < D)
        sm.gd[tid] = gz * p.dt_bias[(size_t)h * D + tid];   // visible after the first tile barrier
    __nv_bfloat16 *outp = p.out + ((size_t)bos * H + h) * D + vv;

    for (int tile = 0; tile < ntiles; ++tile) {
        const int buf = tile & 1;
        const int cnt = min(RC_L, len - tile * RC_L);
        if (tid < RC_L)
            sm.rawb[tid] = bcur;      // the previous tile's prep pass has read rawb (barrier before its loop)
        uint16_t bnext = 0;
        if (tile + 1 < ntiles) {
            issue_tile(tile + 1, buf ^ 1);   // raw[buf ^ 1] was read by the previous prep pass
            bnext = load_beta(tile + 1);
            cp_async_wait_1();
        } else {
            cp_async_wait_all();
        }
        __syncthreads();   // raw[buf] and rawb complete; the previous serial loop is done with sm.prep

        // -------- prep pass: warp w prepares tokens w and w + 8 (channels 4 lane .. 4 lane + 3)
        for (int tt = warp; tt < cnt; tt += RC_WARPS) {
            const uint2 qw = *reinterpret_cast<const uint2 *>(&sm.raw[buf].q[tt][4 * lane]);
            const uint2 kw = *reinterpret_cast<const uint2 *>(&sm.raw[buf].k[tt][4 * lane]);
            const uint2 gw = *reinterpret_cast<const uint2 *>(&sm.raw[buf].g[tt][4 * lane]);
            const float q4[4] = {bf16_lo(qw.x), bf16_hi(qw.x), bf16_lo(qw.y), bf16_hi(qw.y)};
            const float k4[4] = {bf16_lo(kw.x), bf16_hi(kw.x), bf16_lo(kw.y), bf16_hi(kw.y)};
            const float g4[4] = {bf16_lo(gw.x), bf16_hi(gw.x), bf16_lo(gw.y), bf16_hi(gw.y)};
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                sq = fmaf(q4[j], q4[j], sq);
                sk = fmaf(k4[j], k4[j], sk);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            const float rq = rsqrtf(sq + 1e-6f) * p.scale, rk = rsqrtf(sk + 1e-6f);
            const float4 gd4 = *reinterpret_cast<const float4 *>(&sm.gd[4 * lane]);
            const float gd[4] = {gd4.x, gd4.y, gd4.z, gd4.w};
            float a4[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                a4[j] = ex2_approx(p.lb_log2e * rcp_approx(1.f + ex2_approx(fmaf(g4[j], gz, gd[j]))));
            *reinterpret_cast<float4 *>(&sm.prep.qh[tt][4 * lane]) =
                make_float4(q4[0] * rq, q4[1] * rq, q4[2] * rq, q4[3] * rq);
            *reinterpret_cast<float4 *>(&sm.prep.kh[tt][4 * lane]) =
                make_float4(k4[0] * rk, k4[1] * rk, k4[2] * rk, k4[3] * rk);
            *reinterpret_cast<float4 *>(&sm.prep.al[tt][4 * lane]) = make_float4(a4[0], a4[1], a4[2], a4[3]);
            if (lane == 0)
                sm.prep.b[tt] = sigmoid_fast(__uint_as_float((uint32_t)sm.rawb[tt] << 16));
        }
        __syncthreads();

        // -------- serial loop over the tile's tokens (no barriers)
        for (int tt = 0; tt < cnt; ++tt) {
            const float *al = sm.prep.al[tt], *kh = sm.prep.kh[tt], *qh = sm.prep.qh[tt];
            float pk = 0.f, pk2 = 0.f;
#pragma unroll
            for (int f = 0; f < 8; ++f) {
                const int kb = kbase<STATE>(f, kq);
                const float4 a = *reinterpret_cast<const float4 *>(al + kb);
                const float4 kk = *reinterpret_cast<const float4 *>(kh + kb);
                S[4 * f] *= a.x; S[4 * f + 1] *= a.y; S[4 * f + 2] *= a.z; S[4 * f + 3] *= a.w;
                pk = fmaf(S[4 * f], kk.x, pk);
                pk2 = fmaf(S[4 * f + 1], kk.y, pk2);
                pk = fmaf(S[4 * f + 2], kk.z, pk);
                pk2 = fmaf(S[4 * f + 3], kk.w, pk2);
            }
            pk += pk2;
            pk += __shfl_xor_sync(0xffffffffu, pk, 1);
            pk += __shfl_xor_sync(0xffffffffu, pk, 2);
            const float vt = __uint_as_float((uint32_t)sm.raw[buf].v[tt][vl] << 16);
            const float u = sm.prep.b[tt] * (vt - pk);
            float po = 0.f, po2 = 0.f;
#pragma unroll
            for (int f = 0; f < 8; ++f) {
                const int kb = kbase<STATE>(f, kq);
                const float4 kk = *reinterpret_cast<const float4 *>(kh + kb);
                const float4 qq = *reinterpret_cast<const float4 *>(qh + kb);
                S[4 * f] = fmaf(kk.x, u, S[4 * f]);
                S[4 * f + 1] = fmaf(kk.y, u, S[4 * f + 1]);
                S[4 * f + 2] = fmaf(kk.z, u, S[4 * f + 2]);
                S[4 * f + 3] = fmaf(kk.w, u, S[4 * f + 3]);
                po = fmaf(S[4 * f], qq.x, po);
                po2 = fmaf(S[4 * f + 1], qq.y, po2);
                po = fmaf(S[4 * f + 2], qq.z, po);
                po2 = fmaf(S[4 * f + 3], qq.w, po2);
            }
            po += po2;
            po += __shfl_xor_sync(0xffffffffu, po, 1);
            po += __shfl_xor_sync(0xffffffffu, po, 2);
            if (kq == 0)
                *outp = __float2bfloat16_rn(po);
            outp += (size_t)H * D;
        }
        bcur = bnext;
    }

    // -------- final state
    if (STATE == 2 && p.fin) {
        float *dst = static_cast<float *>(p.fin) + srow;
#pragma unroll
        for (int f = 0; f < 8; ++f)
            *reinterpret_cast<float4 *>(dst + kbase<2>(f, kq)) =
                make_float4(S[4 * f], S[4 * f + 1], S[4 * f + 2], S[4 * f + 3]);
    } else if (STATE == 1 && p.fin) {
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.fin) + srow;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            uint32_t w[4];
#pragma unroll
            for (int f = 0; f < 4; ++f) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(S[8 * e + 2 * f], S[8 * e + 2 * f + 1]);
                w[f] = *reinterpret_cast<const uint32_t *>(&b2);
            }
            *reinterpret_cast<uint4 *>(dst + 32 * e + 8 * kq) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

template <int S, bool V>
cudaError_t launch_one(const Problem &p, cudaStream_t stream)
{
    static bool configured[64] = {};
    const int smem = (int)sizeof(RcSmem);
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev >= 64 || !configured[dev]) {
        err = cudaFuncSetAttribute(kda_recurrent_kernel<S, V>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess)
            return err;
        if (dev < 64)
            configured[dev] = true;
    }
    kda_recurrent_kernel<S, V><<<dim3((unsigned)(p.N * p.H), D / RC_VALUES), RC_THREADS, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t recurrent_smem_bytes() { return sizeof(RcSmem); }

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

}  // namespace kda
