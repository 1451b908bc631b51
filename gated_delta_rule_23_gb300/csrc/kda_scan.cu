// The serial level of the chunk-transition scan along T: the start states of the groups of chunks.
//
// Without the scan the recurrence kernel walks all chunks of a (sequence, head) pair in one CTA, a chain
// as long as the sequence, while the other SMs wait once the prep kernel is done (the guancyxx.cn FlashKDA
// article, section 2.2).  With it the chunks of every pair are cut into G groups of L chunks:
//   1. per group, in parallel (recurrence kernel, compose form): the group's chunks map a start state S to
//      M S + B, with M the product of the chunks' transitions Diag(Gamma_C) - K~^T W and B the state
//      reached from S = 0;
//   2. serially over the groups (this kernel): S_{g+1} = M_g S_g + B_g from the initial state;
//   3. per group, in parallel (recurrence kernel, grouped form): the outputs of the group's chunks from S_g.
//
// The compose launches store M_g and B_g transposed like a state (a_g[j][k] = M_g[k][j], b_g[v][k] =
// B_g[k][v]), and states are stored transposed (st[v][k] = S[k][v]), so that
//   st_{g+1} = st_g a_g + b_g,
// in which row v of st_{g+1} depends on row v of st_g only.  One CTA per (pair, block of rows) keeps its
// rows in shared memory and walks g = 0 .. G - 2 in fp32 FMAs (no operand rounding: the whole state passes
// through every step), with a_g staged in shared memory by cp.async and its b_g entries in registers, both
// one group ahead.  The step is bound by shared-memory reads of a_g, so each a_g element read serves four rows.
#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int SC_PITCH = D + 4;   // fp32 pitch of the rows (rows 4 apart fall on other banks)
template <int R>
constexpr int sc_smem() { return (2 * D * D + R * SC_PITCH + 4 * R * D) * 4; }

// CTA: R rows of st for one pair (R = 8 or 16), 16 R threads in 4 R / 8 warps.  Warp w takes the quarter
// jq = w % 4 of the sum index j (32 values) for the row octet w / 4; lane: rows 4 (lane / 16) .. + 3 of the
// octet, columns 4 cg .. 4 cg + 3 and 64 + 4 cg .. 64 + 4 cg + 3 (cg = lane % 16), a 4 x 8 register tile, so
// that each a_g element read from shared memory serves four rows and a_g is read once per CTA and step.  The
// four quarters' partial sums meet in shared memory, where thread t adds them (in quarter order) and b_g for
// row t / 16, the same 8 columns.  The launch picks R from the pair count so that the CTAs (one per SM) fit
// in one wave.
template <int R>
__global__ void __launch_bounds__(16 * R) kda_scan_kernel(const float *init0, const float *a, const float *b, float *s,
                                                         int pairs, int groups)
{
    constexpr int BLOCKS = D / R;   // CTAs per pair
    constexpr int NT = 16 * R;
    extern __shared__ __align__(16) float sc[];
    float *abuf = sc;                        // [2][128][128]: a_g in buffer g % 2
    float *rows = sc + 2 * D * D;            // [R][SC_PITCH]: rows of st_g
    float *part = rows + R * SC_PITCH;       // [4 quarters][R][128]: partial sums
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int pair = blockIdx.x / BLOCKS, rb = blockIdx.x - pair * BLOCKS;
    const int jq = warp & 3, r0 = 8 * (warp >> 2) + 4 * (lane >> 4), cg = lane & 15;
    // the reduction: row tr of the block, the same 8 columns
    const int tr = tid >> 4, tcg = tid & 15, v = rb * R + tr;
    const size_t mat = (size_t)D * D;

    auto load_a = [&](int g) {
        const float *src = a + ((size_t)g * pairs + pair) * mat;
        const uint32_t dst = smem_u32(abuf + (g & 1) * mat);
        for (int i = tid; i < D * D / 4; i += NT)
            cp_async16(dst + 16 * i, src + 4 * i, true);
        cp_async_commit();
    };
    // the reduction thread's 8 entries of b_g (row v), loaded one step ahead
    auto load_b = [&](int g, float4 &b0, float4 &b1) {
        const float *src = b + ((size_t)g * pairs + pair) * mat + (size_t)v * D;
        b0 = *reinterpret_cast<const float4 *>(src + 4 * tcg);
        b1 = *reinterpret_cast<const float4 *>(src + 64 + 4 * tcg);
    };
    load_a(0);
    float4 nb0, nb1;
    load_b(0, nb0, nb1);
    for (int i = tid; i < R * D; i += NT) {
        const int rr = i / D, cc = i - rr * D;
        rows[rr * SC_PITCH + cc] = init0 ? init0[(size_t)pair * mat + (size_t)(rb * R + rr) * D + cc] : 0.f;
    }
    for (int g = 0; g + 1 < groups; ++g) {
        // a_{g + 1} streams in while a_g is used (its buffer was last read in step g - 1, before that step's
        // partial-sum barrier)
        if (g + 2 < groups) {
            load_a(g + 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            cp_async_wait_all();
        }
        __syncthreads();
        const float4 b0 = nb0, b1 = nb1;
        if (g + 2 < groups)
            load_b(g + 1, nb0, nb1);
        float acc[4][8];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[i][e] = 0.f;
        const float *am = abuf + (g & 1) * mat + (size_t)(32 * jq) * D + 4 * cg;
        const float *xr = rows + r0 * SC_PITCH + 32 * jq;
#pragma unroll 4
        for (int j = 0; j < 32; ++j) {
            const float4 a0 = *reinterpret_cast<const float4 *>(am + j * D);
            const float4 a1 = *reinterpret_cast<const float4 *>(am + j * D + 64);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float x = xr[i * SC_PITCH + j];
                acc[i][0] = fmaf(x, a0.x, acc[i][0]);
                acc[i][1] = fmaf(x, a0.y, acc[i][1]);
                acc[i][2] = fmaf(x, a0.z, acc[i][2]);
                acc[i][3] = fmaf(x, a0.w, acc[i][3]);
                acc[i][4] = fmaf(x, a1.x, acc[i][4]);
                acc[i][5] = fmaf(x, a1.y, acc[i][5]);
                acc[i][6] = fmaf(x, a1.z, acc[i][6]);
                acc[i][7] = fmaf(x, a1.w, acc[i][7]);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float *pp = part + ((size_t)jq * R + r0 + i) * D;
            *reinterpret_cast<float4 *>(pp + 4 * cg) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            *reinterpret_cast<float4 *>(pp + 64 + 4 * cg) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
        }
        __syncthreads();   // the partial sums are complete; every thread has read the rows of st_g
        float4 o0 = b0, o1 = b1;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float *pp = part + ((size_t)q * R + tr) * D;
            const float4 p0 = *reinterpret_cast<const float4 *>(pp + 4 * tcg);
            const float4 p1 = *reinterpret_cast<const float4 *>(pp + 64 + 4 * tcg);
            o0 = make_float4(o0.x + p0.x, o0.y + p0.y, o0.z + p0.z, o0.w + p0.w);
            o1 = make_float4(o1.x + p1.x, o1.y + p1.y, o1.z + p1.z, o1.w + p1.w);
        }
        *reinterpret_cast<float4 *>(rows + tr * SC_PITCH + 4 * tcg) = o0;
        *reinterpret_cast<float4 *>(rows + tr * SC_PITCH + 64 + 4 * tcg) = o1;
        float *dst = s + ((size_t)g * pairs + pair) * mat + (size_t)v * D;   // st_{g + 1}
        *reinterpret_cast<float4 *>(dst + 4 * tcg) = o0;
        *reinterpret_cast<float4 *>(dst + 64 + 4 * tcg) = o1;
    }
}

template <int R>
cudaError_t launch_scan_r(const float *init0, const float *a, const float *b, float *s, int pairs, int groups,
                          cudaStream_t stream)
{
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev >= 64 || !configured[dev]) {
        err = cudaFuncSetAttribute(kda_scan_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, sc_smem<R>());
        if (err != cudaSuccess)
            return err;
        if (dev < 64)
            configured[dev] = true;
    }
    kda_scan_kernel<R><<<pairs * (D / R), 16 * R, sc_smem<R>(), stream>>>(init0, a, b, s, pairs, groups);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan_states(const float *init0, const float *a, const float *b, float *s, int pairs, int groups,
                               cudaStream_t stream)
{
    if (groups < 2 || pairs < 1)
        return cudaSuccess;
    // the fewest rows per CTA that keep the CTAs (one per SM: two 64 KB matrix buffers) within one wave of a GB300
    if (pairs * (D / 8) <= 152)
        return launch_scan_r<8>(init0, a, b, s, pairs, groups, stream);
    return launch_scan_r<16>(init0, a, b, s, pairs, groups, stream);
}

}  // namespace kda
