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
// in which row v of st_{g+1} depends on row v of st_g only.  One CTA per (pair, block of 16 rows) keeps
// its rows in shared memory and walks g = 0 .. G - 2 in fp32 FMAs (no operand rounding: the whole state
// passes through every step), with a_g staged in shared memory by cp.async one group ahead.
#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int SC_THREADS = 256;
constexpr int SC_ROWS = 16;                    // rows of st per CTA
constexpr int SC_BLOCKS = D / SC_ROWS;         // CTAs per pair
constexpr int SC_PITCH = D + 4;                // fp32 pitch of the rows (two rows a warp reads: other banks)
constexpr int SC_SMEM = 2 * D * D * 4 + SC_ROWS * SC_PITCH * 4;

// thread: row 16 rb + tid / 16, columns 4 cg .. 4 cg + 3 and 64 + 4 cg .. 64 + 4 cg + 3 (cg = tid % 16), so
// that the 16 threads of a row read one contiguous 256-byte run of a_g per float4 load
__global__ void __launch_bounds__(SC_THREADS) kda_scan_kernel(const float *init0, const float *a, const float *b,
                                                              float *s, int pairs, int groups)
{
    extern __shared__ __align__(16) float sc[];
    float *abuf = sc;                     // [2][128][128]: a_g in buffer g % 2
    float *rows = sc + 2 * D * D;         // [16][SC_PITCH]: rows of st_g
    const int tid = threadIdx.x;
    const int pair = blockIdx.x / SC_BLOCKS, rb = blockIdx.x - pair * SC_BLOCKS;
    const int r = tid >> 4, cg = tid & 15, v = rb * SC_ROWS + r;
    const size_t mat = (size_t)D * D;

    auto load_a = [&](int g) {
        const float *src = a + ((size_t)g * pairs + pair) * mat;
        const uint32_t dst = smem_u32(abuf + (g & 1) * mat);
        for (int i = tid; i < D * D / 4; i += SC_THREADS)
            cp_async16(dst + 16 * i, src + 4 * i, true);
        cp_async_commit();
    };
    load_a(0);
    for (int i = tid; i < SC_ROWS * D; i += SC_THREADS) {
        const int rr = i / D, cc = i - rr * D;
        rows[rr * SC_PITCH + cc] = init0 ? init0[(size_t)pair * mat + (size_t)(rb * SC_ROWS + rr) * D + cc] : 0.f;
    }
    for (int g = 0; g + 1 < groups; ++g) {
        // a_{g + 1} streams in while a_g is used (its buffer was last read in step g - 1, before that step's
        // closing barrier)
        if (g + 2 < groups) {
            load_a(g + 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            cp_async_wait_all();
        }
        __syncthreads();
        const size_t base = ((size_t)g * pairs + pair) * mat + (size_t)v * D;
        float acc[8];
        {
            const float4 b0 = *reinterpret_cast<const float4 *>(b + base + 4 * cg);
            const float4 b1 = *reinterpret_cast<const float4 *>(b + base + 64 + 4 * cg);
            acc[0] = b0.x, acc[1] = b0.y, acc[2] = b0.z, acc[3] = b0.w;
            acc[4] = b1.x, acc[5] = b1.y, acc[6] = b1.z, acc[7] = b1.w;
        }
        const float *am = abuf + (g & 1) * mat + 4 * cg;
        const float *xr = rows + r * SC_PITCH;
#pragma unroll 8
        for (int j = 0; j < D; ++j) {
            const float x = xr[j];
            const float4 a0 = *reinterpret_cast<const float4 *>(am + j * D);
            const float4 a1 = *reinterpret_cast<const float4 *>(am + j * D + 64);
            acc[0] = fmaf(x, a0.x, acc[0]);
            acc[1] = fmaf(x, a0.y, acc[1]);
            acc[2] = fmaf(x, a0.z, acc[2]);
            acc[3] = fmaf(x, a0.w, acc[3]);
            acc[4] = fmaf(x, a1.x, acc[4]);
            acc[5] = fmaf(x, a1.y, acc[5]);
            acc[6] = fmaf(x, a1.z, acc[6]);
            acc[7] = fmaf(x, a1.w, acc[7]);
        }
        __syncthreads();   // every thread has read the rows of st_g
        const float4 o0 = make_float4(acc[0], acc[1], acc[2], acc[3]), o1 = make_float4(acc[4], acc[5], acc[6], acc[7]);
        *reinterpret_cast<float4 *>(rows + r * SC_PITCH + 4 * cg) = o0;
        *reinterpret_cast<float4 *>(rows + r * SC_PITCH + 64 + 4 * cg) = o1;
        *reinterpret_cast<float4 *>(s + base + 4 * cg) = o0;   // st_{g + 1}
        *reinterpret_cast<float4 *>(s + base + 64 + 4 * cg) = o1;
    }
}

}  // namespace

cudaError_t launch_scan_states(const float *init0, const float *a, const float *b, float *s, int pairs, int groups,
                               cudaStream_t stream)
{
    if (groups < 2 || pairs < 1)
        return cudaSuccess;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev >= 64 || !configured[dev]) {
        err = cudaFuncSetAttribute(kda_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SC_SMEM);
        if (err != cudaSuccess)
            return err;
        if (dev < 64)
            configured[dev] = true;
    }
    kda_scan_kernel<<<pairs * SC_BLOCKS, SC_THREADS, SC_SMEM, stream>>>(init0, a, b, s, pairs, groups);
    return cudaGetLastError();
}

}  // namespace kda
