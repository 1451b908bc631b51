// Varlen bookkeeping shared by the kernels that read cu_seqlens and by the host-side test that
// restates the chunk plan (plain C++: no CUDA types, so a host compiler can include it).
//
// cu_seqlens is device-resident and not checked before the launch.  These helpers clamp every
// sequence into [0, T] and every chunk-table write into the table, so that a malformed array can
// only give wrong results (reported through a device flag), never an access outside the buffers.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define KDA_HD __host__ __device__ __forceinline__
#else
#define KDA_HD inline
#endif

namespace kda {

constexpr int PLAN_CHUNK = 64;   // tokens per chunk of the chunked path

// Token range [bos, bos + len) of sequence n (0 <= n < N) from cu_seqlens, clamped into [0, T] with
// len >= 0.  Returns true when cu broke its contract at this sequence: cu[n] or cu[n + 1] outside
// [0, T], cu[n + 1] < cu[n], cu[0] != 0 or cu[N] != T.
KDA_HD bool seq_range(const int64_t *cu, int n, int N, int64_t T, int64_t &bos, int64_t &len)
{
    const int64_t a = cu[n], b = cu[n + 1];
    const int64_t lo = a < 0 ? 0 : (a > T ? T : a);
    const int64_t hi = b < lo ? lo : (b > T ? T : b);
    bos = lo;
    len = hi - lo;
    return a != lo || b != hi || (n == 0 && a != 0) || (n == N - 1 && b != T);
}

// Chunks of a sequence of len tokens (the last one may be partial).
KDA_HD int64_t seq_chunks(int64_t len) { return (len + PLAN_CHUNK - 1) / PLAN_CHUNK; }

// Chunk-table capacity of a varlen call: with a valid cu_seqlens, sum_n ceil(len_n / 64) <= (T + 63 N) / 64.
KDA_HD int64_t varlen_chunk_capacity(int N, int64_t T) { return (T + (int64_t)(PLAN_CHUNK - 1) * N) / PLAN_CHUNK; }

// How many of a sequence's `count` chunks, the first at table index `first`, fit in a table of
// `capacity` entries (all of them when cu_seqlens is valid).
KDA_HD int64_t usable_chunks(int64_t first, int64_t count, int64_t capacity)
{
    if (first >= capacity)
        return 0;
    return count < capacity - first ? count : capacity - first;
}

// Sequence owning table index c: the last n with chunk_off[n] <= c (chunk_off non-decreasing, chunk_off[0] = 0).
KDA_HD int owner_of_chunk(const int64_t *chunk_off, int N, int64_t c)
{
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] <= c)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

}  // namespace kda
