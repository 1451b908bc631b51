// C ABI of the KDA forward library (include/kda.h): argument checks, workspace layout and the
// launch sequence  [plan (varlen only)] -> prep -> recurrence  on the caller's stream.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "kda.h"
#include "kda_device.cuh"
#include "kda_internal.h"
#include "kda_plan.h"

// Set by the varlen plan kernel when cu_seqlens breaks its contract (read by kda_device_status).
__device__ unsigned int g_kda_plan_error;

namespace kda {
namespace {

constexpr int PLAN_THREADS = 1024;
std::atomic<uint32_t> g_wait_polls{KDA_DEFAULT_WAIT_POLLS};   // kda_set_wait_limit
constexpr int LPT_MAX_SEQS = 2048;   // longest-first ordering of varlen sequences up to this count

// Varlen plan, one CTA: chunk_off[n] = sum_{m < n} ceil(len_m / 64) (exclusive scan, [N + 1]);
// chunk_info[c] = (first token, tokens left in the sequence) of every chunk c < chunk_off[N] and (0, 0)
// for the launched chunk indices past it (c < n_info), so that a prep CTA finds its chunk, or that it
// has none, with one load; and, when order != nullptr, order[rank] =
// sequence with that rank by length (longest first, ties by index), so that the recurrence CTAs
// that start first take the longest sequences.  Sequences are the clamped ranges of seq_range and
// the table writes stop at n_info, so a malformed cu_seqlens cannot move an access out of its buffer;
// it sets DEVERR_CU_SEQLENS instead.
__global__ void __launch_bounds__(PLAN_THREADS) kda_plan_kernel(const int64_t *cu, int N, int64_t T,
                                                              int64_t *chunk_off, longlong2 *chunk_info,
                                                              int64_t n_info, int *order)
{
    __shared__ int64_t wsum[PLAN_THREADS / 32];
    __shared__ int64_t carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    bool bad = false;
    if (tid == 0)
        carry = 0;
    __syncthreads();
    for (int base = 0; base < N; base += PLAN_THREADS) {
        const int n = base + tid;
        int64_t cnt = 0;
        if (n < N) {
            int64_t bos, len;
            bad |= seq_range(cu, n, N, T, bos, len);
            cnt = seq_chunks(len);
        }
        int64_t x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += y;
        }
        if (lane == 31)
            wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int64_t w = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o)
                    w += y;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        const int64_t excl = carry + (warp > 0 ? wsum[warp - 1] : 0) + x - cnt;
        if (n < N)
            chunk_off[n] = excl;
        __syncthreads();
        if (tid == PLAN_THREADS - 1)
            carry = excl + cnt;
        __syncthreads();
    }
    if (tid == 0)
        chunk_off[N] = carry;
    __syncthreads();   // chunk_off is complete (global writes of this CTA, ordered by the barrier)
    const int64_t used = carry < n_info ? carry : n_info;   // carry > n_info only for a malformed cu_seqlens
    bad |= tid == 0 && carry > n_info;
    for (int64_t c = tid; c < used; c += PLAN_THREADS) {
        const int s = owner_of_chunk(chunk_off, N, c);
        int64_t bos, len;
        seq_range(cu, s, N, T, bos, len);
        const int64_t tok0 = bos + (c - chunk_off[s]) * CH;
        chunk_info[c] = make_longlong2(tok0, bos + len - tok0);
    }
    for (int64_t c = used + tid; c < n_info; c += PLAN_THREADS)
        chunk_info[c] = make_longlong2(0, 0);
    if (order) {
        // longest-first order: a bitonic sort (descending) of the keys length * 4096 + (4095 - index) in shared
        // memory, padded with -1 to m entries (the power of two from N up, at most LPT_MAX_SEQS); ties keep the
        // lower index first.  Each of the log2(m) (log2(m) + 1) / 2 stages is one compare-exchange in each of the
        // first m / 2 threads.
        static_assert(LPT_MAX_SEQS == 2 * PLAN_THREADS && LPT_MAX_SEQS <= 4096, "bitonic sort layout");
        __shared__ int64_t keys[LPT_MAX_SEQS];
        int m = 2;
        while (m < N)
            m <<= 1;
        for (int s = tid; s < m; s += PLAN_THREADS) {
            int64_t bs, ls = -1;
            if (s < N)
                seq_range(cu, s, N, T, bs, ls);
            keys[s] = s < N ? ls * 4096 + (4095 - s) : -1;
        }
        __syncthreads();
        for (int k = 2; k <= m; k <<= 1)
            for (int j = k >> 1; j > 0; j >>= 1) {
                if (tid < (m >> 1)) {
                    const int i = 2 * j * (tid / j) + (tid % j), ixj = i + j;
                    const int64_t x = keys[i], y = keys[ixj];
                    if ((i & k) == 0 ? x < y : x > y) {
                        keys[i] = y;
                        keys[ixj] = x;
                    }
                }
                __syncthreads();
            }
        for (int r = tid; r < N; r += PLAN_THREADS)
            order[r] = 4095 - (int)(keys[r] & 4095);
    }
    if (__syncthreads_or(bad) && tid == 0)
        atomicOr(&g_kda_plan_error, DEVERR_CU_SEQLENS);
}

bool aligned(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int64_t max_chunks(int N, int64_t T, bool varlen)
{
    // varlen: sum_n ceil(len_n / 64) <= (T + 63 N) / 64
    return varlen ? varlen_chunk_capacity(N, T) : (int64_t)N * ((T + CH - 1) / CH);
}

// Long fixed-length problems on few (sequence, head) pairs run in pieces of whole chunks along T: the
// recurrence over piece i (one CTA per pair, on a part of the SMs) runs beside the prep kernel of piece
// i + 1 on the SMs it leaves free, and the state passes from piece to piece in fp32, exactly as the
// recurrence keeps it between chunks, so the results are the same bits as one launch over all chunks.
// With P pieces the overlap hides about (1 - 1/P) of the shorter of two times: the recurrence's (≈1.43 us
// per chunk step on GB300) scaled by the fraction of SMs it leaves free, and the prep kernel's (≈5.9 us
// per (chunk, head) item per SM); each piece costs about 12 us (the prep kernel's last wave and the
// recurrence's start), so the best P is near sqrt(hidden time / 12 us), rounded down.  With more than 64
// pairs the recurrence already draws most of the HBM bandwidth and the pieces measured no gain.
#ifndef KDA_PIECE_MAX_PAIRS
#define KDA_PIECE_MAX_PAIRS 64
#endif
#ifndef KDA_PIECES_FORCE
#define KDA_PIECES_FORCE 0   // > 0: this many pieces wherever piece_mode holds (measurement builds)
#endif
constexpr int MAX_PIECES = 8;
constexpr int64_t PIECE_MIN_CHUNKS = 16;   // chunks per piece at least
constexpr double CHUNK_STEP_US = 1.43;     // the recurrence's chain per 64-token chunk, measured on GB300

bool piece_mode(int N, int64_t T, int H, bool varlen)
{
    return !varlen && (int64_t)N * H <= KDA_PIECE_MAX_PAIRS && (T + CH - 1) / CH >= 2 * PIECE_MIN_CHUNKS;
}

// pieces for a problem of nch chunks per sequence and `pairs` (sequence, head) pairs on nsm SMs
int piece_count(int64_t nch, int64_t pairs, int nsm)
{
    const int64_t most = std::min<int64_t>(MAX_PIECES, nch / PIECE_MIN_CHUNKS);
    int64_t n = KDA_PIECES_FORCE;
    if (n <= 0 && nsm > 0) {
        const double recur_us = CHUNK_STEP_US * (double)nch * (double)std::max<int64_t>(nsm - pairs, 0) / nsm;
        const double prep_us = 5.9 * (double)nch * (double)pairs / nsm;
        n = (int64_t)std::sqrt(std::min(recur_us, prep_us) / 12.0);
    }
    return (int)std::max<int64_t>(1, std::min<int64_t>(n, most));
}

// Fixed-length problems on at most 16 (sequence, head) pairs with long sequences replace the serial chain of the
// recurrence by the chunk-transition scan along T (kda_scan.cu): G groups of L chunks per pair, composed in
// parallel (2 (G - 1) CTAs per pair at ≈1.38 us per chunk step, or G - 1 CTAs that carry both states at ≈2.32 us,
// whichever finishes first in waves of 152 CTAs), chained serially (G - 1 fp32 steps of ≈1.7 us), then run in
// parallel (G CTAs per pair).  G comes from a cost model of those three launches against the
// serial chain (≈1.43 us per chunk, less what the pieces hide) on the 152 SMs of a GB300, with the step
// costs measured there; it depends only on N, T and H, like the workspace that holds the scan's matrices.
#ifndef KDA_SCAN_GROUPS_FORCE
#define KDA_SCAN_GROUPS_FORCE 0   // > 0: this many groups wherever the scan may run (measurement builds)
#endif
constexpr int SCAN_MAX_PAIRS = 16;
constexpr int SCAN_MAX_GROUPS = 32;
constexpr int MODEL_SMS = 152;
constexpr double COMPOSE_STEP_US = 1.38, COMPOSE2_STEP_US = 2.32, SCAN_STEP_US = 1.7, SCAN_FIXED_US = 10.0;

int64_t model_waves(int64_t ctas) { return (ctas + MODEL_SMS - 1) / MODEL_SMS; }
// the compose form for G groups: true = one CTA per (group, pair) carrying both states
bool compose_two_tiles(int64_t pairs, int G)
{
    return (double)model_waves((G - 1) * pairs) * COMPOSE2_STEP_US <
           (double)model_waves(2 * (G - 1) * pairs) * COMPOSE_STEP_US;
}

// (groups, chunks per group) for a scan over nch chunks with about g groups: every group but the last full
int64_t scan_len(int64_t nch, int g) { return (nch + g - 1) / g; }
int scan_groups_of(int64_t nch, int g) { return (int)((nch + scan_len(nch, g) - 1) / scan_len(nch, g)); }

// groups of the scan for this problem; 1 when the recurrence runs as one chain per pair
int scan_groups(int N, int64_t T, int H, bool varlen)
{
    const int64_t pairs = (int64_t)N * H, nch = (T + CH - 1) / CH;
    if (varlen || pairs > SCAN_MAX_PAIRS || nch < 2 * PIECE_MIN_CHUNKS)
        return 1;
    if (KDA_SCAN_GROUPS_FORCE > 1)
        return scan_groups_of(nch, (int)std::min<int64_t>(KDA_SCAN_GROUPS_FORCE, nch));
    // the serial chain, with what the pieces hide behind it
    const double recur_us = CHUNK_STEP_US * (double)nch;
    const double prep_us = 5.9 * (double)nch * (double)pairs / MODEL_SMS;
    const int pc = piece_count(nch, pairs, MODEL_SMS);
    const double hidden = pc > 1 ? std::min(recur_us * (MODEL_SMS - pairs) / MODEL_SMS, prep_us) * (1.0 - 1.0 / pc) -
                                       12.0 * pc : 0.0;
    double best = recur_us - std::max(hidden, 0.0);
    int best_g = 1;
    for (int g = 2; g <= SCAN_MAX_GROUPS && g <= nch; ++g) {
        const int G = scan_groups_of(nch, g);
        const double L = (double)scan_len(nch, g);
        const double compose = compose_two_tiles(pairs, G) ? model_waves((G - 1) * pairs) * COMPOSE2_STEP_US
                                                           : model_waves(2 * (G - 1) * pairs) * COMPOSE_STEP_US;
        const double t = compose * L + (G - 1) * SCAN_STEP_US + model_waves(G * pairs) * L * CHUNK_STEP_US +
                         SCAN_FIXED_US;
        if (t < best) {
            best = t;
            best_g = G;
        }
    }
    return best_g;
}

// workspace: a header, then the operand slots (256-byte aligned).  varlen: the plan, [chunk_off: (N + 1)
// int64][order: N int32][chunk_info: max_chunks x (int64, int64), 16-byte aligned]; fixed length with the
// scan: [initial state][M_g][B_g][start states], fp32 [N][H][128][128] each, the last three for G - 1 groups;
// fixed length in pieces: the fp32 state passed between pieces, [N][H][128][128]; otherwise nothing.
size_t info_offset(int N) { return round_up((size_t)(N + 1) * 8 + (size_t)N * 4, 16); }
size_t header_bytes(int N, int64_t T, int H, bool varlen)
{
    if (varlen)
        return round_up(info_offset(N) + (size_t)max_chunks(N, T, true) * 16, 256);
    const size_t state = (size_t)N * H * D * D * sizeof(float);
    const int G = scan_groups(N, T, H, false);
    if (G > 1)
        return (1 + 3 * (size_t)(G - 1)) * state;
    return piece_mode(N, T, H, false) ? state : 0;
}

}  // namespace

// Fixed-length problems of at most SHORT_T tokens per sequence (decode steps, short speculative runs) are
// evaluated token by token by the kernels of kda_fwd_recurrent: they stream the state once and need no
// workspace.  With one chunk per sequence the chunked path pays its per-chunk costs whatever T is, and the
// token-by-token cost grows with T: measured on GB300 at 8 to 256 sequences x 96 heads, the token-recurrent
// kernels are faster up to 16 tokens (2.6x at 5, 1.1x at 16) and slower from 24.
constexpr int64_t SHORT_T = 16;
bool short_problem(int N, int64_t T, int H, bool varlen)
{
    return !varlen && T >= 1 && T <= SHORT_T && 2 * (int64_t)N * H <= INT32_MAX;
}

size_t workspace_bytes(int N, int64_t T, int H, bool varlen)
{
    if (short_problem(N, T, H, varlen))
        return 0;
    // checked arguments: N >= 1, H >= 1, 0 <= T <= 2^40, so the varlen chunk bound fits; the fixed-length
    // count and the slot bytes may not fit in 64 bits
    uint64_t chunks = 0;
    if (varlen)
        chunks = (uint64_t)max_chunks(N, T, true);
    else if (__builtin_mul_overflow((uint64_t)N, ((uint64_t)T + CH - 1) / CH, &chunks))
        return SIZE_MAX;
    uint64_t slots = 0, bytes = 0, total = 0;
    if (__builtin_mul_overflow(chunks, (uint64_t)H, &slots) || __builtin_mul_overflow(slots, (uint64_t)SLOT_BYTES, &bytes) ||
        __builtin_add_overflow(bytes, (uint64_t)header_bytes(N, T, H, varlen), &total) || total > (uint64_t)SIZE_MAX)
        return SIZE_MAX;
    return (size_t)total;
}

kda_status_t check_size(int N, int64_t T, int H, bool varlen)
{
    if (short_problem(N, T, H, varlen))
        return KDA_OK;
    if (workspace_bytes(N, T, H, varlen) == SIZE_MAX)
        return KDA_ERR_UNSUPPORTED;
    // one prep CTA per (chunk, head): the grid and the kernels' item arithmetic are 32-bit
    const uint64_t items = (uint64_t)(varlen ? max_chunks(N, T, true) : (int64_t)N * ((T + CH - 1) / CH)) * (uint64_t)H;
    return items > (uint64_t)INT32_MAX ? KDA_ERR_UNSUPPORTED : KDA_OK;
}

namespace {

std::mutex g_pool_mu;
cudaMemPool_t g_pools[64] = {};

// A memory pool owned by this library (one per device) that keeps what it has reserved, so
// repeated calls reuse the same workspace memory without a device synchronisation.
cudaError_t get_pool(int dev, cudaMemPool_t *out)
{
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_pool_mu);
    if (!g_pools[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool;
        cudaError_t err = cudaMemPoolCreate(&pool, &props);
        if (err != cudaSuccess)
            return err;
        uint64_t keep = UINT64_MAX;
        err = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (err != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return err;
        }
        g_pools[dev] = pool;
    }
    *out = g_pools[dev];
    return cudaSuccess;
}

}  // namespace

cudaError_t pool_alloc(void **p, size_t bytes, cudaStream_t stream)
{
    *p = nullptr;
    if (bytes == 0)
        return cudaSuccess;
    int dev = 0;
    cudaMemPool_t pool;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess)
        err = get_pool(dev, &pool);
    if (err == cudaSuccess)
        err = cudaMallocFromPoolAsync(p, bytes, pool, stream);
    return err;
}

kda_status_t check_args(const void *q, const void *k, const void *v, const void *g, const void *beta, float scale,
                        const void *out, const float *A_log, const float *dt_bias, float lower_bound,
                        const void *initial_state, const void *final_state, kda_dtype_t state_dtype,
                        const int64_t *cu_seqlens, int N, int64_t T, int H)
{
    if (N < 1 || H < 1 || T < 0)
        return KDA_ERR_INVALID_ARGUMENT;
    // with no tokens at all the token tensors may be empty (NULL)
    if (T > 0 && (!q || !k || !v || !g || !beta || !out))
        return KDA_ERR_INVALID_ARGUMENT;
    if (!A_log || !dt_bias)
        return KDA_ERR_INVALID_ARGUMENT;
    if ((int64_t)N * H > INT32_MAX || T > ((int64_t)1 << 40))
        return KDA_ERR_INVALID_ARGUMENT;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(g, 16) || !aligned(out, 16) ||
        !aligned(beta, 2) || !aligned(A_log, 4) || !aligned(dt_bias, 16) || !aligned(cu_seqlens, 8))
        return KDA_ERR_INVALID_ARGUMENT;
    if (initial_state || final_state) {
        if (state_dtype != KDA_DTYPE_BF16 && state_dtype != KDA_DTYPE_FP32)
            return KDA_ERR_INVALID_ARGUMENT;
        if (!aligned(initial_state, 16) || !aligned(final_state, 16))
            return KDA_ERR_INVALID_ARGUMENT;
    }
    if (!(lower_bound >= -5.0f && lower_bound <= 0.0f))
        return KDA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale))
        return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

namespace {

// The kernels' view of one call (pointers and sizes; the workspace fields are set by the caller).
Problem make_problem(const void *q, const void *k, const void *v, const void *g, const void *beta, float scale,
                     void *out, const float *A_log, const float *dt_bias, float lower_bound, const void *initial_state,
                     void *final_state, const int64_t *cu_seqlens, int N, int64_t T, int H)
{
    Problem p;
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
    p.nch_fixed = (T + CH - 1) / CH;
    p.ch_base = 0;
    p.groups = 1;
    p.group_len = p.nch_fixed;
    p.sc_a = p.sc_b = nullptr;
    p.sc_s = nullptr;
    p.chunk_off = nullptr;
    p.chunk_info = nullptr;
    p.order = nullptr;
    p.slots = nullptr;
    p.prep_pf = 0;
    p.chunk_cap = cu_seqlens ? varlen_chunk_capacity(N, T) : 0;
    p.wait_polls = g_wait_polls.load(std::memory_order_relaxed);
    p.variant = 0;
    return p;
}

int state_kind(const void *initial_state, const void *final_state, kda_dtype_t state_dtype)
{
    return (initial_state || final_state) ? (state_dtype == KDA_DTYPE_FP32 ? 2 : 1) : 0;
}

// SMs of the current device (looked up once per device)
cudaError_t sm_count(int *nsm)
{
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    int n = dev >= 0 && dev < 64 ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (n == 0) {
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            cache[dev].store(n, std::memory_order_relaxed);
    }
    *nsm = n;
    return cudaSuccess;
}

// pieces of a (checked) problem on the current device; 1 without pieces
cudaError_t pieces_on_device(int N, int64_t T, int H, bool varlen, int *pieces)
{
    *pieces = 1;
    if (!piece_mode(N, T, H, varlen) || scan_groups(N, T, H, varlen) > 1)
        return cudaSuccess;
    int nsm = 0;
    const cudaError_t e = sm_count(&nsm);
    if (e == cudaSuccess)
        *pieces = piece_count((T + CH - 1) / CH, (int64_t)N * H, nsm);
    return e;
}

// The chunk-transition scan (see scan_groups): prep over every chunk, the groups' transitions, their start
// states, then the grouped recurrence.  The initial state is first copied (fp32) or converted (bf16) into
// the header, so that the last group's final state may overwrite the caller's initial state (in place)
// while other groups start; a bf16 final state goes through the last start-state buffer, which only the
// last group's CTAs read (each its own rows, before writing them).
cudaError_t run_scan(const Problem &p, int groups, int state_kind, kda_dtype_t state_dtype, unsigned char *ws,
                     cudaStream_t stream)
{
    const size_t mat = (size_t)D * D, pairs = (size_t)p.N * p.H;
    float *st0 = reinterpret_cast<float *>(ws);
    float *ma = st0 + pairs * mat, *mb = ma + (groups - 1) * pairs * mat, *ss = mb + (groups - 1) * pairs * mat;
    const bool bf16 = state_kind != 0 && state_dtype == KDA_DTYPE_BF16;
    const float *init0 = nullptr;
    cudaError_t e = cudaSuccess;
    if (p.init) {
        e = bf16 ? launch_convert(p.init, st0, pairs * mat, true, stream)
                 : cudaMemcpyAsync(st0, p.init, pairs * mat * sizeof(float), cudaMemcpyDeviceToDevice, stream);
        init0 = st0;
    }
    if (e == cudaSuccess)
        e = launch_prep(p, (int64_t)p.N * p.nch_fixed, stream);
    Problem q = p;
    q.groups = groups;
    q.group_len = scan_len(p.nch_fixed, groups);
    q.sc_a = ma;
    q.sc_b = mb;
    q.sc_s = ss;
    q.init = init0;
    float *last = ss + (size_t)(groups - 2) * pairs * mat;
    q.fin = bf16 ? (p.fin ? last : nullptr) : p.fin;
    if (e == cudaSuccess)
        e = launch_compose(q, compose_two_tiles((int64_t)pairs, groups), stream);
    if (e == cudaSuccess)
        e = launch_scan_states(init0, ma, mb, ss, (int)pairs, groups, stream);
    if (e == cudaSuccess)
        e = launch_recur(q, 2, stream);
    if (e == cudaSuccess && bf16 && p.fin)
        e = launch_convert(last, p.fin, pairs * mat, false, stream);
    return e;
}

// Piece i covers chunks [nch i / P, nch (i + 1) / P) of every sequence; everything runs on the caller's
// stream.  The prep kernel of piece i + 1 (one CTA per item, so that it takes SMs as they come free) is launched as a programmatic dependent of the
// recurrence over piece i: it starts once every recurrence CTA runs (one per pair, on a part of the SMs),
// fills the SMs they leave free, and its last CTA waits for that recurrence to complete before it exits.
// The recurrence over piece i + 1 is a normal launch after that prep kernel, so it starts after both.  The
// state between pieces is the workspace header (fp32); a bf16 initial or final state is converted into or
// out of it.
cudaError_t run_pieces(const Problem &p, int pieces, int state_kind, kda_dtype_t state_dtype, unsigned char *ws,
                       cudaStream_t stream)
{
    float *st = reinterpret_cast<float *>(ws);
    const size_t st_elems = (size_t)p.N * p.H * D * D;
    const bool bf16 = state_kind != 0 && state_dtype == KDA_DTYPE_BF16;
    const void *init0 = p.init;
    cudaError_t e = cudaSuccess;
    if (bf16 && p.init) {
        e = launch_convert(p.init, st, st_elems, true, stream);
        init0 = st;
    }
    const int64_t nch = p.nch_fixed;
    for (int i = 0; i < pieces && e == cudaSuccess; ++i) {
        const int64_t c0 = nch * i / pieces, c1 = nch * (i + 1) / pieces;
        Problem q = p;
        q.ch_base = c0;
        q.nch_fixed = c1 - c0;
        q.group_len = c1 - c0;
        q.slots = p.slots + (size_t)p.N * c0 * p.H * SLOT_BYTES;
        q.init = i == 0 ? init0 : st;
        q.fin = i < pieces - 1 ? st : (bf16 ? (p.fin ? st : nullptr) : p.fin);
        // piece 0 has the GPU to itself (persistent grid); later pieces run beside a recurrence
        e = launch_prep(q, (int64_t)p.N * (c1 - c0), stream, i == 0, i > 0);
        if (e == cudaSuccess)
            e = launch_recur(q, 2, stream);
    }
    if (e == cudaSuccess && bf16 && p.fin)
        e = launch_convert(st, p.fin, st_elems, false, stream);
    return e;
}

}  // namespace

kda_status_t run(const void *q, const void *k, const void *v, const void *g, const void *beta, float scale,
                 void *out, const float *A_log, const float *dt_bias, float lower_bound, const void *initial_state,
                 void *final_state, kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H,
                 unsigned char *ws, cudaStream_t stream, void *const *stage_events, uint32_t variant,
                 bool single_launch)
{
    const bool varlen = cu_seqlens != nullptr;
    auto mark = [&](int i) -> cudaError_t {
        return stage_events && stage_events[i] ? cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), stream)
                                               : cudaSuccess;
    };
    Problem p = make_problem(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, final_state,
                             cu_seqlens, N, T, H);
    if (short_problem(N, T, H, varlen)) {
        const int sk = state_kind(initial_state, final_state, state_dtype);
        cudaError_t e = mark(0);
        if (e == cudaSuccess)
            e = decode_applies(p, sk) ? launch_decode(p, sk, stream) : launch_recurrent(p, sk, stream);
        if (e == cudaSuccess)
            e = mark(1);
        if (e == cudaSuccess)
            e = mark(2);
        return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    }
    p.variant = variant;
    p.slots = ws + header_bytes(N, T, H, varlen);
    // the measurement variants keep the single-launch schedule
    if (!varlen && variant == 0 && !single_launch) {
        const int groups = scan_groups(N, T, H, false);
        if (groups > 1)
            return run_scan(p, groups, state_kind(initial_state, final_state, state_dtype), state_dtype, ws, stream) ==
                           cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    }
    if (piece_mode(N, T, H, varlen) && variant == 0 && !single_launch) {
        int pieces = 0;
        if (pieces_on_device(N, T, H, false, &pieces) != cudaSuccess)
            return KDA_ERR_CUDA;
        if (pieces > 1)
            return run_pieces(p, pieces, state_kind(initial_state, final_state, state_dtype), state_dtype, ws,
                              stream) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    }
    cudaError_t err = cudaSuccess;
    if (varlen) {
        int64_t *chunk_off = reinterpret_cast<int64_t *>(ws);
        int *order = N > 1 && N <= LPT_MAX_SEQS ? reinterpret_cast<int *>(ws + (size_t)(N + 1) * 8) : nullptr;
        longlong2 *chunk_info = reinterpret_cast<longlong2 *>(ws + info_offset(N));
        kda_plan_kernel<<<1, PLAN_THREADS, 0, stream>>>(cu_seqlens, N, T, chunk_off, chunk_info,
                                                        max_chunks(N, T, true), order);
        err = cudaGetLastError();
        p.chunk_off = chunk_off;
        p.chunk_info = chunk_info;
        p.order = order;
    }
    if (err == cudaSuccess)
        err = mark(0);
    if (err == cudaSuccess)
        err = launch_prep(p, max_chunks(N, T, varlen), stream);
    if (err == cudaSuccess)
        err = mark(1);
    const int st = state_kind(initial_state, final_state, state_dtype);
    if (err == cudaSuccess)
        err = launch_recur(p, st, stream);
    if (err == cudaSuccess)
        err = mark(2);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda

using namespace kda;

extern "C" size_t kda_fwd_workspace_size(int N, int64_t T, int H, int varlen)
{
    if (N < 1 || H < 1 || T < 0 || T > ((int64_t)1 << 40) || (int64_t)N * H > INT32_MAX ||
        check_size(N, T, H, varlen != 0) != KDA_OK)
        return 0;
    return workspace_bytes(N, T, H, varlen != 0);
}

extern "C" int kda_fwd_pieces(int N, int64_t T, int H, int varlen)
{
    if (N < 1 || H < 1 || T < 0 || T > ((int64_t)1 << 40) || (int64_t)N * H > INT32_MAX ||
        check_size(N, T, H, varlen != 0) != KDA_OK)
        return 0;
    int pieces = 0;
    return pieces_on_device(N, T, H, varlen != 0, &pieces) == cudaSuccess ? pieces : 0;
}

extern "C" int kda_fwd_scan_groups(int N, int64_t T, int H, int varlen)
{
    if (N < 1 || H < 1 || T < 0 || T > ((int64_t)1 << 40) || (int64_t)N * H > INT32_MAX ||
        check_size(N, T, H, varlen != 0) != KDA_OK)
        return 0;
    return scan_groups(N, T, H, varlen != 0);
}

extern "C" kda_status_t kda_fwd_ws(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                   float scale, void *out, const float *A_log, const float *dt_bias,
                                   float lower_bound, const void *initial_state, void *final_state,
                                   kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H,
                                   void *workspace, size_t workspace_bytes_, kda_stream_t stream)
{
    kda_status_t s = check_args(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                                final_state, state_dtype, cu_seqlens, N, T, H);
    if (s == KDA_OK)
        s = check_size(N, T, H, cu_seqlens != nullptr);
    if (s != KDA_OK)
        return s;
    const size_t need = workspace_bytes(N, T, H, cu_seqlens != nullptr);
    if (need > 0 && (!workspace || !aligned(workspace, 256) || workspace_bytes_ < need))
        return KDA_ERR_INVALID_ARGUMENT;
    return run(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, final_state, state_dtype,
               cu_seqlens, N, T, H, static_cast<unsigned char *>(workspace), reinterpret_cast<cudaStream_t>(stream));
}

extern "C" kda_status_t kda_fwd_ws_profiled(const void *q, const void *k, const void *v, const void *g,
                                            const void *beta, float scale, void *out, const float *A_log,
                                            const float *dt_bias, float lower_bound, const void *initial_state,
                                            void *final_state, kda_dtype_t state_dtype, const int64_t *cu_seqlens,
                                            int N, int64_t T, int H, void *workspace, size_t workspace_bytes_,
                                            void *const *stage_events, kda_stream_t stream)
{
    kda_status_t s = check_args(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                                final_state, state_dtype, cu_seqlens, N, T, H);
    if (s == KDA_OK)
        s = check_size(N, T, H, cu_seqlens != nullptr);
    if (s != KDA_OK)
        return s;
    const size_t need = workspace_bytes(N, T, H, cu_seqlens != nullptr);
    if (need > 0 && (!workspace || !aligned(workspace, 256) || workspace_bytes_ < need))
        return KDA_ERR_INVALID_ARGUMENT;
    return run(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, final_state, state_dtype,
               cu_seqlens, N, T, H, static_cast<unsigned char *>(workspace), reinterpret_cast<cudaStream_t>(stream),
               stage_events, 0, true);
}

extern "C" kda_status_t kda_fwd_ws_variant(const void *q, const void *k, const void *v, const void *g,
                                           const void *beta, float scale, void *out, const float *A_log,
                                           const float *dt_bias, float lower_bound, const void *initial_state,
                                           void *final_state, kda_dtype_t state_dtype, const int64_t *cu_seqlens,
                                           int N, int64_t T, int H, void *workspace, size_t workspace_bytes_,
                                           unsigned variant, kda_stream_t stream)
{
    kda_status_t s = check_args(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                                final_state, state_dtype, cu_seqlens, N, T, H);
    if (s == KDA_OK)
        s = check_size(N, T, H, cu_seqlens != nullptr);
    if (s != KDA_OK)
        return s;
    if (variant & ~(unsigned)(KDA_VARIANT_BF16_STATE | KDA_VARIANT_NEUMANN_INVERSE))
        return KDA_ERR_INVALID_ARGUMENT;
    const size_t need = workspace_bytes(N, T, H, cu_seqlens != nullptr);
    if (need > 0 && (!workspace || !aligned(workspace, 256) || workspace_bytes_ < need))
        return KDA_ERR_INVALID_ARGUMENT;
    return run(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, final_state, state_dtype,
               cu_seqlens, N, T, H, static_cast<unsigned char *>(workspace), reinterpret_cast<cudaStream_t>(stream),
               nullptr, variant);
}

extern "C" kda_status_t kda_fwd(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                float scale, void *out, const float *A_log, const float *dt_bias,
                                float lower_bound, const void *initial_state, void *final_state,
                                kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H,
                                kda_stream_t stream)
{
    kda_status_t s = check_args(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                                final_state, state_dtype, cu_seqlens, N, T, H);
    if (s == KDA_OK)
        s = check_size(N, T, H, cu_seqlens != nullptr);
    if (s != KDA_OK)
        return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t need = workspace_bytes(N, T, H, cu_seqlens != nullptr);
    void *ws = nullptr;
    if (need > 0) {
        int dev = 0;
        cudaMemPool_t pool;
        if (cudaGetDevice(&dev) != cudaSuccess || get_pool(dev, &pool) != cudaSuccess ||
            cudaMallocFromPoolAsync(&ws, need, pool, st) != cudaSuccess)
            return KDA_ERR_CUDA;
    }
    s = run(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, final_state, state_dtype,
            cu_seqlens, N, T, H, static_cast<unsigned char *>(ws), st);
    if (ws && cudaFreeAsync(ws, st) != cudaSuccess && s == KDA_OK)
        s = KDA_ERR_CUDA;
    return s;
}

extern "C" kda_status_t kda_fwd_recurrent(const void *q, const void *k, const void *v, const void *g,
                                          const void *beta, float scale, void *out, const float *A_log,
                                          const float *dt_bias, float lower_bound, const void *initial_state,
                                          void *final_state, kda_dtype_t state_dtype, const int64_t *cu_seqlens,
                                          int N, int64_t T, int H, kda_stream_t stream)
{
    kda_status_t s = check_args(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                                final_state, state_dtype, cu_seqlens, N, T, H);
    if (s != KDA_OK)
        return s;
    if (T > INT32_MAX || 2 * (int64_t)N * H > INT32_MAX)
        return KDA_ERR_UNSUPPORTED;
    const Problem p = make_problem(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                                   final_state, cu_seqlens, N, T, H);
    const int sk = state_kind(initial_state, final_state, state_dtype);
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t err = decode_applies(p, sk) ? launch_decode(p, sk, st) : launch_recurrent(p, sk, st);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

extern "C" kda_status_t kda_fwd_host(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                     float scale, void *out, const float *A_log, const float *dt_bias,
                                     float lower_bound, const void *initial_state, void *final_state,
                                     kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H)
{
    kda_status_t s = check_args(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                                final_state, state_dtype, cu_seqlens, N, T, H);
    if (s == KDA_OK)
        s = check_size(N, T, H, cu_seqlens != nullptr);
    if (s != KDA_OK)
        return s;
    if (cu_seqlens && kda_check_cu_seqlens(cu_seqlens, N, T) != KDA_OK)
        return KDA_ERR_INVALID_ARGUMENT;
    return run_host(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, final_state, state_dtype,
                    cu_seqlens, N, T, H);
}

extern "C" kda_status_t kda_workspace_trim(void)
{
    std::lock_guard<std::mutex> lock(g_pool_mu);
    for (cudaMemPool_t pool : g_pools)
        if (pool && cudaMemPoolTrimTo(pool, 0) != cudaSuccess)
            return KDA_ERR_CUDA;
    return KDA_OK;
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
    case KDA_ERR_NONFINITE: return "non-finite state (fp16 operand range exceeded or inf/NaN input)";
    }
    return "unknown status";
}

extern "C" void kda_set_wait_limit(uint32_t polls) { g_wait_polls.store(polls, std::memory_order_relaxed); }

extern "C" size_t kda_fwd_smem_bytes(void)
{
    const size_t a = prep_smem_bytes(), b = recur_smem_bytes();
    return a > b ? a : b;
}

extern "C" kda_status_t kda_device_status(kda_stream_t stream)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KDA_ERR_CUDA;
    unsigned int flag = 0, flag2 = 0, flag3 = 0, flag4 = 0, flag5 = 0;
    if (read_and_clear_device_error(&flag) != cudaSuccess || prep_read_and_clear_error(&flag2) != cudaSuccess ||
        recurrent_read_and_clear_error(&flag3) != cudaSuccess || decode_read_and_clear_error(&flag4) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&flag5, g_kda_plan_error, sizeof flag5) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (flag5) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_kda_plan_error, &zero, sizeof zero) != cudaSuccess)
            return KDA_ERR_CUDA;
    }
    const unsigned int bits = flag | flag2 | flag3 | flag4 | flag5;
    if (bits & DEVERR_TIMEOUT)
        return KDA_ERR_TIMEOUT;
    if (bits & DEVERR_CU_SEQLENS)
        return KDA_ERR_INVALID_ARGUMENT;
    if (bits & DEVERR_NONFINITE)
        return KDA_ERR_NONFINITE;
    return KDA_OK;
}
