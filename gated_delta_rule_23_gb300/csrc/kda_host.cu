// Host-buffer entry point (kda_fwd_host): the forward pass on host memory, with the host-to-device
// copies, the kernels and the device-to-host copies pipelined over pieces of the sequence.
//
// Fixed-length problems are cut into pieces of whole 64-token chunks (big pieces, then a tail that
// halves, so that little work follows the last copy in).  Piece p's rows of q, k, v, g, beta go to a
// device ring slot on a copy-in stream, the forward pass for the piece runs on a compute stream with
// the state chained between pieces in fp32, and the piece's output rows go back on a copy-out stream,
// so the copies of neighbouring pieces overlap the kernels.  Because the pieces start at chunk
// boundaries and the chained state is fp32 (the state the recurrence keeps internally), the results
// are bit-identical to one kda_fwd call over the whole problem (unless either takes the scan along T,
// whose grouping differs).  Varlen problems (cu_seqlens) are cut into pieces of whole sequences, which
// share no state: each piece is a varlen call of its own, with its cu_seqlens shifted to start at 0 and
// its sequences' slices of the states; the longest sequence comes last, in pieces of whole chunks with
// its state chained in fp32.  The results are again the bits of one call (every (sequence, head) pair
// is computed alone, its chunks where one call puts them).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <vector>

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int HOST_RING = 2;            // device piece buffers in flight
constexpr int64_t HOST_MAX_PIECES = 8;  // varlen pieces; fixed-length big pieces
constexpr int64_t HOST_MIN_PIECE = 512; // tokens
constexpr int64_t HOST_TAIL_MIN = 2;    // chunks of the last piece of a halving tail

// Chunks per fixed-length piece.  Copying a token in takes about twice as long as computing it and copying its
// output back, so a piece's compute and copy-out hide behind the copy-in of the pieces after it only if those
// are at least about half its size: up to HOST_MAX_PIECES big pieces of about nch / 8 chunks (at least
// HOST_MIN_PIECE tokens), then a tail that halves down to HOST_TAIL_MIN chunks, so that little work follows the
// last copy in.  One piece when T <= HOST_MIN_PIECE.
std::vector<int64_t> host_piece_chunks(int64_t nch)
{
    if (nch * CH <= HOST_MIN_PIECE)
        return {nch};
    const int64_t big = std::max<int64_t>(HOST_MIN_PIECE / CH, (nch + HOST_MAX_PIECES - 1) / HOST_MAX_PIECES);
    std::vector<int64_t> tail;
    int64_t tail_sum = 0;
    for (int64_t t = HOST_TAIL_MIN; t < big && tail_sum + t <= nch - big; t *= 2) {
        tail.push_back(t);
        tail_sum += t;
    }
    const int64_t rest = nch - tail_sum, nbig = (rest + big - 1) / big;
    std::vector<int64_t> plan;
    for (int64_t i = 0; i < nbig; ++i)
        plan.push_back(rest / nbig + (i < rest % nbig ? 1 : 0));
    plan.insert(plan.end(), tail.rbegin(), tail.rend());
    return plan;
}

// Token starts of the pieces of a problem of T tokens per batch row: host_piece_chunks when `split`, else one
// piece; the last entry is the end (T, or past it when the last chunk is partial).
std::vector<int64_t> piece_starts(int64_t T, bool split)
{
    std::vector<int64_t> first{0};
    if (split) {
        for (int64_t ch : host_piece_chunks((T + CH - 1) / CH))
            first.push_back(first.back() + ch * CH);
    } else {
        first.push_back(T);
    }
    return first;
}

__global__ void bf16_to_f32_kernel(const __nv_bfloat16 *src, float *dst, size_t n)
{
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = __bfloat162float(src[i]);
}
__global__ void f32_to_bf16_kernel(const float *src, __nv_bfloat16 *dst, size_t n)
{
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = __float2bfloat16_rn(src[i]);
}

// streams and events of the pipeline, one set per device, created on first use
struct HostCtx {
    cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
    cudaEvent_t e_in[HOST_RING] = {}, e_comp[HOST_RING] = {}, e_out[HOST_RING] = {}, e_start = nullptr;
    bool ready = false;
};
std::mutex g_host_mu;
HostCtx g_host[64];

cudaError_t host_ctx(int dev, HostCtx **out)
{
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    HostCtx &c = g_host[dev];
    if (!c.ready) {
        cudaError_t e = cudaSuccess;
        for (cudaStream_t *s : {&c.s_in, &c.s_comp, &c.s_out})
            if (e == cudaSuccess)
                e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
        for (int i = 0; i < HOST_RING && e == cudaSuccess; ++i) {
            e = cudaEventCreateWithFlags(&c.e_in[i], cudaEventDisableTiming);
            if (e == cudaSuccess)
                e = cudaEventCreateWithFlags(&c.e_comp[i], cudaEventDisableTiming);
            if (e == cudaSuccess)
                e = cudaEventCreateWithFlags(&c.e_out[i], cudaEventDisableTiming);
        }
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&c.e_start, cudaEventDisableTiming);
        if (e != cudaSuccess)
            return e;
        c.ready = true;
    }
    *out = &c;
    return cudaSuccess;
}

// device allocations of one call, from the library's pool on the compute stream, returned at the end
struct DevBufs {
    void *ptr[64] = {};
    int n = 0;
    cudaStream_t s = nullptr;
    cudaError_t get(void **p, size_t bytes)
    {
        *p = nullptr;
        if (bytes == 0)
            return cudaSuccess;
        if (n == 64)
            return cudaErrorMemoryAllocation;
        const cudaError_t e = pool_alloc(p, bytes, s);
        if (e == cudaSuccess)
            ptr[n++] = *p;
        return e;
    }
    ~DevBufs()
    {
        for (int i = 0; i < n; ++i)
            cudaFreeAsync(ptr[i], s);
    }
};

}  // namespace

cudaError_t launch_convert(const void *src, void *dst, size_t n, bool to_f32, cudaStream_t s)
{
    if (n == 0)
        return cudaSuccess;
    const int grid = (int)std::min<size_t>((n + 255) / 256, 4096);
    if (to_f32)
        bf16_to_f32_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(src), static_cast<float *>(dst), n);
    else
        f32_to_bf16_kernel<<<grid, 256, 0, s>>>(static_cast<const float *>(src), static_cast<__nv_bfloat16 *>(dst), n);
    return cudaGetLastError();
}

namespace {

// Varlen pipeline: pieces of whole sequences [s0, s1), each about T / P tokens (P at most HOST_MAX_PIECES, pieces
// of at least HOST_MIN_PIECE tokens where the lengths allow).  A piece's token rows [cu[s0], cu[s1]) are contiguous
// in every token tensor, its states are the contiguous slices of sequences s0 .. s1 - 1, and its cu_seqlens is
// cu[s0 .. s1] - cu[s0] (all pieces' arrays go to the device in one copy).  The longest sequence (the last of equals),
// when it spans at least 2 HOST_TAIL_MIN chunks, is in no such piece: it comes last, as a halving tail of pieces of
// whole chunks (each a one-sequence varlen call), its state chained between them in fp32 as in the fixed-length
// pipeline, so that little compute and copy-out follows the last copy in; its chunks start where the sequence's do,
// so the results are the bits of one call.
struct VarlenPiece {
    int64_t t0, pt;   // token rows [t0, t0 + pt)
    int s0, ns;       // sequences s0 .. s0 + ns - 1 (a tail piece: the longest sequence, ns = 1)
    size_t cu_off;    // its cu_seqlens in the device array
    bool tail;        // a part of the longest sequence, its state in the fp32 chain
    bool first_tail, last_tail;
};

// The pieces of a varlen call (N > 1 sequences) in pipeline order, and their cu_seqlens arrays one after another;
// returns the sequence cut into the tail (-1: none).
int varlen_plan(const int64_t *cu, int N, int64_t T, std::vector<VarlenPiece> &pl, std::vector<int64_t> &cus)
{
    // the longest sequence's chunks, cut into a halving tail, when it has enough of them
    int star = 0;
    for (int s = 1; s < N; ++s)
        if (cu[s + 1] - cu[s] >= cu[star + 1] - cu[star])
            star = s;
    std::vector<int64_t> tail_chunks;
    {
        int64_t rem = (cu[star + 1] - cu[star] + CH - 1) / CH;
        if (rem >= 2 * HOST_TAIL_MIN) {
            for (; rem >= 2 * HOST_TAIL_MIN; rem /= 2)
                tail_chunks.push_back(rem - rem / 2);
            tail_chunks.push_back(rem);
        } else {
            star = -1;
        }
    }
    // pieces of whole sequences around it, closed once they reach about 1 / want of the tokens left
    const int64_t Tv = T - (star >= 0 ? cu[star + 1] - cu[star] : 0);
    const int Nv = N - (star >= 0 ? 1 : 0);
    const int64_t want = std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(HOST_MAX_PIECES, Nv),
                                                                (Tv + HOST_MIN_PIECE - 1) / HOST_MIN_PIECE));
    const int64_t target = (Tv + want - 1) / want;
    std::vector<std::pair<int, int>> ranges;
    {
        int s0 = 0;
        for (int s = 0; s < N; ++s) {
            if (s == star) {
                if (s > s0)
                    ranges.push_back({s0, s});
                s0 = s + 1;
            } else if (s > s0 && cu[s] - cu[s0] >= target && (int64_t)ranges.size() + 1 < want) {
                ranges.push_back({s0, s});
                s0 = s;
            }
        }
        if (N > s0)
            ranges.push_back({s0, N});
    }
    for (const auto &r : ranges) {
        const int s0 = r.first, s1 = r.second;
        pl.push_back({cu[s0], cu[s1] - cu[s0], s0, s1 - s0, cus.size(), false, false, false});
        for (int s = s0; s <= s1; ++s)
            cus.push_back(cu[s] - cu[s0]);
    }
    for (size_t i = 0; i < tail_chunks.size(); ++i) {
        const int64_t t = i == 0 ? cu[star] : pl.back().t0 + pl.back().pt;
        const int64_t pt = std::min<int64_t>(tail_chunks[i] * CH, cu[star + 1] - t);
        pl.push_back({t, pt, star, 1, cus.size(), true, i == 0, i + 1 == tail_chunks.size()});
        cus.push_back(0);
        cus.push_back(pt);
    }
    return star;
}

kda_status_t run_host_varlen(HostCtx *c, const void *q, const void *k, const void *v, const void *g, const void *beta,
                             float scale, void *out, const float *A_log, const float *dt_bias, float lower_bound,
                             const void *initial_state, void *final_state, kda_dtype_t state_dtype,
                             const int64_t *cu, int N, int64_t T, int H)
{
    const size_t row = (size_t)H * D;                  // elements of one token's q / k / v / g / out
    const size_t smat = (size_t)H * D * D;             // state elements of one sequence
    const size_t sbytes = state_dtype == KDA_DTYPE_FP32 ? 4 : 2;
    std::vector<VarlenPiece> pl;
    std::vector<int64_t> cus;
    const int star = varlen_plan(cu, N, T, pl, cus);
    int64_t max_t = 0;
    int max_n = 0;
    size_t max_ws = 0;
    for (const VarlenPiece &pc : pl) {
        max_t = std::max(max_t, pc.pt);
        if (!pc.tail)
            max_n = std::max(max_n, pc.ns);
        max_ws = std::max(max_ws, workspace_bytes(pc.ns, pc.pt, H, true));
    }
    const int pieces = (int)pl.size();
    const int ring = pieces > 1 ? HOST_RING : 1;
    const bool chain = star >= 0;   // the tail sequence's state passes between its pieces

    cudaStream_t sc = c->s_comp;
    DevBufs bufs;
    bufs.s = sc;
    void *dq[HOST_RING] = {}, *dk[HOST_RING] = {}, *dv[HOST_RING] = {}, *dg[HOST_RING] = {}, *db[HOST_RING] = {},
         *dout[HOST_RING] = {}, *dinit[HOST_RING] = {}, *dfin[HOST_RING] = {};
    void *dalog = nullptr, *ddt = nullptr, *dcu = nullptr, *dws = nullptr, *dchain = nullptr, *dtail16 = nullptr;
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < ring && e == cudaSuccess; ++i) {
        e = bufs.get(&dq[i], (size_t)max_t * row * 2);
        if (e == cudaSuccess) e = bufs.get(&dk[i], (size_t)max_t * row * 2);
        if (e == cudaSuccess) e = bufs.get(&dv[i], (size_t)max_t * row * 2);
        if (e == cudaSuccess) e = bufs.get(&dg[i], (size_t)max_t * row * 2);
        if (e == cudaSuccess) e = bufs.get(&db[i], (size_t)max_t * H * 2);
        if (e == cudaSuccess) e = bufs.get(&dout[i], (size_t)max_t * row * 2);
        if (e == cudaSuccess && initial_state) e = bufs.get(&dinit[i], (size_t)max_n * smat * sbytes);
        if (e == cudaSuccess && final_state) e = bufs.get(&dfin[i], (size_t)max_n * smat * sbytes);
    }
    if (e == cudaSuccess) e = bufs.get(&dalog, (size_t)H * 4);
    if (e == cudaSuccess) e = bufs.get(&ddt, (size_t)H * D * 4);
    if (e == cudaSuccess) e = bufs.get(&dcu, cus.size() * 8);
    if (e == cudaSuccess) e = bufs.get(&dws, max_ws);
    // the last sequence's state between its tail pieces (fp32), and its bf16 image at the ends
    if (e == cudaSuccess && chain) e = bufs.get(&dchain, smat * 4);
    if (e == cudaSuccess && chain && state_dtype == KDA_DTYPE_BF16 && (initial_state || final_state))
        e = bufs.get(&dtail16, smat * 2);
    // parameters and every piece's cu_seqlens (compute stream), then the copy streams start
    if (e == cudaSuccess) e = cudaMemcpyAsync(dalog, A_log, (size_t)H * 4, cudaMemcpyHostToDevice, sc);
    if (e == cudaSuccess) e = cudaMemcpyAsync(ddt, dt_bias, (size_t)H * D * 4, cudaMemcpyHostToDevice, sc);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dcu, cus.data(), cus.size() * 8, cudaMemcpyHostToDevice, sc);
    const char *hi = static_cast<const char *>(initial_state);
    char *hf = static_cast<char *>(final_state);
    if (e == cudaSuccess) e = cudaEventRecord(c->e_start, sc);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->s_in, c->e_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->s_out, c->e_start, 0);
    if (e != cudaSuccess) {
        cudaStreamSynchronize(sc);
        return KDA_ERR_CUDA;
    }

    const char *hq = static_cast<const char *>(q), *hk = static_cast<const char *>(k);
    const char *hv = static_cast<const char *>(v), *hg = static_cast<const char *>(g);
    const char *hb = static_cast<const char *>(beta);
    char *ho = static_cast<char *>(out);
    kda_status_t st = KDA_OK;
    for (int p = 0; p < pieces && st == KDA_OK; ++p) {
        const VarlenPiece &pc = pl[p];
        const int slot = p % ring;
        const int64_t t0 = pc.t0, pt = pc.pt;
        const size_t w = (size_t)pt * row * 2, o = (size_t)t0 * row * 2;
        const size_t sw = (size_t)pc.ns * smat * sbytes, so = (size_t)pc.s0 * smat * sbytes;
        // copy in (after the slot's previous piece has been computed)
        if (p >= ring) e = cudaStreamWaitEvent(c->s_in, c->e_comp[slot], 0);
        if (pt > 0) {
            if (e == cudaSuccess) e = cudaMemcpyAsync(dq[slot], hq + o, w, cudaMemcpyHostToDevice, c->s_in);
            if (e == cudaSuccess) e = cudaMemcpyAsync(dk[slot], hk + o, w, cudaMemcpyHostToDevice, c->s_in);
            if (e == cudaSuccess) e = cudaMemcpyAsync(dv[slot], hv + o, w, cudaMemcpyHostToDevice, c->s_in);
            if (e == cudaSuccess) e = cudaMemcpyAsync(dg[slot], hg + o, w, cudaMemcpyHostToDevice, c->s_in);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(db[slot], hb + (size_t)t0 * H * 2, (size_t)pt * H * 2, cudaMemcpyHostToDevice, c->s_in);
        }
        if (e == cudaSuccess && initial_state && !pc.tail)
            e = cudaMemcpyAsync(dinit[slot], hi + so, sw, cudaMemcpyHostToDevice, c->s_in);
        // the tail sequence's initial state with its first piece (into the fp32 chain, or its bf16 image)
        if (e == cudaSuccess && initial_state && pc.first_tail)
            e = cudaMemcpyAsync(state_dtype == KDA_DTYPE_FP32 ? dchain : dtail16, hi + so, smat * sbytes,
                                cudaMemcpyHostToDevice, c->s_in);
        if (e == cudaSuccess) e = cudaEventRecord(c->e_in[slot], c->s_in);
        // compute (after the copy in, and after the slot's previous results have been copied out)
        if (e == cudaSuccess) e = cudaStreamWaitEvent(sc, c->e_in[slot], 0);
        if (e == cudaSuccess && p >= ring) e = cudaStreamWaitEvent(sc, c->e_out[slot], 0);
        if (e == cudaSuccess && initial_state && pc.first_tail && state_dtype == KDA_DTYPE_BF16)
            e = launch_convert(dtail16, dchain, smat, true, sc);
        if (e != cudaSuccess) {
            st = KDA_ERR_CUDA;
            break;
        }
        const void *init_p = pc.tail ? ((pc.first_tail && !initial_state) ? nullptr : dchain) : dinit[slot];
        void *fin_p = pc.tail ? dchain : dfin[slot];
        const kda_dtype_t sdt = pc.tail ? KDA_DTYPE_FP32
                                        : ((initial_state || final_state) ? state_dtype : KDA_DTYPE_NONE);
        st = run(dq[slot], dk[slot], dv[slot], dg[slot], db[slot], scale, dout[slot], static_cast<const float *>(dalog),
                 static_cast<const float *>(ddt), lower_bound, init_p, fin_p, sdt,
                 static_cast<const int64_t *>(dcu) + pc.cu_off, pc.ns, pt, H, static_cast<unsigned char *>(dws), sc);
        if (st != KDA_OK)
            break;
        // the last sequence's final state, once its last tail piece is computed (compute stream)
        e = cudaSuccess;
        if (pc.last_tail && final_state) {
            if (state_dtype == KDA_DTYPE_BF16) e = launch_convert(dchain, dtail16, smat, false, sc);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(hf + so, state_dtype == KDA_DTYPE_BF16 ? dtail16 : dchain, smat * sbytes,
                                    cudaMemcpyDeviceToHost, sc);
        }
        if (e == cudaSuccess) e = cudaEventRecord(c->e_comp[slot], sc);
        // copy out
        if (e == cudaSuccess) e = cudaStreamWaitEvent(c->s_out, c->e_comp[slot], 0);
        if (e == cudaSuccess && pt > 0) e = cudaMemcpyAsync(ho + o, dout[slot], w, cudaMemcpyDeviceToHost, c->s_out);
        if (e == cudaSuccess && final_state && !pc.tail)
            e = cudaMemcpyAsync(hf + so, dfin[slot], sw, cudaMemcpyDeviceToHost, c->s_out);
        if (e == cudaSuccess) e = cudaEventRecord(c->e_out[slot], c->s_out);
        if (e != cudaSuccess)
            st = KDA_ERR_CUDA;
    }
    const cudaError_t e1 = cudaStreamSynchronize(sc), e2 = cudaStreamSynchronize(c->s_out),
                      e3 = cudaStreamSynchronize(c->s_in);
    if (st == KDA_OK && (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess))
        st = KDA_ERR_CUDA;
    return st;
}

}  // namespace

kda_status_t run_host(const void *q, const void *k, const void *v, const void *g, const void *beta, float scale,
                      void *out, const float *A_log, const float *dt_bias, float lower_bound, const void *initial_state,
                      void *final_state, kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_host_mu);   // one pipeline per device at a time
    HostCtx *c = nullptr;
    if (host_ctx(dev, &c) != cudaSuccess)
        return KDA_ERR_CUDA;
    const bool varlen = cu_seqlens != nullptr;
    if (varlen && N > 1 && T > HOST_MIN_PIECE)
        return run_host_varlen(c, q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, final_state,
                               state_dtype, cu_seqlens, N, T, H);
    const int B = varlen ? 1 : N;
    const size_t row = (size_t)H * D;                  // elements of one token's q / k / v / g / out
    const size_t state_elems = (size_t)N * H * D * D;
    const size_t sbytes = state_dtype == KDA_DTYPE_FP32 ? 4 : 2;
    const bool has_state = initial_state || final_state;

    // pieces of whole 64-token chunks (host_piece_chunks); piece p starts at token first[p]
    const std::vector<int64_t> first = piece_starts(T, !varlen && T > HOST_MIN_PIECE);
    const int64_t pieces = (int64_t)first.size() - 1;
    int64_t PT = 0;   // tokens of the largest piece
    for (int64_t p = 0; p < pieces; ++p)
        PT = std::max(PT, first[p + 1] - first[p]);
    const int ring = pieces > 1 ? HOST_RING : 1;
    const size_t tok_cap = (size_t)B * (size_t)PT;     // tokens of one piece (all batch rows)

    // device buffers (stream-ordered on the compute stream; the other streams start after them)
    cudaStream_t sc = c->s_comp;
    DevBufs bufs;
    bufs.s = sc;
    void *dq[HOST_RING] = {}, *dk[HOST_RING] = {}, *dv[HOST_RING] = {}, *dg[HOST_RING] = {}, *db[HOST_RING] = {},
         *dout[HOST_RING] = {};
    void *dalog = nullptr, *ddt = nullptr, *dcu = nullptr, *dstate = nullptr, *dinit = nullptr, *dfin = nullptr,
         *dws = nullptr;
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < ring && e == cudaSuccess; ++i) {
        e = bufs.get(&dq[i], tok_cap * row * 2);
        if (e == cudaSuccess) e = bufs.get(&dk[i], tok_cap * row * 2);
        if (e == cudaSuccess) e = bufs.get(&dv[i], tok_cap * row * 2);
        if (e == cudaSuccess) e = bufs.get(&dg[i], tok_cap * row * 2);
        if (e == cudaSuccess) e = bufs.get(&db[i], tok_cap * H * 2);
        if (e == cudaSuccess) e = bufs.get(&dout[i], tok_cap * row * 2);
    }
    if (e == cudaSuccess) e = bufs.get(&dalog, (size_t)H * 4);
    if (e == cudaSuccess) e = bufs.get(&ddt, (size_t)H * D * 4);
    if (e == cudaSuccess && varlen) e = bufs.get(&dcu, (size_t)(N + 1) * 8);
    // the chained state: fp32 whenever the problem has more than one piece
    const bool chain = pieces > 1;
    if (e == cudaSuccess && chain) e = bufs.get(&dstate, state_elems * 4);
    if (e == cudaSuccess && !chain && initial_state) e = bufs.get(&dinit, state_elems * sbytes);
    if (e == cudaSuccess && !chain && final_state) e = bufs.get(&dfin, state_elems * sbytes);
    if (e == cudaSuccess && chain && initial_state && state_dtype == KDA_DTYPE_BF16) e = bufs.get(&dinit, state_elems * 2);
    if (e == cudaSuccess && chain && final_state && state_dtype == KDA_DTYPE_BF16) e = bufs.get(&dfin, state_elems * 2);
    size_t ws_bytes = 0;   // the largest of the pieces' workspaces (a shorter piece may take another schedule)
    for (int64_t p = 0; p < pieces; ++p)
        ws_bytes = std::max(ws_bytes, workspace_bytes(N, varlen ? T : std::min<int64_t>(first[p + 1], T) - first[p], H, varlen));
    if (e == cudaSuccess) e = bufs.get(&dws, ws_bytes);
    // parameters and cu_seqlens (compute stream) before the copy streams start: issued after the first piece's
    // inputs, the copy engine could serve them only after those, and the first compute would wait for it
    if (e == cudaSuccess) e = cudaMemcpyAsync(dalog, A_log, (size_t)H * 4, cudaMemcpyHostToDevice, sc);
    if (e == cudaSuccess) e = cudaMemcpyAsync(ddt, dt_bias, (size_t)H * D * 4, cudaMemcpyHostToDevice, sc);
    if (e == cudaSuccess && varlen) e = cudaMemcpyAsync(dcu, cu_seqlens, (size_t)(N + 1) * 8, cudaMemcpyHostToDevice, sc);
    if (e == cudaSuccess) e = cudaEventRecord(c->e_start, sc);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->s_in, c->e_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->s_out, c->e_start, 0);
    if (e != cudaSuccess) {
        cudaStreamSynchronize(sc);
        return KDA_ERR_CUDA;
    }

    const char *hq = static_cast<const char *>(q), *hk = static_cast<const char *>(k);
    const char *hv = static_cast<const char *>(v), *hg = static_cast<const char *>(g);
    const char *hb = static_cast<const char *>(beta);
    char *ho = static_cast<char *>(out);
    kda_status_t st = KDA_OK;
    for (int64_t p = 0; p < pieces && st == KDA_OK; ++p) {
        const int slot = (int)(p % ring);
        const int64_t t0 = first[p], pt = std::min<int64_t>(first[p + 1], T) - t0;
        const size_t w = (size_t)pt * row * 2, wb = (size_t)pt * H * 2;                 // bytes per batch row
        const size_t sp = (size_t)T * row * 2, spb = (size_t)T * H * 2;                 // host pitches
        const size_t o = (size_t)t0 * row * 2, ob = (size_t)t0 * H * 2;                 // host offsets
        // copy in (after the slot's previous piece has been computed)
        if (p >= ring) e = cudaStreamWaitEvent(c->s_in, c->e_comp[slot], 0);
        if (pt > 0) {
            if (e == cudaSuccess) e = cudaMemcpy2DAsync(dq[slot], w, hq + o, sp, w, B, cudaMemcpyHostToDevice, c->s_in);
            if (e == cudaSuccess) e = cudaMemcpy2DAsync(dk[slot], w, hk + o, sp, w, B, cudaMemcpyHostToDevice, c->s_in);
            if (e == cudaSuccess) e = cudaMemcpy2DAsync(dv[slot], w, hv + o, sp, w, B, cudaMemcpyHostToDevice, c->s_in);
            if (e == cudaSuccess) e = cudaMemcpy2DAsync(dg[slot], w, hg + o, sp, w, B, cudaMemcpyHostToDevice, c->s_in);
            if (e == cudaSuccess) e = cudaMemcpy2DAsync(db[slot], wb, hb + ob, spb, wb, B, cudaMemcpyHostToDevice, c->s_in);
        }
        // the initial state with the first piece's inputs (into the fp32 chain, or its bf16 image, converted below)
        void *init_dst = !chain ? dinit : (state_dtype == KDA_DTYPE_FP32 ? dstate : dinit);
        if (e == cudaSuccess && p == 0 && initial_state)
            e = cudaMemcpyAsync(init_dst, initial_state, state_elems * sbytes, cudaMemcpyHostToDevice, c->s_in);
        if (e == cudaSuccess) e = cudaEventRecord(c->e_in[slot], c->s_in);
        // compute (after the copy in, and after the slot's previous output has been copied out)
        if (e == cudaSuccess) e = cudaStreamWaitEvent(sc, c->e_in[slot], 0);
        if (e == cudaSuccess && p >= ring) e = cudaStreamWaitEvent(sc, c->e_out[slot], 0);
        if (e == cudaSuccess && p == 0 && initial_state && chain && state_dtype == KDA_DTYPE_BF16)
            e = launch_convert(dinit, dstate, state_elems, true, sc);
        if (e != cudaSuccess) {
            st = KDA_ERR_CUDA;
            break;
        }
        const void *init_p;
        void *fin_p;
        kda_dtype_t sdt;
        if (chain) {
            init_p = (p == 0 && !initial_state) ? nullptr : dstate;
            fin_p = has_state || p + 1 < pieces ? dstate : nullptr;
            sdt = KDA_DTYPE_FP32;
        } else {
            init_p = initial_state ? dinit : nullptr;
            fin_p = final_state ? dfin : nullptr;
            sdt = state_dtype;
        }
        st = run(dq[slot], dk[slot], dv[slot], dg[slot], db[slot], scale, dout[slot],
                 static_cast<const float *>(dalog), static_cast<const float *>(ddt), lower_bound, init_p, fin_p,
                 (init_p || fin_p) ? sdt : KDA_DTYPE_NONE, varlen ? static_cast<const int64_t *>(dcu) : nullptr, N,
                 varlen ? T : pt, H, static_cast<unsigned char *>(dws), sc);
        if (st != KDA_OK)
            break;
        e = cudaEventRecord(c->e_comp[slot], sc);
        // copy out
        if (e == cudaSuccess) e = cudaStreamWaitEvent(c->s_out, c->e_comp[slot], 0);
        if (e == cudaSuccess && pt > 0)
            e = cudaMemcpy2DAsync(ho + o, sp, dout[slot], w, w, B, cudaMemcpyDeviceToHost, c->s_out);
        if (e == cudaSuccess) e = cudaEventRecord(c->e_out[slot], c->s_out);
        if (e != cudaSuccess)
            st = KDA_ERR_CUDA;
    }
    // final state
    if (st == KDA_OK && final_state) {
        e = cudaSuccess;
        if (chain && state_dtype == KDA_DTYPE_BF16)
            e = launch_convert(dstate, dfin, state_elems, false, sc);
        const void *src = chain ? (state_dtype == KDA_DTYPE_BF16 ? dfin : dstate) : dfin;
        if (e == cudaSuccess) e = cudaMemcpyAsync(final_state, src, state_elems * sbytes, cudaMemcpyDeviceToHost, sc);
        if (e != cudaSuccess)
            st = KDA_ERR_CUDA;
    }
    // wait for everything (the buffers go back to the pool, in stream order, on return)
    const cudaError_t e1 = cudaStreamSynchronize(sc), e2 = cudaStreamSynchronize(c->s_out),
                      e3 = cudaStreamSynchronize(c->s_in);
    if (st == KDA_OK && (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess))
        st = KDA_ERR_CUDA;
    return st;
}

}  // namespace kda

extern "C" int kda_fwd_host_plan(int N, int64_t T, const int64_t *cu_seqlens, int64_t *first_token, int64_t *tokens,
                                 int *first_seq, int *seqs, int max_pieces)
{
    using namespace kda;
    if (N < 1 || T < 0 || T > ((int64_t)1 << 40) || max_pieces < 0 ||
        (max_pieces > 0 && (!first_token || !tokens || !first_seq || !seqs)))
        return -1;
    if (cu_seqlens && kda_check_cu_seqlens(cu_seqlens, N, T) != KDA_OK)
        return -1;
    int n = 0;
    auto put = [&](int64_t t0, int64_t pt, int s0, int ns) {
        if (n < max_pieces) {
            first_token[n] = t0;
            tokens[n] = pt;
            first_seq[n] = s0;
            seqs[n] = ns;
        }
        ++n;
    };
    if (cu_seqlens && N > 1 && T > HOST_MIN_PIECE) {   // the choice run_host makes
        std::vector<VarlenPiece> pl;
        std::vector<int64_t> cus;
        varlen_plan(cu_seqlens, N, T, pl, cus);
        for (const VarlenPiece &pc : pl)
            put(pc.t0, pc.pt, pc.s0, pc.ns);
    } else {
        const std::vector<int64_t> first = piece_starts(T, !cu_seqlens && T > HOST_MIN_PIECE);
        for (size_t p = 0; p + 1 < first.size(); ++p)
            put(first[p], std::min<int64_t>(first[p + 1], T) - first[p], 0, N);
    }
    return n;
}
