// Host-side entry points of the KDA kernels (one translation unit each), used by kda_api.cu.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "kda.h"

namespace kda {

// Host-side argument checks of kda_fwd (no CUDA calls).
kda_status_t check_args(const void *q, const void *k, const void *v, const void *g, const void *beta, float scale,
                        const void *out, const float *A_log, const float *dt_bias, float lower_bound,
                        const void *initial_state, const void *final_state, kda_dtype_t state_dtype,
                        const int64_t *cu_seqlens, int N, int64_t T, int H);
// Workspace bytes of one call (kda_fwd_workspace_size); SIZE_MAX when the count does not fit in 64 bits.
size_t workspace_bytes(int N, int64_t T, int H, bool varlen);
// KDA_ERR_UNSUPPORTED when the chunked path cannot take the problem size (workspace size not
// representable, or more than 2^31 - 1 (chunk, head) items); KDA_OK otherwise.  No CUDA calls.
kda_status_t check_size(int N, int64_t T, int H, bool varlen);
// The launch sequence on `stream` with workspace `ws` (checked arguments).  single_launch: one prep launch
// over every chunk, then one recurrence launch, also where the problem would run in pieces.
kda_status_t run(const void *q, const void *k, const void *v, const void *g, const void *beta, float scale,
                 void *out, const float *A_log, const float *dt_bias, float lower_bound, const void *initial_state,
                 void *final_state, kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H,
                 unsigned char *ws, cudaStream_t stream, void *const *stage_events = nullptr, uint32_t variant = 0,
                 bool single_launch = false);

// Stream-ordered allocation from the library's memory pool of the current device (kept between calls).
cudaError_t pool_alloc(void **p, size_t bytes, cudaStream_t stream);
// kda_fwd_host: host buffers in and out, copies and kernels pipelined over pieces (checked arguments).
kda_status_t run_host(const void *q, const void *k, const void *v, const void *g, const void *beta, float scale,
                      void *out, const float *A_log, const float *dt_bias, float lower_bound, const void *initial_state,
                      void *final_state, kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H);

struct Problem;

// Prep kernel over max_chunks x H (chunk, head) items; CTAs past the real chunk count exit.  persistent:
// at most two CTAs per SM walking the items; otherwise one CTA per item.  early: launched as a programmatic
// dependent of the recurrence kernel before it on `stream` (it reads nothing that recurrence writes), so it
// starts once every recurrence CTA runs, on the SMs they leave free, and completes after that recurrence.
cudaError_t launch_prep(const Problem &p, int64_t max_chunks, cudaStream_t stream, bool persistent = true,
                        bool early = false);
// Elementwise bf16 <-> fp32 conversion of n values on `stream` (to_f32: bf16 src to fp32 dst).
cudaError_t launch_convert(const void *src, void *dst, size_t n, bool to_f32, cudaStream_t stream);
// Recurrence kernel over N x H (sequence, head) pairs (x p.groups without cu_seqlens); state_kind 0 none,
// 1 bf16, 2 fp32.
cudaError_t launch_recur(const Problem &p, int state_kind, cudaStream_t stream);
// The chunk-transition scan: each group's transition (recurrence kernel, compose form; groups 0 .. p.groups - 2
// into p.sc_a / p.sc_b), then the group start states, serially over the groups (p.sc_s, from the fp32 initial
// state init0 or zeros).
// two_tiles: one CTA per (group, sequence, head) carries both the transition and the offset; otherwise two CTAs.
cudaError_t launch_compose(const Problem &p, bool two_tiles, cudaStream_t stream);
cudaError_t launch_scan_states(const float *init0, const float *a, const float *b, float *s, int pairs, int groups,
                               cudaStream_t stream);
// Token-recurrent kernel, persistent over the N x H x 2 (sequence, head, value half) items; no workspace.
cudaError_t launch_recurrent(const Problem &p, int state_kind, cudaStream_t stream);
size_t recurrent_smem_bytes();
// Decode kernel (fixed-length problems of 1 to 4 tokens per sequence), persistent over the same items.
bool decode_applies(const Problem &p, int state_kind);
cudaError_t launch_decode(const Problem &p, int state_kind, cudaStream_t stream);
size_t decode_smem_bytes();
cudaError_t decode_read_and_clear_error(unsigned int *flag);
size_t prep_smem_bytes();
size_t recur_smem_bytes();
// Read the device-side "bounded wait expired" words of the recurrence / prep kernels and clear them.
cudaError_t read_and_clear_device_error(unsigned int *flag);
cudaError_t prep_read_and_clear_error(unsigned int *flag);
cudaError_t recurrent_read_and_clear_error(unsigned int *flag);

}  // namespace kda
