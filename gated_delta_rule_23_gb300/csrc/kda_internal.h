// Host-side entry points of the KDA kernels (one translation unit each), used by kda_api.cu.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace kda {

struct Problem;

// Prep kernel over max_chunks x H (chunk, head) items; CTAs past the real chunk count exit.
cudaError_t launch_prep(const Problem &p, int64_t max_chunks, cudaStream_t stream);
// Recurrence kernel over N x H (sequence, head) pairs; state_kind 0 none, 1 bf16, 2 fp32.
cudaError_t launch_recur(const Problem &p, int state_kind, cudaStream_t stream);
size_t prep_smem_bytes();
size_t recur_smem_bytes();
// Read the device-side "bounded wait expired" words of the recurrence / prep kernels and clear them.
cudaError_t read_and_clear_device_error(unsigned int *flag);
cudaError_t prep_read_and_clear_error(unsigned int *flag);

}  // namespace kda
