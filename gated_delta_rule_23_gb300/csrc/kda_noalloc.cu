// kda_fwd_noalloc: the forward pass with its workspace in a fixed, statically sized device array
// of this translation unit instead of memory the library allocates per call.
//
// The array exists once per device: the driver creates it when this library's module is loaded
// on that device, and it stays there until the process exits.  In host code the name of the
// array only stands for it; the device address is looked up once per device (with that device
// current) by cudaGetSymbolAddress, on the first call that needs a workspace, and cached.  Every
// call on a device shares the array, so calls whose kernels overlap on the GPU race; problems
// whose workspace exceeds the array are rejected before anything is launched.
#include <mutex>

#include "kda.h"
#include "kda_internal.h"

static __device__ __align__(256) unsigned char g_kda_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int MAX_DEVICES = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[MAX_DEVICES] = {};

// Device address of this device's copy of the array (looked up on first use, then cached).
cudaError_t scratch_address(void **addr)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= MAX_DEVICES)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_kda_noalloc_scratch);
        if (err != cudaSuccess)
            return err;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" kda_status_t kda_fwd_noalloc(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                        float scale, void *out, const float *A_log, const float *dt_bias,
                                        float lower_bound, const void *initial_state, void *final_state,
                                        kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H,
                                        kda_stream_t stream)
{
    kda_status_t s = kda::check_args(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                                     final_state, state_dtype, cu_seqlens, N, T, H);
    if (s == KDA_OK)
        s = kda::check_size(N, T, H, cu_seqlens != nullptr);
    if (s != KDA_OK)
        return s;
    const size_t need = kda::workspace_bytes(N, T, H, cu_seqlens != nullptr);
    if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES)
        return KDA_ERR_UNSUPPORTED;
    void *scratch = nullptr;   // decode-sized problems need no workspace: no lookup at all
    if (need > 0 && scratch_address(&scratch) != cudaSuccess)
        return KDA_ERR_CUDA;
    // Every byte of the workspace that the kernels read is written earlier in the same call (the
    // varlen plan, then the operand slots), so the array needs no clearing between calls.
    return kda::run(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, final_state,
                    state_dtype, cu_seqlens, N, T, H, static_cast<unsigned char *>(scratch),
                    reinterpret_cast<cudaStream_t>(stream));
}
