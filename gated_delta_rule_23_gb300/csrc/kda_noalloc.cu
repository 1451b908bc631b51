// kda_fwd_noalloc: the forward pass with its workspace in a fixed, statically sized device array
// of this translation unit instead of memory the library allocates per call.  The array exists
// once per device context (it is created when this unit's module is first used on a device) and
// is shared by every call on that device, so calls must be ordered (one stream, or serialised by
// the caller).  Problems whose workspace exceeds it are rejected before anything is launched.
#include "kda.h"
#include "kda_internal.h"

static __device__ __align__(256) unsigned char g_kda_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

extern "C" kda_status_t kda_fwd_noalloc(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                        float scale, void *out, const float *A_log, const float *dt_bias,
                                        float lower_bound, const void *initial_state, void *final_state,
                                        kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H,
                                        kda_stream_t stream)
{
    kda_status_t s = kda::check_args(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                                     final_state, state_dtype, cu_seqlens, N, T, H);
    if (s != KDA_OK)
        return s;
    if (kda::workspace_bytes(N, T, H, cu_seqlens != nullptr) > (size_t)KDA_NOALLOC_SCRATCH_BYTES)
        return KDA_ERR_UNSUPPORTED;
    void *scratch = nullptr;   // this device's copy of the array
    if (cudaGetSymbolAddress(&scratch, g_kda_noalloc_scratch) != cudaSuccess)
        return KDA_ERR_CUDA;
    return kda::run(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, final_state,
                    state_dtype, cu_seqlens, N, T, H, static_cast<unsigned char *>(scratch),
                    reinterpret_cast<cudaStream_t>(stream));
}
