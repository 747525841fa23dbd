// kda_fwd_noalloc: the chunked KDA forward for callers that cannot allocate
// device memory at all -- for example code running inside a custom
// allocator's own callback (allocating there would re-enter the allocator),
// a plug-in inside a host application that owns every allocation itself, or
// an embedded runtime with a fixed memory budget decided up front.  It
// runs the same kernels as kda_fwd, with the workspace taken from a static
// device array that is part of this library (every GPU that loads the
// library holds it until the process exits) instead of from the caller.
#include <mutex>

#include "../../include/kda.h"

namespace {

// The scratch array.  Its size is fixed when the library is built; problems
// whose workspace does not fit are rejected with KDA_ERR_TOO_LARGE.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::once_flag g_setup_once[kMaxDevices];
void* g_scratch_ptr[kMaxDevices];
cudaError_t g_setup_err[kMaxDevices];

}  // namespace

extern "C" kda_status kda_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                      const float* beta, float scale, const float* h0,
                                      const int32_t* cu_seqlens, void* o, float* ht, int B, int T, int H, int K,
                                      int V, int N, unsigned flags, cudaStream_t stream) {
    if (flags & KDA_FLAG_SAVE_FOR_BWD) return KDA_ERR_INVALID_ARG;   // the saved states need a caller workspace
    const size_t need = kda_fwd_workspace_bytes(B, T, H, K, V, N);
    if (need == 0) return (K != 128 || V != 128) ? KDA_ERR_UNSUPPORTED : KDA_ERR_INVALID_ARG;
    if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_TOO_LARGE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    // Once per device, with that device current: the host-side name of the
    // array is only a stand-in, so look up its device address.
    std::call_once(g_setup_once[dev], [dev]() {
        void* ptr = nullptr;
        g_setup_err[dev] = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        g_scratch_ptr[dev] = ptr;
    });
    if (g_setup_err[dev] != cudaSuccess || g_scratch_ptr[dev] == nullptr) return KDA_ERR_CUDA;

    // kda_fwd clears the status word at the start of the array; nothing else
    // in the workspace needs to start at zero.
    return kda_fwd(q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, B, T, H, K, V, N, flags, g_scratch_ptr[dev],
                   (size_t)KDA_NOALLOC_SCRATCH_BYTES, stream);
}
