// chunk_fwd_noalloc.cu -- the context-parallel prefill for callers that cannot
// allocate device memory.
//
// The scratch that kda_chunk_fwd's context-parallel path takes from a caller
// workspace (segment table, per-segment transitions M and N, per-segment
// initial states) lives here in one fixed file-scope device array instead.
// Every GPU that loads this library holds the array until the process exits.
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

#include "../../include/kda.h"

namespace {

__device__ __align__(256) unsigned char g_cp_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_cp_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
int scratch_for_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_cp_scratch) != cudaSuccess || !p) return KDA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" int kda_chunk_fwd_cp_noalloc(const void *q, const void *k, const void *v, const float *g,
                                        const float *beta, const int32_t *cu_seqlens, int N, int T, int H,
                                        int dk, int dv, const float *initial_state, float *final_state,
                                        void *o, float scale, float g_min, int in_dtype, int segment_len,
                                        uint32_t *status, void *stream) {
    if (N < 1 || T < 0 || H < 1 || segment_len < 0) return KDA_ERR_INVALID_ARG;
    size_t need = kda_chunk_fwd_workspace_size(N, T, H, dk, dv, KDA_CP_ON, segment_len);
    if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    int rc = scratch_for_current_device(&scratch);
    if (rc != KDA_OK) return rc;
    // Nothing in the scratch needs to start at zero: the segment-table kernel
    // writes every table entry and count it later reads, the transition kernel
    // writes every M and N tile, and the composition writes every S_in tile.
    // When the rest of the array holds the two-kernel area, its slot list is
    // cleared by the launch that fills it, a carried state is written by the
    // walk of one piece before the next piece reads it, and every operand blob
    // is written by the chunk-local kernel before the walk of its piece reads it.
    return kda_chunk_fwd(q, k, v, g, beta, cu_seqlens, N, T, H, dk, dv, initial_state, final_state, o, scale,
                         g_min, in_dtype, KDA_CP_ON, segment_len, scratch, (size_t)KDA_NOALLOC_SCRATCH_BYTES,
                         status, stream);
}
