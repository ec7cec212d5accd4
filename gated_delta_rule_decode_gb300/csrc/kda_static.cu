// Allocation-free chunked prefill: the same kernels as kda_prefill_chunked,
// with the scratch memory in a fixed device array owned by the library, for
// callers that cannot allocate device memory when they call.
#include <mutex>

#include "kda.h"
#include "kda_internal.h"

namespace {

// The scratch of kda_prefill_chunked_static.  Every GPU that loads the
// library reserves it until the process exits.
__device__ __align__(256) unsigned char g_static_scratch[KDA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_lock;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device.  In host code the
// array's name is only a host-side stand-in (a kernel handed it would fault or
// silently use the wrong memory), so the address is asked for once per device,
// with that device current.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> guard(g_lock);
    if (g_scratch_addr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr)
            return KDA_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" {

size_t kda_static_scratch_bytes(void) { return KDA_STATIC_SCRATCH_BYTES; }

int kda_prefill_chunked_static(const kda_dims *dims, int32_t num_seqs, const int32_t *cu_seqlens,
                               int64_t total_tokens, const void *q, const void *k, const void *v,
                               const float *g, const void *b, const int32_t *slot_ids, float *pool,
                               int64_t num_slots, int32_t init_from_pool, void *out, int32_t *err_flag,
                               void *stream) {
    const size_t need = kda_prefill_workspace_bytes(dims, num_seqs, total_tokens);
    if (need > KDA_STATIC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0) {
        const int st = scratch_address(&scratch);
        if (st != KDA_OK) return st;
    }
    return kda_prefill_chunked(dims, num_seqs, cu_seqlens, total_tokens, q, k, v, g, b, slot_ids, pool,
                               num_slots, init_from_pool, out, scratch, need > 0 ? KDA_STATIC_SCRATCH_BYTES : 0,
                               err_flag, stream);
}

}  // extern "C"
