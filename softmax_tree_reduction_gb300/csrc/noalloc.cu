// tree_attn_decode_noalloc: decode attention for callers that must not
// allocate device memory.  The partial states that tree_attn_decode keeps in
// a caller-provided workspace live here in a fixed buffer that the library
// reserves statically on every device that loads it.
#include <mutex>

#include "../../include/tree_attn.h"
#include "common.cuh"

namespace {

// The scratch buffer.  In host code this name is only a stand-in for the
// symbol: its device address is looked up per device below and that address
// is what the kernels receive.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];

// One-time set-up per device, with that device current.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return TA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return TA_OK;
}

}  // namespace

extern "C" int tree_attn_decode_noalloc(const ta_shape* shape, const void* q, const void* k_cache,
                                        const void* v_cache, const int32_t* seqlens, float* out,
                                        float* lse, int num_splits, void* stream) {
    int rc = tree_attn_check_shape(shape);
    if (rc != TA_OK) return rc;
    if (num_splits > TA_MAX_SPLITS) return TA_ERR_SPLITS;
    int P = num_splits;
    if (P <= 0) {
        P = tree_attn_pick_splits(shape, nullptr, 0);
        if (P < 0) return P;
    }
    const size_t need = tree_attn_workspace_bytes(shape, P);
    if (need > TA_NOALLOC_SCRATCH_BYTES) return TA_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    if (P > 1 && (rc = scratch_address(&scratch)) != TA_OK) return rc;
    // A split count left to the library stays 0: tree_attn_decode then picks the
    // same P (and may merge short rows through a thread-block cluster).
    return tree_attn_decode(shape, q, k_cache, v_cache, seqlens, out, lse, num_splits <= 0 ? 0 : P, scratch,
                            P > 1 ? static_cast<size_t>(TA_NOALLOC_SCRATCH_BYTES) : 0, stream);
}
