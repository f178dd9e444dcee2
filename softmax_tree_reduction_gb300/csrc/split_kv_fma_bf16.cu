// FP32-FMA split-KV kernels for BF16 K/V caches (q in BF16 or FP32).
#include "split_kv_fma.cuh"

namespace ta {

Geometry fma_geometry(int kv_elem_bytes, int head_dim) {
    return Geometry{32768 / (2 * head_dim * kv_elem_bytes), head_dim, 0, 0};
}

cudaError_t launch_split_fma_bf16(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const SplitParams& p, cudaStream_t stream) {
    return fma_detail::launch_fma<__nv_bfloat16>(head_dim, tk, tv, p, stream);
}

}  // namespace ta
