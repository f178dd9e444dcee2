// FP32-FMA split-KV kernels for FP32 K/V caches (q in BF16 or FP32).
#include "split_kv_fma.cuh"

namespace ta {

cudaError_t launch_split_fma_f32(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const SplitParams& p, cudaStream_t stream) {
    return fma_detail::launch_fma<float>(head_dim, tk, tv, p, stream);
}

}  // namespace ta
