// Host-side view of the kernels: tile geometry and launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"

namespace ta {

// Raises a kernel's dynamic shared-memory limit once per device (the setting
// persists), instead of on every launch.  `done` is the kernel's own bit set
// of devices already configured.
template <typename Kernel>
cudaError_t set_smem_once(Kernel kernel, int bytes, std::atomic<unsigned long long>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// How a split-KV kernel wants its K/V tiles delivered by TMA.
struct Geometry {
    int tile_tokens;   // tokens per pipeline stage (slices are cut at multiples of this)
    int box_x;         // channels per TMA box (64 with 128-byte swizzle, else head_dim)
    int swizzle128;    // 1: CU_TENSOR_MAP_SWIZZLE_128B, 0: no swizzle
    int halves5d = 0;  // 1: 5-D view whose box brings every 64-channel half at once
    int heads_per_block = 1;  // KV heads a block serves; each box spans all of them
    int split_halves = 0;  // 1 (with halves5d): the box brings one 64-channel half; one copy per half
};

Geometry mma_geometry(int head_dim, int heads_per_block);
Geometry fma_geometry(int kv_elem_bytes, int head_dim);
Geometry fp8_geometry(int heads_per_block);

// Per-slice kernels.  Grid (P, Hkv / hb, B); `tk`/`tv` are tensor maps over
// (channel, token, KV head, batch row or page) with the box of the kernel's
// Geometry (hb = p.hb KV heads per box).
cudaError_t launch_split_mma(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv,
                             const SplitParams& p, cudaStream_t stream);
// Clusters of `cluster_size` blocks of the BF16 tensor-core kernel that can be
// resident at once on the current device (the GPCs bound it; the FP8 kernel's
// blocks, also one per SM, fit the same way).  0 if the query fails.
int mma_cluster_capacity(int cluster_size);
cudaError_t launch_split_fma_bf16(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const SplitParams& p, cudaStream_t stream);
cudaError_t launch_split_fma_f32(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const SplitParams& p, cudaStream_t stream);
// Fifth-generation tensor cores (tcgen05, accumulators in TMEM): BF16 q and
// cache, head_dim 128, up to 64 columns per KV head, one KV head per block.
Geometry tc05_geometry(int page_size);
cudaError_t launch_split_tc05(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                              cudaStream_t stream);
// FP8 (E4M3) caches on the tcgen05 tensor cores: head_dim 128, BF16 q, up to
// 32 columns per KV head, one KV head per block.
Geometry tc05_fp8_geometry();
cudaError_t launch_split_tc05_fp8(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                                  cudaStream_t stream);
// FP8 (E4M3) caches, head_dim 128, BF16 q, up to 16 columns per KV head.
cudaError_t launch_split_fp8(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                             cudaStream_t stream);

// Cross-block tree combine of P partial states per (b, h) plus normalisation.
// With `dependent` set it is launched as a programmatic dependent of the
// previous kernel on the stream (it waits for that grid before reading).
cudaError_t launch_combine(int head_dim, const float* po, const float* pm, const float* pl,
                           float* out, float* lse, int B, int Hq, int P, bool dependent,
                           cudaStream_t stream);

}  // namespace ta
