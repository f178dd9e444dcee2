// Cross-block tree combine ("The Tree Reduction Merge Operator" over the P
// partial states of every (b, h), then the root normalisation O = o / l).
//
// One block per (h, b): 128 threads for up to 64 states, 512 for more (the
// fold is bound by loads in flight, so larger P gets more of them).  The root
// maximum M = max_p m_p is found first (a block max-reduction), so every
// leaf's rescale factor exp(m_p - M) is applied directly -- the merge tree
// with its maxima already resolved.  The numerators are then folded by groups
// of threads (group r takes p = r, r + groups, ...; each thread owns four
// channels; eight loads in flight per thread) and the group sums are merged
// pairwise in shared memory.  An empty slice (m = -inf, l = 0)
// contributes nothing; all-empty rows give out = 0, lse = -inf; NaN inputs
// propagate to the row's outputs.
#include "common.cuh"
#include "kernels.h"

namespace ta {
namespace {

template <int D, int kCombineThreads>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const float* __restrict__ po, const float* __restrict__ pm,
                   const float* __restrict__ pl, float* __restrict__ out, float* __restrict__ lse,
                   int Hq, int P) {
    constexpr int kTPR = D / 4;                      // threads per row of channels
    constexpr int kGroups = kCombineThreads / kTPR;  // p-folding groups
    __shared__ float red[kCombineThreads / 32];
    __shared__ float4 acc_s[kGroups][kTPR];
    __shared__ float l_s[kGroups];

    wait_primary();  // no-op unless launched as a programmatic dependent

    const int h = blockIdx.x, b = blockIdx.y;
    const size_t row = static_cast<size_t>(b) * Hq + h;
    const float* m = pm + row * P;
    const float* l = pl + row * P;
    const float4* o = reinterpret_cast<const float4*>(po + row * P * D);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // root maximum
    float M = -INFINITY;
    for (int q = tid; q < P; q += kCombineThreads) M = fmaxf(M, m[q]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int w = 1; w < kCombineThreads / 32; ++w) M = fmaxf(M, red[w]);
    const float Ms = (M == -INFINITY) ? 0.f : M;

    // leaves folded per group
    const int c4 = tid % kTPR, grp = tid / kTPR;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lacc = 0.f;
#pragma unroll 8
    for (int q = grp; q < P; q += kGroups) {
        const float mq = m[q];
        const float w = (mq == -INFINITY) ? 0.f : ex2((mq - Ms) * kLog2e);
        const float4 v = o[static_cast<size_t>(q) * kTPR + c4];
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
        lacc = fmaf(w, l[q], lacc);
    }
    acc_s[grp][c4] = acc;
    if (c4 == 0) l_s[grp] = lacc;
    __syncthreads();
    // pairwise tree over the groups
    for (int stride = kGroups / 2; stride > 0; stride >>= 1) {
        if (grp < stride) {
            float4 a = acc_s[grp][c4];
            const float4 bq = acc_s[grp + stride][c4];
            a.x += bq.x;
            a.y += bq.y;
            a.z += bq.z;
            a.w += bq.w;
            acc_s[grp][c4] = a;
            if (c4 == 0) l_s[grp] += l_s[grp + stride];
        }
        __syncthreads();
    }
    if (grp == 0) {
        const float L = l_s[0];
        float4 r = acc_s[0][c4];
        if (L > 0.f) {
            r.x /= L;
            r.y /= L;
            r.z /= L;
            r.w /= L;
        } else if (L == 0.f) {
            r = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        reinterpret_cast<float4*>(out + row * D)[c4] = r;
        if (c4 == 0 && lse) lse[row] = (L > 0.f) ? M + logf(L) : (L == 0.f ? -INFINITY : L);
    }
}

template <int D, int kCombineThreads>
cudaError_t launch_impl(const float* po, const float* pm, const float* pl, float* out, float* lse,
                        int B, int Hq, int P, bool dependent, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(Hq, B, 1);
    cfg.blockDim = dim3(kCombineThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, combine_kernel<D, kCombineThreads>, po, pm, pl, out, lse, Hq, P);
}

}  // namespace

cudaError_t launch_combine(int head_dim, const float* po, const float* pm, const float* pl,
                           float* out, float* lse, int B, int Hq, int P, bool dependent,
                           cudaStream_t stream) {
    const bool wide = P > 64;
    switch (head_dim) {
        case 64:
            return wide ? launch_impl<64, 512>(po, pm, pl, out, lse, B, Hq, P, dependent, stream)
                        : launch_impl<64, 128>(po, pm, pl, out, lse, B, Hq, P, dependent, stream);
        case 128:
            return wide ? launch_impl<128, 512>(po, pm, pl, out, lse, B, Hq, P, dependent, stream)
                        : launch_impl<128, 128>(po, pm, pl, out, lse, B, Hq, P, dependent, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ta
