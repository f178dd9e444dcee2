// Split-KV partial attention on the CUDA cores (FP32 FMA), for any dtype
// combination.  Same block decomposition and pipeline as the tensor-core
// kernel: grid (slice p, KV head g, batch row b); warp 0 streams K/V tiles
// (unswizzled TMA boxes of tile x head_dim) into a ring of stages; the other
// 8 warps compute.
//
// Consumer layout: a warp is split into 4 groups of 8 lanes; a group owns one
// token per step and each lane holds head_dim/8 channels of it (16-byte
// shared-memory reads, conflict-free).  q.k is a per-lane FMA chain reduced
// over the group by three shuffles.  Every group keeps its own running state
// (m, l, o) per head -- the leaves of the block's merge tree -- which are
// merged inside the warp by shuffles and across warps in shared memory.
// With G > 4 query heads per KV head the warps also split the heads.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "emit.cuh"
#include "kernels.h"
#include "sched.cuh"

namespace ta {
namespace fma_detail {

template <typename KV, int D>
struct FmaCfg {
    static constexpr int kES = sizeof(KV);
    static constexpr int kWarps = 8;                        // consumer warps
    static constexpr int kRowBytes = D * kES;
    static constexpr int kTile = 32768 / (2 * kRowBytes);   // tokens per stage (32 KB of K+V)
    static constexpr int kKBytes = kTile * kRowBytes;
    static constexpr int kStageBytes = 2 * kKBytes;
    static constexpr int kStages = 3;
    static constexpr int kCPL = kRowBytes / 128;            // 16-byte chunks per lane per row
    static constexpr int kEPC = 16 / kES;                   // elements per chunk
    static constexpr int kEPL = kCPL * kEPC;                // channels per lane (= D / 8)
    static constexpr int kMergeFloats = kWarps * 4 * D + 2 * 64;
    static constexpr int kBarBytes = 2 * kStages * 8 + kStages * 8 + 32;
    static constexpr int kSmem = 1024 + kStages * kStageBytes + kMergeFloats * 4 + kBarBytes;
    static constexpr int kThreads = 32 * (kWarps + 1);
    static_assert(kTile >= 32, "a stage must hold at least 32 tokens");
};

template <typename KV>
__device__ __forceinline__ void unpack16(const uint4& raw, float* f);

template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4& raw, float* f) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

template <>
__device__ __forceinline__ void unpack16<float>(const uint4& raw, float* f) {
    f[0] = __uint_as_float(raw.x);
    f[1] = __uint_as_float(raw.y);
    f[2] = __uint_as_float(raw.z);
    f[3] = __uint_as_float(raw.w);
}

template <typename KV, int D, int GC>
__global__ void __launch_bounds__(FmaCfg<KV, D>::kThreads, 1)
    split_kv_fma_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const SplitParams p) {
    using C = FmaCfg<KV, D>;
    constexpr int EPL = C::kEPL, EPC = C::kEPC, CPL = C::kCPL;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = smem;
    float* mg_o = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes);
    float* mg_m = mg_o + C::kWarps * 4 * D;   // [NTS][G] (NTS*G <= 64)
    float* mg_l = mg_m + 64;
    uint64_t* full = reinterpret_cast<uint64_t*>(mg_l + 64);
    uint64_t* empty = full + C::kStages;
    volatile StageMeta* meta = reinterpret_cast<volatile StageMeta*>(empty + C::kStages);
    int* abort_flag = const_cast<int*>(reinterpret_cast<volatile int*>(meta + C::kStages));
    int* last_flag = abort_flag + 1;
    volatile unsigned* claim_sink = reinterpret_cast<volatile unsigned*>(abort_flag + 2);
    volatile int* bad_page = reinterpret_cast<volatile int*>(abort_flag + 3);
    uint64_t* prod_done = reinterpret_cast<uint64_t*>(abort_flag + 4);  // the copy warp's last claim is made

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::kWarps);
        }
        mbar_init(prod_done, 1);
        *abort_flag = 0;
        *bad_page = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    int n_hint = -1;  // row length read before the dependency wait (a hint)
    if (warp == 0) {  // first tiles into L2 while the previous grid drains
        const int page_mask = (1 << p.page_shift) - 1;
        n_hint = prefetch_row_head(p, b, split, C::kTile, p.prefetch_tiles, [&](int y, int j, int page) {
            if (!p.block_table) {
                tma_prefetch_4d(&tmK, 0, y, g, b);
                tma_prefetch_4d(&tmV, 0, y, g, b);
                return;
            }
            const int ty = (y + j * p.box_rows) & page_mask;
            tma_prefetch_4d(&tmK, 0, ty, g, page);
            tma_prefetch_4d(&tmV, 0, ty, g, page);
        });
    }
    __syncthreads();
    // Launched as a programmatic dependent: apart from the address hints of
    // the prefetch, nothing an earlier kernel may write is read before this.
    wait_primary();

    const int n_raw = p.seqlens[b];  // validated by each side where it is used

    if (warp == 0) {
        if (p.stall) {  // diagnostic: publish nothing, so the consumers' waits give up
            if (lane == 0) mbar_arrive(prod_done);
            allow_dependents();
            return;
        }
        {
            const uint64_t pol = l2_policy_evict_first();
            const bool paged = p.block_table != nullptr;
            const int page_mask = (1 << p.page_shift) - 1;
            produce_row<C::kStages>(
                p, b, b * p.Hkv + g, n_raw, n_hint, split, C::kTile, full, empty, meta, claim_sink, bad_page,
                C::kStageBytes, [&](int s, int y, int j, int page) {
                    uint8_t* st = stages + s * C::kStageBytes;
                    if (!paged) {
                        tma_load_4d(st, &tmK, 0, y, g, b, &full[s], pol);
                        tma_load_4d(st + C::kKBytes, &tmV, 0, y, g, b, &full[s], pol);
                        return;
                    }
                    const int ty = (y + j * p.box_rows) & page_mask;
                    const int off = j * p.box_rows * C::kRowBytes;
                    tma_load_4d(st + off, &tmK, 0, ty, g, page, &full[s], pol);
                    tma_load_4d(st + C::kKBytes + off, &tmV, 0, ty, g, page, &full[s], pol);
                });
        }
        if (lane == 0) mbar_arrive(prod_done);  // after its last claim (lane 0 makes them)
        allow_dependents();
        return;
    }

    // ---------------------------------------------------------- consumers
    int N = n_raw;
    const bool bad = (N < 0) || (N > p.S);
    if (bad) {
        if (threadIdx.x == 32) atomicOr(p.err, kErrBadSeqlen);
        N = 0;
    }
    const int G = p.G;
    const int NHC = G / GC;                  // head chunks (1, 2 or 4)
    const int NTS = C::kWarps / NHC;         // token slices of a stage
    const int cw = warp - 1;
    const int hc = cw % NHC, ts = cw / NHC;
    const int grp = lane >> 3, j = lane & 7;
    const int tok_per_slice = C::kTile / NTS;
    const int steps = tok_per_slice / 4;

    // this lane's channels: chunk (j + 8c), element e -> (j + 8c) * EPC + e
    float qf[GC][EPL];
    {
        const size_t qrow = static_cast<size_t>(b) * p.Hq + g * G + hc * GC;
#pragma unroll
        for (int i = 0; i < GC; ++i)
#pragma unroll
            for (int c = 0; c < CPL; ++c)
#pragma unroll
                for (int e = 0; e < EPC; ++e) {
                    const size_t idx = (qrow + i) * D + (j + 8 * c) * EPC + e;
                    const float qv = !in_bounds(idx, p.q_elems, p.err) ? 0.f
                        : p.q_is_bf16
                            ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.q)[idx])
                            : static_cast<const float*>(p.q)[idx];
                    qf[i][c * EPC + e] = qv * p.scale_log2;
                }
    }
    // causal limits of this warp's virtual heads (query i of nq sees tokens < N - nq + 1 + i)
    int lim[GC];
#pragma unroll
    for (int i = 0; i < GC; ++i)
        lim[i] = p.causal ? N - p.nq + 1 + (hc * GC + i) % p.nq : 0x7fffffff;
    float m[GC], l[GC], o[GC][EPL];
#pragma unroll
    for (int i = 0; i < GC; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[i][e] = 0.f;
    }
    bool timed_out = false;

    for (int it = 0;; ++it) {
        const int s = it % C::kStages;
        if (!mbar_wait(&full[s], (it / C::kStages) & 1, p.err)) {
            timed_out = true;
            break;
        }
        const int tile_valid = meta[s].nvalid;
        if (tile_valid < 0) break;  // end of this block's work
        const int tile_tok0 = meta[s].tok0;
        const uint8_t* kst = stages + s * C::kStageBytes;
        const uint8_t* vst = kst + C::kKBytes;
        for (int step = 0; step < steps; ++step) {
            const int row = ts * tok_per_slice + step * 4 + grp;
            const bool valid = row < tile_valid;
            float kf[EPL];
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const uint4 raw =
                    *reinterpret_cast<const uint4*>(kst + row * C::kRowBytes + (j + 8 * c) * 16);
                unpack16<KV>(raw, &kf[c * EPC]);
            }
            float pv[GC];
#pragma unroll
            for (int i = 0; i < GC; ++i) {
                float dot = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) dot = fmaf(qf[i][e], kf[e], dot);
                dot += __shfl_xor_sync(0xffffffffu, dot, 1);
                dot += __shfl_xor_sync(0xffffffffu, dot, 2);
                dot += __shfl_xor_sync(0xffffffffu, dot, 4);
                const bool vi = valid && tile_tok0 + row < lim[i];
                const float sc = vi ? dot : -INFINITY;
                if (sc > m[i]) {
                    const float al = ex2(m[i] - sc);
                    m[i] = sc;
                    l[i] *= al;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) o[i][e] *= al;
                }
                pv[i] = vi ? ex2(sc - m[i]) : 0.f;
                l[i] += pv[i];
            }
            if (valid) {
                float vf[EPL];
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(vst + row * C::kRowBytes +
                                                                      (j + 8 * c) * 16);
                    unpack16<KV>(raw, &vf[c * EPC]);
                }
#pragma unroll
                for (int i = 0; i < GC; ++i)
#pragma unroll
                    for (int e = 0; e < EPL; ++e) o[i][e] = fmaf(pv[i], vf[e], o[i][e]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (timed_out) atomicOr(abort_flag, 1);

    // merge the four groups of the warp (lanes j, j+8, j+16, j+24)
#pragma unroll
    for (int i = 0; i < GC; ++i) {
        float M = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], 8));
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 16));
        const float w = (M == -INFINITY) ? 0.f : ex2(m[i] - M);
        float li = l[i] * w;
        li += __shfl_xor_sync(0xffffffffu, li, 8);
        li += __shfl_xor_sync(0xffffffffu, li, 16);
        l[i] = li;
        m[i] = M;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            float oe = o[i][e] * w;
            oe += __shfl_xor_sync(0xffffffffu, oe, 8);
            oe += __shfl_xor_sync(0xffffffffu, oe, 16);
            o[i][e] = oe;
        }
    }
    if (grp == 0) {
#pragma unroll
        for (int i = 0; i < GC; ++i) {
            const int h = hc * GC + i;
#pragma unroll
            for (int c = 0; c < CPL; ++c)
#pragma unroll
                for (int e = 0; e < EPC; ++e)
                    mg_o[(ts * G + h) * D + (j + 8 * c) * EPC + e] = o[i][c * EPC + e];
            if (j == 0) {
                mg_m[ts * G + h] = m[i];
                mg_l[ts * G + h] = l[i];
            }
        }
    }
    consumer_sync(C::kWarps * 32);
    const bool poison = bad || (*abort_flag != 0) || (*bad_page != 0);
    const int ct = threadIdx.x - 32;
    for (int idx = ct; idx < G * D; idx += C::kWarps * 32) {
        const int h = idx / D, dd = idx - h * D;
        float M = -INFINITY;
        for (int t = 0; t < NTS; ++t) M = fmaxf(M, mg_m[t * G + h]);
        const float Ms = (M == -INFINITY) ? 0.f : M;
        float ov = 0.f, lv = 0.f;
        for (int t = 0; t < NTS; ++t) {
            const float wt = ex2(mg_m[t * G + h] - Ms);
            ov += wt * mg_o[(t * G + h) * D + dd];
            lv += wt * mg_l[t * G + h];
        }
        emit_state(p, b, g * G + h, split, D, dd, ov, lv, M, poison);
    }
    if (p.done)
        finish_row<D>(p, b * p.Hkv + g, static_cast<size_t>(b) * p.Hq + static_cast<size_t>(g) * p.G, p.G,
                      reinterpret_cast<float*>(stages), last_flag, prod_done, ct, C::kWarps * 32);
    allow_dependents();
}

template <typename KV, int D, int GC>
cudaError_t launch_one(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                       cudaStream_t stream) {
    using C = FmaCfg<KV, D>;
    static std::atomic<unsigned long long> configured{0};
    cudaError_t e = set_smem_once(split_kv_fma_kernel<KV, D, GC>, C::kSmem, configured);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.P, p.Hkv, p.B);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_kv_fma_kernel<KV, D, GC>, tk, tv, p);
}

template <typename KV, int D>
cudaError_t launch_d(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                     cudaStream_t stream) {
    switch (p.G) {
        case 1: return launch_one<KV, D, 1>(tk, tv, p, stream);
        case 2: return launch_one<KV, D, 2>(tk, tv, p, stream);
        case 4:
        case 8:
        case 16: return launch_one<KV, D, 4>(tk, tv, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <typename KV>
cudaError_t launch_fma(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv,
                       const SplitParams& p, cudaStream_t stream) {
    switch (head_dim) {
        case 64: return launch_d<KV, 64>(tk, tv, p, stream);
        case 128: return launch_d<KV, 128>(tk, tv, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fma_detail
}  // namespace ta
