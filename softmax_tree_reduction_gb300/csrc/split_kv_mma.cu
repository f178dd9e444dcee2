// Split-KV partial attention on the tensor cores (BF16 q and KV, FP32 state).
//
// One thread block per (slice p, KV head g, batch row b) computes the partial
// state (o, l, m) of its slice of the sequence for the G query heads that
// share KV head g ("Local Independent Partial Attention" on the Tree
// Attention pages), then merges the states of its warps with the merge
// operator ("The Tree Reduction Merge Operator").
//
//  warp 0      producer: streams K and V tiles (128 tokens x all channels,
//              as 128-byte-swizzled halves of 64 channels) HBM -> shared memory
//              with TMA into a ring of stages guarded by full/empty mbarriers.
//  warps 1..8  consumers: each owns 16 tokens of every 128-token stage (two
//              warps per SM sub-partition hide each other's latencies).
//     S^T[16 tok x 8 heads] = K_blk . Q^T      mma.m16n8k16 (A = K via ldmatrix,
//                                              B = q, resident in registers)
//     online softmax over the block            FP32, base 2, per head
//     O^T[d x 8 heads] += V_blk^T . P^T        mma.m16n8k16 (A = V via
//                                              ldmatrix.trans, B = P moved into
//                                              place by movmatrix.trans)
//  P is fed to the second product as BF16 hi + lo parts (two mma), so the
//  weights keep ~16 significant bits; every accumulation is FP32.
//  Heads beyond G in the 8-wide n dimension are zero and never written.
#include <cuda_bf16.h>

#include "common.cuh"
#include "emit.cuh"
#include "kernels.h"
#include "sched.cuh"

namespace ta {
namespace {

template <int D>
struct MmaCfg {
    static constexpr int kWarps = 8;                 // consumer warps (two per SM sub-partition)
    static constexpr int kTile = 16 * kWarps;        // tokens per stage
    static constexpr int kHalves = D / 64;           // 128-byte column blocks per row
    static constexpr int kKBytes = kHalves * kTile * 128;
    static constexpr int kStageBytes = 2 * kKBytes;  // K and V
    static constexpr int kStages = (D == 128) ? 3 : 6;
    static constexpr int kBarBytes = 2 * kStages * 8 + kStages * 8 + 32;
    // the warps' states are merged in the stage buffers once streaming is over
    static constexpr int kSmem = 1024 + kStages * kStageBytes + kBarBytes;
    static constexpr int kThreads = 32 * (kWarps + 1);
    static_assert(kWarps * 8 * (D + 2) * 4 <= kStages * kStageBytes, "merge buffer");
    static_assert(kTile <= 256, "TMA box height");
};

// Pairwise tree sum of N values (N a power of two).
template <int N>
__device__ __forceinline__ float tree_sum(const float* v) {
    if constexpr (N == 1) {
        return v[0];
    } else {
        return tree_sum<N / 2>(v) + tree_sum<N / 2>(v + N / 2);
    }
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 v) {
    return *reinterpret_cast<uint32_t*>(&v);
}

template <int D>
__global__ void __launch_bounds__(MmaCfg<D>::kThreads, 1)
    split_kv_mma_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const SplitParams p) {
    using C = MmaCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = smem;
    float* mg_o = reinterpret_cast<float*>(stages);  // [W][8][D], after streaming
    float* mg_m = mg_o + C::kWarps * 8 * D;          // [W][8]
    float* mg_l = mg_m + C::kWarps * 8;              // [W][8]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
    uint64_t* empty = full + C::kStages;
    volatile StageMeta* meta = reinterpret_cast<volatile StageMeta*>(empty + C::kStages);
    int* abort_flag = const_cast<int*>(reinterpret_cast<volatile int*>(meta + C::kStages));
    int* last_flag = abort_flag + 1;
    volatile unsigned* claim_sink = reinterpret_cast<volatile unsigned*>(abort_flag + 2);
    volatile int* bad_page = reinterpret_cast<volatile int*>(abort_flag + 3);

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::kWarps);
        }
        *abort_flag = 0;
        *bad_page = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    __syncthreads();
    // Launched as a programmatic dependent: nothing an earlier kernel may
    // write (q, the caches, the lengths, the outputs) is touched before this.
    wait_primary();

    int N = p.seqlens[b];
    const bool bad = (N < 0) || (N > p.S);
    if (bad) {
        if (threadIdx.x == 0) atomicOr(p.err, kErrBadSeqlen);
        N = 0;
    }

    if (warp == 0) {
        // ------------------------------------------------------ producer
        {
            const uint64_t pol = l2_policy_evict_first();
            const bool paged = p.block_table != nullptr;
            const int page_mask = (1 << p.page_shift) - 1;
            const int box_bytes = C::kHalves * p.box_rows * 128;
            produce_row<C::kStages>(
                p, b, b * p.Hkv + g, N, split, C::kTile, full, empty, meta, claim_sink, bad_page,
                C::kStageBytes, [&](int s, int y, int j, int page) {
                    // One box = box_rows tokens x all channels, laid out in shared
                    // memory as [half][box_rows][128 B]; box j of a tile at j*box_bytes.
                    uint8_t* st = stages + s * C::kStageBytes;
                    const int off = j * box_bytes;
                    if (!paged) {
                        tma_load_5d(st + off, &tmK, 0, y, 0, g, b, &full[s], pol);
                        tma_load_5d(st + C::kKBytes + off, &tmV, 0, y, 0, g, b, &full[s], pol);
                        return;
                    }
                    // paged: (channel, token in page, half, KV head, physical page)
                    const int ty = (y + j * p.box_rows) & page_mask;
                    tma_load_5d(st + off, &tmK, 0, ty, 0, g, page, &full[s], pol);
                    tma_load_5d(st + C::kKBytes + off, &tmV, 0, ty, 0, g, page, &full[s], pol);
                });
        }
        allow_dependents();
        return;
    }

    // ---------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int gid = lane >> 2, tig = lane & 3;
    const int r8 = lane & 7;

    // q as the B operand of S^T = K Q^T: column n = head gid of this group.
    uint32_t qb[D / 16][2];
    {
        const bool hv = gid < p.G;
        const int hq = g * p.G + (hv ? gid : 0);
        const __nv_bfloat16* qh =
            static_cast<const __nv_bfloat16*>(p.q) + (static_cast<size_t>(b) * p.Hq + hq) * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qb[kk][0] = hv ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 2 * tig) : 0u;
            qb[kk][1] = hv ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 8 + 2 * tig) : 0u;
        }
    }

    // Running state for heads (2*tig, 2*tig+1): maxima (log2 units, equal in
    // all lanes of a column), per-lane partial denominators, O^T fragments.
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float oacc[D / 16][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;

    // ldmatrix row addresses (swizzled 16-byte chunk = chunk ^ (row & 7)).  A
    // stage holds tile/R boxes of [half][R rows][128 B] (R = box_rows >= 16), so
    // this warp's 16 rows sit in one box.
    const int R = p.box_rows;
    const uint32_t half_bytes = R * 128;
    const int r0 = cw * 16;
    const uint32_t warp_base = (r0 / R) * (C::kHalves * half_bytes) + (r0 % R) * 128;
    const uint32_t k_row = warp_base + (r8 + 8 * ((lane >> 3) & 1)) * 128;
    const int k_chi = lane >> 4;
    const uint32_t v_row = warp_base + (r8 + 8 * (lane >> 4)) * 128;
    const int v_chi = (lane >> 3) & 1;
    const float sl2 = p.scale_log2;
    bool timed_out = false;

    for (int it = 0;; ++it) {
        const int s = it % C::kStages;
        if (!mbar_wait(&full[s], (it / C::kStages) & 1, p.err)) {
            timed_out = true;
            break;
        }
        const int tile_valid = meta[s].nvalid;
        if (tile_valid < 0) break;  // end of this block's work
        const uint32_t kbase = smem_u32(stages + s * C::kStageBytes);
        const uint32_t vbase = kbase + C::kKBytes;
        const int nvalid = tile_valid - cw * 16;  // valid tokens of this warp's 16-token block

        if (nvalid > 0) {
            // S^T = K_blk Q^T (two accumulators to shorten the dependency chain)
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int c = 2 * (kk & 3) + k_chi;
                uint32_t a[4];
                ldsm_x4(a, kbase + (kk >> 2) * half_bytes + k_row + ((c ^ r8) << 4));
                if (kk & 1)
                    mma_bf16(sb, a, qb[kk][0], qb[kk][1]);
                else
                    mma_bf16(sa, a, qb[kk][0], qb[kk][1]);
            }
            float s0 = (sa[0] + sb[0]) * sl2, s1 = (sa[1] + sb[1]) * sl2;
            float s2 = (sa[2] + sb[2]) * sl2, s3 = (sa[3] + sb[3]) * sl2;
            if (nvalid < 16) {
                if (gid >= nvalid) s0 = s1 = -INFINITY;
                if (gid + 8 >= nvalid) s2 = s3 = -INFINITY;
            }
            // block maximum per head over the 16 tokens (lanes differing in gid)
            float bm0 = fmaxf(s0, s2), bm1 = fmaxf(s1, s3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
                bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
            }
            const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
            const float ms0 = (mn0 == -INFINITY) ? 0.f : mn0;
            const float ms1 = (mn1 == -INFINITY) ? 0.f : mn1;
            const float al0 = ex2(m0 - ms0), al1 = ex2(m1 - ms1);
            const float p0 = ex2(s0 - ms0), p1 = ex2(s1 - ms1);
            const float p2 = ex2(s2 - ms0), p3 = ex2(s3 - ms1);
            l0 = l0 * al0 + (p0 + p2);
            l1 = l1 * al1 + (p1 + p3);
            m0 = mn0;
            m1 = mn1;
            if (__any_sync(0xffffffffu, (al0 != 1.f) || (al1 != 1.f))) {
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    oacc[mt][0] *= al0;
                    oacc[mt][1] *= al1;
                    oacc[mt][2] *= al0;
                    oacc[mt][3] *= al1;
                }
            }
            // P^T as B fragments (k = token, n = head), BF16 hi + lo parts.
            const __nv_bfloat162 h01 = __floats2bfloat162_rn(p0, p1);
            const __nv_bfloat162 h23 = __floats2bfloat162_rn(p2, p3);
            const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
            const __nv_bfloat162 e01 = __floats2bfloat162_rn(p0 - f01.x, p1 - f01.y);
            const __nv_bfloat162 e23 = __floats2bfloat162_rn(p2 - f23.x, p3 - f23.y);
            const uint32_t bh0 = movtrans(bf16x2_bits(h01)), bh1 = movtrans(bf16x2_bits(h23));
            const uint32_t bl0 = movtrans(bf16x2_bits(e01)), bl1 = movtrans(bf16x2_bits(e23));
            // V rows past the slice may hold anything (even NaN): zero them.
            uint32_t vm01 = 0xffffffffu, vm23 = 0xffffffffu;
            if (nvalid < 16) {
                const int ta = 2 * tig, tb = 8 + 2 * tig;
                vm01 = (ta < nvalid ? 0x0000ffffu : 0u) | (ta + 1 < nvalid ? 0xffff0000u : 0u);
                vm23 = (tb < nvalid ? 0x0000ffffu : 0u) | (tb + 1 < nvalid ? 0xffff0000u : 0u);
            }
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const int c = 2 * (mt & 3) + v_chi;
                uint32_t a[4];
                ldsm_x4_t(a, vbase + (mt >> 2) * half_bytes + v_row + ((c ^ r8) << 4));
                a[0] &= vm01;
                a[1] &= vm01;
                a[2] &= vm23;
                a[3] &= vm23;
                mma_bf16(oacc[mt], a, bh0, bh1);
                mma_bf16(oacc[mt], a, bl0, bl1);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (timed_out) atomicOr(abort_flag, 1);

    // ------------------------------------------- merge the warps' states
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    consumer_sync(C::kWarps * 32);  // every warp is done reading the stages
    float* mo = mg_o + cw * 8 * D;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        mo[(2 * tig) * D + 16 * mt + gid] = oacc[mt][0];
        mo[(2 * tig + 1) * D + 16 * mt + gid] = oacc[mt][1];
        mo[(2 * tig) * D + 16 * mt + gid + 8] = oacc[mt][2];
        mo[(2 * tig + 1) * D + 16 * mt + gid + 8] = oacc[mt][3];
    }
    if (gid == 0) {
        mg_m[cw * 8 + 2 * tig] = m0;
        mg_m[cw * 8 + 2 * tig + 1] = m1;
        mg_l[cw * 8 + 2 * tig] = l0;
        mg_l[cw * 8 + 2 * tig + 1] = l1;
    }
    consumer_sync(C::kWarps * 32);
    const bool poison = bad || (*abort_flag != 0) || (*bad_page != 0);
    const int ct = threadIdx.x - 32;
    for (int idx = ct; idx < p.G * D; idx += C::kWarps * 32) {
        const int h = idx / D, dd = idx - h * D;
        float mw[C::kWarps];
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::kWarps; ++w) {
            mw[w] = mg_m[w * 8 + h];
            M = fmaxf(M, mw[w]);
        }
        const float Ms = (M == -INFINITY) ? 0.f : M;
        float ow[C::kWarps], lw[C::kWarps];
#pragma unroll
        for (int w = 0; w < C::kWarps; ++w) {
            const float wt = ex2(mw[w] - Ms);
            ow[w] = wt * mg_o[(w * 8 + h) * D + dd];
            lw[w] = wt * mg_l[w * 8 + h];
        }
        // pairwise tree over the warps
        const float o = tree_sum<C::kWarps>(ow);
        const float l = tree_sum<C::kWarps>(lw);
        emit_state(p, b, g * p.G + h, split, D, dd, o, l, M, poison);
    }
    if (p.done) finish_row<D>(p, b, g, reinterpret_cast<float*>(stages), last_flag, ct, C::kWarps * 32);
    allow_dependents();
}

template <int D>
cudaError_t launch_impl(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                        cudaStream_t stream) {
    using C = MmaCfg<D>;
    cudaError_t e = cudaFuncSetAttribute(split_kv_mma_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
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
    return cudaLaunchKernelEx(&cfg, split_kv_mma_kernel<D>, tk, tv, p);
}

}  // namespace

Geometry mma_geometry(int head_dim) {
    (void)head_dim;
    return Geometry{MmaCfg<128>::kTile, 64, 1};
}

cudaError_t launch_split_mma(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv,
                             const SplitParams& p, cudaStream_t stream) {
    switch (head_dim) {
        case 64: return launch_impl<64>(tk, tv, p, stream);
        case 128: return launch_impl<128>(tk, tv, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ta
