// Split-KV partial attention over an FP8 (E4M3) KV cache with one scale per KV
// head, on the tensor cores (one or two n-tiles of 8 columns per KV head).
// Same blocks, scheduler, warp merge and row merge as the BF16 kernel; what
// changes is how the operands reach the mma.
//
// TMA brings 128-token tiles of 128-byte FP8 rows (128-byte swizzle).  There
// is no widening pass through shared memory: each thread loads its fragment
// bytes with 16-byte shared loads and converts E4M3 -> FP16 in registers
// (exact), feeding FP16 mma.m16n8k16 with FP32 accumulation.
//
//  S^T = K Q^T   The channel order of the contraction is permuted so that
//                thread (gid, tig) needs bytes [32 tig, 32 tig + 32) of rows
//                gid and gid + 8: in k-step kk its k-elements (2tig, 2tig+1)
//                and (2tig+8, 2tig+9) are channels 32tig + 4kk + {0,1} and
//                {2,3}.  q is loaded in the same order.
//  O^T += V^T P^T  Output channels are permuted instead: row gid (gid + 8) of
//                m-tile mt is channel 16 gid + 2 mt (+1), so a thread reads one
//                16-byte chunk of each of its four token rows, and byte pairs
//                of two token rows are interleaved with prmt before the
//                conversion.
// q is scaled by an exact power of two into the FP16 range (folded back into
// the logit scale with the KV head's K scale); P is scaled by 2^14 before its
// FP16 hi + lo split so that small weights keep their precision; the V scale
// and 2^-14 are applied to the merged numerator.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "emit.cuh"
#include "kernels.h"
#include "sched.cuh"
#include "warp_mma.cuh"

namespace ta {
namespace {

// HB KV heads per block: a stage holds kTile tokens of each (256 rows of
// 128 B per operand), and kWarps / HB consumer warps serve each head.
template <int HB>
struct Fp8Cfg {
    static constexpr int D = 128;
    static constexpr int kWarps = 8;                 // consumer warps
    static constexpr int kSub = 2;                   // 16-token slabs per warp per stage
    static constexpr int kRows = 16 * kWarps * kSub; // rows per operand per stage
    static constexpr int kTile = kRows / HB;         // tokens per stage
    static constexpr int kWPH = kWarps / HB;         // consumer warps per KV head
    static constexpr int kKBytes = kRows * D;        // one byte per element
    static constexpr int kStageBytes = 2 * kKBytes;  // K and V
    static constexpr int kStages = 6 / kSub;
    static constexpr int kBarBytes = 2 * kStages * 8 + kStages * 8 + 32;
    static constexpr int kSmem = 1024 + kStages * kStageBytes + kBarBytes;
    static constexpr int kThreads = 32 * (kWarps + 1);
    // Merge buffer: a warp state's row holds channel c at position
    // (c % 16) * 8 + c / 16, with 4 floats of padding per row, so the
    // fragment stores (rows 2 tig, 2 tig + 1; channels 16 gid + 2 mt (+1))
    // hit 32 distinct banks and the merge reads consecutive positions.
    static constexpr int kMergeStride = D + 4;
    static_assert(kWarps * 16 * (kMergeStride + 2) * 4 <= kStages * kStageBytes, "merge buffer (two n-tiles)");
    // cluster row merge: the block's merged state, [HB*16 heads][D] + 2 x [HB*16]
    static_assert((kWarps * 16 * (kMergeStride + 2) + HB * 16 * (D + 2)) * 4 <= kStages * kStageBytes,
                  "cluster state buffer");
};

constexpr float kPScale = 16384.f;  // 2^14

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t pair16) {
    uint32_t r;
    const uint16_t x = static_cast<uint16_t>(pair16);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(x));
    return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

template <int HB, int NT>
__global__ void __launch_bounds__(Fp8Cfg<HB>::kThreads, 1)
    split_kv_fp8_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const SplitParams p) {
    using C = Fp8Cfg<HB>;
    constexpr int D = C::D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = smem;
    float* mg_o = reinterpret_cast<float*>(stages);  // [W][8*NT][D (+pad)], after streaming
    float* mg_m = mg_o + C::kWarps * 8 * NT * C::kMergeStride;  // [W][8*NT]
    float* mg_l = mg_m + C::kWarps * 8 * NT;                    // [W][8*NT]
    float* cs_o = mg_l + C::kWarps * 8 * NT;  // cluster merge: [HB*G][D], m, l [HB*G]
    float* cs_m = cs_o + HB * 16 * D;
    float* cs_l = cs_m + HB * 16;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
    uint64_t* empty = full + C::kStages;
    volatile StageMeta* meta = reinterpret_cast<volatile StageMeta*>(empty + C::kStages);
    int* abort_flag = const_cast<int*>(reinterpret_cast<volatile int*>(meta + C::kStages));
    int* last_flag = abort_flag + 1;
    volatile unsigned* claim_sink = reinterpret_cast<volatile unsigned*>(abort_flag + 2);
    volatile int* bad_page = reinterpret_cast<volatile int*>(abort_flag + 3);
    uint64_t* prod_done = reinterpret_cast<uint64_t*>(abort_flag + 4);  // the copy warp's last claim is made

    // KV heads g0 .. g0 + HB - 1 of batch row b; schedule row `row`
    const int split = blockIdx.x, g0 = blockIdx.y * HB, b = blockIdx.z;
    const int row = b * (p.Hkv / HB) + blockIdx.y;
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
                tma_prefetch_4d(&tmK, 0, y, g0, b);
                tma_prefetch_4d(&tmV, 0, y, g0, b);
                return;
            }
            const int ty = (y + j * p.box_rows) & page_mask;
            tma_prefetch_4d(&tmK, 0, ty, g0, page);
            tma_prefetch_4d(&tmV, 0, ty, g0, page);
        });
    }
    __syncthreads();
    wait_primary();  // apart from the prefetch's address hints, nothing an earlier kernel writes is read before this

    const int n_raw = p.seqlens[b];  // validated by each side where it is used

    if (warp == 0) {
        if (p.stall) {  // diagnostic: publish nothing, so the consumers' waits give up
            if (lane == 0) mbar_arrive(prod_done);
            allow_dependents();
            if (p.cluster) {  // the cluster barriers of the row merge
                cluster_sync_all();
                cluster_sync_all();
            }
            return;
        }
        const uint64_t pol = l2_policy_evict_first();
        const bool paged = p.block_table != nullptr;
        const int page_mask = (1 << p.page_shift) - 1;
        // box j = box_rows tokens of the HB heads, [head][row][128 B], at j * box_bytes
        const int box_bytes = HB * p.box_rows * D;
        produce_row<C::kStages>(
            p, b, row, n_raw, n_hint, split, C::kTile, full, empty, meta, claim_sink, bad_page,
            C::kStageBytes, [&](int s, int y, int j, int page) {
                uint8_t* st = stages + s * C::kStageBytes;
                const int off = j * box_bytes;
                if (!in_bounds(off + box_bytes - 1, C::kKBytes, p.err)) return;
                if (!paged) {
                    tma_load_4d(st + off, &tmK, 0, y, g0, b, &full[s], pol);
                    tma_load_4d(st + C::kKBytes + off, &tmV, 0, y, g0, b, &full[s], pol);
                    return;
                }
                const int ty = (y + j * p.box_rows) & page_mask;
                tma_load_4d(st + off, &tmK, 0, ty, g0, page, &full[s], pol);
                tma_load_4d(st + C::kKBytes + off, &tmV, 0, ty, g0, page, &full[s], pol);
            });
        if (lane == 0) mbar_arrive(prod_done);  // after its last claim (lane 0 makes them)
        allow_dependents();
        if (p.cluster) {  // the cluster barriers of the row merge
            cluster_sync_all();
            cluster_sync_all();
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    int N = n_raw;
    const bool bad = (N < 0) || (N > p.S);
    if (bad) {
        if (threadIdx.x == 32) atomicOr(p.err, kErrBadSeqlen);
        N = 0;
    }
    const int cw = warp - 1;
    const int gid = lane >> 2, tig = lane & 3;
    const int hw = cw / C::kWPH, wi = cw % C::kWPH;  // this warp's head within the block
    const int g = g0 + hw;
    // scales first, so their loads overlap those of q
    const float ks = p.k_scale[g];
    float vsc[HB];  // V scales of the block's heads (applied in the merge), / 2^14
#pragma unroll
    for (int i = 0; i < HB; ++i) vsc[i] = p.v_scale[g0 + i] / kPScale;

    // q (BF16): column c = 8 nt + gid of n-tile nt (a query head, or a (head,
    // query) pair when several queries share the cache), channels 32 tig ..
    // 32 tig + 31 in the permuted order.
    // (kept as BF16 pairs: element 2 i of the chunk in the low half of word i)
    uint32_t qw[NT][16];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int c = nt * 8 + gid;
        const int hq = g * p.G + (c < p.G ? c : 0);
        const bool hv = c < p.G && in_bounds((static_cast<size_t>(b) * p.Hq + hq + 1) * D - 1, p.q_elems, p.err);
        const uint4* qh = reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(p.q) + (static_cast<size_t>(b) * p.Hq + hq) * D + 32 * tig);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = hv ? qh[i] : make_uint4(0u, 0u, 0u, 0u);
            qw[nt][4 * i] = v.x;
            qw[nt][4 * i + 1] = v.y;
            qw[nt][4 * i + 2] = v.z;
            qw[nt][4 * i + 3] = v.w;
        }
    }
    auto lo = [](uint32_t w) { return __uint_as_float(w << 16); };
    auto hi = [](uint32_t w) { return __uint_as_float(w & 0xffff0000u); };
    // exact power-of-two scale bringing max|q| into [2^14, 2^15): every q value
    // of the group is held by some lane of this warp
    float amax = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fmaxf(fabsf(lo(qw[nt][i])), fabsf(hi(qw[nt][i]))));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    int qexp = 0;
    if (amax > 0.f) {
        int e;
        frexpf(amax, &e);  // amax = f * 2^e, f in [0.5, 1)
        qexp = max(-100, min(100, 15 - e));
    }
    const float qs = ldexpf(1.f, qexp);
    uint32_t qb[NT][D / 16][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qb[nt][kk][0] = half2_bits(__floats2half2_rn(lo(qw[nt][2 * kk]) * qs, hi(qw[nt][2 * kk]) * qs));
            qb[nt][kk][1] =
                half2_bits(__floats2half2_rn(lo(qw[nt][2 * kk + 1]) * qs, hi(qw[nt][2 * kk + 1]) * qs));
        }
    const float sl2 = p.scale_log2 * ks / qs;

    // causal limits of this thread's columns (2 tig, 2 tig + 1 of each n-tile)
    const int causal_from = p.causal ? N - p.nq + 1 : 0x7fffffff;
    int lim[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j)
            lim[nt][j] = p.causal ? causal_from + (nt * 8 + 2 * tig + j) % p.nq : 0x7fffffff;

    float m[NT][2], l[NT][2];
    float oacc[NT][D / 16][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m[nt][0] = m[nt][1] = -INFINITY;
        l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
            oacc[nt][mt][0] = oacc[nt][mt][1] = oacc[nt][mt][2] = oacc[nt][mt][3] = 0.f;
    }

    // Rows are 128 B (one swizzle row); chunk c of row r sits at chunk c ^ (r & 7).
    // Offsets within a 16-row slab (slabs start at multiples of 16 rows, so
    // the swizzle phase of a row is the same in every slab).
    const int ra = gid, rb = gid + 8;                           // K rows of this thread
    const uint32_t k_a0 = ra * 128 + (((2 * tig) ^ (ra & 7)) << 4);
    const uint32_t k_a1 = ra * 128 + (((2 * tig + 1) ^ (ra & 7)) << 4);
    const uint32_t k_b0 = rb * 128 + (((2 * tig) ^ (rb & 7)) << 4);
    const uint32_t k_b1 = rb * 128 + (((2 * tig + 1) ^ (rb & 7)) << 4);
    const int tv0 = 2 * tig;                                    // V rows of this thread
    const uint32_t v_0 = tv0 * 128 + ((gid ^ (tv0 & 7)) << 4);
    const uint32_t v_1 = (tv0 + 1) * 128 + ((gid ^ ((tv0 + 1) & 7)) << 4);
    const uint32_t v_2 = (tv0 + 8) * 128 + ((gid ^ ((tv0 + 8) & 7)) << 4);
    const uint32_t v_3 = (tv0 + 9) * 128 + ((gid ^ ((tv0 + 9) & 7)) << 4);
    // This warp's slabs: tokens r0 .. r0 + 15 of the tile (r0 = 16 (sub * kWPH + wi)),
    // in box r0 / R at row r0 % R of its head's [R rows][128 B] part.
    static_assert(C::kSub == 2, "two slabs per warp per stage");
    const int R = p.box_rows;
    auto slab_offset = [&](int r0) -> uint32_t {
        return (r0 / R) * (HB * R * 128) + hw * (R * 128) + (r0 % R) * 128;
    };
    const uint32_t slab_off0 = slab_offset(wi * 16), slab_off1 = slab_offset((C::kWPH + wi) * 16);
    bool timed_out = false;

    for (int it = 0;; ++it) {
        const int s = it % C::kStages;
        if (!mbar_wait(&full[s], (it / C::kStages) & 1, p.err)) {
            timed_out = true;
            break;
        }
        const int tile_valid = meta[s].nvalid;
        if (tile_valid < 0) break;
        const int tile_tok0 = meta[s].tok0;
#pragma unroll 1
        for (int sub = 0; sub < C::kSub; ++sub) {
            const int r0 = (sub * C::kWPH + wi) * 16;  // first token of this warp's slab
            const int blk0 = tile_tok0 + r0;
            uint32_t kbase = smem_u32(stages + s * C::kStageBytes);
            if constexpr (HB == 1)
                kbase += r0 * 128;  // one box of the whole tile
            else
                kbase += (sub == 0 ? slab_off0 : slab_off1);
            const uint32_t vbase = kbase + C::kKBytes;
            const int nvalid = tile_valid - r0;

            if (nvalid > 0) {
                const uint4 ka0 = lds128(kbase + k_a0), ka1 = lds128(kbase + k_a1);
                const uint4 kb0 = lds128(kbase + k_b0), kb1 = lds128(kbase + k_b1);
                const uint32_t wa[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
                const uint32_t wb[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
                float sa[NT][4], sb[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sa[nt][e] = sb[nt][e] = 0.f;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint32_t a[4];
                    a[0] = e4m3x2_to_f16x2(wa[kk] & 0xffffu);
                    a[1] = e4m3x2_to_f16x2(wb[kk] & 0xffffu);
                    a[2] = e4m3x2_to_f16x2(wa[kk] >> 16);
                    a[3] = e4m3x2_to_f16x2(wb[kk] >> 16);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (kk & 1)
                            mma_f16(sb[nt], a, qb[nt][kk][0], qb[nt][kk][1]);
                        else
                            mma_f16(sa[nt], a, qb[nt][kk][0], qb[nt][kk][1]);
                    }
                }
                const bool causal_blk = blk0 + 16 > causal_from;
                uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float s0 = (sa[nt][0] + sb[nt][0]) * sl2, s1 = (sa[nt][1] + sb[nt][1]) * sl2;
                    float s2 = (sa[nt][2] + sb[nt][2]) * sl2, s3 = (sa[nt][3] + sb[nt][3]) * sl2;
                    if (nvalid < 16) {
                        if (gid >= nvalid) s0 = s1 = -INFINITY;
                        if (gid + 8 >= nvalid) s2 = s3 = -INFINITY;
                    }
                    if (causal_blk) {
                        const int ta = blk0 + gid, tb = ta + 8;
                        if (ta >= lim[nt][0]) s0 = -INFINITY;
                        if (ta >= lim[nt][1]) s1 = -INFINITY;
                        if (tb >= lim[nt][0]) s2 = -INFINITY;
                        if (tb >= lim[nt][1]) s3 = -INFINITY;
                    }
                    float bm0 = fmaxf(s0, s2), bm1 = fmaxf(s1, s3);
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
                        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
                    }
                    const float mn0 = fmaxf(m[nt][0], bm0), mn1 = fmaxf(m[nt][1], bm1);
                    const float ms0 = (mn0 == -INFINITY) ? 0.f : mn0;
                    const float ms1 = (mn1 == -INFINITY) ? 0.f : mn1;
                    const float al0 = ex2(m[nt][0] - ms0), al1 = ex2(m[nt][1] - ms1);
                    const float p0 = ex2(s0 - ms0), p1 = ex2(s1 - ms1);
                    const float p2 = ex2(s2 - ms0), p3 = ex2(s3 - ms1);
                    l[nt][0] = l[nt][0] * al0 + (p0 + p2);
                    l[nt][1] = l[nt][1] * al1 + (p1 + p3);
                    m[nt][0] = mn0;
                    m[nt][1] = mn1;
                    if (__any_sync(0xffffffffu, (al0 != 1.f) || (al1 != 1.f))) {
#pragma unroll
                        for (int mt = 0; mt < D / 16; ++mt) {
                            oacc[nt][mt][0] *= al0;
                            oacc[nt][mt][1] *= al1;
                            oacc[nt][mt][2] *= al0;
                            oacc[nt][mt][3] *= al1;
                        }
                    }
                    // P^T (scaled by 2^14) as FP16 hi + lo B fragments
                    const float q0 = p0 * kPScale, q1 = p1 * kPScale, q2 = p2 * kPScale, q3 = p3 * kPScale;
                    const __half2 h01 = __floats2half2_rn(q0, q1), h23 = __floats2half2_rn(q2, q3);
                    const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
                    const __half2 e01 = __floats2half2_rn(q0 - f01.x, q1 - f01.y);
                    const __half2 e23 = __floats2half2_rn(q2 - f23.x, q3 - f23.y);
                    bh[nt][0] = movtrans(half2_bits(h01));
                    bh[nt][1] = movtrans(half2_bits(h23));
                    bl[nt][0] = movtrans(half2_bits(e01));
                    bl[nt][1] = movtrans(half2_bits(e23));
                }
                // V: tokens 2tig, 2tig+1, 2tig+8, 2tig+9 of the block, channels 16 gid .. 16 gid + 15;
                // rows past the valid range may hold anything (even NaN codes): zero them
                uint4 va = lds128(vbase + v_0), vb = lds128(vbase + v_1);
                uint4 vc = lds128(vbase + v_2), vd = lds128(vbase + v_3);
                if (nvalid < 16) {
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                    if (2 * tig >= nvalid) va = z;
                    if (2 * tig + 1 >= nvalid) vb = z;
                    if (2 * tig + 8 >= nvalid) vc = z;
                    if (2 * tig + 9 >= nvalid) vd = z;
                }
                const uint32_t xa[4] = {va.x, va.y, va.z, va.w}, xb[4] = {vb.x, vb.y, vb.z, vb.w};
                const uint32_t xc[4] = {vc.x, vc.y, vc.z, vc.w}, xd[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t p01 = prmt(xa[w], xb[w], 0x5140u), p23 = prmt(xa[w], xb[w], 0x7362u);
                    const uint32_t r01 = prmt(xc[w], xd[w], 0x5140u), r23 = prmt(xc[w], xd[w], 0x7362u);
                    uint32_t a[4];
                    a[0] = e4m3x2_to_f16x2(p01 & 0xffffu);
                    a[1] = e4m3x2_to_f16x2(p01 >> 16);
                    a[2] = e4m3x2_to_f16x2(r01 & 0xffffu);
                    a[3] = e4m3x2_to_f16x2(r01 >> 16);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_f16(oacc[nt][2 * w], a, bh[nt][0], bh[nt][1]);
                        mma_f16(oacc[nt][2 * w], a, bl[nt][0], bl[nt][1]);
                    }
                    a[0] = e4m3x2_to_f16x2(p23 & 0xffffu);
                    a[1] = e4m3x2_to_f16x2(p23 >> 16);
                    a[2] = e4m3x2_to_f16x2(r23 & 0xffffu);
                    a[3] = e4m3x2_to_f16x2(r23 >> 16);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_f16(oacc[nt][2 * w + 1], a, bh[nt][0], bh[nt][1]);
                        mma_f16(oacc[nt][2 * w + 1], a, bl[nt][0], bl[nt][1]);
                    }
                }
            }
        }  // slabs
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (timed_out) atomicOr(abort_flag, 1);

    // ------------------------------------------- merge the warps' states
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], off);
            l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], off);
        }
    consumer_sync(C::kWarps * 32);  // every warp is done reading the stages
    constexpr int MS = C::kMergeStride;
    constexpr int kCols = 8 * NT;  // columns per warp state
    float* mo = mg_o + cw * kCols * MS;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int c0 = nt * 8 + 2 * tig;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            // fragment rows gid / gid + 8 are channels 16 gid + 2 mt (+1), stored at
            // positions (2 mt) * 8 + gid and (2 mt + 1) * 8 + gid
            const int pos = 16 * mt + gid;
            mo[c0 * MS + pos] = oacc[nt][mt][0];
            mo[(c0 + 1) * MS + pos] = oacc[nt][mt][1];
            mo[c0 * MS + pos + 8] = oacc[nt][mt][2];
            mo[(c0 + 1) * MS + pos + 8] = oacc[nt][mt][3];
        }
        if (gid == 0) {
            mg_m[cw * kCols + c0] = m[nt][0];
            mg_m[cw * kCols + c0 + 1] = m[nt][1];
            mg_l[cw * kCols + c0] = l[nt][0];
            mg_l[cw * kCols + c0 + 1] = l[nt][1];
        }
    }
    consumer_sync(C::kWarps * 32);
    const bool poison = bad || (*abort_flag != 0) || (*bad_page != 0);
    const int ct = threadIdx.x - 32;
    // states of the warps serving one head, merged per (head, column, channel)
    for (int idx = ct; idx < HB * p.G * D; idx += C::kWarps * 32) {
        int hh = 0, rem = idx;
        if constexpr (HB > 1) {
            hh = idx / (p.G * D);
            rem = idx - hh * (p.G * D);
        }
        const int h = rem / D, pos = rem - h * D;
        const int dd = (pos & 7) * 16 + (pos >> 3);  // channel stored at `pos`
        const int w0 = hh * C::kWPH;
        float mw[C::kWPH];
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::kWPH; ++w) {
            mw[w] = mg_m[(w0 + w) * kCols + h];
            M = fmaxf(M, mw[w]);
        }
        const float Ms = (M == -INFINITY) ? 0.f : M;
        float ow[C::kWPH], lw[C::kWPH];
#pragma unroll
        for (int w = 0; w < C::kWPH; ++w) {
            const float wt = ex2(mw[w] - Ms);
            ow[w] = wt * mg_o[((w0 + w) * kCols + h) * MS + pos];
            lw[w] = wt * mg_l[(w0 + w) * kCols + h];
        }
        float osc = vsc[0];
#pragma unroll
        for (int i = 1; i < HB; ++i) osc = (hh == i) ? vsc[i] : osc;
        const float o = tree_sum<C::kWPH>(ow) * osc;
        const float lsum = tree_sum<C::kWPH>(lw);
        if (p.cluster) {  // kept for the cluster row merge
            const float nan = __int_as_float(0x7fc00000);
            const int hb_h = hh * p.G + h;
            cs_o[hb_h * D + dd] = poison ? nan : o;
            if (dd == 0) {
                cs_m[hb_h] = poison ? nan : M;
                cs_l[hb_h] = poison ? nan : lsum;
            }
        } else {
            emit_state(p, b, (g0 + hh) * p.G + h, split, D, dd, o, lsum, M, poison);
        }
    }
    const size_t hq0 = static_cast<size_t>(b) * p.Hq + static_cast<size_t>(g0) * p.G;
    if (p.cluster) {
        cluster_sync_all();  // every block's state is in its shared memory; every claim is made
        if (p.claim && ct == 0 && cluster_rank() == 0) atomicExch(p.claim + row, 0u);
        cluster_merge_row<D, 8>(p, hq0, HB * p.G, cs_o, cs_m, cs_l, ct, C::kWarps * 32);
        cluster_sync_all();  // no block's state goes away while a peer reads it
    } else if (p.done) {
        finish_row<D>(p, row, hq0, HB * p.G, reinterpret_cast<float*>(stages), last_flag, prod_done, ct, C::kWarps * 32);
    }
    allow_dependents();
}

template <int HB, int NT>
cudaError_t launch_hb(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                      cudaStream_t stream) {
    using C = Fp8Cfg<HB>;
    static std::atomic<unsigned long long> configured{0};
    cudaError_t e = set_smem_once(split_kv_fp8_kernel<HB, NT>, C::kSmem, configured);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.P, p.Hkv / HB, p.B);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;  // a row's P blocks form one cluster
    attr[1].val.clusterDim.x = static_cast<unsigned>(p.P);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.cluster ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, split_kv_fp8_kernel<HB, NT>, tk, tv, p);
}

}  // namespace

Geometry fp8_geometry(int heads_per_block) {
    switch (heads_per_block) {
        case 2: return Geometry{Fp8Cfg<2>::kTile, Fp8Cfg<2>::D, 1, 0, 2};
        case 4: return Geometry{Fp8Cfg<4>::kTile, Fp8Cfg<4>::D, 1, 0, 4};
        default: return Geometry{Fp8Cfg<1>::kTile, Fp8Cfg<1>::D, 1, 0, 1};
    }
}

cudaError_t launch_split_fp8(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                             cudaStream_t stream) {
    // one n-tile of 8 columns per KV head group, two for up to 16
    const bool two = p.G > 8;
    switch (p.hb) {
        case 1: return two ? launch_hb<1, 2>(tk, tv, p, stream) : launch_hb<1, 1>(tk, tv, p, stream);
        case 2: return two ? launch_hb<2, 2>(tk, tv, p, stream) : launch_hb<2, 1>(tk, tv, p, stream);
        case 4: return two ? launch_hb<4, 2>(tk, tv, p, stream) : launch_hb<4, 1>(tk, tv, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ta
