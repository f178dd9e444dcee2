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
//  The n dimension holds the group's G query heads (or (head, query) pairs
//  when several queries share the cache), 8 per n-tile, one or two n-tiles;
//  unused columns are zero and never written.
#include <cuda_bf16.h>

#include "common.cuh"
#include "emit.cuh"
#include "kernels.h"
#include "sched.cuh"
#include "warp_mma.cuh"

namespace ta {
namespace {

// Consumer warps are split into groups.  HB KV heads per block: a stage
// holds kTile tokens of each (128 rows per operand) and each head has its
// group of warps, one 16-token slab per warp.  CG column groups (more than 16
// columns per KV head, HB = 1): each group of warps owns 16 columns and every
// warp takes CG slabs of each 128-token stage.
template <int D, int HB, int CG = 1>
struct MmaCfg {
    static_assert(HB == 1 || CG == 1, "heads per block or column groups");
    static constexpr int kWarps = 8;                 // consumer warps (two per SM sub-partition)
    static constexpr int kRows = 16 * kWarps;        // rows per operand per stage
    static constexpr int kTile = kRows / HB;         // tokens per stage
    static constexpr int kGroups = HB * CG;          // warp groups (heads or column groups)
    static constexpr int kWPG = kWarps / kGroups;    // consumer warps per group
    static constexpr int kSub = CG;                  // 16-token slabs per warp per stage
    static constexpr int kLocalHeads = 16 * HB * CG; // most (head, column) states a block holds
    static constexpr int kHalves = D / 64;           // 128-byte column blocks per row
    static constexpr int kKBytes = kHalves * kRows * 128;
    static constexpr int kStageBytes = 2 * kKBytes;  // K and V
    static constexpr int kStages = (D == 128) ? 3 : 6;
    static constexpr int kBarBytes = 2 * kStages * 8 + kStages * 8 + 32;
    // Column groups keep q in shared memory ([column][d] rows padded by 16
    // bytes, so the 8 rows an ldmatrix reads fall in distinct banks) and load
    // its fragments per k-step, which leaves the registers to the running state.
    static constexpr bool kQSmem = CG > 1;
    static constexpr int kQRowBytes = (D + 8) * 2;
    static constexpr int kQOff = (kStages * kStageBytes + kBarBytes + 127) / 128 * 128;
    static constexpr int kQBytes = kQSmem ? 16 * CG * kQRowBytes : 0;
    // the warps' states are merged in the stage buffers once streaming is over
    static constexpr int kSmem = 1024 + (kQSmem ? kQOff + kQBytes : kStages * kStageBytes + kBarBytes);
    static_assert(kSmem <= 227 * 1024, "shared memory per block");
    static constexpr int kThreads = 32 * (kWarps + 1);
    // Row stride of a warp state in the merge buffer: 4 floats of padding make
    // the fragment stores (rows 2 tig, 2 tig + 1; channels 16 mt + gid) hit 32
    // distinct banks.
    static constexpr int kMergeStride = D + 4;
    static_assert(kWarps * 16 * (kMergeStride + 2) * 4 <= kStages * kStageBytes, "merge buffer (two n-tiles)");
    // cluster row merge: the block's merged state, [kLocalHeads][D] + 2 x [kLocalHeads]
    static_assert((kWarps * 16 * (kMergeStride + 2) + kLocalHeads * (D + 2)) * 4 <= kStages * kStageBytes,
                  "cluster state buffer");
    static_assert(kTile <= 256, "TMA box height");
};

template <int D, int NT, int HB, int CG>
__global__ void __launch_bounds__(MmaCfg<D, HB, CG>::kThreads, 1)
    split_kv_mma_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const SplitParams p) {
    using C = MmaCfg<D, HB, CG>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = smem;
    float* mg_o = reinterpret_cast<float*>(stages);  // [W][8*NT][D (+pad)], after streaming
    float* mg_m = mg_o + C::kWarps * 8 * NT * C::kMergeStride;  // [W][8*NT]
    float* mg_l = mg_m + C::kWarps * 8 * NT;         // [W][8*NT]
    float* cs_o = mg_l + C::kWarps * 8 * NT;         // cluster merge: [HB*G][D], m, l [HB*G]
    float* cs_m = cs_o + C::kLocalHeads * D;
    float* cs_l = cs_m + C::kLocalHeads;
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
    if (warp == 0) {
        const int page_mask = (1 << p.page_shift) - 1;
        n_hint = prefetch_row_head(p, b, split, C::kTile, p.prefetch_tiles, [&](int y, int j, int page) {
            if (!p.block_table) {
                tma_prefetch_5d(&tmK, 0, y, 0, g0, b);
                tma_prefetch_5d(&tmV, 0, y, 0, g0, b);
                return;
            }
            const int ty = (y + j * p.box_rows) & page_mask;
            tma_prefetch_5d(&tmK, 0, ty, 0, g0, page);
            tma_prefetch_5d(&tmV, 0, ty, 0, g0, page);
        });
    }
    __syncthreads();
    // Launched as a programmatic dependent: apart from the address hints of
    // the prefetch, nothing an earlier kernel may write (q, the caches, the
    // lengths, the outputs) is read before this.
    wait_primary();

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
        // ------------------------------------------------------ producer
        {
            const uint64_t pol = l2_policy_evict_first();
            const bool paged = p.block_table != nullptr;
            const int page_mask = (1 << p.page_shift) - 1;
            const int box_bytes = HB * C::kHalves * p.box_rows * 128;
            produce_row<C::kStages>(
                p, b, row, n_raw, n_hint, split, C::kTile, full, empty, meta, claim_sink, bad_page,
                C::kStageBytes, [&](int s, int y, int j, int page) {
                    // One box = box_rows tokens x all channels of the HB heads, laid out
                    // in shared memory as [head][half][box_rows][128 B]; box j of a
                    // tile at j*box_bytes.
                    uint8_t* st = stages + s * C::kStageBytes;
                    const int off = j * box_bytes;
                    if (!in_bounds(off + box_bytes - 1, C::kKBytes, p.err)) return;
                    if (!paged) {
                        tma_load_5d(st + off, &tmK, 0, y, 0, g0, b, &full[s], pol);
                        tma_load_5d(st + C::kKBytes + off, &tmV, 0, y, 0, g0, b, &full[s], pol);
                        return;
                    }
                    // paged: (channel, token in page, half, KV head, physical page)
                    const int ty = (y + j * p.box_rows) & page_mask;
                    tma_load_5d(st + off, &tmK, 0, ty, 0, g0, page, &full[s], pol);
                    tma_load_5d(st + C::kKBytes + off, &tmV, 0, ty, 0, g0, page, &full[s], pol);
                });
        }
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
    const int r8 = lane & 7;
    const int grp = cw / C::kWPG, wi = cw % C::kWPG;  // this warp's group, rank in the group
    const int hw = (CG > 1) ? 0 : grp;                 // its head within the block
    const int cbase = (CG > 1) ? grp * 16 : 0;         // its first column of the head's group
    const int g = g0 + hw;

    // q as the B operand of S^T = K Q^T.  Column n of n-tile t is virtual head
    // c = 8t + n of this KV head's group: a query head, or a (head, query) pair
    // when several queries share the cache (q rows are [head][query]).
    uint32_t qb[NT][D / 16][2];
    uint32_t q_lane = 0;  // kQSmem: this lane's ldmatrix row address (k-step 0)
    if constexpr (C::kQSmem) {
        // all groups' columns, [column][d] bf16 pairs; padding columns are zero
        uint8_t* qs = smem + C::kQOff;
        const uint32_t* q32 = static_cast<const uint32_t*>(p.q);
        for (int idx = threadIdx.x - 32; idx < 16 * CG * (D / 2); idx += C::kWarps * 32) {
            const int c = idx / (D / 2), w = idx - c * (D / 2);
            const size_t qi = (static_cast<size_t>(b) * p.Hq + g0 * p.G + c) * (D / 2) + w;
            const uint32_t v = (c < p.G && in_bounds(2 * qi + 1, p.q_elems, p.err)) ? q32[qi] : 0u;
            *reinterpret_cast<uint32_t*>(qs + c * C::kQRowBytes + 4 * w) = v;
        }
        consumer_sync(C::kWarps * 32);
        // matrices of an x4 load: (n-tile 0, k 0..7), (0, 8..15), (1, 0..7), (1, 8..15)
        q_lane = smem_u32(qs) + (cbase + 8 * (lane >> 4) + r8) * C::kQRowBytes + 16 * ((lane >> 3) & 1);
    }
#pragma unroll
    for (int nt = 0; nt < NT && !C::kQSmem; ++nt) {
        const int c = cbase + nt * 8 + gid;
        const int hq = g * p.G + (c < p.G ? c : 0);
        const bool hv = c < p.G && in_bounds((static_cast<size_t>(b) * p.Hq + hq + 1) * D - 1, p.q_elems, p.err);
        const __nv_bfloat16* qh =
            static_cast<const __nv_bfloat16*>(p.q) + (static_cast<size_t>(b) * p.Hq + hq) * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qb[nt][kk][0] = hv ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 2 * tig) : 0u;
            qb[nt][kk][1] = hv ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 8 + 2 * tig) : 0u;
        }
    }
    // Causal limits of this thread's columns (query i of nq sees tokens < N - nq + 1 + i);
    // masking applies only to blocks reaching past N - nq + 1.
    const int causal_from = p.causal ? N - p.nq + 1 : 0x7fffffff;
    // (recomputed where used: only blocks that reach the causal edge need them)
    auto lim = [&](int nt, int j) { return causal_from + (cbase + nt * 8 + 2 * tig + j) % p.nq; };

    // Running state for columns (2*tig, 2*tig+1) of each n-tile: maxima (log2
    // units, equal in all lanes of a column), per-lane partial denominators,
    // O^T fragments.
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

    // ldmatrix row addresses (swizzled 16-byte chunk = chunk ^ (row & 7)).  A
    // stage holds tile/R boxes of [head][half][R rows][128 B] (R = box_rows >=
    // 16), so each 16-token slab of a head (r0 .. r0 + 15) sits in one box.
    const int R = p.box_rows;
    const uint32_t half_bytes = R * 128;
    auto slab_base = [&](int r0) -> uint32_t {
        return (r0 / R) * (HB * C::kHalves * half_bytes) + hw * (C::kHalves * half_bytes) + (r0 % R) * 128;
    };
    const uint32_t k_lane = (r8 + 8 * ((lane >> 3) & 1)) * 128;
    const int k_chi = lane >> 4;
    const uint32_t v_lane = (r8 + 8 * (lane >> 4)) * 128;
    const int v_chi = (lane >> 3) & 1;
    uint32_t sbase[C::kSub];  // this warp's slab offsets within a stage (fixed for the whole loop)
#pragma unroll
    for (int sub = 0; sub < C::kSub; ++sub) sbase[sub] = slab_base((sub * C::kWPG + wi) * 16);
    const float sl2 = p.scale_log2;
    constexpr int J = (C::kSub >= 2) ? 2 : 1;  // slabs taken together
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
        // A warp's slabs of the stage are taken J at a time as one block of
        // 16 J tokens: the J score products are independent chains, and the
        // block maximum, the rescale and the denominator update happen once.
#pragma unroll
        for (int sp = 0; sp < C::kSub; sp += J) {
            int blk0[J], nvalid[J];  // first token, valid tokens of each slab
            uint32_t k_row[J], v_row[J];
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int r0 = ((sp + j) * C::kWPG + wi) * 16;  // this warp's slab of the stage
                blk0[j] = meta[s].tok0 + r0;
                nvalid[j] = tile_valid - r0;
                k_row[j] = sbase[sp + j] + k_lane;
                v_row[j] = sbase[sp + j] + v_lane;
            }

            if (nvalid[0] > 0) {  // later slabs of the block hold later tokens
                // S^T = K_blk Q^T, two accumulators per slab and n-tile to
                // shorten the chains (one with four slabs a stage, where the
                // registers are short: measured slower with two).
                constexpr int kAcc = (C::kSub <= 2) ? 2 : 1;
                float sacc[kAcc][J][NT][4];
#pragma unroll
                for (int u = 0; u < kAcc; ++u)
#pragma unroll
                    for (int j = 0; j < J; ++j)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) sacc[u][j][nt][e] = 0.f;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int c = 2 * (kk & 3) + k_chi;
                    uint32_t qf[4];  // kQSmem: B fragments of both n-tiles for this k-step
                    if constexpr (C::kQSmem) ldsm_x4(qf, q_lane + 32 * kk);
#pragma unroll
                    for (int j = 0; j < J; ++j) {
                        uint32_t a[4];
                        ldsm_x4(a, kbase + (kk >> 2) * half_bytes + k_row[j] + ((c ^ r8) << 4));
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            if constexpr (C::kQSmem)
                                mma_bf16(sacc[(kAcc == 2) ? (kk & 1) : 0][j][nt], a, qf[2 * nt], qf[2 * nt + 1]);
                            else
                                mma_bf16(sacc[(kAcc == 2) ? (kk & 1) : 0][j][nt], a, qb[nt][kk][0], qb[nt][kk][1]);
                        }
                    }
                }
                uint32_t bh[J][NT][2], bl[J][NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float sc[J][4];
                    float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
                    for (int j = 0; j < J; ++j) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            sc[j][e] = ((kAcc == 2) ? sacc[0][j][nt][e] + sacc[kAcc - 1][j][nt][e]
                                                    : sacc[0][j][nt][e]) * sl2;
                        if (nvalid[j] < 16) {
                            if (gid >= nvalid[j]) sc[j][0] = sc[j][1] = -INFINITY;
                            if (gid + 8 >= nvalid[j]) sc[j][2] = sc[j][3] = -INFINITY;
                        }
                        if (blk0[j] + 16 > causal_from) {
                            const int ta = blk0[j] + gid, tb = ta + 8;
                            const int l0 = lim(nt, 0), l1 = lim(nt, 1);
                            if (ta >= l0) sc[j][0] = -INFINITY;
                            if (ta >= l1) sc[j][1] = -INFINITY;
                            if (tb >= l0) sc[j][2] = -INFINITY;
                            if (tb >= l1) sc[j][3] = -INFINITY;
                        }
                        bm0 = fmaxf(bm0, fmaxf(sc[j][0], sc[j][2]));
                        bm1 = fmaxf(bm1, fmaxf(sc[j][1], sc[j][3]));
                    }
                    // block maximum per column over its 16 J tokens (lanes differing in gid)
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
                        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
                    }
                    const float mn0 = fmaxf(m[nt][0], bm0), mn1 = fmaxf(m[nt][1], bm1);
                    const float ms0 = (mn0 == -INFINITY) ? 0.f : mn0;
                    const float ms1 = (mn1 == -INFINITY) ? 0.f : mn1;
                    const float al0 = ex2(m[nt][0] - ms0), al1 = ex2(m[nt][1] - ms1);
                    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
                    for (int j = 0; j < J; ++j) {
                        const float p0 = ex2(sc[j][0] - ms0), p1 = ex2(sc[j][1] - ms1);
                        const float p2 = ex2(sc[j][2] - ms0), p3 = ex2(sc[j][3] - ms1);
                        ps0 += p0 + p2;
                        ps1 += p1 + p3;
                        // P^T as B fragments (k = token, n = column), BF16 hi + lo parts.
                        const __nv_bfloat162 h01 = __floats2bfloat162_rn(p0, p1);
                        const __nv_bfloat162 h23 = __floats2bfloat162_rn(p2, p3);
                        const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
                        const __nv_bfloat162 e01 = __floats2bfloat162_rn(p0 - f01.x, p1 - f01.y);
                        const __nv_bfloat162 e23 = __floats2bfloat162_rn(p2 - f23.x, p3 - f23.y);
                        bh[j][nt][0] = movtrans(bf16x2_bits(h01));
                        bh[j][nt][1] = movtrans(bf16x2_bits(h23));
                        bl[j][nt][0] = movtrans(bf16x2_bits(e01));
                        bl[j][nt][1] = movtrans(bf16x2_bits(e23));
                    }
                    l[nt][0] = l[nt][0] * al0 + ps0;
                    l[nt][1] = l[nt][1] * al1 + ps1;
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
                }
#pragma unroll
                for (int j = 0; j < J; ++j) {
                    // V rows past the slice may hold anything (even NaN): zero them.
                    uint32_t vm01 = 0xffffffffu, vm23 = 0xffffffffu;
                    if (nvalid[j] < 16) {
                        const int ta = 2 * tig, tb = 8 + 2 * tig;
                        vm01 = (ta < nvalid[j] ? 0x0000ffffu : 0u) | (ta + 1 < nvalid[j] ? 0xffff0000u : 0u);
                        vm23 = (tb < nvalid[j] ? 0x0000ffffu : 0u) | (tb + 1 < nvalid[j] ? 0xffff0000u : 0u);
                    }
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        const int c = 2 * (mt & 3) + v_chi;
                        uint32_t a[4];
                        ldsm_x4_t(a, vbase + (mt >> 2) * half_bytes + v_row[j] + ((c ^ r8) << 4));
                        a[0] &= vm01;
                        a[1] &= vm01;
                        a[2] &= vm23;
                        a[3] &= vm23;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma_bf16(oacc[nt][mt], a, bh[j][nt][0], bh[j][nt][1]);
                            mma_bf16(oacc[nt][mt], a, bl[j][nt][0], bl[j][nt][1]);
                        }
                    }
                }
            }
        }  // slabs
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (timed_out) atomicOr(abort_flag, 1);

    // ------------------------------------------- merge the warps' states
    constexpr int kCols = 8 * NT;  // columns per warp state
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], off);
            l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], off);
        }
    consumer_sync(C::kWarps * 32);  // every warp is done reading the stages
    constexpr int MS = C::kMergeStride;
    float* mo = mg_o + cw * kCols * MS;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int c0 = nt * 8 + 2 * tig;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            mo[c0 * MS + 16 * mt + gid] = oacc[nt][mt][0];
            mo[(c0 + 1) * MS + 16 * mt + gid] = oacc[nt][mt][1];
            mo[c0 * MS + 16 * mt + gid + 8] = oacc[nt][mt][2];
            mo[(c0 + 1) * MS + 16 * mt + gid + 8] = oacc[nt][mt][3];
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
    // states of the warps of one group, merged per (group, column, channel);
    // lh = the column's query head within the block's g0 * G ..
    const int cpg = (CG > 1) ? 16 : p.G;  // columns per group
    for (int idx = ct; idx < C::kGroups * cpg * D; idx += C::kWarps * 32) {
        int hh = 0, rem = idx;
        if constexpr (C::kGroups > 1) {
            hh = idx / (cpg * D);
            rem = idx - hh * (cpg * D);
        }
        const int h = rem / D, dd = rem - h * D;
        const int lh = (CG > 1) ? hh * 16 + h : hh * p.G + h;
        if (CG > 1 && lh >= p.G) continue;  // padding columns of the last group
        const int w0 = hh * C::kWPG;
        float mw[C::kWPG];
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::kWPG; ++w) {
            mw[w] = mg_m[(w0 + w) * kCols + h];
            M = fmaxf(M, mw[w]);
        }
        const float Ms = (M == -INFINITY) ? 0.f : M;
        float ow[C::kWPG], lw[C::kWPG];
#pragma unroll
        for (int w = 0; w < C::kWPG; ++w) {
            const float wt = ex2(mw[w] - Ms);
            ow[w] = wt * mg_o[((w0 + w) * kCols + h) * MS + dd];
            lw[w] = wt * mg_l[(w0 + w) * kCols + h];
        }
        // pairwise tree over the warps
        const float o = tree_sum<C::kWPG>(ow);
        const float lsum = tree_sum<C::kWPG>(lw);
        if (p.cluster) {  // kept for the cluster row merge
            const float nan = __int_as_float(0x7fc00000);
            cs_o[lh * D + dd] = poison ? nan : o;
            if (dd == 0) {
                cs_m[lh] = poison ? nan : M;
                cs_l[lh] = poison ? nan : lsum;
            }
        } else {
            emit_state(p, b, g0 * p.G + lh, split, D, dd, o, lsum, M, poison);
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

template <int D, int NT, int HB, int CG = 1>
cudaError_t launch_impl(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                        cudaStream_t stream) {
    using C = MmaCfg<D, HB, CG>;
    static std::atomic<unsigned long long> configured{0};
    cudaError_t e = set_smem_once(split_kv_mma_kernel<D, NT, HB, CG>, C::kSmem, configured);
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
    return cudaLaunchKernelEx(&cfg, split_kv_mma_kernel<D, NT, HB, CG>, tk, tv, p);
}

}  // namespace

int mma_cluster_capacity(int cluster_size) {
    using C = MmaCfg<128, 1>;
    static std::atomic<unsigned long long> configured{0};
    if (set_smem_once(split_kv_mma_kernel<128, 1, 1, 1>, C::kSmem, configured) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster_size, 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = static_cast<unsigned>(cluster_size);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, split_kv_mma_kernel<128, 1, 1, 1>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// Several KV heads per block only at head_dim 128 (small pages).
Geometry mma_geometry(int head_dim, int heads_per_block) {
    const int hb = (head_dim == 128 && heads_per_block == 2) ? 2 : 1;
    return Geometry{MmaCfg<128, 1>::kRows / hb, 64, 1, 1, hb};
}

cudaError_t launch_split_mma(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv,
                             const SplitParams& p, cudaStream_t stream) {
    // one n-tile of 8 columns per KV head group, two for up to 16; beyond, 2 or
    // 4 column groups of 16 (head_dim 128, one KV head per block)
    if (p.G > 16) {
        if (head_dim != 128 || p.hb != 1 || p.G > 64) return cudaErrorInvalidValue;
        return p.G > 32 ? launch_impl<128, 2, 1, 4>(tk, tv, p, stream) : launch_impl<128, 2, 1, 2>(tk, tv, p, stream);
    }
    const bool two = p.G > 8;
    if (p.hb == 2 && head_dim == 128)
        return two ? launch_impl<128, 2, 2>(tk, tv, p, stream) : launch_impl<128, 1, 2>(tk, tv, p, stream);
    if (p.hb != 1) return cudaErrorInvalidValue;
    switch (head_dim) {
        case 64:
            return two ? launch_impl<64, 2, 1>(tk, tv, p, stream) : launch_impl<64, 1, 1>(tk, tv, p, stream);
        case 128:
            return two ? launch_impl<128, 2, 1>(tk, tv, p, stream) : launch_impl<128, 1, 1>(tk, tv, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ta
