// Split-KV partial attention on the fifth-generation tensor cores (tcgen05),
// for KV heads shared by many columns: BF16 q and cache, head_dim 128, up to
// 64 columns per KV head (query heads of a GQA or MQA group, or (head, query)
// pairs when several queries share the cache).
//
// One thread block per (slice p, KV head g, batch row b) computes the partial
// state (o, l, m) of its slice for every column of the group ("Local
// Independent Partial Attention" on the Tree Attention pages) and writes it
// for the row merge ("The Tree Reduction Merge Operator").  The columns are
// the M dimension of both products, so each column's scores sit in one TMEM
// lane, read by a pair of softmax threads (half of the tokens each): its
// running maximum and denominator need one shuffle per stage:
//
//   S  [64 columns x 128 tokens]  = Q . K^T   tcgen05.mma, FP32 in TMEM
//   P  = 2^(S scale log2e - m)                 softmax warps, FP32
//   O  [64 columns x 128 channels] += P . V   tcgen05.mma, FP32 in TMEM,
//                                              P as BF16 hi + lo parts
//
//  warp 0     copies: K and V tiles of 128 tokens (128-byte swizzled halves
//             of 64 channels) HBM -> shared memory by TMA, 3-stage ring
//  warp 1     allocates 512 TMEM columns (two S buffers, O) and issues every
//             MMA from one thread; each MMA group is committed to an mbarrier
//  warps 2-5  softmax: read S from TMEM, online softmax with a lazy rescale
//             (the reference maximum moves only when a column's maximum grows
//             by more than 2^8, so O in TMEM is rarely touched), write P into
//             the stage's K half (free once S is computed) as the A operand
//             of the second product, and finally read O and emit the state.
//
// Operands in shared memory (128-byte swizzle, 1024-byte atoms of 8 rows):
//   Q   [half][64 rows][128 B]        A of S = Q K^T, K-major
//   K   [half][128 tokens][128 B]     B of S = Q K^T, K-major (as TMA left it)
//   P   [half][64 rows][128 B] x2     A of O += P V, K-major (hi, then lo)
//   V   [half][128 tokens][128 B]     B of O += P V, MN-major (as TMA left it)
// With a paged cache whose pages hold fewer than 128 tokens a stage is
// [page][half][R tokens][128 B]: S is computed per page (N = R) and each
// 16-token K step of P V addresses its page.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "sched.cuh"
#include "tc05.cuh"

namespace ta {
namespace {

struct Tc05Cfg {
    static constexpr int D = 128;
    static constexpr int kTile = 128;                   // tokens per stage
    static constexpr int kStages = 3;
    static constexpr int kKBytes = 2 * kTile * 128;     // K (or V) of a stage
    static constexpr int kStageBytes = 2 * kKBytes;
    static constexpr int kRows = 64;                    // M of both products (columns of the group)
    static constexpr int kQOff = kStages * kStageBytes;
    static constexpr int kQBytes = 2 * kRows * 128;
    static constexpr int kCtlOff = kQOff + kQBytes;
    static constexpr int kCtlBytes = 256;
    static constexpr int kSmem = 1024 + kCtlOff + kCtlBytes;
    static_assert(kSmem <= 227 * 1024, "shared memory per block");
    static_assert(kSmem > 114 * 1024, "one block per SM: the block's TMEM allocation never waits");
    static constexpr int kThreads = 192;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 128;              // S buffer x at columns x * 128 (x = 0, 1)
    static constexpr uint32_t kColO = 256;              // O
    static constexpr float kRescaleLog2 = 8.f;          // lazy-rescale margin (log2 units)
};

// Row r of an M = 64 accumulator is TMEM lane 32 (r / 16) + r % 16: the warp
// reading lane quarter q reaches rows 16 q .. 16 q + 15.

// Bounded wait that also gives up when another role of the block has aborted.
__device__ bool wait_or_abort(uint64_t* bar, unsigned parity, int* err, const volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
}

// Lane 0 waits, the warp follows (warp-uniform outcome).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, unsigned parity, int* err, const volatile int* abort_flag) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = wait_or_abort(bar, parity, err, abort_flag) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// Lane 0 waits until *count >= target (a counter published with release
// semantics by another warp of the block), the warp follows.
__device__ __forceinline__ bool warp_wait_count(int* count, int target, int* err, const volatile int* abort_flag) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0 && ld_acquire_smem(count) < target) {
        const unsigned long long t0 = globaltimer();
        while (ld_acquire_smem(count) < target) {
            if (*abort_flag || globaltimer() - t0 > kWaitLimitNs) {
                if (!*abort_flag) atomicOr(err, kErrTimeout);
                ok = 0;
                break;
            }
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(Tc05Cfg::kThreads, 1)
    split_kv_tc05_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const SplitParams p) {
    using C = Tc05Cfg;
    constexpr int D = C::D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = smem;
    uint8_t* qs = smem + C::kQOff;
    uint8_t* ctl = smem + C::kCtlOff;
    uint64_t* full = reinterpret_cast<uint64_t*>(ctl);           // [3] copies landed
    uint64_t* empty = full + C::kStages;                          // [3] stage released (after O += P V)
    volatile StageMeta* meta = reinterpret_cast<volatile StageMeta*>(ctl + 48);
    int* abort_flag = reinterpret_cast<int*>(ctl + 72);
    int* last_flag = abort_flag + 1;
    volatile unsigned* claim_sink = reinterpret_cast<volatile unsigned*>(abort_flag + 2);
    volatile int* bad_page = reinterpret_cast<volatile int*>(abort_flag + 3);
    uint64_t* prod_done = reinterpret_cast<uint64_t*>(ctl + 88);  // the copy warp's last claim is made
    uint64_t* s_full = reinterpret_cast<uint64_t*>(ctl + 96);     // [2] S of an event computed
    uint64_t* s_free = s_full + 2;                                // [2] S read by the softmax warps
    uint64_t* p_full = s_full + 4;                                // [2] P of an event written
    uint64_t* o_done = s_full + 6;                                // [2] O += P V of an event done
    uint64_t* tmem_free = s_full + 8;                             // softmax warps are done with TMEM
    uint64_t* final_bar = s_full + 9;                             // every MMA has completed
    uint64_t* q_full = s_full + 10;                               // Q is in shared memory
    volatile int* smeta = reinterpret_cast<volatile int*>(ctl + 192);  // [2][4]: tok0, nvalid, stage
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctl + 224);
    // Number of events whose O += P V has completed, published by the issuer
    // (it alone waits on o_done, in order); the softmax warps read it when they
    // must touch O, instead of waiting on a barrier phase that may have moved on.
    int* o_count = reinterpret_cast<int*>(ctl + 228);
    static_assert(228 + 4 <= C::kCtlBytes, "control block");

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int row = b * p.Hkv + g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(prod_done, 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 2);  // the issuer's release of the event, and the MMA commit
            mbar_init(&s_free[x], 4);
            mbar_init(&p_full[x], 4);
        }
        mbar_init(&o_done[0], 1);
        mbar_init(&o_done[1], 1);
        mbar_init(tmem_free, 4);
        mbar_init(final_bar, 1);
        mbar_init(q_full, 4);
        *o_count = 0;
        *abort_flag = 0;
        *bad_page = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
    if (threadIdx.x == 32) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    int n_hint = -1;  // row length read before the dependency wait (a hint)
    if (warp == 0) {
        const int page_mask = (1 << p.page_shift) - 1;
        n_hint = prefetch_row_head(p, b, split, C::kTile, p.prefetch_tiles, [&](int y, int j, int page) {
            if (!p.block_table) {
                tma_prefetch_5d(&tmK, 0, y, 0, g, b);
                tma_prefetch_5d(&tmV, 0, y, 0, g, b);
                return;
            }
            const int ty = (y + j * p.box_rows) & page_mask;
            tma_prefetch_5d(&tmK, 0, ty, 0, g, page);
            tma_prefetch_5d(&tmV, 0, ty, 0, g, page);
        });
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched as a programmatic dependent: apart from the address hints of
    // the prefetch, nothing an earlier kernel may write is read before this.
    wait_primary();
    const int n_raw = p.seqlens[b];  // validated by each side where it is used

    // ---------------------------------------------------------- copies
    if (warp == 0) {
        if (!p.stall) {  // diagnostic stall: publish nothing, so the waits give up
            const uint64_t pol = l2_policy_evict_first();
            const bool paged = p.block_table != nullptr;
            const int page_mask = (1 << p.page_shift) - 1;
            const int box_bytes = 2 * p.box_rows * 128;
            produce_row<C::kStages>(
                p, b, row, n_raw, n_hint, split, C::kTile, full, empty, meta, claim_sink, bad_page,
                C::kStageBytes, [&](int s, int y, int j, int page) {
                    // box j = box_rows tokens x both channel halves, [half][box_rows][128 B]
                    uint8_t* st = stages + s * C::kStageBytes;
                    const int off = j * box_bytes;
                    if (!paged) {
                        tma_load_5d(st + off, &tmK, 0, y, 0, g, b, &full[s], pol);
                        tma_load_5d(st + C::kKBytes + off, &tmV, 0, y, 0, g, b, &full[s], pol);
                        return;
                    }
                    const int ty = (y + j * p.box_rows) & page_mask;
                    tma_load_5d(st + off, &tmK, 0, ty, 0, g, page, &full[s], pol);
                    tma_load_5d(st + C::kKBytes + off, &tmV, 0, ty, 0, g, page, &full[s], pol);
                });
        }
        if (lane == 0) mbar_arrive(prod_done);  // after its last claim (lane 0 makes them)
        allow_dependents();
        return;
    }

    const int R = p.box_rows;        // tokens per box: 128, or the page size when smaller
    const int nbox = C::kTile / R;

    // ---------------------------------------------------------- MMA issuer
    if (warp == 1) {
        if (lane == 0) {
            bool ok = wait_or_abort(q_full, 0, p.err, abort_flag);
            const uint32_t id_s = idesc_bf16(64, R, 0, 0);    // S = Q K^T: both K-major
            const uint32_t id_o = idesc_bf16(64, 128, 0, 1);  // O += P V: V MN-major
            const uint32_t q_addr = smem_u32(qs), st_addr = smem_u32(stages);
            int it = 0;          // copy stage sequence
            int j1 = 0, j2 = 0;  // next event for S = Q K^T; next event for O += P V
            int o_seen = 0;      // events whose O += P V completion was observed and published
            int ev_stage[4];     // stage of each event whose O += P V is outstanding
            bool end = false;
            unsigned long long idle_since = 0;
            // Every barrier is polled without blocking, so that whichever becomes
            // ready first is served.  No barrier can run two phases ahead of its
            // poll: o_done[x] because at most two O += P V are in flight, p_full
            // because a softmax warp arrives on P of event j only after event j - 2's
            // O += P V has completed (o_count), s_full / s_free as the events alternate.
            while (ok) {
                bool progress = false;
                // publish completed O += P V, in order
                if (o_seen < j2 && mbar_test_wait(&o_done[o_seen & 1], (o_seen >> 1) & 1)) {
                    ++o_seen;
                    st_release_smem(o_count, o_seen);
                    progress = true;
                }
                // O += P V for the oldest event whose P is written
                if (j2 < j1 && o_seen >= j2 - 1 && mbar_test_wait(&p_full[j2 & 1], (j2 >> 1) & 1)) {
                    tc_fence_after();
                    const int s = ev_stage[j2 & 3];
                    const uint32_t kb = st_addr + s * C::kStageBytes, vb = kb + C::kKBytes;
#pragma unroll 1
                    for (int kk = 0; kk < C::kTile / 16; ++kk) {
                        const uint32_t aoff = (kk >> 2) * 8192 + (kk & 3) * 32;
                        const int t0 = 16 * kk;
                        const uint64_t vdesc =
                            smem_desc_sw128(vb + (t0 / R) * (256 * R) + (t0 % R) * 128, R * 128, 1024);
                        umma_bf16(tmem + C::kColO, smem_desc_sw128(kb + aoff, 16, 1024), vdesc, id_o,
                                  (j2 > 0 || kk > 0) ? 1u : 0u);
                        umma_bf16(tmem + C::kColO, smem_desc_sw128(kb + 16384 + aoff, 16, 1024), vdesc, id_o, 1u);
                    }
                    umma_commit(&empty[s]);
                    umma_commit(&o_done[j2 & 1]);
                    ++j2;
                    progress = true;
                }
                // S = Q K^T for the next stage once its copies landed and its S buffer is free
                if (!end && mbar_test_wait(&full[it % C::kStages], (it / C::kStages) & 1)) {
                    const int s = it % C::kStages;
                    const int nv = meta[s].nvalid;
                    if (nv < 0) {
                        end = true;
                        progress = true;
                    } else if (nv == 0) {  // a discarded speculative stage
                        mbar_arrive(&empty[s]);
                        ++it;
                        progress = true;
                    } else if (j1 < 2 || mbar_test_wait(&s_free[j1 & 1], ((j1 >> 1) - 1) & 1)) {
                        tc_fence_after();
                        const int x = j1 & 1;
                        smeta[4 * x + 0] = meta[s].tok0;
                        smeta[4 * x + 1] = nv;
                        smeta[4 * x + 2] = s;
                        mbar_arrive(&s_full[x]);
                        const uint32_t kb = st_addr + s * C::kStageBytes;
#pragma unroll 1
                        for (int bx = 0; bx < nbox; ++bx) {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint64_t qdesc =
                                    smem_desc_sw128(q_addr + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024);
                                const uint64_t kdesc = smem_desc_sw128(
                                    kb + bx * (256 * R) + (kk >> 2) * (R * 128) + (kk & 3) * 32, 16, 1024);
                                umma_bf16(tmem + C::kColS * x + bx * R, qdesc, kdesc, id_s, kk > 0 ? 1u : 0u);
                            }
                        }
                        umma_commit(&s_full[x]);
                        ev_stage[j1 & 3] = s;
                        ++j1;
                        ++it;
                        progress = true;
                    }
                }
                if (end && j2 == j1 && o_seen == j2) break;
                if (progress) {
                    idle_since = 0;
                } else if (idle_since == 0) {
                    idle_since = globaltimer();
                } else if (globaltimer() - idle_since > kWaitLimitNs) {
                    atomicOr(p.err, kErrTimeout);
                    ok = false;
                }
            }
            if (ok) {  // the end-of-work event for the softmax warps
                const int x = j1 & 1;
                if (j1 < 2 || wait_or_abort(&s_free[x], ((j1 >> 1) - 1) & 1, p.err, abort_flag)) {
                    smeta[4 * x + 1] = -1;
                    mbar_arrive(&s_full[x]);
                    mbar_arrive(&s_full[x]);
                } else {
                    ok = false;
                }
            }
            if (!ok) atomicOr(abort_flag, 1);
            // TMEM is freed only once no MMA is in flight and the softmax warps are done with it
            umma_commit(final_bar);
            mbar_wait(final_bar, 0, p.err);
            if (!mbar_wait(tmem_free, 0, p.err)) mbar_wait(tmem_free, 0, p.err);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
        allow_dependents();
        return;
    }

    // ---------------------------------------------------------- softmax
    // Row r = 16 quarter + (lane % 16) of S and O belongs to a pair of threads
    // of the warp reading lane quarter `quarter`: half h = lane / 16 takes the
    // row's tokens [64 h, 64 h + 64) of each stage and its channels
    // [64 h, 64 h + 64) of O (the TMEM loads split the row at column 64).
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const int ct = threadIdx.x - 64;              // 0..127
    const int r = 16 * quarter + (lane & 15);     // accumulator row = column of the group
    const int h = lane >> 4;
    const bool act = r < p.G;

    // Q rows (columns of the group; rows past G are zero), 16-byte chunks, swizzled
    {
        const uint4* q16 = static_cast<const uint4*>(p.q);
        for (int idx = ct; idx < C::kRows * 16; idx += 128) {
            const int rr = idx >> 4, ch = idx & 15;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (rr < p.G) v = __ldg(q16 + (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(g) * p.G + rr) * 16 + ch);
            *reinterpret_cast<uint4*>(qs + (ch >> 3) * 8192 + rr * 128 + (((ch & 7) ^ (rr & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_full);
    }

    int N = n_raw;
    const bool bad = (N < 0) || (N > p.S);
    if (bad) {
        if (ct == 0) atomicOr(p.err, kErrBadSeqlen);
        N = 0;
    }
    // causal: query i of nq sees tokens < N - nq + 1 + i
    const int lim = !act ? 0 : (p.causal ? N - p.nq + 1 + r % p.nq : 0x7fffffff);
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY;  // reference maximum (log2 units of the scaled logits), same in both halves
    float lsum = 0.f;         // this half's denominator relative to m_ref
    bool failed = false;
    int j = 0;
    for (;; ++j) {
        const int x = j & 1;
        if (!warp_wait(&s_full[x], (j >> 1) & 1, p.err, abort_flag)) {
            failed = true;
            break;
        }
        const int tok0 = smeta[4 * x + 0], nv = smeta[4 * x + 1], s = smeta[4 * x + 2];
        if (nv < 0) break;
        tc_fence_after();
        float sv[2][32];  // scores of tokens 64 h + 32 k + i
#pragma unroll
        for (int k = 0; k < 2; ++k) tmem_ld16x2_32(tmem + lane_base + C::kColS * x + 32 * k, sv[k]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[x]);

        // this half's valid tokens of the stage, relative to its first: [0, nvc)
        const int nvc = max(0, min(min(nv, lim - tok0) - 64 * h, 64));
        float tmax = -INFINITY;
        if (nvc == 64) {
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
                for (int i = 0; i < 32; ++i) tmax = fmaxf(tmax, sv[k][i]);
        } else {
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (32 * k + i < nvc) tmax = fmaxf(tmax, sv[k][i]);
        }
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
        const float tm = tmax * sl2;
        float alpha = 1.f;
        bool resc = false;
        if (tm != -INFINITY) {
            if (m_ref == -INFINITY) {
                m_ref = tm;
            } else if (tm > m_ref + C::kRescaleLog2) {
                alpha = ex2(m_ref - tm);
                m_ref = tm;
                lsum *= alpha;
                resc = true;
            }
        }
        if (__any_sync(0xffffffffu, resc)) {
            // O += P V of every earlier event must be complete before O is rescaled
            if (!warp_wait_count(o_count, j, p.err, abort_flag)) {
                failed = true;
                break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int k = 0; k < 2; ++k) {
                float ov[32];
                tmem_ld16x2_32(tmem + lane_base + C::kColO + 32 * k, ov);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) ov[i] *= alpha;
                tmem_st16x2_32(tmem + lane_base + C::kColO + 32 * k, ov);
            }
            tmem_wait_st();
        }
        // P = 2^(s sl2 - m_ref) into row r of the A operand (the stage's K half):
        // this half's 64 tokens are the K half h of the operand; hi parts, then
        // lo parts 16 KB further; masked tokens are 0
        uint8_t* pb = stages + s * C::kStageBytes;
        {
            const float ms = (m_ref == -INFINITY) ? 0.f : m_ref;
            float ps = 0.f;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                float pv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int t = 8 * ch + e;
                    pv[e] = (t < nvc) ? ex2(fmaf(sv[t >> 5][t & 31], sl2, -ms)) : 0.f;
                    ps += pv[e];
                }
                uint4 hi, lo;
                uint32_t* hw = reinterpret_cast<uint32_t*>(&hi);
                uint32_t* lw = reinterpret_cast<uint32_t*>(&lo);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    hw[e] = pack_bf16(pv[2 * e], pv[2 * e + 1]);
                    const float h0 = __uint_as_float(hw[e] << 16), h1 = __uint_as_float(hw[e] & 0xffff0000u);
                    lw[e] = pack_bf16(pv[2 * e] - h0, pv[2 * e + 1] - h1);
                }
                const uint32_t off = h * 8192 + r * 128 + ((ch ^ (r & 7)) << 4);
                *reinterpret_cast<uint4*>(pb + off) = hi;
                *reinterpret_cast<uint4*>(pb + 16384 + off) = lo;
            }
            lsum += ps;
        }
        // V rows past the stage's valid tokens may hold anything (even NaN): zero them
        if (nv < C::kTile) {
            uint8_t* vb = pb + C::kKBytes;
            for (int idx = ct; idx < (C::kTile - nv) * 16; idx += 128) {
                const int t = nv + (idx >> 4), ch = idx & 15;
                const int off = (t / R) * (256 * R) + (ch >> 3) * (R * 128) + (t % R) * 128 + (ch & 7) * 16;
                *reinterpret_cast<uint4*>(vb + off) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        // event j - 2's P must have been taken (its O += P V completed) before
        // p_full[x] gets event j's arrivals
        if (j >= 2 && !warp_wait_count(o_count, j - 1, p.err, abort_flag)) {
            failed = true;
            break;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[x]);
    }

    // the block's state: O (relative to m_ref) from TMEM once the last O += P V is done
    float o[2][32];  // channels 64 h + 32 k + i
    if (!failed && j > 0) failed = !warp_wait_count(o_count, j, p.err, abort_flag);
    if (!failed && j > 0) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 2; ++k) tmem_ld16x2_32(tmem + lane_base + C::kColO + 32 * k, o[k]);
        tmem_wait_ld();
    } else {
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int i = 0; i < 32; ++i) o[k][i] = 0.f;
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tmem_free);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);  // the row's denominator

    const bool poison = bad || failed || (*const_cast<volatile int*>(abort_flag) != 0) || (*bad_page != 0);
    if (act) {
        const size_t hrow = static_cast<size_t>(b) * p.Hq + static_cast<size_t>(g) * p.G + r;
        const float nan = __int_as_float(0x7fc00000);
        if (p.P == 1) {
            const float inv = (lsum > 0.f) ? 1.f / lsum : 0.f;
            float4* dst = reinterpret_cast<float4*>(p.out + hrow * D + 64 * h);
#pragma unroll
            for (int c4 = 0; c4 < 16; ++c4) {
                const int k = c4 >> 3, i = (c4 & 7) * 4;
                dst[c4] = poison ? make_float4(nan, nan, nan, nan)
                                 : make_float4(o[k][i] * inv, o[k][i + 1] * inv, o[k][i + 2] * inv, o[k][i + 3] * inv);
            }
            if (p.lse && h == 0) p.lse[hrow] = poison ? nan : (lsum > 0.f ? (m_ref + log2f(lsum)) * kLn2 : -INFINITY);
        } else {
            const size_t pr = hrow * p.P + split;
            float4* dst = reinterpret_cast<float4*>(p.part_o + pr * D + 64 * h);
#pragma unroll
            for (int c4 = 0; c4 < 16; ++c4) {
                const int k = c4 >> 3, i = (c4 & 7) * 4;
                dst[c4] = poison ? make_float4(nan, nan, nan, nan)
                                 : make_float4(o[k][i], o[k][i + 1], o[k][i + 2], o[k][i + 3]);
            }
            if (h == 0) {
                p.part_m[pr] = poison ? nan : (m_ref == -INFINITY || lsum == 0.f ? -INFINITY : m_ref * kLn2);
                p.part_l[pr] = poison ? nan : lsum;
            }
        }
    }
    if (p.done)
        finish_row<D>(p, row, static_cast<size_t>(b) * p.Hq + static_cast<size_t>(g) * p.G, p.G,
                      reinterpret_cast<float*>(stages), last_flag, prod_done, ct, 128);
    allow_dependents();
}

}  // namespace

cudaError_t launch_split_tc05(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                              cudaStream_t stream) {
    using C = Tc05Cfg;
    if (p.G < 1 || p.G > C::kRows || p.hb != 1 || p.cluster || p.box_rows < 16 || p.box_rows > C::kTile)
        return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> configured{0};
    cudaError_t e = set_smem_once(split_kv_tc05_kernel, C::kSmem, configured);
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
    return cudaLaunchKernelEx(&cfg, split_kv_tc05_kernel, tk, tv, p);
}

}  // namespace ta
