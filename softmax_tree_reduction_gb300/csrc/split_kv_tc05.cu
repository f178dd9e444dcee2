// Split-KV partial attention on the fifth-generation tensor cores (tcgen05),
// for KV heads shared by many columns: BF16 q and cache, head_dim 128, up to
// 64 columns per KV head (query heads of a GQA or MQA group, or (head, query)
// pairs when several queries share the cache).
//
// One thread block per (slice p, KV head g, batch row b) computes the partial
// state (o, l, m) of its slice for every column of the group ("Local
// Independent Partial Attention" on the Tree Attention pages) and writes it
// for the row merge ("The Tree Reduction Merge Operator").  Both products put
// 128 rows in the M dimension, so they run at the tensor cores' full rate:
//
//   S^T [128 tokens x NC columns]     = K . Q^T          tcgen05.mma, FP32 in TMEM
//   P^T = 2^(S^T scale log2e - m_c)                        softmax warps, one token each
//   O^T [128 channels x 2 NC] += V^T . [P_hi | P_lo]^T   tcgen05.mma, FP32 in TMEM
//
// (NC = the group's columns rounded up to 32 or 64.)  P's BF16 hi and lo
// parts are two halves of the second product's N dimension, so one MMA per K
// step carries both, and O = O_hi + O_lo at the end.
//
//  warp 0     copies: K and V tiles of 128 tokens, [half][128 tokens][128 B]
//             (128-byte swizzle), HBM -> shared memory by TMA, 3-stage ring
//  warp 1     allocates TMEM (two S^T buffers, O^T) and issues the O^T
//             products from one thread
//  warp 2     issues the S^T products from one thread; each MMA group is
//             committed to an mbarrier
//  warps 3-   softmax: 4 warps per 16 columns (8 up to 32 columns in the
//             group, 16 up to 64), one token of the stage and 16 of its
//             columns per thread:
//             exponentials against one reference maximum per column, shared
//             by all threads in shared memory.  The reference moves only when a column's
//             logits exceed it by more than 2^8 (one barrier reduction per
//             stage tells), and then O^T in TMEM is rescaled.  Each thread
//             keeps per-column partial denominators, summed once at the end;
//             P^T goes into the stage's K half (free once S^T is computed).
//
// Operands in shared memory (128-byte swizzle, 1024-byte atoms of 8 rows):
//   K    [half][128 tokens][128 B]    A of S^T, K-major (as TMA left it)
//   Q    [half][64 rows][128 B]       B of S^T, K-major
//   V    [half][128 tokens][128 B]    A of O^T, MN-major (as TMA left it)
//   P^T  [block][128 tokens][128 B]   B of O^T, MN-major: N = [hi | lo] columns,
//                                     64 per block
// Paged caches with pages of fewer than 128 tokens land each page's two
// channel halves with one copy each, so a stage has the same layout.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "sched.cuh"
#include "tc05.cuh"

namespace ta {
namespace {

template <int NCP, int CPT>
struct Tc05Cfg {
    static_assert(NCP == 32 || NCP == 64, "columns per MMA");
    static_assert(CPT == 16 || CPT == 32, "columns per softmax thread");
    static constexpr int D = 128;
    static constexpr int kTile = 128;                   // tokens per stage (M of S^T)
    static constexpr int kStages = 3;
    static constexpr int kKBytes = 2 * kTile * 128;     // K (or V) of a stage: [half][tile][128 B]
    static constexpr int kStageBytes = 2 * kKBytes;
    static constexpr int kPBlocks = 2 * NCP / 64;       // 64-column blocks of [hi | lo]
    static_assert(kPBlocks * kTile * 128 <= kKBytes, "P^T fits the stage's K half");
    static constexpr int kQOff = kStages * kStageBytes;
    static constexpr int kQBytes = 2 * 64 * 128;
    static constexpr int kCtlOff = kQOff + kQBytes;
    static constexpr int kCtlBytes = 384;
    // m_ref, m_fin, alpha, shift [64]; per-warp partials [4][64]; causal column masks [4][16]
    static constexpr int kRedOff = kCtlOff + kCtlBytes;
    static constexpr int kRedBytes = (4 * 64 + 4 * 64 + 64 + 4) * 4;
    static constexpr int kSmem = 1024 + kRedOff + kRedBytes;
    static_assert(kSmem <= 227 * 1024, "shared memory per block");
    static_assert(kSmem > 114 * 1024, "one block per SM: the block's TMEM allocation never waits");
    static constexpr int kSoftmaxWarps = 4 * NCP / CPT;  // a thread takes CPT columns of one token
    static constexpr int kSoftmax0 = 3;                  // first softmax warp
    static constexpr int kThreads = 32 * (kSoftmax0 + kSoftmaxWarps);
    static constexpr uint32_t kColS = NCP;              // S^T buffer x at columns x * NCP (x = 0, 1)
    static constexpr uint32_t kColO = 2 * NCP;          // O^T: [hi | lo], 2 NCP columns
    static constexpr uint32_t kTmemCols = 4 * NCP;      // 128 or 256
    static constexpr float kRescaleLog2 = 8.f;          // lazy-rescale margin (log2 units)
    // the row merge's loads in flight per thread (4 registers each; fewer when
    // the block's threads leave about 100 registers each)
    static constexpr int kMergeBatch = kThreads > 400 ? 8 : 20;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

template <int NCP, int CPT>
__global__ void __launch_bounds__(Tc05Cfg<NCP, CPT>::kThreads, 1)
    split_kv_tc05_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const SplitParams p) {
    using C = Tc05Cfg<NCP, CPT>;
    constexpr int D = C::D;
    constexpr int kS = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = smem;
    uint8_t* qs = smem + C::kQOff;
    uint8_t* ctl = smem + C::kCtlOff;
    uint64_t* full = reinterpret_cast<uint64_t*>(ctl);            // [kS] copies landed
    uint64_t* empty = full + kS;                                   // [kS] stage released (after O^T += ...)
    volatile StageMeta* meta = reinterpret_cast<volatile StageMeta*>(empty + kS);
    int* abort_flag = const_cast<int*>(reinterpret_cast<volatile int*>(meta + kS));
    int* last_flag = abort_flag + 1;
    volatile unsigned* claim_sink = reinterpret_cast<volatile unsigned*>(abort_flag + 2);
    volatile int* bad_page = reinterpret_cast<volatile int*>(abort_flag + 3);
    uint64_t* prod_done = reinterpret_cast<uint64_t*>(abort_flag + 4);  // the copy warp's last claim is made
    uint64_t* s_full = prod_done + 1;                              // [2] S^T of an event computed
    uint64_t* s_free = s_full + 2;                                 // [2] S^T read by the softmax warps
    // p_full[j % 4]: P^T of event j written.  The O^T issuer has waited on the
    // same barrier for event j - 4 before the softmax warps arrive for event j:
    // event j's stage was last used by event j - 3 and released by its O^T
    // product, issued after event j - 4's.
    uint64_t* p_full = s_full + 4;                                 // [4]
    // o_done[j % 4]: event j's O^T product done.  The softmax warps wait on it
    // for the event just before theirs, and a barrier can only move on past
    // that event once they have written P^T of an event four later, so the
    // phase they wait for is never overtaken.
    uint64_t* o_done = s_full + 8;                                 // [4]
    uint64_t* tmem_free = s_full + 12;                             // softmax warps are done with TMEM
    uint64_t* final_bar = s_full + 13;                             // every MMA has completed
    uint64_t* q_full = s_full + 14;                                // Q is in shared memory
    volatile int* smeta = reinterpret_cast<volatile int*>(s_full + 15);  // [2][4]: tok0, nvalid, stage
    uint32_t* tmem_slot = const_cast<uint32_t*>(reinterpret_cast<volatile uint32_t*>(smeta + 8));
    int* ev_total = reinterpret_cast<int*>(tmem_slot + 1);  // events of the block (-1 until known)
    volatile int* ev_stage = ev_total + 1;  // [4] stage of each event whose O^T product is outstanding
    static_assert(3 * kS * 8 + 16 + 8 + 15 * 8 + 32 + 4 + 4 + 16 <= C::kCtlBytes, "control block");
    float* m_ref = reinterpret_cast<float*>(smem + C::kRedOff);   // [64] reference maxima (log2 units)
    float* m_fin = m_ref + 64;                                     // [64] m_ref, 0 where it is -inf
    float* alpha_s = m_fin + 64;                                   // [64] scale of a moved reference
    float* shift_s = alpha_s + 64;                                 // [64] offset change of a moved reference
    float* wred = shift_s + 64;                                    // [4][64] per-warp partials
    // cmask[slice][d]: bit i set iff column CPT slice + i of the group sees a
    // token d positions into the causal diagonal, i.e. (CPT slice + i) % nq >= d
    uint32_t* cmask = reinterpret_cast<uint32_t*>(wred + 4 * 64);
    int* fail_rec = reinterpret_cast<int*>(cmask + 64);            // a softmax warp's wait failed

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int row = b * p.Hkv + g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool split_halves = p.block_table != nullptr && p.box_rows < C::kTile;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(prod_done, 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 2);  // the issuer's release of the event, and the MMA commit
            mbar_init(&s_free[x], C::kSoftmaxWarps);
        }
        for (int x = 0; x < 4; ++x) {
            mbar_init(&p_full[x], C::kSoftmaxWarps);
            mbar_init(&o_done[x], 1);
        }
        mbar_init(tmem_free, C::kSoftmaxWarps);
        mbar_init(final_bar, 2);  // both issuing threads' MMAs have completed
        mbar_init(q_full, C::kSoftmaxWarps);
        *ev_total = -1;
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
            for (int hf = 0; hf < (split_halves ? 2 : 1); ++hf) {
                tma_prefetch_5d(&tmK, 0, ty, hf, g, page);
                tma_prefetch_5d(&tmV, 0, ty, hf, g, page);
            }
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
            const int R = p.box_rows;
            produce_row<kS>(
                p, b, row, n_raw, n_hint, split, C::kTile, full, empty, meta, claim_sink, bad_page,
                C::kStageBytes, [&](int s, int y, int j, int page) {
                    // every stage is [half][128 tokens][128 B] for K, then for V
                    uint8_t* st = stages + s * C::kStageBytes;
                    if (!paged) {
                        tma_load_5d(st, &tmK, 0, y, 0, g, b, &full[s], pol);
                        tma_load_5d(st + C::kKBytes, &tmV, 0, y, 0, g, b, &full[s], pol);
                        return;
                    }
                    const int ty = (y + j * R) & page_mask;
                    if (!in_bounds(static_cast<size_t>(j + 1) * R * 128 - 1, C::kTile * 128, p.err)) return;
                    if (!split_halves) {  // one box: both halves of the 128 tokens
                        tma_load_5d(st, &tmK, 0, ty, 0, g, page, &full[s], pol);
                        tma_load_5d(st + C::kKBytes, &tmV, 0, ty, 0, g, page, &full[s], pol);
                        return;
                    }
                    // box j: tokens [j R, j R + R) of one half per copy
                    for (int hf = 0; hf < 2; ++hf) {
                        const int off = hf * (C::kTile * 128) + j * R * 128;
                        tma_load_5d(st + off, &tmK, 0, ty, hf, g, page, &full[s], pol);
                        tma_load_5d(st + C::kKBytes + off, &tmV, 0, ty, hf, g, page, &full[s], pol);
                    }
                });
        }
        if (lane == 0) mbar_arrive(prod_done);  // after its last claim (lane 0 makes them)
        allow_dependents();
        return;
    }

    // ---------------------------------------------------------- MMA issuers
    // Lane 0 of warp 2 issues the S^T products, lane 0 of warp 1 the O^T
    // products: one thread issuing both would keep either waiting while it
    // issues the other.
    if (warp == 2) {
        if (lane == 0) {
            bool ok = wait_or_abort(q_full, 0, p.err, abort_flag);
            constexpr uint32_t id_s = idesc_bf16(128, NCP, 0, 0);  // S^T = K Q^T: both K-major
            // Descriptors of the buffers' first bytes; an operand's descriptor is its
            // buffer's plus the byte offset / 16 (start-address field; no carry, as
            // every shared address is below 256 KB).
            const uint64_t dq = smem_desc_sw128(smem_u32(qs), 16, 1024);
            const uint64_t dk0 = smem_desc_sw128(smem_u32(stages), 16, 1024);
            int j1 = 0;  // next event
            for (int it = 0; ok; ++it) {
                const int s = it % kS;
                if (!wait_or_abort(&full[s], (it / kS) & 1, p.err, abort_flag)) {
                    ok = false;
                    break;
                }
                const int nv = meta[s].nvalid;
                if (nv == 0) {  // a discarded speculative stage
                    mbar_arrive(&empty[s]);
                    continue;
                }
                // S^T buffer j1 % 2 is free once the softmax warps have read event j1 - 2
                const int x = j1 & 1;
                if (j1 >= 2 && !wait_or_abort(&s_free[x], ((j1 >> 1) - 1) & 1, p.err, abort_flag)) {
                    ok = false;
                    break;
                }
                if (nv < 0) {  // the end-of-work event for the softmax warps, the count for the O^T issuer
                    smeta[4 * x + 1] = -1;
                    mbar_arrive(&s_full[x]);
                    mbar_arrive(&s_full[x]);
                    st_release_smem(ev_total, j1);
                    break;
                }
                tc_fence_after();
                smeta[4 * x + 0] = meta[s].tok0;
                smeta[4 * x + 1] = nv;
                smeta[4 * x + 2] = s;
                ev_stage[j1 & 3] = s;  // read by the O^T issuer after P^T of event j1 is written
                mbar_arrive(&s_full[x]);
                const uint64_t dk = dk0 + static_cast<uint64_t>((s * C::kStageBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * (C::kTile * 128) + (kk & 3) * 32;
                    const uint32_t qoff = (kk >> 2) * 8192 + (kk & 3) * 32;
                    umma_f16(tmem + C::kColS * x, dk + (koff >> 4), dq + (qoff >> 4), id_s, kk > 0 ? 1u : 0u);
                }
                umma_commit(&s_full[x]);
                ++j1;
            }
            if (!ok) atomicOr(abort_flag, 1);
            umma_commit(final_bar);  // completes once its S^T products have
        }
        allow_dependents();
        return;
    }
    if (warp == 1) {
        if (lane == 0) {
            bool ok = true;
            constexpr uint32_t id_o = idesc_bf16(128, 2 * NCP, 1, 1);  // O^T += V^T P^T: both MN-major
            const uint64_t dst0 = smem_desc_sw128(smem_u32(stages), C::kTile * 128, 1024);
            // Event by event: P^T of event j2 written (or, at the end of work, the
            // softmax warps' last arrival, after which the event count is known)
            for (int j2 = 0;; ++j2) {
                if (!wait_or_abort(&p_full[j2 & 3], (j2 >> 2) & 1, p.err, abort_flag)) {
                    ok = false;
                    break;
                }
                const int n_ev = ld_acquire_smem(ev_total);
                if (n_ev >= 0 && j2 >= n_ev) break;
                tc_fence_after();
                const int s = ev_stage[j2 & 3];
                const uint64_t pd = dst0 + static_cast<uint64_t>((s * C::kStageBytes) >> 4);
                const uint64_t vd = pd + (C::kKBytes >> 4);
#pragma unroll
                for (int kk = 0; kk < C::kTile / 16; ++kk) {
                    // 16 tokens: two groups of 8 rows; V's channel halves and
                    // P^T's 64-column blocks are 16 KB apart
                    umma_f16(tmem + C::kColO, vd + 128 * kk, pd + 128 * kk, id_o, (j2 > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(&empty[s]);
                umma_commit(&o_done[j2 & 3]);
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
    // Softmax warp sw (of SW) reads TMEM lane quarter `quarter` = warp % 4 and
    // owns the CPT columns [CPT cs, CPT cs + CPT), cs = sw / 4: its thread t =
    // 32 quarter + lane handles token t of each stage and, at the end,
    // channel t of O^T for those columns.
    constexpr int SW = C::kSoftmaxWarps;
    constexpr int NT = 32 * SW;       // softmax threads
    constexpr int NS = NCP / CPT;     // column slices
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const int ct = threadIdx.x - 32 * C::kSoftmax0;  // 0 .. NT - 1
    const int cs = (warp - C::kSoftmax0) >> 2;       // column slice
    const int c_base = CPT * cs;
    const int t = 32 * quarter + lane;
    const int G = p.G;

    // Q rows (columns of the group; rows past G are zero), 16-byte chunks,
    // swizzled; reference maxima start empty
    {
        const uint4* q16 = static_cast<const uint4*>(p.q);
        for (int idx = ct; idx < 64 * 16; idx += NT) {
            const int rr = idx >> 4, ch = idx & 15;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            const size_t qi = (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(g) * G + rr) * 16 + ch;
            if (rr < G && in_bounds(8 * qi + 7, p.q_elems, p.err)) v = __ldg(q16 + qi);
            *reinterpret_cast<uint4*>(qs + (ch >> 3) * 8192 + rr * 128 + (((ch & 7) ^ (rr & 7)) << 4)) = v;
        }
        if (ct < 64) {
            m_ref[ct] = -INFINITY;
            m_fin[ct] = 0.f;
        }
        if (ct == 0) *fail_rec = 0;
        if (ct < 64) {  // cmask[slice][d] over slices of CPT columns, d < 16
            const int sl = ct >> 4, d = ct & 15;
            uint32_t m = 0;
            for (int i = 0; i < CPT; ++i) m |= static_cast<uint32_t>((CPT * sl + i) % p.nq >= d) << i;
            cmask[ct] = m;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_full);
    }
    consumer_sync(NT);  // m_ref, m_fin and cmask initialised
    // bit i of gmask: column c_base + i exists in the group
    const uint32_t gmask = G >= c_base + CPT ? (CPT == 32 ? 0xffffffffu : (1u << CPT) - 1u)
                                             : (G <= c_base ? 0u : (1u << (G - c_base)) - 1u);
    const uint32_t* cm = cmask + 16 * cs;
    uint32_t mneg = gmask;  // bit i: column c_base + i has no reference yet (m_ref = -inf)

    int N = n_raw;
    const bool bad = (N < 0) || (N > p.S);
    if (bad) {
        if (ct == 0) atomicOr(p.err, kErrBadSeqlen);
        N = 0;
    }
    // causal: query i of nq sees tokens < N - nq + 1 + i
    const int causal_from = p.causal ? N - p.nq + 1 : 0x7fffffff;
    const float sl2 = p.scale_log2;
    float lp[CPT];  // this thread's partial denominators of its columns, relative to m_ref
#pragma unroll
    for (int i = 0; i < CPT; ++i) lp[i] = 0.f;
    // Every exit from this loop is decided together by the softmax warps after
    // the stage's one barrier reduction (a warp leaving alone would strand the
    // others at the next named barrier): a warp whose wait failed records it in
    // shared memory before the reduction and votes, and all warps read the
    // record after it.
    bool failed = false;
    int j = 0;
    for (;; ++j) {
        const int x = j & 1;
        const bool ok = warp_wait(&s_full[x], (j >> 1) & 1, p.err, abort_flag);
        int tok0 = 0, nv = -1, s = 0;
        if (ok) {
            tok0 = smeta[4 * x + 0];
            nv = smeta[4 * x + 1];
            s = smeta[4 * x + 2];
        } else if (lane == 0) {
            *fail_rec = 1;
        }
        float xs[CPT];       // this token's logits of the warp's columns, then their offsets from the references
        uint32_t vmask = 0;  // bit i: column c_base + i counts this token
        bool over = !ok;
        const bool tok_ok = t < nv;
        if (ok && nv >= 0) {
            tc_fence_after();
            tmem_ld_cols<CPT>(tmem + lane_base + C::kColS * x + c_base, xs);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[x]);

            // column c counts this token iff c < G, t < nv and (causal) tok0 + t <
            // causal_from + c % nq, i.e. c % nq >= d for the token's depth d into the diagonal
            vmask = tok_ok ? gmask : 0u;
            const int d = tok0 + t - causal_from + 1;  // <= 0 before the diagonal (and without causality)
            if (d > 0) vmask &= cm[min(d, 15)];
            // offsets from the references (0 where there is none yet); a logit past
            // its reference by more than the margin, or a column's first logits,
            // move the reference (rare)
            float xm[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int i4 = 0; i4 < CPT / 4; ++i4) {
                const float4 m4 = *reinterpret_cast<const float4*>(m_fin + c_base + 4 * i4);
                const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
                float y[4];
                fma2(y[0], y[1], xs[4 * i4], xs[4 * i4 + 1], sl2, sl2, -mv[0], -mv[1]);
                fma2(y[2], y[3], xs[4 * i4 + 2], xs[4 * i4 + 3], sl2, sl2, -mv[2], -mv[3]);
#pragma unroll
                for (int e = 0; e < 4; ++e) xs[4 * i4 + e] = y[e];
            }
            // columns that do not count this token get -inf (exponential 0); a
            // stage whose tokens all count in every column (the usual one) skips this
            constexpr uint32_t kAll = CPT == 32 ? 0xffffffffu : (1u << CPT) - 1u;
            if (!__all_sync(0xffffffffu, vmask == kAll)) {
#pragma unroll
                for (int i = 0; i < CPT; ++i) xs[i] = ((vmask >> i) & 1) ? xs[i] : -INFINITY;
            }
#pragma unroll
            for (int i = 0; i < CPT; i += 2) xm[(i >> 1) & 1] = max3(xm[(i >> 1) & 1], xs[i], xs[i + 1]);
            over = (fmaxf(xm[0], xm[1]) > C::kRescaleLog2) || (vmask & mneg);
        }
        const bool any_over = softmax_any<NT>(over);  // the stage's barrier reduction
        if (*const_cast<volatile int*>(fail_rec)) {
            failed = true;
            break;
        }
        if (nv < 0) {  // every warp's wait succeeded and saw the same end-of-work event
            if (lane == 0) mbar_arrive(&p_full[j & 3]);  // a last arrival wakes the O^T issuer
            break;
        }
        bool rescale_o = false;  // O^T needs the moved references' scales (after P^T is written)
        if (any_over) {
            // new references: per column, the maximum over the stage's counted tokens
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                const float wm = warp_max(xs[i]);
                if (lane == 0) wred[quarter * 64 + c_base + i] = wm;
            }
            consumer_sync(NT);
            float alpha = 1.f;
            if (ct < NCP) {  // one thread per column decides its new reference
                const int c = ct;
                const float tx = fmaxf(fmaxf(wred[c], wred[64 + c]), fmaxf(wred[128 + c], wred[192 + c]));
                const float m_old = m_ref[c];
                const float base = m_fin[c];  // xs = logit - base
                float m_new = m_old;
                if (tx != -INFINITY && (m_old == -INFINITY || tx > C::kRescaleLog2)) m_new = tx + base;
                alpha = (m_old == -INFINITY || m_new == m_old) ? 1.f : ex2(m_old - m_new);
                alpha_s[c] = alpha;
                shift_s[c] = (m_new == -INFINITY) ? 0.f : base - m_new;
                m_ref[c] = m_new;
                m_fin[c] = (m_new == -INFINITY) ? 0.f : m_new;
            }
            const bool resc = softmax_any<NT>(alpha != 1.f);  // also publishes the new references
            mneg = 0;
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                lp[i] *= alpha_s[c_base + i];
                xs[i] += shift_s[c_base + i];
                mneg |= static_cast<uint32_t>(m_ref[c_base + i] == -INFINITY) << i;
            }
            mneg &= gmask;
            rescale_o = resc && j > 0;  // the same decision in every thread
        }
        // P^T row t of the B operand in the stage's K half: element n of
        // [hi | lo] at block n / 64, 16-byte chunk (n % 64) / 8 (swizzled)
        uint8_t* pb = stages + s * C::kStageBytes;
#pragma unroll
        for (int k = 0; k < CPT / 8; ++k) {  // hi columns c_base + 8k .. + 7, lo columns NCP + the same
            float pv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) pv[e] = ex2(xs[8 * k + e]);
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                add2(lp[8 * k + 2 * e], lp[8 * k + 2 * e + 1], lp[8 * k + 2 * e], lp[8 * k + 2 * e + 1], pv[2 * e],
                     pv[2 * e + 1]);
                hw[e] = pack_bf16(pv[2 * e], pv[2 * e + 1]);
                float l0, l1;
                sub2(l0, l1, pv[2 * e], pv[2 * e + 1], __uint_as_float(hw[e] << 16),
                     __uint_as_float(hw[e] & 0xffff0000u));
                lw[e] = pack_bf16(l0, l1);
            }
            const int nh = c_base + 8 * k, nl = NCP + c_base + 8 * k;
            const uint32_t oh = (nh / 64) * (C::kTile * 128) + t * 128 + ((((nh % 64) / 8) ^ (t & 7)) << 4);
            const uint32_t ol = (nl / 64) * (C::kTile * 128) + t * 128 + ((((nl % 64) / 8) ^ (t & 7)) << 4);
            if (in_bounds(oh + 15, C::kKBytes, p.err))
                *reinterpret_cast<uint4*>(pb + oh) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            if (in_bounds(ol + 15, C::kKBytes, p.err))
                *reinterpret_cast<uint4*>(pb + ol) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        // V rows past the stage's valid tokens may hold anything (even NaN): zero
        // them, the row's 16 chunks shared among the column slices
        if (!tok_ok) {
            uint4* vr = reinterpret_cast<uint4*>(pb + C::kKBytes + t * 128);
#pragma unroll
            for (int q = 0; q < 16 / NS; ++q) {
                const int ch = cs * (16 / NS) + q;  // chunk ch of the row: half ch / 8
                vr[(ch >> 3) * C::kTile * 8 + (ch & 7)] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if (rescale_o) {
            // every earlier O^T product must be complete before O^T is rescaled:
            // this warp's columns, hi and lo
            failed |= !warp_wait(&o_done[(j - 1) & 3], ((j - 1) >> 2) & 1, p.err, abort_flag);
            if (failed && lane == 0) *fail_rec = 1;  // the next stage's reduction ends the loop
            if (!failed) {
                tc_fence_after();
#pragma unroll 1
                for (int k = 0; k < 2; ++k) {
                    float ov[CPT];
                    const uint32_t col = C::kColO + k * NCP + c_base;
                    tmem_ld_cols<CPT>(tmem + lane_base + col, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < CPT; ++i) ov[i] *= alpha_s[c_base + i];
                    tmem_st_cols<CPT>(tmem + lane_base + col, ov);
                }
                tmem_wait_st();
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !failed) mbar_arrive(&p_full[j & 3]);
        if (lane == 0 && failed) *fail_rec = 1;
    }
    if (failed && lane == 0) atomicOr(abort_flag, 1);  // the issuer stops polling too

    // the block's state: the denominators summed over the threads, then O^T
    // (relative to m_ref) from TMEM once the last product is done
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const float ws = warp_sum(lp[i]);
        if (lane == 0) wred[quarter * 64 + c_base + i] = ws;
    }
    if (!failed && j > 0) failed = !warp_wait(&o_done[(j - 1) & 3], ((j - 1) >> 2) & 1, p.err, abort_flag);
    float o[CPT];  // channel t of the warp's columns
    if (!failed && j > 0) {
        tc_fence_after();
        float lo[CPT];
        tmem_ld_cols<CPT>(tmem + lane_base + C::kColO + c_base, o);
        tmem_ld_cols<CPT>(tmem + lane_base + C::kColO + NCP + c_base, lo);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < CPT; ++i) o[i] += lo[i];
    } else {
#pragma unroll
        for (int i = 0; i < CPT; ++i) o[i] = 0.f;
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tmem_free);
    const bool any_failed = softmax_any<NT>(failed);  // also publishes the partial sums

    const bool poison = bad || any_failed || (*const_cast<volatile int*>(abort_flag) != 0) || (*bad_page != 0);
    const float nan = __int_as_float(0x7fc00000);
    const size_t hrow0 = static_cast<size_t>(b) * p.Hq + static_cast<size_t>(g) * G;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int c = c_base + i;
        if (c >= G) break;
        const float L = (wred[c] + wred[64 + c]) + (wred[128 + c] + wred[192 + c]);
        const size_t hrow = hrow0 + c;
        if (p.P == 1) {
            if (in_bounds(hrow * D + t, p.out_elems, p.err))
                p.out[hrow * D + t] = poison ? nan : (L > 0.f ? o[i] / L : 0.f);
        } else if (in_bounds(hrow * p.P + split, p.part_rows, p.err)) {
            p.part_o[(hrow * p.P + split) * D + t] = poison ? nan : o[i];
        }
    }
    if (ct < G) {  // one thread per column: maximum and denominator
        const float L = (wred[ct] + wred[64 + ct]) + (wred[128 + ct] + wred[192 + ct]);
        const float m = m_ref[ct];
        const size_t hrow = hrow0 + ct;
        if (p.P == 1) {
            if (p.lse && in_bounds(hrow, p.rows, p.err))
                p.lse[hrow] = poison ? nan : (L > 0.f ? (m + log2f(L)) * kLn2 : -INFINITY);
        } else if (in_bounds(hrow * p.P + split, p.part_rows, p.err)) {
            const size_t pr = hrow * p.P + split;
            p.part_m[pr] = poison ? nan : (m == -INFINITY || L == 0.f ? -INFINITY : m * kLn2);
            p.part_l[pr] = poison ? nan : L;
        }
    }
    if (p.done)
        finish_row<D, C::kMergeBatch>(p, row, hrow0, G, reinterpret_cast<float*>(stages), last_flag, prod_done,
                                      ct, NT);
    allow_dependents();
}

template <int NCP, int CPT>
cudaError_t launch_ncp(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p, cudaStream_t stream) {
    using C = Tc05Cfg<NCP, CPT>;
    static std::atomic<unsigned long long> configured{0};
    cudaError_t e = set_smem_once(split_kv_tc05_kernel<NCP, CPT>, C::kSmem, configured);
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
    return cudaLaunchKernelEx(&cfg, split_kv_tc05_kernel<NCP, CPT>, tk, tv, p);
}

}  // namespace

// Pages of fewer than 128 tokens land each channel half with a copy of its own.
Geometry tc05_geometry(int page_size) {
    constexpr int kTile = Tc05Cfg<64, 16>::kTile;
    Geometry geo{kTile, 64, 1, 1, 1};
    geo.split_halves = (page_size > 0 && page_size < kTile) ? 1 : 0;
    return geo;
}

cudaError_t launch_split_tc05(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                              cudaStream_t stream) {
    constexpr int kTile = Tc05Cfg<64, 16>::kTile;
    if (p.G < 1 || p.G > 64 || p.hb != 1 || p.cluster || p.box_rows < 16 || p.box_rows > kTile)
        return cudaErrorInvalidValue;
    if (p.block_table == nullptr && p.box_rows != kTile) return cudaErrorInvalidValue;
    // up to 32 columns: 8 softmax warps of 16 columns (16 warps of 8 measured
    // slower: 92.2 vs 91.2 us on the 131072-token layer); up to 64: 16 warps of
    // 16 columns (8 warps of 32: 105.7 vs 104.0 us)
    return p.G <= 32 ? launch_ncp<32, 16>(tk, tv, p, stream) : launch_ncp<64, 16>(tk, tv, p, stream);
}

}  // namespace ta
