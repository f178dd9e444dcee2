// Split-KV partial attention over an FP8 (E4M3) KV cache with one scale per
// KV head, on the fifth-generation tensor cores (tcgen05), for KV heads
// shared by up to 32 columns (query heads of a group, or (head, query) pairs
// when several queries share the cache; the automatic choice above 16).  BF16
// q, head_dim 128.
//
// One thread block per (slice p, KV head g, batch row b) computes the partial
// state (o, l, m) of its slice for every column of the group ("Local
// Independent Partial Attention" on the Tree Attention pages) and writes it
// for the row merge ("The Tree Reduction Merge Operator").  Per stage of 128
// tokens:
//
//   S^T [128 tokens x 2 NC]  = K8 . [Q1 | Q2]^T     tcgen05.mma kind::f8f6f4, FP32 in TMEM
//   logits = S1 + S2 / 16                            (q = Q1 + Q2 / 16 in E4M3, exact)
//   P^T = 2^(logits - m_c)                           softmax warps, one token each
//   O^T [128 channels x 64] += V16^T . [P_hi | P_lo]^T   tcgen05.mma kind::f16 (FP16), FP32 in TMEM
//
// (NC = the group's columns rounded up to 16 or 32.)  K is used as the copy
// left it: the E4M3 x E4M3 product needs no widening, and q, scaled by a power
// of two into [2^7, 2^8), is two E4M3 terms -- the first rounds q to 4
// significant bits, the second holds the rest times 16, which fits 4 bits
// again, so BF16 q is represented exactly wherever both terms are normal.
// The weights need 16-bit precision, so V is widened to FP16 (exact) in
// shared memory and P is FP16, scaled by 2^6 and split into hi + lo parts.
//
//  warp 0       copies: K and V tiles of 128 tokens x 128 B (E4M3, 128-byte
//               swizzle), HBM -> shared memory by TMA, 5-stage ring
//  warp 1       allocates TMEM (two S^T buffers, O^T accumulators) and issues
//               the O^T products from one thread; each releases its stage
//  warp 2       issues the S^T products from one thread
//  warps 3-6    widen V in place: one token row each, E4M3 -> FP16, written
//               over the stage once its S^T product is done -- channel half
//               0 over the K tile (no longer needed), half 1 over the
//               thread's own V row (already in its registers)
//  warps 7-     softmax: one token of the stage and CPT columns per thread,
//               with lazily moved per-column reference maxima as in the BF16
//               tcgen05 kernel; P^T goes into one of three 16 KB buffers
//
// Operands in shared memory (128-byte swizzle, 1024-byte atoms of 8 rows):
//   K8   [128 tokens][128 B]          A of S^T, K-major (as TMA left it)
//   Q8   [2 terms][NC rows][128 B]    B of S^T, K-major
//   V16  [half][128 tokens][128 B]    A of O^T, MN-major (the whole stage)
//   P^T  [128 tokens][128 B]          B of O^T, MN-major: N = 64 columns,
//                                     hi at [0, NC), lo at [NC, 2 NC)
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "sched.cuh"
#include "tc05.cuh"

namespace ta {
namespace {

template <int NCP, int CPT>
struct Tc05F8Cfg {
    static_assert(NCP == 16 || NCP == 32, "columns per MMA");
    static_assert(CPT == 8 || CPT == 16, "columns per softmax thread");
    static constexpr int D = 128;
    static constexpr int kTile = 128;                   // tokens per stage
    static constexpr int kStages = 5;
    static constexpr int kK8Bytes = kTile * 128;        // K (or V) of a stage: [128 tokens][128 B]
    static constexpr int kStageBytes = 2 * kK8Bytes;
    static constexpr int kPBytes = kTile * 128;         // [128 tokens][64 FP16 columns]
    static constexpr int kPBufs = 3;
    static constexpr int kPOff = kStages * kStageBytes;
    static constexpr int kQOff = kPOff + kPBufs * kPBytes;
    static constexpr int kQBytes = 2 * NCP * 128;       // [2 terms][NCP rows][128 B]
    static constexpr int kCtlOff = kQOff + kQBytes;
    static constexpr int kCtlBytes = 512;
    // m_ref, m_fin, alpha, shift [64]; per-warp partials [4][64]; causal column masks [4][16]
    static constexpr int kRedOff = kCtlOff + kCtlBytes;
    static constexpr int kRedBytes = (4 * 64 + 4 * 64 + 64 + 4) * 4;
    static constexpr int kSmem = 1024 + kRedOff + kRedBytes;
    static_assert(kSmem <= 227 * 1024, "shared memory per block");
    static_assert(kSmem > 114 * 1024, "one block per SM: the block's TMEM allocation never waits");
    static constexpr int kWidenWarps = 4;
    static constexpr int kWiden0 = 3;                   // first widening warp
    static constexpr int kSoftmaxWarps = 4 * NCP / CPT;
    static constexpr int kSoftmax0 = kWiden0 + kWidenWarps;  // first softmax warp
    static constexpr int kThreads = 32 * (kSoftmax0 + kSoftmaxWarps);
    static constexpr uint32_t kColS = 2 * NCP;          // S^T buffer x at columns x * 2 NCP: [term 1 | term 2]
    // O^T in kOAcc accumulators of 64 columns ([hi | lo] in the first 2 NCP),
    // so that consecutive products do not wait on one another: accumulator
    // 2 (j % 2) + h takes the token half h of event j's product.
    static constexpr int kOAcc = 4;
    static constexpr uint32_t kColO = 4 * NCP;
    static constexpr uint32_t kTmemCols = kColO + 64 * kOAcc <= 256 ? 256 : 512;
    static constexpr float kRescaleLog2 = 8.f;          // lazy-rescale margin (log2 units)
    static constexpr float kPScale = 64.f;              // P' = 2^6 P: up to 2^14, FP16-safe
    static constexpr int kMergeBatch = 20;
};

// Two E4M3 codes of (lo, hi), round to nearest, saturating: lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two E4M3 codes (low byte first) -> two FP16 values (exact), low half first.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t pair16) {
    uint32_t r;
    const uint16_t x = static_cast<uint16_t>(pair16);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(x));
    return r;
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t pair16) {
    const uint32_t h = e4m3x2_to_f16x2(pair16);
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

template <int NCP, int CPT>
__global__ void __launch_bounds__(Tc05F8Cfg<NCP, CPT>::kThreads, 1)
    split_kv_tc05_fp8_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                             const SplitParams p) {
    using C = Tc05F8Cfg<NCP, CPT>;
    constexpr int D = C::D;
    constexpr int kS = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = smem;
    uint8_t* pbuf = smem + C::kPOff;
    uint8_t* qs = smem + C::kQOff;
    uint8_t* ctl = smem + C::kCtlOff;
    uint64_t* full = reinterpret_cast<uint64_t*>(ctl);             // [kS] copies landed
    uint64_t* empty = full + kS;                                    // [kS] the stage's O^T product done
    volatile StageMeta* meta = reinterpret_cast<volatile StageMeta*>(empty + kS);
    int* abort_flag = const_cast<int*>(reinterpret_cast<volatile int*>(meta + kS));
    int* last_flag = abort_flag + 1;
    volatile unsigned* claim_sink = reinterpret_cast<volatile unsigned*>(abort_flag + 2);
    volatile int* bad_page = reinterpret_cast<volatile int*>(abort_flag + 3);
    uint64_t* prod_done = reinterpret_cast<uint64_t*>(abort_flag + 4);  // the copy warp's last claim is made
    uint64_t* k_done = prod_done + 1;                               // [kS] the stage's S^T product done
    uint64_t* v_full = k_done + kS;                                 // [kS] the stage's V widened in place
    uint64_t* s_full = v_full + kS;                                 // [2] S^T of an event computed
    uint64_t* s_free = s_full + 2;                                  // [2] S^T read by the softmax warps
    uint64_t* p_full = s_full + 4;                                  // [3] P^T of an event written
    // o_done[j % 4]: event j's O^T product done.  The softmax warps wait on it
    // for an event at most three behind theirs, and a barrier can only move on
    // past that event once they have written P^T of an event four later.
    uint64_t* o_done = s_full + 7;                                  // [4]
    uint64_t* tmem_free = s_full + 11;                              // softmax warps are done with TMEM
    uint64_t* final_bar = s_full + 12;                              // every MMA has completed
    uint64_t* q_full = s_full + 13;                                 // Q8 is in shared memory
    volatile int* smeta = reinterpret_cast<volatile int*>(s_full + 14);  // [2][4]: tok0, nvalid
    uint32_t* tmem_slot = const_cast<uint32_t*>(reinterpret_cast<volatile uint32_t*>(smeta + 8));
    int* ev_total = reinterpret_cast<int*>(tmem_slot + 1);         // events of the block (-1 until known)
    // [8] each event's stage and the parity of that stage's use, until its O^T
    // product is issued (at most kS events are outstanding: a stage is reused
    // only after its product)
    volatile int* ev_stage = ev_total + 1;
    volatile int* ev_par = ev_stage + 8;
    static_assert(3 * kS * 8 + 16 + 8 + 2 * kS * 8 + 14 * 8 + 32 + 8 + 64 <= C::kCtlBytes, "control block");
    float* m_ref = reinterpret_cast<float*>(smem + C::kRedOff);    // [64] reference maxima (log2 units)
    float* m_fin = m_ref + 64;                                      // [64] m_ref, 0 where it is -inf
    float* alpha_s = m_fin + 64;                                    // [64] scale of a moved reference
    float* shift_s = alpha_s + 64;                                  // [64] offset change of a moved reference
    float* wred = shift_s + 64;                                     // [4][64] per-warp partials
    uint32_t* cmask = reinterpret_cast<uint32_t*>(wred + 4 * 64);   // [slice][depth] causal column masks
    int* fail_rec = reinterpret_cast<int*>(cmask + 64);             // a softmax warp's wait failed

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int row = b * p.Hkv + g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&k_done[s], 1);
            mbar_init(&v_full[s], C::kWidenWarps);
        }
        mbar_init(prod_done, 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 2);  // the issuer's release of the event, and the MMA commit
            mbar_init(&s_free[x], C::kSoftmaxWarps);
        }
        for (int x = 0; x < 4; ++x) mbar_init(&o_done[x], 1);
        for (int x = 0; x < C::kPBufs; ++x) mbar_init(&p_full[x], C::kSoftmaxWarps);
        mbar_init(tmem_free, C::kSoftmaxWarps);
        mbar_init(final_bar, 2);  // both issuing threads' MMAs have completed
        mbar_init(q_full, C::kSoftmaxWarps);
        *ev_total = -1;
        *abort_flag = 0;
        *bad_page = 0;
        fence_barrier_init();
    }
    if (2 * NCP < 64) {  // P^T columns past [hi | lo] take part in the product: keep them zero
        for (int i = threadIdx.x; i < C::kPBufs * C::kPBytes / 16; i += blockDim.x)
            reinterpret_cast<uint4*>(pbuf)[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
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
                tma_prefetch_4d(&tmK, 0, y, g, b);
                tma_prefetch_4d(&tmV, 0, y, g, b);
                return;
            }
            const int ty = (y + j * p.box_rows) & page_mask;
            tma_prefetch_4d(&tmK, 0, ty, g, page);
            tma_prefetch_4d(&tmV, 0, ty, g, page);
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
            produce_row<kS>(p, b, row, n_raw, n_hint, split, C::kTile, full, empty, meta, claim_sink, bad_page,
                            C::kStageBytes, [&](int s, int y, int j, int page) {
                                uint8_t* st = stages + s * C::kStageBytes;
                                if (!paged) {
                                    tma_load_4d(st, &tmK, 0, y, g, b, &full[s], pol);
                                    tma_load_4d(st + C::kK8Bytes, &tmV, 0, y, g, b, &full[s], pol);
                                    return;
                                }
                                // box j: tokens [j R, j R + R) of the stage
                                const int off = j * R * 128;
                                if (!in_bounds(static_cast<size_t>(off) + R * 128 - 1, C::kK8Bytes, p.err)) return;
                                const int ty = (y + j * R) & page_mask;
                                tma_load_4d(st + off, &tmK, 0, ty, g, page, &full[s], pol);
                                tma_load_4d(st + C::kK8Bytes + off, &tmV, 0, ty, g, page, &full[s], pol);
                            });
        }
        if (lane == 0) mbar_arrive(prod_done);  // after its last claim (lane 0 makes them)
        allow_dependents();
        return;
    }

    // ---------------------------------------------------------- MMA issuers
    // Lane 0 of warp 2 issues the S^T products, lane 0 of warp 1 the O^T
    // products: one thread issuing both would keep either waiting while it
    // issues the other.  Descriptors are those of the buffers' first bytes plus
    // the byte offset / 16 (start-address field; no carry, as every shared
    // address is below 256 KB).
    if (warp == 2) {
        if (lane == 0) {
            bool ok = wait_or_abort(q_full, 0, p.err, abort_flag);
            constexpr uint32_t id_s = idesc_e4m3(128, 2 * NCP, 0, 0);  // S^T = K8 Q8^T: both K-major
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
                if (nv == 0) {  // a discarded speculative stage: its barriers still move one phase
                    mbar_arrive(&k_done[s]);
                    mbar_arrive(&empty[s]);
                    continue;
                }
                // S^T buffer j1 % 2 is free once the softmax warps have read event j1 - 2
                const int x = j1 & 1;
                if (j1 >= 2 && !wait_or_abort(&s_free[x], ((j1 >> 1) - 1) & 1, p.err, abort_flag)) {
                    ok = false;
                    break;
                }
                if (nv < 0) {  // the count for the O^T issuer, the end-of-work event for the softmax warps
                    st_release_smem(ev_total, j1);
                    smeta[4 * x + 1] = -1;
                    mbar_arrive(&s_full[x]);
                    mbar_arrive(&s_full[x]);
                    break;
                }
                tc_fence_after();
                smeta[4 * x + 0] = meta[s].tok0;
                smeta[4 * x + 1] = nv;
                ev_stage[j1 & 7] = s;  // read by the O^T issuer once P^T of event j1 is written
                ev_par[j1 & 7] = (it / kS) & 1;
                mbar_arrive(&s_full[x]);
                const uint64_t dk = dk0 + static_cast<uint64_t>((s * C::kStageBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk)  // 32 channels (32 B) per K step
                    umma_e4m3(tmem + C::kColS * x, dk + 2 * kk, dq + 2 * kk, id_s, kk > 0 ? 1u : 0u);
                umma_commit(&s_full[x]);
                umma_commit(&k_done[s]);
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
            constexpr uint32_t id_o = idesc_f16(128, 64, 1, 1);  // O^T += V16^T P^T: both MN-major
            const uint64_t dst0 = smem_desc_sw128(smem_u32(stages), C::kTile * 128, 1024);
            const uint64_t dp0 = smem_desc_sw128(smem_u32(pbuf), C::kTile * 128, 1024);
            // Event by event: P^T of event j2 written (or, at the end of work, the
            // softmax warps' last arrival, after which the event count is known),
            // then the event's stage widened
            for (int j2 = 0;; ++j2) {
                if (!wait_or_abort(&p_full[j2 % C::kPBufs], (j2 / C::kPBufs) & 1, p.err, abort_flag)) {
                    ok = false;
                    break;
                }
                const int n_ev = ld_acquire_smem(ev_total);
                if (n_ev >= 0 && j2 >= n_ev) break;
                const int s = ev_stage[j2 & 7];
                if (!wait_or_abort(&v_full[s], static_cast<unsigned>(ev_par[j2 & 7]), p.err, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t dp = dp0 + static_cast<uint64_t>(((j2 % C::kPBufs) * C::kPBytes) >> 4);
                const uint64_t dv = dst0 + static_cast<uint64_t>((s * C::kStageBytes) >> 4);
#pragma unroll
                for (int i = 0; i < C::kTile / 16; ++i) {
                    // 16 tokens: two groups of 8 rows; V16's channel halves are 16 KB
                    // apart.  The two token halves alternate between two accumulators.
                    const int h = i & 1, kk = 4 * h + (i >> 1);
                    const uint32_t acc = C::kColO + 64 * (2 * (j2 & 1) + h);
                    umma_f16(tmem + acc, dv + 128 * kk, dp + 128 * kk, id_o, (j2 >= 2 || (kk & 3) > 0) ? 1u : 0u);
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

    // ---------------------------------------------------------- widening
    // Thread tw widens token row tw of each stage's V in place: 16-byte chunk c
    // of the E4M3 row (channels 16c .. 16c + 15) becomes chunks 2 (c % 4) and
    // 2 (c % 4) + 1 of channel half c / 4 in FP16; half 0 goes over the K tile
    // (free once the stage's S^T product is done), half 1 over the thread's own
    // E4M3 row, read beforehand.  Rows past the stage's valid tokens may hold
    // anything (even NaN) and are written as zeros.
    if (warp < C::kSoftmax0) {
        const int tw = threadIdx.x - 32 * C::kWiden0;  // 0 .. 127
        const uint32_t sw = static_cast<uint32_t>(tw & 7);
        bool ok = true;
        for (int it = 0;; ++it) {
            const int s = it % kS;
            const unsigned par = (it / kS) & 1;
            if (!warp_wait(&full[s], par, p.err, abort_flag)) {
                ok = false;
                break;
            }
            const int nv = meta[s].nvalid;
            if (nv < 0) break;
            if (nv == 0) {  // a discarded speculative stage: no event, but v_full[s] moves one phase
                __syncwarp();
                if (lane == 0) mbar_arrive(&v_full[s]);
                continue;
            }
            uint8_t* st = stages + s * C::kStageBytes;
            const bool row_ok = tw < nv;
            uint4 raw[8];
            if (row_ok) {
                const uint8_t* v8 = st + C::kK8Bytes + tw * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) raw[c] = *reinterpret_cast<const uint4*>(v8 + ((c ^ sw) << 4));
            }
            if (!warp_wait(&k_done[s], par, p.err, abort_flag)) {
                ok = false;
                break;
            }
            uint8_t* vd = st + tw * 128;
            if (row_ok) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 w = raw[c];
                    const uint4 lo4 = make_uint4(e4m3x2_to_f16x2(w.x), e4m3x2_to_f16x2(w.x >> 16),
                                                 e4m3x2_to_f16x2(w.y), e4m3x2_to_f16x2(w.y >> 16));
                    const uint4 hi4 = make_uint4(e4m3x2_to_f16x2(w.z), e4m3x2_to_f16x2(w.z >> 16),
                                                 e4m3x2_to_f16x2(w.w), e4m3x2_to_f16x2(w.w >> 16));
                    uint8_t* half_row = vd + (c >> 2) * C::kK8Bytes;
                    const uint32_t c0 = 2 * (c & 3);
                    *reinterpret_cast<uint4*>(half_row + ((c0 ^ sw) << 4)) = lo4;
                    *reinterpret_cast<uint4*>(half_row + (((c0 + 1) ^ sw) << 4)) = hi4;
                }
            } else {
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    *reinterpret_cast<uint4*>(vd + (c >> 3) * C::kK8Bytes + (c & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&v_full[s]);
        }
        if (!ok && lane == 0) atomicOr(abort_flag, 1);
        allow_dependents();
        return;
    }

    // ---------------------------------------------------------- softmax
    // Softmax warp sw (of SW) reads TMEM lane quarter `quarter` = warp % 4 and
    // owns the CPT columns [CPT cs, CPT cs + CPT), cs = sw / 4: its thread t =
    // 32 quarter + lane handles token t of each stage and, at the end,
    // channel t of O^T for those columns.
    constexpr int SW = C::kSoftmaxWarps;
    constexpr int NT = 32 * SW;  // softmax threads
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const int ct = threadIdx.x - 32 * C::kSoftmax0;  // 0 .. NT - 1
    const int cs = (warp - C::kSoftmax0) >> 2;       // column slice
    const int c_base = CPT * cs;
    const int t = 32 * quarter + lane;
    const int G = p.G;

    // q: the group's columns (rows past G are zero) as BF16, scaled by the power
    // of two that brings max|q| into [2^7, 2^8), written as two E4M3 terms: Q1 =
    // rn(q'), Q2 = rn(16 (q' - Q1)).  Each 16-byte chunk of q (8 channels) fills
    // 8 bytes of a term's 128-byte row.
    const float ks = p.k_scale[g];
    const float vsc = p.v_scale[g] / C::kPScale;
    const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q) +
                              (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(g) * G) * D;
    float amax = 0.f;
    for (int idx = ct; idx < NCP * 16; idx += NT) {
        const int rr = idx >> 4, ch = idx & 15;
        if (rr < G && in_bounds((static_cast<size_t>(b) * p.Hq + static_cast<size_t>(g) * G + rr) * D + 8 * ch + 7,
                                p.q_elems, p.err)) {
            const uint4 v = *reinterpret_cast<const uint4*>(qg + rr * D + 8 * ch);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[e] << 16)), fabsf(__uint_as_float(w[e] & 0xffff0000u))));
        }
    }
    amax = warp_max(amax);
    if (lane == 0) wred[warp - C::kSoftmax0] = amax;
    consumer_sync(NT);
#pragma unroll 1
    for (int i = 0; i < SW; ++i) amax = fmaxf(amax, wred[i]);
    int qexp = 0;
    if (amax > 0.f) {
        int e;
        frexpf(amax, &e);  // amax = f 2^e, f in [0.5, 1)
        qexp = max(-100, min(100, 8 - e));
    }
    const float qsc = ldexpf(1.f, qexp);
    for (int idx = ct; idx < NCP * 16; idx += NT) {
        const int rr = idx >> 4, ch = idx & 15;
        uint32_t t1[2] = {0u, 0u}, t2[2] = {0u, 0u};
        if (rr < G && in_bounds((static_cast<size_t>(b) * p.Hq + static_cast<size_t>(g) * G + rr) * D + 8 * ch + 7,
                                p.q_elems, p.err)) {
            const uint4 v = *reinterpret_cast<const uint4*>(qg + rr * D + 8 * ch);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float a = __uint_as_float(w[e] << 16) * qsc, c = __uint_as_float(w[e] & 0xffff0000u) * qsc;
                const uint32_t p1 = e4m3x2(a, c);
                const float2 r1 = e4m3x2_to_float2(p1);
                const uint32_t p2 = e4m3x2((a - r1.x) * 16.f, (c - r1.y) * 16.f);
                t1[e >> 1] |= p1 << (16 * (e & 1));
                t2[e >> 1] |= p2 << (16 * (e & 1));
            }
        }
        const int off = (ch & 1) * 8;  // 8 channels = half of a 16-byte chunk
        const uint32_t o1 = rr * 128 + ((((ch >> 1) ^ (rr & 7))) << 4) + off;
        const uint32_t o2 = (NCP + rr) * 128 + ((((ch >> 1) ^ (rr & 7))) << 4) + off;
        if (in_bounds(o2 + 7, C::kQBytes, p.err)) {
            *reinterpret_cast<uint2*>(qs + o1) = make_uint2(t1[0], t1[1]);
            *reinterpret_cast<uint2*>(qs + o2) = make_uint2(t2[0], t2[1]);
        }
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
    consumer_sync(NT);  // m_ref, m_fin and cmask initialised
    // bit i of gmask: column c_base + i exists in the group
    const uint32_t gmask = G >= c_base + CPT ? ((1u << CPT) - 1u) : (G <= c_base ? 0u : (1u << (G - c_base)) - 1u);
    const uint32_t* cm = cmask + 16 * cs;
    uint32_t mneg = gmask;  // bit i: column c_base + i has no reference yet (m_ref = -inf)

    int N = n_raw;
    const bool bad = (N < 0) || (N > p.S);
    if (bad) {
        if (ct == 0) atomicOr(p.err, kErrBadSeqlen);
        N = 0;
    }
    const int causal_from = p.causal ? N - p.nq + 1 : 0x7fffffff;
    const float sl2 = p.scale_log2 * ks / qsc;
    float lp[CPT];  // this thread's partial denominators of its columns, relative to m_ref
#pragma unroll
    for (int i = 0; i < CPT; ++i) lp[i] = 0.f;
    // Every exit from this loop is decided together by the softmax warps after
    // the stage's barrier reduction (see the BF16 tcgen05 kernel).
    bool failed = false;
    int j = 0;
    for (;; ++j) {
        const int x = j & 1;
        const bool ok = warp_wait(&s_full[x], (j >> 1) & 1, p.err, abort_flag);
        int tok0 = 0, nv = -1;
        if (ok) {
            tok0 = smeta[4 * x + 0];
            nv = smeta[4 * x + 1];
        } else if (lane == 0) {
            *fail_rec = 1;
        }
        float xs[CPT];       // this token's logits of the warp's columns, then their offsets from the references
        uint32_t vmask = 0;  // bit i: column c_base + i counts this token
        bool over = !ok;
        const bool tok_ok = t < nv;
        if (ok && nv >= 0) {
            float s2[CPT];
            tc_fence_after();
            tmem_ld_cols<CPT>(tmem + lane_base + C::kColS * x + c_base, xs);
            tmem_ld_cols<CPT>(tmem + lane_base + C::kColS * x + NCP + c_base, s2);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[x]);
#pragma unroll
            for (int i = 0; i < CPT; i += 2) fma2(xs[i], xs[i + 1], s2[i], s2[i + 1], 0.0625f, 0.0625f, xs[i], xs[i + 1]);

            vmask = tok_ok ? gmask : 0u;
            const int d = tok0 + t - causal_from + 1;  // <= 0 before the diagonal (and without causality)
            if (d > 0) vmask &= cm[min(d, 15)];
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
            // columns that do not count this token get -inf (exponential 0); with 16
            // columns a thread, a stage whose tokens all count in every column (the
            // usual one) skips this (with 8 the warp vote measured slower than the selects)
            constexpr uint32_t kAll = CPT == 32 ? 0xffffffffu : (1u << CPT) - 1u;
            if (CPT < 16 || !__all_sync(0xffffffffu, vmask == kAll)) {
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
            // a last arrival wakes the O^T issuer (after event j - 3's product, as for any event)
            if (j >= C::kPBufs)
                failed = !warp_wait(&o_done[(j - C::kPBufs) & 3], ((j - C::kPBufs) >> 2) & 1, p.err, abort_flag);
            if (lane == 0 && !failed) mbar_arrive(&p_full[j % C::kPBufs]);
            break;
        }
        bool rescale_o = false;
        if (any_over) {
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
                const float base = m_fin[c];
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
            rescale_o = resc && j > 0;
        }
        // P^T buffer j % 3 was last read by event j - 3's product
        if (j >= C::kPBufs && !failed)
            failed = !warp_wait(&o_done[(j - C::kPBufs) & 3], ((j - C::kPBufs) >> 2) & 1, p.err, abort_flag);
        if (!failed) {
            // P^T row t: element n of [hi | lo] at 16-byte chunk n / 8 (swizzled)
            uint8_t* pb = pbuf + (j % C::kPBufs) * C::kPBytes + t * 128;
#pragma unroll
            for (int k = 0; k < CPT / 8; ++k) {
                float pv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) pv[e] = ex2(xs[8 * k + e]);
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    add2(lp[8 * k + 2 * e], lp[8 * k + 2 * e + 1], lp[8 * k + 2 * e], lp[8 * k + 2 * e + 1],
                         pv[2 * e], pv[2 * e + 1]);
                    float a, c;
                    mul2(a, c, pv[2 * e], pv[2 * e + 1], C::kPScale, C::kPScale);
                    hw[e] = pack_f16(a, c);
                    const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hw[e]));
                    float l0, l1;
                    sub2(l0, l1, a, c, hf.x, hf.y);
                    lw[e] = pack_f16(l0, l1);
                }
                const int nh = c_base + 8 * k, nl = NCP + c_base + 8 * k;
                const uint32_t oh = ((nh / 8) ^ (t & 7)) << 4, ol = ((nl / 8) ^ (t & 7)) << 4;
                *reinterpret_cast<uint4*>(pb + oh) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(pb + ol) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
        }
        if (rescale_o && !failed) {
            // every earlier O^T product must be complete before O^T is rescaled
            failed = !warp_wait(&o_done[(j - 1) & 3], ((j - 1) >> 2) & 1, p.err, abort_flag);
            if (!failed) {
                tc_fence_after();
#pragma unroll 1
                for (int k = 0; k < 2 * C::kOAcc; ++k) {  // hi and lo of every accumulator
                    float ov[CPT];
                    const uint32_t col = C::kColO + 64 * (k >> 1) + (k & 1) * NCP + c_base;
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
        if (lane == 0 && !failed) mbar_arrive(&p_full[j % C::kPBufs]);
        if (lane == 0 && failed) *fail_rec = 1;  // the next stage's reduction ends the loop
    }
    if (failed && lane == 0) atomicOr(abort_flag, 1);  // the other roles stop waiting too

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
#pragma unroll
        for (int i = 0; i < CPT; ++i) o[i] = 0.f;
        // the accumulators of odd events exist once there were two events
#pragma unroll 1
        for (int k = 0; k < 2 * (j > 1 ? C::kOAcc : C::kOAcc / 2); ++k) {
            float part[CPT];
            tmem_ld_cols<CPT>(tmem + lane_base + C::kColO + 64 * (k >> 1) + (k & 1) * NCP + c_base, part);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < CPT; ++i) o[i] += part[i];
        }
#pragma unroll
        for (int i = 0; i < CPT; ++i) o[i] *= vsc;
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
cudaError_t launch_fp8_ncp(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                           cudaStream_t stream) {
    using C = Tc05F8Cfg<NCP, CPT>;
    static std::atomic<unsigned long long> configured{0};
    cudaError_t e = set_smem_once(split_kv_tc05_fp8_kernel<NCP, CPT>, C::kSmem, configured);
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
    return cudaLaunchKernelEx(&cfg, split_kv_tc05_fp8_kernel<NCP, CPT>, tk, tv, p);
}

}  // namespace

// 128-token stages of 128-byte E4M3 rows; pages of fewer than 128 tokens
// take one box each.
Geometry tc05_fp8_geometry() {
    constexpr int kTile = Tc05F8Cfg<16, 8>::kTile;
    return Geometry{kTile, 128, 1, 0, 1};
}

cudaError_t launch_split_tc05_fp8(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                                  cudaStream_t stream) {
    constexpr int kTile = Tc05F8Cfg<16, 8>::kTile;
    if (p.G < 1 || p.G > 32 || p.hb != 1 || p.cluster || p.box_rows < 16 || p.box_rows > kTile ||
        !p.k_scale || !p.v_scale)
        return cudaErrorInvalidValue;
    if (p.block_table == nullptr && p.box_rows != kTile) return cudaErrorInvalidValue;
    return p.G <= 16 ? launch_fp8_ncp<16, 8>(tk, tv, p, stream) : launch_fp8_ncp<32, 16>(tk, tv, p, stream);
}

}  // namespace ta
