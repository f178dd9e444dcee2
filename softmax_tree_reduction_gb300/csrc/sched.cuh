// Work distribution inside a schedule row -- one batch row and the KV head
// (or the hb KV heads sharing each copy) its blocks serve -- and the row's
// final merge, shared by the split-KV kernels.
//
// Scheduling.  With run-time balancing (the default) each of a row's P blocks
// first streams a contiguous slice holding 7/8 of its fair share of the row
// (contiguous streaming keeps DRAM pages and translations local); the last
// eighth of the row is cut into chunks of `chunk_tiles` tiles that blocks
// claim from a per-row counter as they run dry, so blocks on SMs that receive
// more bandwidth stream more and a row's blocks finish together.  Each block
// ends with one partial state over the tokens it streamed; the merge operator
// is commutative, so this changes nothing in the result.  Without balancing
// (P == 1, or the deterministic flag) block p streams the contiguous slice
// [p*c, (p+1)*c), c = ceil(N/P) rounded up to a tile.
//
// The row merge: for up to 20 splits each thread merges one channel of one
// head from a single round trip of loads; beyond that the maxima and
// denominators are reduced per head in shared memory first.
//
// Counters start at zero.  Claims are atomicAdds issued up to two ahead, when
// the block has at most two chunks of work left in hand, so their latency
// hides behind streaming; a block stops at its first claim past the pool
// (later ones fail too: the counter only grows).  Every block then takes the
// row's ticket (an acquire-release atomicInc wrapping after P tickets); the
// block holding the last ticket -- when every claim of the row has been made
// -- resets the claim counter, so a completed call leaves both counters at
// zero.
//
// The producer lane publishes each stage's token range in shared memory
// before arming the stage's full barrier; consumers read it after the wait.
// A stage whose `nvalid` is negative marks the end of the block's work.
#pragma once

#include "common.cuh"

namespace ta {

struct StageMeta {
    int tok0;    // first token of the tile
    int nvalid;  // valid tokens in the tile (1..tile); < 0: no more tiles
};

// Box needs no page (past the row's end, or no tile).
constexpr int kNoPage = -2147483647 - 1;

// Block-table entry for box `j` of the tile at token t (paged caches), or
// kNoPage.  The load is only started here; the entry is checked when the tile
// is issued.
__device__ __forceinline__ int load_box_page(const SplitParams& p, int b, int N, int t, int tile,
                                             int j) {
    if (t < 0 || !p.block_table) return kNoPage;
    const int tj = t + j * p.box_rows;
    if (j >= tile / p.box_rows || tj >= N) return kNoPage;
    const size_t e = static_cast<size_t>(b) * p.max_pages + (tj >> p.page_shift);
    if (!in_bounds(e, p.bt_elems, p.err)) return kNoPage;
    return __ldg(p.block_table + e);
}

// The contiguous slice [*t, *t_end) that block `split` streams first, and the
// first token of the row's claimed pool (*base; N without balancing).
__device__ __forceinline__ void slice_bounds(const SplitParams& p, int N, int split, int tile, int* t,
                                             int* t_end, int* base) {
    const int P = p.P;
    long long slice;
    if (p.claim != nullptr) {
        const int C = tile * p.chunk_tiles;
        slice = (static_cast<long long>(N) * 7 / 8) / P / C * C;
    } else {
        slice = (static_cast<long long>(N) + P - 1) / P;
        slice = (slice + tile - 1) / tile * tile;
    }
    *t = static_cast<int>(min(static_cast<long long>(split) * slice, static_cast<long long>(N)));
    *t_end = static_cast<int>(min(static_cast<long long>(split + 1) * slice, static_cast<long long>(N)));
    *base = p.claim != nullptr
                ? static_cast<int>(min(static_cast<long long>(P) * slice, static_cast<long long>(N)))
                : N;
}

// Producer warp, before the block waits for the previous grid on the stream:
// prefetch the first `ntiles` tiles of the block's slice into L2 through
// `pf(t, j, page)` (box j of the tile at token t).  The previous grid may
// still be writing the lengths, block table or caches, so what is read here
// only picks addresses (clamped to the row and the pool); the data itself is
// loaded after the wait, from L2, which holds any newer writes.  This fills
// the time in which the previous grid's last blocks merge and DRAM is idle.
// Returns the row length it read (the hint), in [0, S].
template <typename Prefetch>
__device__ int prefetch_row_head(const SplitParams& p, int b, int split, int tile, int ntiles,
                                 Prefetch&& pf) {
    const int lane = threadIdx.x & 31;
    const int N = max(0, min(ld_relaxed(p.seqlens + b), p.S));
    int t, t_end, base;
    slice_bounds(p, N, split, tile, &t, &t_end, &base);
    const int nbox = p.block_table ? tile / p.box_rows : 1;
    if (lane >= nbox) return N;
    for (int i = 0; i < ntiles && t < t_end; ++i, t += tile) {
        int page = 0;
        if (p.block_table) {
            const int tj = t + lane * p.box_rows;
            if (tj >= N) break;
            const size_t e = static_cast<size_t>(b) * p.max_pages + (tj >> p.page_shift);
            if (!in_bounds(e, p.bt_elems, p.err)) break;
            page = ld_relaxed(p.block_table + e);
            if (page < 0 || page >= p.num_pages) break;
        }
        pf(t, lane, page);
    }
    return N;
}

// Producer warp (all 32 lanes): stream this block's tiles into the stage ring.
// Lane 0 keeps the schedule (slices, claims, barriers, stage descriptors);
// lane j issues the TMA copies of box j of each tile via `issue(s, t, j, page)`
// (page = physical page for paged caches, else unused) after lane 0 has armed
// the stage's full barrier with `stage_bytes`.  Tiles are generated one ahead
// so each lane's block-table entry loads while the previous tile is issued.
// Returns false if a wait timed out (the error word is set; the warp still
// drains).
//
// Dense caches: the first ring of tiles is issued from `N_hint` (the length
// read before the dependency wait, or -1) while the real length N is still
// in flight.  Those stages get their transaction bytes but not the arrive
// that completes them; once N is known they are released as they are (same
// tiles) or with nvalid = 0 (the consumers skip them), and the schedule
// continues after them.
template <int kStages, typename Issue>
__device__ bool produce_row(const SplitParams& p, int b, int row, const int& N_ref, int N_hint, int split,
                            int tile, uint64_t* full, uint64_t* empty, volatile StageMeta* meta,
                            volatile unsigned* sink, volatile int* bad_flag, unsigned stage_bytes,
                            Issue&& issue) {
    const int lane = threadIdx.x & 31;
    const int C = tile * p.chunk_tiles;  // tokens per claimed chunk
    const bool dynamic = p.claim != nullptr;
    const int nbox = p.block_table ? tile / p.box_rows : 1;
    int spec = 0, spec_t = 0, spec_end = 0;
    if (p.mishint && N_hint > 0) N_hint = N_hint / 2 + 1;  // diagnostic: a stale hint
    if (!p.block_table && N_hint > 0) {
        int hb_;
        slice_bounds(p, N_hint, split, tile, &spec_t, &spec_end, &hb_);
        spec = min(kStages, (spec_end - spec_t + tile - 1) / tile);
        for (int i = 0; i < spec; ++i) {
            const int t0 = spec_t + i * tile;
            if (lane == 0) {
                meta[i].tok0 = t0;
                meta[i].nvalid = min(tile, spec_end - t0);
                mbar_expect_tx(&full[i], stage_bytes);
            }
            __syncwarp();
            if (lane < nbox) issue(i, t0, lane, 0);
        }
    }
    // the real length (its load was issued before the copies above); a length
    // outside [0, S] streams nothing (the consumers report it)
    const int N = (N_ref < 0 || N_ref > p.S) ? 0 : N_ref;
    int t, t_end, base;
    slice_bounds(p, N, split, tile, &t, &t_end, &base);
    int it = 0;
    if (spec > 0) {
        // same tiles iff the slice starts at the same token and the covered
        // ranges end at the same place
        const bool same = (spec_t == t) && (min(spec_end, spec_t + spec * tile) == min(t_end, t + spec * tile));
        if (lane == 0) {
            for (int i = 0; i < spec; ++i) {
                if (!same) meta[i].nvalid = 0;
                mbar_arrive(&full[i]);
            }
        }
        if (same) t += spec * tile;
        it = spec;
    }
    const int npool = dynamic ? (N - base + C - 1) / C : 0;  // chunks handed out by the counter
    bool exhausted = (npool == 0);
    unsigned pend0 = 0, pend1 = 0;  // claims in flight (lane 0's registers), oldest first
    int npend = 0;
    bool claimed = false;

    // Next tile to stream, or -1; its token range ends at *end.  Warp-uniform:
    // only lane 0 performs claims, and a claim's value is broadcast when used.
    auto next_tile = [&](int* end) -> int {
        if (t >= t_end) {
            if (exhausted) return -1;
            if (npend == 0) {
                if (lane == 0) pend0 = atomicAdd(p.claim + row, 1u);
                npend = 1;
                claimed = true;
            }
            const unsigned j = __shfl_sync(0xffffffffu, pend0, 0);
            pend0 = pend1;
            --npend;
            if (static_cast<int>(j) >= npool) {
                exhausted = true;
                return -1;
            }
            t = base + static_cast<int>(j) * C;
            t_end = min(t + C, N);
        }
        const int r = t;
        *end = t_end;
        t += tile;
        if (!exhausted && npend < 2 && t_end - t <= 2 * C) {
            if (lane == 0) {
                const unsigned v = atomicAdd(p.claim + row, 1u);
                if (npend == 0) pend0 = v; else pend1 = v;
            }
            ++npend;
            claimed = true;
        }
        return r;
    };

    bool bad = false;
    bool ok = true;
    int cur_end = 0, nxt_end = 0;
    int cur = next_tile(&cur_end);
    int pg_a = load_box_page(p, b, N, cur, tile, lane), pg_b = kNoPage;
    // Issue `cur` (this lane's page in `now`) after starting the load for the tile after it.
    auto step = [&](int& now, int& ahead) -> bool {
        const int nxt = next_tile(&nxt_end);
        ahead = load_box_page(p, b, N, nxt, tile, lane);
        const int s = it % kStages;
        if (it >= kStages) {
            // lane 0 waits; the outcome is broadcast so the warp stays converged
            int waited = 1;
            if (lane == 0) waited = mbar_wait(&empty[s], ((it / kStages) - 1) & 1, p.err) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, waited, 0)) return false;
        }
        int page = p.num_pages;  // past the row's end, or out of range: the TMA unit zero-fills
        if (now != kNoPage) {
            if (now >= 0 && now < p.num_pages) page = now; else bad = true;
        }
        if (lane == 0) {
            meta[s].tok0 = cur;
            meta[s].nvalid = min(tile, cur_end - cur);
            mbar_arrive_expect_tx(&full[s], stage_bytes);
        }
        __syncwarp();
        if (lane < nbox) issue(s, cur, lane, page);
        ++it;
        cur = nxt;
        cur_end = nxt_end;
        return true;
    };
    while (cur >= 0) {
        if (!step(pg_a, pg_b)) { ok = false; break; }
        if (cur < 0) break;
        if (!step(pg_b, pg_a)) { ok = false; break; }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) {
        *bad_flag = 1;
        atomicOr(p.err, kErrBadSeqlen);
    }
    // Every claim must have been performed before the block takes its ticket
    // (the last ticket resets the counter): consume the outstanding results.
    if (claimed && lane == 0) *sink = pend0 + pend1;
    if (lane != 0) return ok;
    int first_pending = it > kStages ? it - kStages : 0;
    if (ok) {
        // end-of-work marker in the next stage
        const int s = it % kStages;
        if (it < kStages || mbar_wait(&empty[s], ((it / kStages) - 1) & 1, p.err)) {
            meta[s].tok0 = 0;
            meta[s].nvalid = -1;
            mbar_arrive(&full[s]);
            first_pending = it >= kStages ? it - kStages + 1 : 0;
        } else {
            ok = false;
        }
    }
    // Do not leave while copies into this block's shared memory are in flight.
    for (int j = first_pending; j < it; ++j) mbar_wait(&full[j % kStages], (j / kStages) & 1, p.err);
    return ok;
}

// Ticket with acquire-release semantics at GPU scope: the block's partial
// writes (ordered before it by the preceding block barrier) are published,
// and the last taker sees every other block's writes.
__device__ __forceinline__ unsigned ticket_acq_rel(unsigned* p, unsigned limit) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(limit)
                 : "memory");
    return old;
}

// Row merge through the cluster's distributed shared memory (a row's P
// blocks form one thread-block cluster; block rank = slice).  Every block has
// written its merged state -- numerators cs_o [nh][D], maxima cs_m (log2
// units) and denominators cs_l [nh] -- to its own shared memory and passed a
// cluster barrier; each block then merges a share of the row's (head,
// channel) outputs from all P states, normalises and writes them.  The
// caller ends with a second cluster barrier, so no block's state goes away
// while a peer still reads it.
template <int D, int kMaxP>
__device__ void cluster_merge_row(const SplitParams& p, size_t hq0, int nh, const float* cs_o,
                                  const float* cs_m, const float* cs_l, int tid, int nthr) {
    const int P = p.P;
    const int rank = static_cast<int>(cluster_rank());
    const int items = nh * D;
    const int per = (items + P - 1) / P;
    const int i0 = rank * per, i1 = min(items, i0 + per);
    for (int idx = i0 + tid; idx < i1; idx += nthr) {
        const int h = idx / D, dd = idx - h * D;
        float mq[kMaxP], lq[kMaxP], oq[kMaxP];
#pragma unroll
        for (int q = 0; q < kMaxP; ++q) {
            if (q < P) {
                mq[q] = ld_dsmem(dsmem_addr(cs_m + h, q));
                lq[q] = ld_dsmem(dsmem_addr(cs_l + h, q));
                oq[q] = ld_dsmem(dsmem_addr(cs_o + idx, q));
            } else {
                mq[q] = -INFINITY;
                lq[q] = 0.f;
                oq[q] = 0.f;
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int q = 0; q < kMaxP; ++q) M = fmaxf(M, mq[q]);
        const float Ms = (M == -INFINITY) ? 0.f : M;
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int q = 0; q < kMaxP; ++q) {
            const float w = (mq[q] == -INFINITY) ? 0.f : ex2(mq[q] - Ms);
            L = fmaf(w, lq[q], L);
            O = fmaf(w, oq[q], O);
        }
        const size_t r = hq0 + h;
        if (!in_bounds(r, p.rows, p.err)) continue;
        p.out[r * D + dd] = (L == 0.f) ? 0.f : O / L;  // NaN inputs propagate
        if (dd == 0 && p.lse) p.lse[r] = (L > 0.f) ? (M + log2f(L)) * kLn2 : (L == 0.f ? -INFINITY : L);
    }
}

// `row`: the block's schedule row (ticket and claim counters); the row's
// blocks hold the states of query heads [hq0, hq0 + G) (flat b * Hq + h).
// `prod_done`: the mbarrier the block's copy warp arrives on once it has made
// its last claim.  The ticket is taken only after that arrival, so when the
// last ticket resets the claim counter every claim of the row has landed --
// also when the compute warps left the stage ring early after a timed-out
// wait -- and a finished call leaves both counters at zero.
// kBatch: leaf numerators each thread keeps in flight (registers: 4 per leaf).
template <int D, int kBatch = 20>
__device__ void finish_row(const SplitParams& p, int row, size_t hq0, int G, float* scratch,
                           int* flag, uint64_t* prod_done, int tid, int nthr) {
    consumer_sync(nthr);
    if (tid == 0) {
        if (!mbar_wait(prod_done, 0, p.err)) atomicOr(p.err, kErrCounters);
        const unsigned t = ticket_acq_rel(p.done + row, static_cast<unsigned>(p.P - 1));
        const bool last = (t == static_cast<unsigned>(p.P - 1));
        if (last && p.claim) atomicExch(p.claim + row, 0u);
        *flag = last;
    }
    consumer_sync(nthr);
    if (!*flag || !p.fuse) return;
    const int P = p.P;
    const size_t row0 = hq0;
    constexpr int D4 = D / 4;
    if (P <= kBatch) {
        // Few leaves: each thread loads its channel's numerators together with
        // its head's maxima and denominators (one round trip to L2) and merges
        // them on its own: no block barrier on the way to the outputs.
        for (int idx = tid; idx < G * D4; idx += nthr) {
            const int h = idx / D4, d4 = idx - h * D4;
            if (!in_bounds((row0 + h) * P + P - 1, p.part_rows, p.err) || !in_bounds(row0 + h, p.rows, p.err))
                continue;
            const float4* o = reinterpret_cast<const float4*>(p.part_o + (row0 + h) * P * D) + d4;
            const float* mrow = p.part_m + (row0 + h) * P;
            const float* lrow = p.part_l + (row0 + h) * P;
            float4 v[kBatch];
            float mq[kBatch], lq[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                v[k] = k < P ? __ldcg(o + static_cast<size_t>(k) * D4) : make_float4(0.f, 0.f, 0.f, 0.f);
                mq[k] = k < P ? __ldcg(mrow + k) : -INFINITY;
                lq[k] = k < P ? __ldcg(lrow + k) : 0.f;
            }
            float M = -INFINITY;
#pragma unroll
            for (int k = 0; k < kBatch; ++k) M = fmaxf(M, mq[k]);
            const float Ms = (M == -INFINITY) ? 0.f : M;
            float L = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const float w = (mq[k] == -INFINITY) ? 0.f : ex2((mq[k] - Ms) * kLog2e);
                L = fmaf(w, lq[k], L);
                acc.x = fmaf(w, v[k].x, acc.x);
                acc.y = fmaf(w, v[k].y, acc.y);
                acc.z = fmaf(w, v[k].z, acc.z);
                acc.w = fmaf(w, v[k].w, acc.w);
            }
            if (L == 0.f) {
                acc = make_float4(0.f, 0.f, 0.f, 0.f);
            } else {  // NaN inputs propagate
                acc.x /= L;
                acc.y /= L;
                acc.z /= L;
                acc.w /= L;
            }
            reinterpret_cast<float4*>(p.out + (row0 + h) * D)[d4] = acc;
            if (d4 == 0 && p.lse) p.lse[row0 + h] = (L > 0.f) ? M + logf(L) : (L == 0.f ? -INFINITY : L);
        }
        return;
    }
    if (!in_bounds((row0 + G) * P - 1, p.part_rows, p.err) || !in_bounds(row0 + G - 1, p.rows, p.err))
        return;  // (bounds-checking build) the row's states are not where they should be
    float* sw = scratch;           // [G][P]  maxima, then leaf weights
    float* sl = scratch + G * P;   // [G][P]  denominators
    float* sr = sl + G * P;        // [G] root maxima, [G] root denominators
    // The first batch of each thread's numerators is loaded together with the
    // maxima and denominators, so the merge costs one round trip to L2.
    const int idx0 = tid;
    const bool has0 = idx0 < G * D4;
    const int h0 = has0 ? idx0 / D4 : 0, d40 = has0 ? idx0 - h0 * D4 : 0;
    const float4* o0 = reinterpret_cast<const float4*>(p.part_o + (row0 + h0) * P * D) + d40;
    float4 v[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
        v[k] = (has0 && k < P) ? __ldcg(o0 + static_cast<size_t>(k) * D4) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = tid; i < G * P; i += nthr) {
        sw[i] = __ldcg(p.part_m + row0 * P + i);
        sl[i] = __ldcg(p.part_l + row0 * P + i);
    }
    consumer_sync(nthr);
    const int warp = tid >> 5, lane = tid & 31, nw = nthr >> 5;
    for (int h = warp; h < G; h += nw) {
        float M = -INFINITY;
        for (int q = lane; q < P; q += 32) M = fmaxf(M, sw[h * P + q]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float Ms = (M == -INFINITY) ? 0.f : M;
        float L = 0.f;
        for (int q = lane; q < P; q += 32) {
            const float mq = sw[h * P + q];
            const float w = (mq == -INFINITY) ? 0.f : ex2((mq - Ms) * kLog2e);
            sw[h * P + q] = w;
            L = fmaf(w, sl[h * P + q], L);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
        if (lane == 0) {
            sr[h] = M;
            sr[G + h] = L;
        }
    }
    consumer_sync(nthr);
    for (int idx = tid; idx < G * D4; idx += nthr) {
        const int h = idx / D4, d4 = idx - h * D4;
        const float4* o = reinterpret_cast<const float4*>(p.part_o + (row0 + h) * P * D) + d4;
        const float* w = sw + h * P;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q0 = 0; q0 < P; q0 += kBatch) {
            if (idx != idx0 || q0 != 0) {
#pragma unroll
                for (int k = 0; k < kBatch; ++k)
                    v[k] = (q0 + k < P) ? __ldcg(o + static_cast<size_t>(q0 + k) * D4)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const float wk = (q0 + k < P) ? w[q0 + k] : 0.f;
                acc.x = fmaf(wk, v[k].x, acc.x);
                acc.y = fmaf(wk, v[k].y, acc.y);
                acc.z = fmaf(wk, v[k].z, acc.z);
                acc.w = fmaf(wk, v[k].w, acc.w);
            }
        }
        const float L = sr[G + h];
        if (L == 0.f) {
            acc = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {  // NaN inputs propagate
            acc.x /= L;
            acc.y /= L;
            acc.z /= L;
            acc.w /= L;
        }
        reinterpret_cast<float4*>(p.out + (row0 + h) * D)[d4] = acc;
        if (d4 == 0 && p.lse) p.lse[row0 + h] = (L > 0.f) ? sr[h] + logf(L) : (L == 0.f ? -INFINITY : L);
    }
}

}  // namespace ta
