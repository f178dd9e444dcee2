// Device-side building blocks shared by the split-KV kernels and the combine:
// mbarrier waits with a time limit, TMA tile loads, base-2 exponentials and
// the parameter block every per-slice kernel receives.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ta {

// Error bits of the device error word.
constexpr int kErrBadSeqlen = 1;  // a sequence length outside [0, max_seqlen], or a bad page
constexpr int kErrTimeout = 2;    // a bounded barrier wait gave up
constexpr int kErrCounters = 4;   // a row's copy warp outlived its bounded hand-over, so the
                                  // row's scheduling counters may not be back at zero
constexpr int kErrBounds = 8;     // (bounds-checking builds) an index outside its buffer was
                                  // caught and the access skipped

// log2(e) and ln(2): the kernels evaluate exp(x) as 2^(x * log2 e).
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// A bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Parameters of one per-slice launch.  Grid: (num_splits, Hkv, B).
struct SplitParams {
    const void* q;          // [B][Hq][d]
    int q_is_bf16;          // 1: q is BF16, 0: FP32
    const int32_t* seqlens; // [B]
    float* out;             // [B][Hq][d]      (num_splits == 1)
    float* lse;             // [B][Hq] or null (num_splits == 1)
    float* part_o;          // [B][Hq][P][d]   (num_splits > 1)
    float* part_m;          // [B][Hq][P]
    float* part_l;          // [B][Hq][P]
    int* err;               // device error word
    unsigned* claim;        // [B*Hkv/hb] chunk counters (null: static chunk assignment)
    unsigned* done;         // [B*Hkv/hb] row tickets (null: no ticket is taken)
    int fuse;               // the row's last block merges the partial states
    const float* k_scale;   // [Hkv] FP8 caches: K = k_scale[g] * e4m3 code
    const float* v_scale;   // [Hkv] likewise for V
    const int32_t* block_table;  // [B][max_pages] (null: dense cache, coordinate w = batch row)
    int max_pages;          // block_table columns
    int page_shift;         // log2(page_size)
    int num_pages;          // pages in the pool (an out-of-range page reads zeros)
    int box_rows;           // tokens per TMA box: the tile, or the page when it is smaller
    int hb;                 // KV heads per block (a box brings box_rows tokens of each)
    int stall;              // diagnostic: the producer publishes nothing (waits give up)
    int mishint;            // diagnostic: the producer's length hint is made wrong
    int cluster;            // a row's P blocks form a cluster and merge through its shared memory
    int B, Hq, Hkv, G, S, P; // Hq, G count virtual heads: query heads x queries per row
    int nq;                 // queries per row (q rows are [head][query])
    int causal;             // query i of nq sees tokens < N - nq + 1 + i
    int chunk_tiles;        // tiles per scheduled chunk
    int prefetch_tiles;     // tiles of its slice a block prefetches into L2 before its wait
    float scale_log2;       // logit scale * log2(e)
    // buffer extents, checked by the bounds-checking build only
    size_t q_elems;         // elements of q
    size_t out_elems;       // elements of out (B * Hq * d)
    size_t rows;            // rows of lse (B * Hq)
    size_t part_rows;       // rows of the partial states (B * Hq * P; 0 when P == 1)
    size_t bt_elems;        // entries of the block table
};

// Bounds checks of the bounds-checking build (TA_DEBUG_BOUNDS): an index
// outside [0, n) sets kErrBounds in *err and the caller skips the access.
// In the normal build the check is the constant true and compiles away.
#ifdef TA_DEBUG_BOUNDS
__device__ __forceinline__ bool in_bounds(size_t idx, size_t n, int* err) {
    if (idx < n) return true;
    atomicOr(err, kErrBounds);
    return false;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(size_t, size_t, int*) { return true; }
#endif

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

// Adds `bytes` to the transaction count of the current phase without
// arriving: the phase cannot complete before a later arrive.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// sets the timeout bit of *err) if that takes longer than kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > kWaitLimitNs) {
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
}

// ------------------------------------------------------------------- TMA
// 4-D tiled load (x = channel, y = token, z = KV head, w = batch row) into
// shared memory, completing `bytes` of the mbarrier's transaction count.
__device__ __forceinline__ void tma_load_4d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)),
        "l"(policy)
        : "memory");
}

// 5-D tiled load (x = channel within a 64-channel half, y = token, z = half,
// w = KV head, v = batch row or physical page).
__device__ __forceinline__ void tma_load_5d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, int v, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(v),
        "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// L2 prefetch of one box of a tiled tensor (no shared memory, no barrier);
// boxes reaching past the tensor fetch only what lies inside it.
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* map, int x, int y, int z, int w) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}

__device__ __forceinline__ void tma_prefetch_5d(const CUtensorMap* map, int x, int y, int z, int w,
                                                int v) {
    asm volatile("cp.async.bulk.prefetch.tensor.5d.L2.global.tile [%0, {%1, %2, %3, %4, %5}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(w), "r"(v)
                 : "memory");
}

// Relaxed GPU-scope load: a value another grid may still be writing (used
// only as a hint).
__device__ __forceinline__ int ld_relaxed(const int* ptr) {
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Named barrier over the consumer warps only (id 1; id 0 is __syncthreads).
__device__ __forceinline__ void consumer_sync(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Programmatic dependent launch: let the combine grid start its launch early.
// ------------------------------------------------------------ clusters
// Barrier over every thread of the thread-block cluster (writes to shared
// memory before it are visible to loads from any block of the cluster after).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ unsigned cluster_rank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of this block's shared-memory word `local` in block `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, unsigned rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_dsmem(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace ta
