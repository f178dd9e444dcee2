// C ABI of libtreeattn.so (declared in include/tree_attn.h): argument
// validation, the split-count heuristic, TMA descriptors, kernel dispatch and
// the device error word.  Every step of the computation runs in the kernels
// of this library; this file only checks, plans and enqueues.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <iterator>
#include <memory>
#include <mutex>
#include <new>
#include <queue>
#include <vector>

#include "../../include/tree_attn.h"
#include "kernels.h"

namespace {

using ta::Geometry;

__device__ int g_error_word;  // bits ta::kErrBadSeqlen | kErrTimeout | kErrCounters | kErrBounds

// Scheduling counters (chunk claims and row tickets) of the split kernels.
// Zero at load; each call reserves two consecutive slots per schedule row
// (B * Hkv / heads_per_block rows) and leaves them at zero when it
// completes -- also when one of its waits gave up, because a row's ticket is
// taken only after the block's copy warp has made its last claim -- so slots
// are reused as the cursor wraps.
constexpr unsigned kRingSlots = 1u << 20;
__device__ unsigned g_sched_ring[kRingSlots];

// Tokens per run-time scheduled chunk of a row (rounded to whole tiles).
constexpr int kChunkTokens = 128;
// Tokens of its slice each block prefetches into L2 before waiting on the
// previous grid (fills the DRAM time of that grid's merge tail).  Measured
// optima: 1152 for BF16 caches (576 KB per KV head), 768 for FP8 (192 KB;
// 512 / 1152 / 1792 / 2304 were slower on the 8B-shaped layer).
constexpr int kPrefetchTokens = 1152;
constexpr int kPrefetchTokensFp8 = 768;
// The tcgen05 kernel's steps are longer (many columns per KV head), so less of
// the prefetch hides behind the previous step's merge: 256 tokens measured
// best (0 / 256 / 512 / 1152: 94.2 / 93.6 / 94.5 / 95.2 us with 32 columns).
constexpr int kPrefetchTokensTc05 = 256;
// The row's last block merges the partial states itself when there are few
// of them (its merge costs about one L2 round trip per 20 states, serially);
// more splits go to the combine kernel, which spreads the merge over (h, b)
// blocks.  G*P states must also fit in the block's idle stage buffers.
constexpr int kFusedMaxSplits = 40;
// Chunks are balanced at run time only for grids of at most this many waves.
constexpr int64_t kBalanceMaxWaves = 4;
constexpr int kFusedMaxStates = 8192;

bool fuse_merge(int G, int P) {
    return P <= kFusedMaxSplits && static_cast<int64_t>(G) * P <= kFusedMaxStates;
}
// A block serving several KV heads merges heads_per_block * G states per
// slice; within the split limit that never changes the decision (G <= 16,
// at most 4 heads per block), so the launch count needs no page size.
static_assert(kFusedMaxSplits * 16 * 4 <= kFusedMaxStates, "fused-merge decision independent of heads per block");

// Paged caches with 16-token pages: one TMA box spans the same tokens of
// several KV heads (a block serves them all), so a box is 4-16 KB instead of
// 2-4 KB.  (Measured on GB300: FP8 16-token pages 55.8 -> 49.1 us on the
// 131072-token layer in either pool layout; BF16 gains only in token-major
// pools, and FP8 32-token pages not at all.)
constexpr int kFp8HeadsPage16 = 4;   // FP8 cache
constexpr int kMmaHeadsPage16 = 2;   // BF16 tensor-core kernel, token-major pools

constexpr int kKnownFlags =
    TA_FLAG_DETERMINISTIC | TA_FLAG_DIAG_STALL | TA_FLAG_DIAG_MISHINT | TA_FLAG_CLUSTER_MERGE;
constexpr int kClusterMaxSplits = 8;  // portable cluster size
// With the split count left to the library, rows whose slices are at most this
// many tokens merge through a thread-block cluster (TA_FLAG_CLUSTER_MERGE):
// there the step is mostly its fixed start and end, and the cluster merge
// drops the ticket and the last block's L2 round trips (about 3 us).  Measured
// on GB300 with CUDA-graph replay: 9-14 % shorter steps on the 8B-shaped layer
// (8 rows) at 1024-4096 tokens, 6-8 % on the 70B-shaped one (32 rows of 4
// slices) at 1024-2048, 1 % at 640 tokens per slice (BF16), and slower from
// 768 tokens per slice (BF16) or 1024 (FP8) on, where 16 slices beat 8.
constexpr int kClusterAutoTokens = 640;
constexpr int kClusterAutoTokensFp8 = 768;

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    int* err = nullptr;        // device address of g_error_word on this device
    unsigned* ring = nullptr;  // device address of g_sched_ring on this device
    unsigned cursor = 0;       // next free ring slot
    int device = 0;            // this entry's CUDA device
    int cluster_cap[kClusterMaxSplits + 1];  // co-resident clusters per size; -1: not queried
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Per-device set-up, once, with that device current.
int device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& s = g_dev[dev];
    if (!s.ready) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TA_ERR_CUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return TA_ERR_CUDA;
        void* r = nullptr;
        if (cudaGetSymbolAddress(&r, g_sched_ring) != cudaSuccess) return TA_ERR_CUDA;
        s.num_sms = sms;
        s.device = dev;
        s.err = static_cast<int*>(p);
        s.ring = static_cast<unsigned*>(r);
        std::fill(std::begin(s.cluster_cap), std::end(s.cluster_cap), -1);
        s.ready = true;
    }
    *out = &s;
    return TA_OK;
}

// Clusters of `size` split-kernel blocks that fit on the device at once.
int cluster_capacity(DeviceState* s, int size) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (s->cluster_cap[size] < 0) s->cluster_cap[size] = ta::mma_cluster_capacity(size);
    return s->cluster_cap[size];
}

// Reserve `n` consecutive counter slots for one call (nullptr if n exceeds the ring).
unsigned* reserve_slots(DeviceState* s, unsigned n) {
    if (n == 0 || n > kRingSlots) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (s->cursor + n > kRingSlots) s->cursor = 0;
    unsigned* r = s->ring + s->cursor;
    s->cursor += n;
    return r;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_bytes(int dtype) { return dtype == TA_BF16 ? 2 : (dtype == TA_E4M3 ? 1 : 4); }

// Internal kernel families for FP8 caches: the warp-level tensor-core kernel
// (TA_KERNEL_MMA) and the tcgen05 kernel (TA_KERNEL_TC05).
constexpr int kKernelFp8 = 4;
constexpr int kKernelTc05Fp8 = 5;
static_assert(kKernelFp8 != TA_KERNEL_AUTO && kKernelFp8 != TA_KERNEL_FMA && kKernelFp8 != TA_KERNEL_MMA &&
                  kKernelFp8 != TA_KERNEL_TC05 && kKernelTc05Fp8 > kKernelFp8,
              "internal kernel id");
// FP8 caches with more than this many columns per KV head take the tcgen05
// kernel by default (up to 16 the warp-level kernel is faster: 59.8 against
// 66.2 us with 16 columns on the 131072-token 8B-shaped layer).
constexpr int kFp8Tc05MinCols = 16;

struct Strides {
    int64_t b, h, t;
};

// Validate the shape; on success fill the resolved KV strides (elements).
// `page_size` > 0: the strides describe a page pool whose default layout is
// [num_pages][page_size][Hkv][d] (kv_stride_b = stride between pages).
int check_shape(const ta_shape* s, Strides* st, int page_size = 0) {
    if (!s) return TA_ERR_NULL;
    if (s->batch < 1 || s->num_q_heads < 1 || s->num_kv_heads < 1 || s->max_seqlen < 1)
        return TA_ERR_SHAPE;
    if (s->num_q_heads % s->num_kv_heads != 0) return TA_ERR_SHAPE;
    const int G = s->num_q_heads / s->num_kv_heads;
    if (G < 1 || G > 64) return TA_ERR_SHAPE;
    if (s->head_dim != 64 && s->head_dim != 128) return TA_ERR_SHAPE;
    if ((s->q_dtype != TA_F32 && s->q_dtype != TA_BF16) ||
        (s->kv_dtype != TA_F32 && s->kv_dtype != TA_BF16 && s->kv_dtype != TA_E4M3))
        return TA_ERR_DTYPE;
    if (!(s->scale >= 0.f) || std::isinf(s->scale)) return TA_ERR_SHAPE;
    Strides r;
    const int64_t d = s->head_dim, S = s->max_seqlen, H = s->num_kv_heads;
    if (s->kv_stride_b == 0 && s->kv_stride_h == 0 && s->kv_stride_t == 0) {
        if (page_size > 0) {
            r.h = d;
            r.t = H * d;
            r.b = static_cast<int64_t>(page_size) * H * d;
        } else {
            r.t = d;
            r.h = S * d;
            r.b = H * S * d;
        }
    } else {
        r.b = s->kv_stride_b;
        r.h = s->kv_stride_h;
        r.t = s->kv_stride_t;
        if (r.b <= 0 || r.h <= 0 || r.t <= 0) return TA_ERR_SHAPE;
    }
    const int64_t es = elem_bytes(s->kv_dtype);
    const int64_t lim = int64_t(1) << 40;
    for (int64_t x : {r.b, r.h, r.t}) {
        if ((x * es) % 16 != 0) return TA_ERR_ALIGN;
        if (x * es >= lim) return TA_ERR_SHAPE;
    }
    if (st) *st = r;
    return TA_OK;
}

// Kernel family for a shape (num_q_heads counts (head, query) pairs for
// multi-query calls): the warp-level tensor-core kernel takes BF16 q and cache
// with up to 16 columns per KV head (64 at head_dim 128, in column groups of
// 16); the tcgen05 kernel BF16 q and cache at head_dim 128 with up to 64
// columns, and is the automatic choice above 16 columns (the cluster merge
// is built into the warp-level kernels only); the FMA kernel any dtypes with
// a power-of-two group up to 16.
int resolve_kernel(const ta_shape* s, int requested, bool cluster = false) {
    const int G = s->num_q_heads / s->num_kv_heads;
    if (s->kv_dtype == TA_E4M3) {
        if (s->q_dtype != TA_BF16 || s->head_dim != 128 || requested == TA_KERNEL_FMA) return TA_ERR_DTYPE;
        const bool mma_ok = G <= 16, tc05_ok = G <= 32 && !cluster;
        switch (requested) {
            case TA_KERNEL_AUTO:
                if (tc05_ok && G > kFp8Tc05MinCols) return kKernelTc05Fp8;
                return mma_ok ? kKernelFp8 : static_cast<int>(TA_ERR_SHAPE);
            case TA_KERNEL_MMA: return mma_ok ? kKernelFp8 : static_cast<int>(TA_ERR_SHAPE);
            case TA_KERNEL_TC05: return tc05_ok ? kKernelTc05Fp8 : static_cast<int>(TA_ERR_SHAPE);
            default: return TA_ERR_SHAPE;
        }
    }
    const bool bf16 = s->q_dtype == TA_BF16 && s->kv_dtype == TA_BF16;
    const bool mma_ok = bf16 && (G <= 16 || (G <= 64 && s->head_dim == 128));
    const bool tc05_ok = bf16 && G <= 64 && s->head_dim == 128;
    const bool fma_ok = (G & (G - 1)) == 0 && G <= 16;
    switch (requested) {
        case TA_KERNEL_AUTO:
            if (tc05_ok && G > 16 && !cluster) return TA_KERNEL_TC05;
            return mma_ok ? static_cast<int>(TA_KERNEL_MMA)
                          : (fma_ok ? static_cast<int>(TA_KERNEL_FMA) : static_cast<int>(TA_ERR_SHAPE));
        case TA_KERNEL_FMA: return fma_ok ? static_cast<int>(TA_KERNEL_FMA) : static_cast<int>(TA_ERR_SHAPE);
        case TA_KERNEL_MMA: return mma_ok ? static_cast<int>(TA_KERNEL_MMA) : static_cast<int>(TA_ERR_DTYPE);
        case TA_KERNEL_TC05:
            if (!tc05_ok) return bf16 ? static_cast<int>(TA_ERR_SHAPE) : static_cast<int>(TA_ERR_DTYPE);
            return cluster ? static_cast<int>(TA_ERR_SHAPE) : static_cast<int>(TA_KERNEL_TC05);
        default: return TA_ERR_SHAPE;
    }
}

Geometry geometry_hb(const ta_shape* s, int kernel, int hb) {
    if (kernel == kKernelFp8) return ta::fp8_geometry(hb);
    if (kernel == kKernelTc05Fp8) return ta::tc05_fp8_geometry();  // one KV head per block
    if (kernel == TA_KERNEL_TC05) return ta::tc05_geometry(0);    // one KV head per block
    return kernel == TA_KERNEL_MMA ? ta::mma_geometry(s->head_dim, hb)
                                   : ta::fma_geometry(elem_bytes(s->kv_dtype), s->head_dim);
}

int pick_splits_hb(const ta_shape* s, const int32_t* host_seqlens, int num_sms, int kernel, int hb);

// KV heads per block for a kernel family and page size (0: dense cache).
// The BF16 kernel uses several only in token-major pools ([page][token][head]
// [d]: the KV heads of a token lie closer together than the tokens of a
// head).  The largest candidate is taken whose split count for full-length
// rows keeps the row merge fused, when one head per block does (more splits
// would add a combine launch).
int heads_per_block(const ta_shape* s, int kernel, int page_size, int num_sms) {
    if (page_size <= 0 || page_size > 16) return 1;
    const int64_t sh = s->kv_stride_h ? s->kv_stride_h : static_cast<int64_t>(s->head_dim);
    const int64_t st = s->kv_stride_t ? s->kv_stride_t : static_cast<int64_t>(s->num_kv_heads) * s->head_dim;
    int want = 1;
    if (kernel == kKernelFp8)
        want = kFp8HeadsPage16;
    else if (kernel == TA_KERNEL_MMA && s->head_dim == 128 && sh < st && s->num_q_heads <= 16 * s->num_kv_heads)
        want = kMmaHeadsPage16;
    const int splits1 = pick_splits_hb(s, nullptr, num_sms, kernel, 1);
    const bool fused1 = splits1 <= kFusedMaxSplits;
    // With two n-tiles (9..16 columns) the consumers carry twice the work per
    // token: sharing a block between heads pays only when it does not also
    // shorten every block's slice (more splits).
    const bool wide = s->num_q_heads > 8 * s->num_kv_heads;
    for (; want > 1; want /= 2) {
        if (s->num_kv_heads % want != 0) continue;
        const int splits = pick_splits_hb(s, nullptr, num_sms, kernel, want);
        if (wide && splits > splits1) continue;
        if (!fused1 || splits <= kFusedMaxSplits) break;
    }
    return want;
}

Geometry geometry_of(const ta_shape* s, int kernel, int page_size, int num_sms) {
    if (kernel == TA_KERNEL_TC05) return ta::tc05_geometry(page_size);
    if (kernel == kKernelTc05Fp8) return ta::tc05_fp8_geometry();
    return geometry_hb(s, kernel, heads_per_block(s, kernel, page_size, num_sms));
}

// Resident thread blocks per SM of each kernel family (shared memory bound:
// the MMA kernel's ring is 192 KB; the FMA kernel's ~113 KB with 288 threads
// of ~170 registers).
int blocks_per_sm(const ta_shape* s, int kernel) {
    (void)s;
    (void)kernel;
    return 1;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
    size_t o, m, l, total;
};

WsLayout workspace_layout(const ta_shape* s, int P) {
    const size_t rows = static_cast<size_t>(s->batch) * s->num_q_heads * P;
    WsLayout w;
    w.o = 0;
    w.m = round256(rows * s->head_dim * sizeof(float));
    w.l = w.m + round256(rows * sizeof(float));
    w.total = w.l + round256(rows * sizeof(float));
    return w;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------------ heuristic
// Estimated step time for P slices, in units of "one block streaming one
// token of one KV head": a block's fixed cost (pipeline fill, epilogue) is
// worth kBlockCost tokens; a second (combine) launch kBlockCost more plus its
// traffic (partials written and read back) spread over the whole GPU.  A
// block serving hb KV heads streams hb such units per token.  512 matches the
// measured split sweeps on GB300: it keeps the best counts of the uniform
// layers (19 on 152 SMs) and picks the best one of the ragged batch (5; 256
// picked 16, measured 7 % slower).
constexpr double kBlockCost = 512.0;

double estimate(const ta_shape* s, const std::vector<int64_t>& lens, bool uniform, int P,
                int tile, int slots, int hb) {
    const int Hkv = s->num_kv_heads / hb;
    const double bytes_per_token = 2.0 * s->head_dim * elem_bytes(s->kv_dtype);
    double comb = 0.0;
    if (P > 1) {
        const double comb_bytes =
            2.0 * s->batch * s->num_q_heads * static_cast<double>(P) * (s->head_dim + 2) * 4;
        comb = kBlockCost + comb_bytes / bytes_per_token / slots;
    }
    if (uniform) {
        const int64_t N = lens[0];
        const int64_t c = ceil_div(ceil_div(N, P), tile) * tile;
        const int64_t blocks = static_cast<int64_t>(s->batch) * Hkv * P;
        const int64_t waves = ceil_div(blocks, slots);
        return static_cast<double>(waves) * (static_cast<double>(std::min<int64_t>(c, N)) * hb + kBlockCost) +
               comb;
    }
    // Ragged rows: list-schedule the blocks in launch order (slice fastest,
    // then KV head, then batch row) onto the earliest free slot.
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    for (int i = 0; i < slots; ++i) free_at.push(0.0);
    double makespan = 0.0;
    for (int b = 0; b < s->batch; ++b) {
        const int64_t N = lens[b];
        const int64_t c = N > 0 ? ceil_div(ceil_div(N, P), tile) * tile : 0;
        for (int g = 0; g < Hkv; ++g) {
            for (int p = 0; p < P; ++p) {
                const int64_t a = c * p;
                const int64_t len = (a >= N) ? 0 : std::min<int64_t>(c, N - a);
                const double t = free_at.top() + static_cast<double>(len) * hb + kBlockCost;
                free_at.pop();
                free_at.push(t);
                makespan = std::max(makespan, t);
            }
        }
    }
    return makespan + comb;
}

int pick_splits_hb(const ta_shape* s, const int32_t* host_seqlens, int num_sms, int kernel, int hb) {
    const Geometry geo = geometry_hb(s, kernel, hb);
    const int tile = geo.tile_tokens;
    const int slots = std::max(1, num_sms) * blocks_per_sm(s, kernel);
    std::vector<int64_t> lens(s->batch);
    bool uniform = true;
    int64_t maxN = 0;
    for (int b = 0; b < s->batch; ++b) {
        int64_t n = host_seqlens ? host_seqlens[b] : s->max_seqlen;
        n = std::max<int64_t>(0, std::min<int64_t>(n, s->max_seqlen));
        lens[b] = n;
        maxN = std::max(maxN, n);
        if (n != lens[0]) uniform = false;
    }
    if (maxN == 0) return 1;
    // slices of at least 256 tokens; no more than 64 waves of blocks
    int64_t pmax = std::max<int64_t>(1, ceil_div(maxN, 256));
    pmax = std::min<int64_t>(pmax, TA_MAX_SPLITS);
    const int64_t rows = static_cast<int64_t>(s->batch) * (s->num_kv_heads / hb);
    pmax = std::min<int64_t>(pmax, std::max<int64_t>(1, 64 * static_cast<int64_t>(slots) / rows));
    int best = 1;
    double best_t = estimate(s, lens, uniform, 1, tile, slots, hb);
    for (int P = 2; P <= pmax; ++P) {
        const double t = estimate(s, lens, uniform, P, tile, slots, hb);
        if (t < best_t * (1.0 - 1e-9)) {
            best_t = t;
            best = P;
        }
    }
    return best;
}

int pick_splits_impl(const ta_shape* s, const int32_t* host_seqlens, int num_sms, int kernel,
                     int page_size) {
    return pick_splits_hb(s, host_seqlens, num_sms, kernel,
                          heads_per_block(s, kernel, page_size, num_sms));
}

// Whether a call whose split count the library picked (P) merges each row
// through a cluster of min(P, 8) blocks instead: short slices, a kernel with
// the cluster merge, and every row's cluster resident in one wave.
bool auto_cluster(DeviceState* ds, const ta_shape* s, int kernel, int P, int page_size,
                  const ta_options* options) {
    if (P < 2 || (kernel != TA_KERNEL_MMA && kernel != kKernelFp8)) return false;
    if (options && (options->flags & (TA_FLAG_DIAG_STALL | TA_FLAG_DIAG_MISHINT))) return false;
    const int pc = std::min(P, kClusterMaxSplits);
    const int limit = s->kv_dtype == TA_E4M3 ? kClusterAutoTokensFp8 : kClusterAutoTokens;
    if (ceil_div(s->max_seqlen, pc) > limit) return false;
    const int64_t rows = static_cast<int64_t>(s->batch) *
                         (s->num_kv_heads / heads_per_block(s, kernel, page_size, ds->num_sms));
    return rows <= cluster_capacity(ds, pc);
}

// 4-D map over (channel, token, KV head, batch row) -- or, for a page pool,
// (channel, token in page, KV head, physical page).  Box: box_x channels x
// `rows` tokens.
int encode_kv_map_uncached(CUtensorMap* map, const void* base, const ta_shape* s, const Strides& st,
                           const Geometry& geo, const ta_paged_kv* paged, int rows) {
    auto fn = encode_fn();
    if (!fn) return TA_ERR_CUDA;
    const int64_t es = elem_bytes(s->kv_dtype);
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(s->head_dim),
                          static_cast<cuuint64_t>(paged ? paged->page_size : s->max_seqlen),
                          static_cast<cuuint64_t>(s->num_kv_heads),
                          static_cast<cuuint64_t>(paged ? paged->num_pages : s->batch)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.t * es), static_cast<cuuint64_t>(st.h * es),
                             static_cast<cuuint64_t>(st.b * es)};
    const cuuint32_t hb = static_cast<cuuint32_t>(geo.heads_per_block);
    cuuint32_t box[4] = {static_cast<cuuint32_t>(geo.box_x), static_cast<cuuint32_t>(rows), hb, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    if (geo.halves5d) {
        // 5-D view (channel in half, token, half, KV head, row/page): one box
        // brings every 64-channel half of `rows` tokens, [half][rows][128 B].
        const cuuint64_t halves = static_cast<cuuint64_t>(s->head_dim / 64);
        cuuint64_t dims5[5] = {64, dims[1], halves, dims[2], dims[3]};
        cuuint64_t strides5[4] = {strides[0], 128, strides[1], strides[2]};
        cuuint32_t box5[5] = {64, static_cast<cuuint32_t>(rows),
                              geo.split_halves ? 1u : static_cast<cuuint32_t>(halves), hb, 1};
        const CUresult r5 = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base),
                               dims5, strides5, box5, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        return r5 == CUDA_SUCCESS ? TA_OK : TA_ERR_CUDA;
    }
    const CUresult r = fn(map,
                          s->kv_dtype == TA_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                          : s->kv_dtype == TA_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          4, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          geo.swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TA_OK : TA_ERR_CUDA;
}

// Every input of a tensor-map encode: a map is a pure function of these, so a
// cached map stays valid for as long as the same inputs come back (decode
// steps reuse the same cache buffers and sizes).
struct MapKey {
    const void* base;
    int64_t dims[4], strides[3];
    int32_t dtype, rows, box_x, swizzle128, halves5d, hb, split_halves;
};

struct MapSlot {
    MapKey key;
    CUtensorMap map;
    bool valid;
};

constexpr int kMapSlots = 1024;  // direct-mapped, per device (allocated on first use)

std::unique_ptr<MapSlot[]> g_maps[kMaxDevices];

uint64_t hash_key(const MapKey& k) {
    const unsigned char* b = reinterpret_cast<const unsigned char*>(&k);
    uint64_t h = 1469598103934665603ull;  // FNV-1a
    for (size_t i = 0; i < sizeof k; ++i) h = (h ^ b[i]) * 1099511628211ull;
    return h;
}

int encode_kv_map(int dev, CUtensorMap* map, const void* base, const ta_shape* s, const Strides& st,
                  const Geometry& geo, const ta_paged_kv* paged, int rows) {
    MapKey k;
    std::memset(&k, 0, sizeof k);  // padding bytes take part in the hash and the compare
    k.base = base;
    k.dims[0] = s->head_dim;
    k.dims[1] = paged ? paged->page_size : s->max_seqlen;
    k.dims[2] = s->num_kv_heads;
    k.dims[3] = paged ? paged->num_pages : s->batch;
    k.strides[0] = st.t;
    k.strides[1] = st.h;
    k.strides[2] = st.b;
    k.dtype = s->kv_dtype;
    k.rows = rows;
    k.box_x = geo.box_x;
    k.swizzle128 = geo.swizzle128;
    k.halves5d = geo.halves5d;
    k.split_halves = geo.split_halves;
    k.hb = geo.heads_per_block;
    const size_t i = hash_key(k) % kMapSlots;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_maps[dev]) g_maps[dev].reset(new (std::nothrow) MapSlot[kMapSlots]());
        if (g_maps[dev] && g_maps[dev][i].valid && std::memcmp(&g_maps[dev][i].key, &k, sizeof k) == 0) {
            *map = g_maps[dev][i].map;
            return TA_OK;
        }
    }
    const int rc = encode_kv_map_uncached(map, base, s, st, geo, paged, rows);
    if (rc != TA_OK) return rc;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_maps[dev]) {
        g_maps[dev][i].key = k;
        g_maps[dev][i].map = *map;
        g_maps[dev][i].valid = true;
    }
    return TA_OK;
}

}  // namespace

namespace {

int check_paged(const ta_shape* shape, const ta_paged_kv* pg) {
    if (!pg->block_table) return TA_ERR_NULL;
    if (!aligned(pg->block_table, 4)) return TA_ERR_ALIGN;
    if (pg->reserved != 0) return TA_ERR_SHAPE;
    const int ps = pg->page_size;
    if (ps < 16 || ps > 1024 || (ps & (ps - 1)) != 0) return TA_ERR_SHAPE;
    if (pg->max_pages_per_seq < 1 || pg->num_pages < 1) return TA_ERR_SHAPE;
    if (static_cast<int64_t>(shape->max_seqlen) > static_cast<int64_t>(pg->max_pages_per_seq) * ps)
        return TA_ERR_SHAPE;
    return TA_OK;
}

// `shape` counts (head, query) pairs as query heads when nq > 1.
int decode_impl(const ta_shape* shape, const ta_paged_kv* paged, int nq, int causal, const void* q,
                const void* k_cache, const void* v_cache, const int32_t* seqlens, float* out,
                float* lse, int num_splits, void* workspace, size_t workspace_bytes,
                const ta_options* options, void* stream_ptr) {
    if (!shape) return TA_ERR_NULL;
    Strides st;
    int rc = paged ? check_paged(shape, paged) : TA_OK;
    if (rc != TA_OK) return rc;
    rc = check_shape(shape, &st, paged ? paged->page_size : 0);
    if (rc != TA_OK) return rc;
    if (!q || !k_cache || !v_cache || !seqlens || !out) return TA_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(seqlens, 4) || (lse && !aligned(lse, 4)))
        return TA_ERR_ALIGN;
    if (options && (options->flags & ~kKnownFlags) != 0) return TA_ERR_SHAPE;
    const bool deterministic = options && (options->flags & TA_FLAG_DETERMINISTIC);
    bool cluster = options && (options->flags & TA_FLAG_CLUSTER_MERGE);
    const int kernel = resolve_kernel(shape, options ? options->kernel : TA_KERNEL_AUTO, cluster);
    if (kernel < 0) return kernel;
    if (cluster && kernel != TA_KERNEL_MMA && kernel != kKernelFp8) return TA_ERR_SHAPE;
    if (cluster && num_splits > kClusterMaxSplits) return TA_ERR_SPLITS;
    if (shape->kv_dtype == TA_E4M3) {
        if (!options || !options->k_scale || !options->v_scale) return TA_ERR_NULL;
        if (!aligned(options->k_scale, 4) || !aligned(options->v_scale, 4)) return TA_ERR_ALIGN;
    }
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

    if (num_splits > TA_MAX_SPLITS) return TA_ERR_SPLITS;
    auto check_ws = [&](int P) {
        if (P <= 1) return static_cast<int>(TA_OK);
        if (!workspace || workspace_bytes < workspace_layout(shape, P).total)
            return static_cast<int>(TA_ERR_WORKSPACE);
        if (!aligned(workspace, 16)) return static_cast<int>(TA_ERR_ALIGN);
        return static_cast<int>(TA_OK);
    };
    // With an explicit split count every argument is checked before any CUDA call.
    if (num_splits > 0 && (rc = check_ws(num_splits)) != TA_OK) return rc;

    DeviceState* ds = nullptr;
    rc = device_state(&ds);
    if (rc != TA_OK) return rc;

    int P = num_splits;
    if (P <= 0) {
        P = pick_splits_impl(shape, nullptr, ds->num_sms, kernel, paged ? paged->page_size : 0);
        if (!cluster && auto_cluster(ds, shape, kernel, P, paged ? paged->page_size : 0, options))
            cluster = true;
        if (cluster) P = std::min(P, kClusterMaxSplits);
        if (P < 1 || P > TA_MAX_SPLITS) return TA_ERR_SPLITS;
        if ((rc = check_ws(P)) != TA_OK) return rc;
    }
    const WsLayout ws = workspace_layout(shape, P);

    const Geometry geo = geometry_of(shape, kernel, paged ? paged->page_size : 0, ds->num_sms);
    const int hb = geo.heads_per_block;
    const int rows = paged ? std::min(geo.tile_tokens, paged->page_size) : geo.tile_tokens;
    if (geo.tile_tokens / rows > 32) return TA_ERR_SHAPE;  // one producer lane per box
    CUtensorMap tk, tv;
    rc = encode_kv_map(ds->device, &tk, k_cache, shape, st, geo, paged, rows);
    if (rc != TA_OK) return rc;
    rc = encode_kv_map(ds->device, &tv, v_cache, shape, st, geo, paged, rows);
    if (rc != TA_OK) return rc;

    ta::SplitParams p;
    std::memset(&p, 0, sizeof p);
    if (options) {
        p.k_scale = options->k_scale;
        p.v_scale = options->v_scale;
    }
    p.q = q;
    p.q_is_bf16 = shape->q_dtype == TA_BF16;
    p.seqlens = seqlens;
    p.err = ds->err;
    p.B = shape->batch;
    p.Hq = shape->num_q_heads;
    p.Hkv = shape->num_kv_heads;
    p.G = shape->num_q_heads / shape->num_kv_heads;
    p.S = shape->max_seqlen;
    p.P = P;
    p.nq = nq;
    p.causal = causal ? 1 : 0;
    const float scale = shape->scale > 0.f ? shape->scale
                                           : 1.0f / std::sqrt(static_cast<float>(shape->head_dim));
    p.scale_log2 = scale * ta::kLog2e;
    p.chunk_tiles = std::max(1, kChunkTokens / geo.tile_tokens);
    p.prefetch_tiles = std::max(1, (kernel == kKernelFp8 || kernel == kKernelTc05Fp8 ? kPrefetchTokensFp8
                                    : kernel == TA_KERNEL_TC05 ? kPrefetchTokensTc05
                                                               : kPrefetchTokens) /
                                       geo.tile_tokens);
    p.box_rows = rows;
    p.hb = hb;
    p.stall = (options && (options->flags & TA_FLAG_DIAG_STALL)) ? 1 : 0;
    p.mishint = (options && (options->flags & TA_FLAG_DIAG_MISHINT)) ? 1 : 0;
    p.num_pages = shape->batch;
    if (paged) {
        p.block_table = paged->block_table;
        p.max_pages = paged->max_pages_per_seq;
        p.num_pages = paged->num_pages;
        int sh = 0;
        while ((1 << sh) < paged->page_size) ++sh;
        p.page_shift = sh;
    }
    p.out = out;
    p.lse = lse;
    p.rows = static_cast<size_t>(shape->batch) * shape->num_q_heads;
    p.q_elems = p.rows * shape->head_dim;
    p.out_elems = p.q_elems;
    p.part_rows = P > 1 ? p.rows * P : 0;
    p.bt_elems = paged ? static_cast<size_t>(shape->batch) * paged->max_pages_per_seq : 0;
    bool fused = false;
    if (P > 1) {
        char* w = static_cast<char*>(workspace);
        p.part_o = reinterpret_cast<float*>(w + ws.o);
        p.part_m = reinterpret_cast<float*>(w + ws.m);
        p.part_l = reinterpret_cast<float*>(w + ws.l);
        const unsigned rows = static_cast<unsigned>(shape->batch) * (shape->num_kv_heads / hb);
        unsigned* slots = reserve_slots(ds, 2 * rows);
        if (slots) {
            // Run-time balancing pays while the grid is a few waves at most; with
            // more waves the block scheduler balances and claims only add latency.
            const int64_t blocks = static_cast<int64_t>(rows) * P;
            const int64_t resident = static_cast<int64_t>(ds->num_sms) * blocks_per_sm(shape, kernel);
            if (!deterministic && blocks <= kBalanceMaxWaves * resident) p.claim = slots;
            if (!cluster) {
                fused = fuse_merge(hb * p.G, P);
                p.fuse = fused ? 1 : 0;
                if (p.claim || fused) p.done = slots + rows;
            }
        }
        if (cluster) {  // the row's blocks merge through the cluster: no ticket, no combine
            p.cluster = 1;
            fused = true;
        }
    }

    if (options && options->split_start_event &&
        cudaEventRecord(static_cast<cudaEvent_t>(options->split_start_event), stream) != cudaSuccess)
        return TA_ERR_CUDA;
    cudaError_t e;
    if (kernel == kKernelFp8)
        e = ta::launch_split_fp8(tk, tv, p, stream);
    else if (kernel == TA_KERNEL_TC05)
        e = ta::launch_split_tc05(tk, tv, p, stream);
    else if (kernel == kKernelTc05Fp8)
        e = ta::launch_split_tc05_fp8(tk, tv, p, stream);
    else if (kernel == TA_KERNEL_MMA)
        e = ta::launch_split_mma(shape->head_dim, tk, tv, p, stream);
    else if (shape->kv_dtype == TA_BF16)
        e = ta::launch_split_fma_bf16(shape->head_dim, tk, tv, p, stream);
    else
        e = ta::launch_split_fma_f32(shape->head_dim, tk, tv, p, stream);
    if (e != cudaSuccess) return TA_ERR_CUDA;
    if (options && options->split_end_event &&
        cudaEventRecord(static_cast<cudaEvent_t>(options->split_end_event), stream) != cudaSuccess)
        return TA_ERR_CUDA;
    if (P > 1 && !fused) {
        e = ta::launch_combine(shape->head_dim, p.part_o, p.part_m, p.part_l, out, lse,
                               shape->batch, shape->num_q_heads, P, /*dependent=*/true, stream);
        if (e != cudaSuccess) return TA_ERR_CUDA;
    }
    return TA_OK;
}

}  // namespace

extern "C" {

const char* tree_attn_status_string(int status) {
    switch (status) {
        case TA_OK: return "ok";
        case TA_ERR_NULL: return "a required pointer is NULL";
        case TA_ERR_ALIGN: return "a pointer or stride is not 16-byte aligned";
        case TA_ERR_SHAPE: return "unsupported or inconsistent sizes";
        case TA_ERR_DTYPE: return "unsupported dtype combination";
        case TA_ERR_SPLITS: return "num_splits outside [1, TA_MAX_SPLITS]";
        case TA_ERR_WORKSPACE: return "workspace missing or too small";
        case TA_ERR_CUDA: return "a CUDA call failed";
        case TA_ERR_DEVICE_DATA: return "a sequence length outside [0, max_seqlen] was found on the device";
        case TA_ERR_DEVICE_TIMEOUT: return "an on-chip wait timed out";
        case TA_ERR_DEVICE_BOUNDS:
            return "an index outside its buffer was caught on the device (bounds-checking build)";
        case TA_ERR_SCRATCH_LIMIT:
            return "the partial states need more than the no-allocation scratch buffer holds "
                   "(TA_NOALLOC_SCRATCH_BYTES); use fewer splits or tree_attn_decode with a workspace";
        default: return "unknown status";
    }
}

int tree_attn_version(void) { return TREE_ATTN_VERSION; }

int tree_attn_check_shape(const ta_shape* shape) {
    const int rc = check_shape(shape, nullptr);
    if (rc != TA_OK) return rc;
    const int kernel = resolve_kernel(shape, TA_KERNEL_AUTO);
    return kernel < 0 ? kernel : TA_OK;
}

size_t tree_attn_workspace_bytes(const ta_shape* shape, int num_splits) {
    if (check_shape(shape, nullptr) != TA_OK) return 0;
    if (num_splits <= 1 || num_splits > TA_MAX_SPLITS) return 0;
    return workspace_layout(shape, num_splits).total;
}

int tree_attn_pick_splits_paged(const ta_shape* shape, int page_size, const int32_t* host_seqlens,
                                int num_sms) {
    const int rc = check_shape(shape, nullptr);
    if (rc != TA_OK) return rc;
    if (page_size > 0 && (page_size < 16 || page_size > 1024 || (page_size & (page_size - 1)) != 0))
        return TA_ERR_SHAPE;
    const int kernel = resolve_kernel(shape, TA_KERNEL_AUTO);
    if (kernel < 0) return kernel;
    if (num_sms <= 0) {
        DeviceState* ds = nullptr;
        const int r = device_state(&ds);
        if (r != TA_OK) return r;
        num_sms = ds->num_sms;
    }
    return pick_splits_impl(shape, host_seqlens, num_sms, kernel, page_size > 0 ? page_size : 0);
}

int tree_attn_pick_splits(const ta_shape* shape, const int32_t* host_seqlens, int num_sms) {
    return tree_attn_pick_splits_paged(shape, 0, host_seqlens, num_sms);
}

int tree_attn_decode_ex(const ta_shape* shape, const void* q, const void* k_cache,
                        const void* v_cache, const int32_t* seqlens, float* out, float* lse,
                        int num_splits, void* workspace, size_t workspace_bytes,
                        const ta_options* options, void* stream) {
    return decode_impl(shape, nullptr, 1, 0, q, k_cache, v_cache, seqlens, out, lse, num_splits,
                       workspace, workspace_bytes, options, stream);
}

int tree_attn_decode_paged(const ta_shape* shape, const ta_paged_kv* paged, const void* q,
                           const void* k_pages, const void* v_pages, const int32_t* seqlens,
                           float* out, float* lse, int num_splits, void* workspace,
                           size_t workspace_bytes, const ta_options* options, void* stream) {
    if (!paged) return TA_ERR_NULL;
    return decode_impl(shape, paged, 1, 0, q, k_pages, v_pages, seqlens, out, lse, num_splits,
                       workspace, workspace_bytes, options, stream);
}

int tree_attn_decode_multi(const ta_shape* shape, const ta_paged_kv* paged, int num_queries,
                           int causal, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* seqlens, float* out, float* lse, int num_splits,
                           void* workspace, size_t workspace_bytes, const ta_options* options,
                           void* stream) {
    if (!shape) return TA_ERR_NULL;
    if (num_queries < 1 || num_queries > 16) return TA_ERR_SHAPE;
    if (static_cast<int64_t>(shape->num_q_heads) * num_queries > (1 << 30)) return TA_ERR_SHAPE;
    ta_shape eff = *shape;  // each (head, query) pair is a query head of the cache
    eff.num_q_heads = shape->num_q_heads * num_queries;
    return decode_impl(&eff, paged, num_queries, causal, q, k_cache, v_cache, seqlens, out, lse,
                       num_splits, workspace, workspace_bytes, options, stream);
}

int tree_attn_launch_count(const ta_shape* shape, int num_splits, const ta_options* options) {
    int rc = check_shape(shape, nullptr);
    if (rc != TA_OK) return rc;
    if (options && (options->flags & ~kKnownFlags) != 0) return TA_ERR_SHAPE;
    const int kernel = resolve_kernel(shape, options ? options->kernel : TA_KERNEL_AUTO,
                                      options && (options->flags & TA_FLAG_CLUSTER_MERGE));
    if (kernel < 0) return kernel;
    int P = num_splits;
    if (P > TA_MAX_SPLITS) return TA_ERR_SPLITS;
    if (P <= 0) {
        DeviceState* ds = nullptr;
        if ((rc = device_state(&ds)) != TA_OK) return rc;
        P = pick_splits_impl(shape, nullptr, ds->num_sms, kernel, 0);
    }
    if (P == 1) return 1;
    if (options && (options->flags & TA_FLAG_CLUSTER_MERGE)) return 1;
    const int64_t G = shape->num_q_heads / shape->num_kv_heads;
    const unsigned rows = static_cast<unsigned>(shape->batch) * shape->num_kv_heads;
    const bool have_slots = 2 * static_cast<uint64_t>(rows) <= kRingSlots;
    return (have_slots && fuse_merge(static_cast<int>(G), P)) ? 1 : 2;
}

int tree_attn_decode(const ta_shape* shape, const void* q, const void* k_cache,
                     const void* v_cache, const int32_t* seqlens, float* out, float* lse,
                     int num_splits, void* workspace, size_t workspace_bytes, void* stream) {
    return tree_attn_decode_ex(shape, q, k_cache, v_cache, seqlens, out, lse, num_splits,
                               workspace, workspace_bytes, nullptr, stream);
}

int tree_attn_combine(const ta_shape* shape, const float* partial_o, const float* partial_m,
                      const float* partial_l, int num_splits, float* out, float* lse,
                      void* stream) {
    if (!shape) return TA_ERR_NULL;
    if (shape->batch < 1 || shape->num_q_heads < 1) return TA_ERR_SHAPE;
    if (shape->head_dim != 64 && shape->head_dim != 128) return TA_ERR_SHAPE;
    if (num_splits < 1 || num_splits > TA_MAX_SPLITS) return TA_ERR_SPLITS;
    if (!partial_o || !partial_m || !partial_l || !out) return TA_ERR_NULL;
    if (!aligned(partial_o, 16) || !aligned(out, 16) || !aligned(partial_m, 4) ||
        !aligned(partial_l, 4) || (lse && !aligned(lse, 4)))
        return TA_ERR_ALIGN;
    if (shape->batch > 65535) return TA_ERR_SHAPE;
    const cudaError_t e =
        ta::launch_combine(shape->head_dim, partial_o, partial_m, partial_l, out, lse, shape->batch,
                           shape->num_q_heads, num_splits, false, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TA_OK : TA_ERR_CUDA;
}

int tree_attn_get_device_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TA_ERR_CUDA;
    DeviceState* ds = nullptr;
    const int rc = device_state(&ds);
    if (rc != TA_OK) return rc;
    int h = 0;
    if (cudaMemcpy(&h, ds->err, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return TA_ERR_CUDA;
    if (h == 0) return TA_OK;
    const int zero = 0;
    if (cudaMemcpy(ds->err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
        return TA_ERR_CUDA;
    if (h & ta::kErrCounters) {
        // A copy warp outlived its bounded hand-over to the row's ticket, so
        // some counters may be off zero.  Only then is the ring cleared, after
        // every stream of the device has drained (no call may be enqueued
        // from another host thread meanwhile).
        if (cudaDeviceSynchronize() != cudaSuccess) return TA_ERR_CUDA;
        if (cudaMemset(ds->ring, 0, sizeof(unsigned) * kRingSlots) != cudaSuccess) return TA_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return TA_ERR_CUDA;
    }
    if (h & (ta::kErrTimeout | ta::kErrCounters)) return TA_ERR_DEVICE_TIMEOUT;
    if (h & ta::kErrBounds) return TA_ERR_DEVICE_BOUNDS;
    return TA_ERR_DEVICE_DATA;
}

}  // extern "C"
