/*
 * tree_attn.h -- C ABI of libtreeattn.so: exact single-query (decode) softmax
 * attention over a long KV cache, computed Tree Attention's way on one GPU.
 *
 * The method (web pages on Tree Attention, arXiv:2408.04093; "Tree Attention
 * Guide: Topology-Aware LLM Decoding"):
 *  - "Local Independent Partial Attention": the sequence axis is cut into P
 *    slices; each slice i yields a partial state T_i = (o_i, l_i, m_i) with
 *    m_i = max(q K_i^T), l_i = sum exp(q K_i^T - m_i),
 *    o_i = sum exp(q K_i^T - m_i) V_i (logits scaled by 1/sqrt(d), as in the
 *    page's implementation listing).
 *  - "The Tree Reduction Merge Operator": states merge by
 *    m = max(m_A, m_B), alpha = exp(m_A - m), beta = exp(m_B - m),
 *    l = alpha l_A + beta l_B, o = alpha o_A + beta o_B; the operator is
 *    associative and commutative, so any tree shape gives the same result.
 *  - Root normalisation: O = o_root / l_root.
 * Here the P slices become P thread blocks per (batch row, KV head) and the
 * tree is an on-chip reduction (lanes -> warps -> blocks) instead of a
 * reduction across devices.
 *
 * Conventions for every entry point:
 *  - All pointers named "device" are CUDA device (or managed) memory owned by
 *    the caller.  The library allocates nothing and frees nothing.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Work is enqueued asynchronously on it; no call synchronises
 *    except tree_attn_get_device_error.
 *  - Argument errors are detected on the host, before anything is enqueued,
 *    and returned as a negative ta_status.  A launch failure returns
 *    TA_ERR_CUDA.  Invalid data found on the device (a sequence length outside
 *    [0, max_seqlen]) never traps: the affected rows become NaN and an error
 *    word is set, reported by tree_attn_get_device_error.
 *  - Outputs `out` and `lse` are fully overwritten; inputs are never written.
 *  - The library sets itself up once per device and process, the first time
 *    it is called with that device current: it looks up the device addresses
 *    of its own fixed buffers (error word, scheduling counters, the
 *    no-allocation scratch) and raises its kernels' shared-memory limits.
 *    That set-up does not survive cudaDeviceReset: after resetting a device,
 *    a process must not call the library on that device again.
 */
#ifndef TREE_ATTN_H
#define TREE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TREE_ATTN_VERSION 1

/* Status codes (0 = success). */
typedef enum {
    TA_OK = 0,
    TA_ERR_NULL = -1,          /* a required pointer is NULL */
    TA_ERR_ALIGN = -2,         /* a pointer or stride breaks the 16-byte rule */
    TA_ERR_SHAPE = -3,         /* unsupported or inconsistent sizes */
    TA_ERR_DTYPE = -4,         /* unsupported dtype combination */
    TA_ERR_SPLITS = -5,        /* num_splits outside [1, TA_MAX_SPLITS] */
    TA_ERR_WORKSPACE = -6,     /* workspace missing or too small */
    TA_ERR_CUDA = -7,          /* a CUDA runtime/driver call failed */
    TA_ERR_DEVICE_DATA = -8,   /* device found a sequence length outside [0, max_seqlen] */
    TA_ERR_DEVICE_TIMEOUT = -9, /* a bounded on-chip wait gave up (outputs are NaN) */
    TA_ERR_SCRATCH_LIMIT = -10, /* tree_attn_decode_noalloc: the partial states need more than
                                   TA_NOALLOC_SCRATCH_BYTES */
    TA_ERR_DEVICE_BOUNDS = -11  /* bounds-checking build only (compiled with TA_DEBUG_BOUNDS):
                                   a kernel caught an index outside its buffer and skipped
                                   the access; the outputs are not to be trusted */
} ta_status;

/* Element types. */
typedef enum {
    TA_F32 = 0,   /* IEEE binary32 */
    TA_BF16 = 1,  /* bfloat16 (upper half of a binary32) */
    TA_E4M3 = 2   /* FP8 E4M3 ("fn": no infinities), KV caches only; the element
                     value is the code times a per-KV-head scale given in
                     ta_options (k_scale, v_scale).  Needs BF16 q, head_dim 128
                     and at most 16 query heads (x queries) per KV head. */
} ta_dtype;

/* Largest accepted num_splits. */
#define TA_MAX_SPLITS 4096

/* Sizes and layout of one decode-attention call.
 *
 *  q       [batch][num_q_heads][head_dim], dense, dtype q_dtype.
 *  k_cache, v_cache: element (b, g, t, i) of KV head g, token t, channel i is
 *          at  b*kv_stride_b + g*kv_stride_h + t*kv_stride_t + i  (elements,
 *          dtype kv_dtype).  All three strides 0 selects the dense layout
 *          [batch][num_kv_heads][max_seqlen][head_dim].  A token-major layout
 *          [batch][max_seqlen][num_kv_heads][head_dim] is expressed with
 *          kv_stride_t = num_kv_heads*head_dim, kv_stride_h = head_dim.
 *          Every stride times the element size must be a multiple of 16 bytes.
 *  Query head h reads KV head h / (num_q_heads / num_kv_heads).
 */
typedef struct {
    int32_t batch;          /* B >= 1 */
    int32_t num_q_heads;    /* Hq >= 1 */
    int32_t num_kv_heads;   /* Hkv >= 1, Hq % Hkv == 0, 1 <= Hq/Hkv <= 16 (a power of two
                               unless q and the cache are BF16); up to 64 with BF16 q
                               and cache at head_dim 128 */
    int32_t head_dim;       /* d: 64 or 128 */
    int32_t max_seqlen;     /* S: cache capacity per sequence, tokens (>= 1) */
    int32_t q_dtype;        /* ta_dtype */
    int32_t kv_dtype;       /* ta_dtype */
    float scale;            /* logit scale; 0 selects 1/sqrt(head_dim) */
    int64_t kv_stride_b;    /* elements; see above */
    int64_t kv_stride_h;
    int64_t kv_stride_t;
} ta_shape;

/* Kernel family for the per-slice step. */
typedef enum {
    TA_KERNEL_AUTO = 0,  /* tensor-core path when it applies, else FMA: TA_KERNEL_TC05 for
                            BF16 q at head_dim 128 with more than 16 columns (query heads x
                            queries) per KV head, on a BF16 cache (up to 64 columns) or an
                            E4M3 cache (up to 32), unless TA_FLAG_CLUSTER_MERGE is set;
                            else TA_KERNEL_MMA where it applies */
    TA_KERNEL_FMA = 1,   /* FP32 FMA on CUDA cores; every dtype combination */
    TA_KERNEL_MMA = 2,   /* warp-level tensor-core mma: BF16 q and kv (Hq/Hkv <= 16, or <= 64
                            at head_dim 128), or BF16 q with an E4M3 cache (Hq/Hkv <= 16,
                            head_dim 128) */
    TA_KERNEL_TC05 = 3   /* fifth-generation tensor cores (tcgen05.mma, accumulators in
                            tensor memory), BF16 q, head_dim 128: BF16 kv with Hq/Hkv <= 64
                            (x queries), or an E4M3 cache with Hq/Hkv <= 32 (x queries;
                            K used as E4M3 against q split into two E4M3 terms, V widened
                            to FP16); not with TA_FLAG_CLUSTER_MERGE */
} ta_kernel;

/* Bits of ta_options.flags. */
#define TA_FLAG_DETERMINISTIC 1  /* give slice p the fixed contiguous range [p*c, (p+1)*c) of
                                    its row instead of balancing the last eighth of the row
                                    between the row's blocks at run time: results are then
                                    bitwise reproducible for a given num_splits (balancing,
                                    used by default when the grid is at most four waves of
                                    blocks, changes the rounding order from run to run) */
#define TA_FLAG_DIAG_STALL 2     /* diagnostic, for testing the failure path: the copy warps
                                    publish no tile, so every compute warp's bounded wait
                                    gives up (after about two seconds); the call completes,
                                    its outputs are NaN and tree_attn_get_device_error
                                    returns TA_ERR_DEVICE_TIMEOUT.  Nothing faults or hangs,
                                    and the device stays usable. */
#define TA_FLAG_CLUSTER_MERGE 8  /* the row's num_splits (2..8) thread blocks run as one
                                    thread-block cluster and merge their partial states
                                    through the cluster's distributed shared memory instead
                                    of the last-arriving block reading them back from L2:
                                    a shorter step end for short contexts.  Tensor-core and
                                    FP8 kernels; a heuristic split count is capped at 8.
                                    Chosen without the flag for short rows when num_splits
                                    <= 0 (see tree_attn_decode) */
#define TA_FLAG_DIAG_MISHINT 4   /* diagnostic, for testing: the copy warps' length hint
                                    (used to start the first copies before the row length
                                    is read) is made wrong, so those copies are discarded
                                    and the step streams its real tiles after them; results
                                    are unchanged */

/* Optional per-call settings (pass NULL for defaults). */
typedef struct {
    int32_t kernel;            /* ta_kernel */
    int32_t flags;             /* TA_FLAG_* bits; other bits must be 0 */
    void *split_start_event;   /* optional cudaEvent_t recorded on `stream` just before the
                                  per-slice kernel is enqueued */
    void *split_end_event;     /* optional cudaEvent_t recorded just after it (before the combine) */
    const float *k_scale;      /* device float [num_kv_heads]: required for TA_E4M3 caches */
    const float *v_scale;      /* device float [num_kv_heads]: required for TA_E4M3 caches */
} ta_options;

/* Text for a status code (static storage; never NULL). */
const char *tree_attn_status_string(int status);

/* Library ABI version (TREE_ATTN_VERSION). */
int tree_attn_version(void);

/* Validate a shape (sizes, dtypes, strides) without touching any pointer.
 * Returns TA_OK or the error tree_attn_decode would return for it. */
int tree_attn_check_shape(const ta_shape *shape);

/* Bytes of device workspace tree_attn_decode needs for `num_splits` slices:
 * partial o [B][Hq][P][d], partial m and l [B][Hq][P], FP32, each region
 * 256-byte aligned.  0 when num_splits == 1 (no partial states are stored)
 * and 0 for an invalid shape or num_splits (see tree_attn_check_shape). */
size_t tree_attn_workspace_bytes(const ta_shape *shape, int num_splits);

/* Split-count heuristic ("Core Innovation 1": the P-way partition of the
 * sequence axis).  Picks P so that the B*Hkv*P thread blocks fill the GPU's
 * `num_sms` multiprocessors in whole waves with slices of >= 256 tokens,
 * trading the combine's cost against wave quantisation.  `host_seqlens`
 * ([batch], host memory) may be NULL, in which case every row is assumed to
 * hold max_seqlen tokens.  num_sms <= 0 queries the current CUDA device.
 * Returns P in [1, TA_MAX_SPLITS], or a negative ta_status. */
int tree_attn_pick_splits(const ta_shape *shape, const int32_t *host_seqlens, int num_sms);

/* The same heuristic for a paged cache of `page_size`-token pages (the value
 * tree_attn_decode_paged and tree_attn_decode_multi use when called with
 * num_splits <= 0).  With 16-token pages one thread block may serve several
 * KV heads of a row (each copy then brings the same tokens of all of them:
 * FP8 caches, and BF16 caches in token-major pools; with more than 8 columns
 * per KV head only where that needs no more slices), which changes the block
 * count and so the best P.  page_size <= 0 is the dense heuristic.  Returns P
 * or a negative ta_status. */
int tree_attn_pick_splits_paged(const ta_shape *shape, int page_size, const int32_t *host_seqlens,
                                int num_sms);

/* One decode-attention step: out[b][h][:] = softmax(scale q K^T) V over the
 * tokens [0, seqlens[b]) of row b, and lse[b][h] = log sum exp of the scaled
 * logits (natural log).  The sequence axis of each (b, KV head) is cut into
 * `num_splits` contiguous slices; every slice yields a partial state and the
 * states are merged by the operator above (partial m in natural-log units),
 * then normalised.  A row with seqlens[b] == 0 gives out = 0, lse = -inf.
 *
 *  shape       sizes/layout (host memory, read during the call only)
 *  q, k_cache, v_cache   device, 16-byte aligned; strides as in ta_shape
 *  seqlens     device int32 [batch], each in [0, max_seqlen]
 *  out         device float32 [batch][num_q_heads][head_dim]
 *  lse         device float32 [batch][num_q_heads], or NULL to skip it
 *  num_splits  P >= 1, or <= 0 to use tree_attn_pick_splits(shape, NULL, 0).
 *              With <= 0 the library also picks the merge: when P >= 2, the
 *              kernel has the cluster merge (BF16 tensor-core kernel up to 16
 *              columns, FP8 kernel), slices of min(P, 8) blocks would hold at
 *              most 640 tokens (768 for FP8 caches) and every row's cluster
 *              fits on the device at once, the row's min(P, 8) blocks merge as
 *              with TA_FLAG_CLUSTER_MERGE (not with the diagnostic flags).  The
 *              workspace for the heuristic's P is then more than enough.
 *  workspace   device, >= tree_attn_workspace_bytes(shape, P) bytes, 16-byte
 *              aligned; may be NULL when P == 1.  Contents on entry are
 *              ignored; calls sharing one workspace must be ordered on the GPU.
 *  stream      cudaStream_t as void*
 */
int tree_attn_decode(const ta_shape *shape, const void *q, const void *k_cache,
                     const void *v_cache, const int32_t *seqlens, float *out, float *lse,
                     int num_splits, void *workspace, size_t workspace_bytes, void *stream);

/* Number of kernels tree_attn_decode_ex enqueues for this shape, split count
 * and options: 1 when the partial states are merged inside the per-slice
 * kernel (num_splits == 1, or num_splits <= 40), else 2 (the per-slice
 * kernel, then the combine).  num_splits <= 0 queries the current
 * device for the heuristic's choice.  Negative ta_status on invalid input. */
int tree_attn_launch_count(const ta_shape *shape, int num_splits, const ta_options *options);

/* tree_attn_decode with per-call options (kernel family, timing events). */
int tree_attn_decode_ex(const ta_shape *shape, const void *q, const void *k_cache,
                        const void *v_cache, const int32_t *seqlens, float *out, float *lse,
                        int num_splits, void *workspace, size_t workspace_bytes,
                        const ta_options *options, void *stream);

/* Paged KV cache: the K and V caches are pools of fixed-size pages, and a
 * block table maps each sequence's logical pages to physical pages (the
 * layout of paged-attention serving engines).  Token t of batch row b lives
 * in physical page block_table[b][t / page_size] at position t % page_size.
 * With this, ta_shape's strides describe one pool: element (page, t_in_page,
 * g, i) is at page*kv_stride_b + t_in_page*kv_stride_t + g*kv_stride_h + i;
 * all three 0 select [num_pages][page_size][num_kv_heads][head_dim]. */
typedef struct {
    const int32_t *block_table;  /* device int32 [batch][max_pages_per_seq] */
    int32_t max_pages_per_seq;   /* columns of block_table; max_seqlen <= this * page_size */
    int32_t page_size;           /* tokens per page: a power of two in [16, 1024] */
    int32_t num_pages;           /* pages in each pool */
    int32_t reserved;            /* must be 0 */
} ta_paged_kv;

/* tree_attn_decode over a paged KV cache.  `k_pages`, `v_pages`: device,
 * 16-byte aligned pools of `paged->num_pages` pages laid out as described
 * above.  Block-table entries of pages that hold valid tokens must be in
 * [0, num_pages); an entry outside that range reads zeros, sets the device
 * error word (TA_ERR_DEVICE_DATA from tree_attn_get_device_error) and makes
 * that row NaN.  Entries past a row's last page are never read.  Results are
 * those of tree_attn_decode on the gathered cache (bitwise equal with
 * TA_FLAG_DETERMINISTIC at the same num_splits). */
int tree_attn_decode_paged(const ta_shape *shape, const ta_paged_kv *paged, const void *q,
                           const void *k_pages, const void *v_pages, const int32_t *seqlens,
                           float *out, float *lse, int num_splits, void *workspace,
                           size_t workspace_bytes, const ta_options *options, void *stream);

/* Several queries per sequence (multi-query decode, e.g. verifying draft
 * tokens): query i of batch row b sits at position seqlens[b] - num_queries + i.
 * With `causal` != 0 it attends to tokens [0, seqlens[b] - num_queries + i];
 * otherwise every query attends to all seqlens[b] tokens.  A query that sees
 * no token gives out = 0, lse = -inf.
 *  q    device [batch][num_q_heads][num_queries][head_dim], dtype q_dtype
 *  out  device float32 [batch][num_q_heads][num_queries][head_dim]
 *  lse  device float32 [batch][num_q_heads][num_queries], or NULL
 *  paged  NULL for dense caches, else as for tree_attn_decode_paged
 * Each (head, query) pair is handled as one query head of the KV group:
 * num_q_heads * num_queries / num_kv_heads must be at most 16 (a power of two
 * unless q and the cache are BF16; up to 64 with BF16 q and cache at head_dim
 * 128), and tree_attn_workspace_bytes,
 * tree_attn_pick_splits and tree_attn_launch_count take the shape with
 * num_q_heads multiplied by num_queries.  num_queries in [1, 16]. */
int tree_attn_decode_multi(const ta_shape *shape, const ta_paged_kv *paged, int num_queries,
                           int causal, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *seqlens, float *out, float *lse, int num_splits,
                           void *workspace, size_t workspace_bytes, const ta_options *options,
                           void *stream);

/* The tree combine on its own ("The Tree Reduction Merge Operator" applied to
 * P states per (b, h), then the root normalisation O = o / l):
 *
 *  partial_o  device float32 [batch][num_q_heads][num_splits][head_dim],
 *             unnormalised numerators
 *  partial_m  device float32 [batch][num_q_heads][num_splits], maxima in
 *             natural-log units of the scaled logits (-inf for an empty slice)
 *  partial_l  device float32 [batch][num_q_heads][num_splits], denominators
 *             (0 for an empty slice)
 *  out        device float32 [batch][num_q_heads][head_dim]
 *  lse        device float32 [batch][num_q_heads] or NULL
 * Only batch, num_q_heads and head_dim of `shape` are used; head_dim must be
 * 64 or 128.  All pointers 16-byte aligned.  All-empty rows give out = 0,
 * lse = -inf. */
int tree_attn_combine(const ta_shape *shape, const float *partial_o, const float *partial_m,
                      const float *partial_l, int num_splits, float *out, float *lse,
                      void *stream);

/* Size of the fixed device buffer behind tree_attn_decode_noalloc (8 MiB per
 * GPU that loads the library, held until the process exits). */
#define TA_NOALLOC_SCRATCH_BYTES (8u << 20)

/* tree_attn_decode for callers that must not allocate device memory.  The
 * Tree Attention pages have no counterpart to this; it is a deployment aid.
 *
 * Some callers cannot call cudaMalloc at decode time: an inference engine's
 * plugin whose device memory is planned before serving starts and whose
 * enqueue must not allocate, or a serving loop that cannot afford
 * cudaMalloc's implicit device-wide synchronisation.  This entry point takes
 * the same inputs and outputs as tree_attn_decode but keeps the partial states
 * in a buffer of TA_NOALLOC_SCRATCH_BYTES that the library reserves statically
 * on each device, so the caller passes no workspace and nothing is allocated.
 *
 *  - The first call on a device looks up that buffer's device address (a
 *    one-time set-up with that device current); make that first call before
 *    any stream capture begins.
 *  - Returns TA_ERR_SCRATCH_LIMIT, with nothing enqueued, when
 *    tree_attn_workspace_bytes(shape, P) exceeds TA_NOALLOC_SCRATCH_BYTES
 *    (P = num_splits, or the heuristic's choice when num_splits <= 0).
 *  - Every call on a device shares the one buffer and it keeps the previous
 *    call's contents.  Nothing in it needs to start at zero (every partial
 *    state is written before it is read), but calls whose work overlaps on
 *    the GPU (different streams without ordering) race on it: order them.
 * Other arguments, errors and results are as for tree_attn_decode. */
int tree_attn_decode_noalloc(const ta_shape *shape, const void *q, const void *k_cache,
                             const void *v_cache, const int32_t *seqlens, float *out, float *lse,
                             int num_splits, void *stream);

/* Synchronise `stream`, then read and clear the current device's error word.
 * Returns TA_OK, TA_ERR_DEVICE_DATA, TA_ERR_DEVICE_TIMEOUT or (bounds-checking
 * build) TA_ERR_DEVICE_BOUNDS, or TA_ERR_CUDA when the synchronisation itself
 * fails.
 *
 * The error word is one per device, shared by every call and stream: it
 * reports what any call since the last read found.  The library's scheduling
 * counters (a fixed per-device ring; each call uses its own slots) are back at
 * zero when a call ends, also after a wait gave up, so a timeout needs no
 * clean-up and calls running on other streams are not disturbed.  Only if a
 * block's copy warp did not end within its own bounded wait either (a second
 * timeout inside the same block) does this function synchronise the whole
 * device and clear the ring; no call may be enqueued from another host thread
 * while it does. */
int tree_attn_get_device_error(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TREE_ATTN_H */
