"""Host-side checks of libtreeattn.so that need no GPU: the library loads, exports
every entry point its header declares, validates arguments before touching
CUDA, sizes the workspace and picks split counts."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tree_attn.h")


@pytest.fixture(scope="module")
def ta():
    from softmax_tree_reduction_gb300 import build
    build.build()
    import softmax_tree_reduction_gb300 as mod
    mod.load()
    return mod


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(tree_attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("tree_attn_decode", "tree_attn_combine", "tree_attn_workspace_bytes",
              "tree_attn_pick_splits", "tree_attn_get_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(ta):
    lib = ctypes.CDLL(ta.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_status_strings(ta):
    assert ta.tree_attn_version() == 1
    for code in range(0, -10, -1):
        s = ta.tree_attn_status_string(code)
        assert s and s != "unknown status"
    assert ta.tree_attn_status_string(-77) == "unknown status"


def shape(ta, **kw):
    base = dict(batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128, max_seqlen=131072,
                q_dtype=1, kv_dtype=1, scale=0.0, kv_stride_b=0, kv_stride_h=0, kv_stride_t=0)
    base.update(kw)
    return ta.TaShape(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(), 0),
    (dict(num_q_heads=12, num_kv_heads=8), -3),      # Hq % Hkv != 0
    (dict(num_q_heads=24, num_kv_heads=8), 0),       # G = 3: tensor-core kernel (BF16)
    (dict(num_q_heads=24, num_kv_heads=8, q_dtype=0, kv_dtype=0), -3),   # G = 3 without BF16: no kernel
    (dict(num_q_heads=128, num_kv_heads=4), 0),      # G = 32: BF16 column groups
    (dict(num_q_heads=256, num_kv_heads=2), -3),     # G = 128 unsupported
    (dict(num_q_heads=128, num_kv_heads=4, head_dim=64), -3),  # G > 16 needs head_dim 128
    (dict(num_q_heads=128, num_kv_heads=4, q_dtype=0, kv_dtype=0), -3),  # FMA: G <= 16
    (dict(head_dim=96), -3),
    (dict(batch=0), -3),
    (dict(max_seqlen=0), -3),
    (dict(q_dtype=2), -4),
    (dict(kv_dtype=7), -4),
    (dict(kv_dtype=2), 0),                            # FP8 cache, BF16 q, d128, G=4
    (dict(kv_dtype=2, q_dtype=0), -4),                # FP8 needs BF16 q
    (dict(kv_dtype=2, head_dim=64), -4),              # FP8 path is d = 128
    (dict(kv_dtype=2, num_q_heads=128), 0),           # FP8 path: G = 16 (two n-tiles)
    (dict(kv_dtype=2, num_q_heads=256), 0),           # FP8 on tcgen05: G = 32
    (dict(kv_dtype=2, num_q_heads=512), -3),          # FP8: G = 64 unsupported
    (dict(scale=-1.0), -3),
    (dict(scale=float("nan")), -3),
    (dict(kv_stride_b=131072 * 8 * 128, kv_stride_h=128, kv_stride_t=8 * 128), 0),  # token-major
    (dict(kv_stride_b=104, kv_stride_h=128, kv_stride_t=1024), 0),
    (dict(kv_stride_b=100, kv_stride_h=128, kv_stride_t=1024), -2),  # 200 B not 16-aligned
    (dict(kv_stride_b=1000, kv_stride_h=129, kv_stride_t=1024), -2),   # 258 B not 16-aligned
    (dict(kv_stride_b=1, kv_stride_h=0, kv_stride_t=1024), -3),
])
def test_check_shape(ta, kw, code):
    assert ta.tree_attn_check_shape(shape(ta, **kw)) == code


def test_workspace_bytes_layout(ta):
    s = shape(ta)
    assert ta.tree_attn_workspace_bytes(s, 1) == 0
    assert ta.tree_attn_workspace_bytes(s, 0) == 0
    assert ta.tree_attn_workspace_bytes(s, 5000) == 0
    for P in (2, 19, 64, 4096):
        rows = 1 * 32 * P
        r256 = lambda x: (x + 255) // 256 * 256
        assert ta.tree_attn_workspace_bytes(s, P) == r256(rows * 128 * 4) + 2 * r256(rows * 4)


def test_pick_splits_fills_whole_waves(ta):
    # 8 (b, kv-head) rows on 152 SMs: 19 slices give exactly one wave of 152 blocks
    assert ta.tree_attn_pick_splits(shape(ta), None, 152) == 19
    # 32 rows (4 x 8): 19 slices give 608 blocks = 4 full waves
    assert ta.tree_attn_pick_splits(shape(ta, batch=4, num_q_heads=64, max_seqlen=262144), None, 152) == 19
    # a different SM count moves the choice with it: the largest single wave
    for sms in (132, 148, 160):
        assert ta.tree_attn_pick_splits(shape(ta), None, sms) == sms // 8


def test_pick_splits_bounds(ta):
    for n in (1, 100, 255, 256, 257, 4096, 65536, 1 << 20):
        P = ta.tree_attn_pick_splits(shape(ta, max_seqlen=n), None, 152)
        assert 1 <= P <= max(1, math.ceil(n / 256))
    assert ta.tree_attn_pick_splits(shape(ta, max_seqlen=64), [0], 152) == 1


def test_pick_splits_ragged_uses_lengths(ta):
    from softmax_tree_reduction_gb300 import workloads
    sl = workloads.seqlens_of(workloads.BATCHED_RAGGED)
    s = shape(ta, batch=16, max_seqlen=65536)
    P = ta.tree_attn_pick_splits(s, sl, 152)
    assert P == 5   # the best of a measured sweep on GB300 (3..19)
    # all rows at the shortest length: the uniform model applies
    P2 = ta.tree_attn_pick_splits(s, np.full(16, 8192), 152)
    assert 1 <= P2 <= 32


def test_pick_splits_rejects_bad_shape(ta):
    with pytest.raises(ta.TreeAttnError):
        ta.tree_attn_pick_splits(shape(ta, head_dim=80), None, 152)


def _decode_raw(ta, s, q=0x1000, k=0x2000, v=0x3000, sl=0x4000, out=0x5000, lse=0x6000, P=1,
                ws=0, wsb=0, opts=None):
    lib = ta.load()
    vp = ctypes.c_void_p
    if opts is None:
        return lib.tree_attn_decode(ctypes.byref(s) if s is not None else None, vp(q), vp(k), vp(v),
                                    vp(sl), vp(out), vp(lse), P, vp(ws), wsb, vp(0))
    return lib.tree_attn_decode_ex(ctypes.byref(s), vp(q), vp(k), vp(v), vp(sl), vp(out), vp(lse),
                                   P, vp(ws), wsb, ctypes.byref(opts), vp(0))


def test_decode_argument_errors_before_any_cuda_call(ta):
    s = shape(ta)
    assert _decode_raw(ta, None) == -1
    assert _decode_raw(ta, s, q=0) == -1
    assert _decode_raw(ta, s, out=0) == -1
    assert _decode_raw(ta, s, sl=0) == -1
    assert _decode_raw(ta, s, k=0x2001) == -2
    assert _decode_raw(ta, s, out=0x5004) == -2
    assert _decode_raw(ta, s, P=5000) == -5
    assert _decode_raw(ta, s, P=4, ws=0, wsb=0) == -6
    need = ta.tree_attn_workspace_bytes(s, 4)
    assert _decode_raw(ta, s, P=4, ws=0x7000, wsb=need - 1) == -6
    assert _decode_raw(ta, s, P=4, ws=0x7008, wsb=need) == -2
    assert _decode_raw(ta, shape(ta, head_dim=32)) == -3
    f32 = shape(ta, q_dtype=0, kv_dtype=0)
    assert _decode_raw(ta, f32, opts=ta.TaOptions(2, 0, None, None, None, None)) == -4   # mma needs bf16
    assert _decode_raw(ta, shape(ta, num_q_heads=256, num_kv_heads=2),
                       opts=ta.TaOptions(2, 0, None, None, None, None)) == -3          # G = 128 > 64
    assert _decode_raw(ta, s, opts=ta.TaOptions(0, 16, None, None, None, None)) == -3  # unknown flag bit
    assert _decode_raw(ta, s, opts=ta.TaOptions(9, 0, None, None, None, None)) == -3  # unknown kernel


def test_combine_argument_errors(ta):
    lib = ta.load()
    vp = ctypes.c_void_p
    s = shape(ta)
    call = lambda s_, po=0x1000, pm=0x2000, pl=0x3000, P=4, out=0x4000, lse=0x5000: \
        lib.tree_attn_combine(ctypes.byref(s_), vp(po), vp(pm), vp(pl), P, vp(out), vp(lse), vp(0))
    assert call(s, po=0) == -1
    assert call(s, out=0) == -1
    assert call(s, P=0) == -5
    assert call(s, P=4097) == -5
    assert call(shape(ta, head_dim=100)) == -3
    assert call(s, po=0x1004) == -2
    assert call(s, pm=0x2002) == -2


def test_binding_refuses_cpu_tensors(ta):
    """Every entry point refuses host tensors before any work: there is no CPU
    fallback on the product path."""
    import torch
    q = torch.zeros(1, 1, 64)
    k = torch.zeros(1, 1, 8, 64)
    sl = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA device"):
        ta.tree_attn_decode(q, k, k, sl)
    with pytest.raises(ValueError, match="CUDA device"):
        ta.tree_attn_decode_multi(q[:, :, None, :], k, k, sl)
    pages = torch.zeros(4, 16, 1, 64)
    bt = torch.zeros(1, 4, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA device"):
        ta.tree_attn_decode_paged(q, pages, pages, bt, sl)
    with pytest.raises(ValueError, match="CUDA device"):
        ta.tree_attn_decode_noalloc(q, k, k, sl, torch.zeros(1, 1, 64))
    with pytest.raises(ValueError, match="CUDA device"):
        ta.tree_attn_combine(torch.zeros(1, 1, 2, 64), torch.zeros(1, 1, 2), torch.zeros(1, 1, 2))


def test_launch_count(ta):
    s = shape(ta)
    assert ta.tree_attn_launch_count(s, 1) == 1
    assert ta.tree_attn_launch_count(s, 19) == 1
    assert ta.tree_attn_launch_count(s, 40) == 1
    assert ta.tree_attn_launch_count(s, 41) == 2
    assert ta.tree_attn_launch_count(s, 4096) == 2
    with pytest.raises(ta.TreeAttnError):
        ta.tree_attn_launch_count(s, 5000)
    with pytest.raises(ta.TreeAttnError):
        ta.tree_attn_launch_count(shape(ta, head_dim=48), 4)


def test_paged_argument_errors(ta):
    lib = ta.load()
    vp = ctypes.c_void_p
    s = shape(ta, max_seqlen=4096)

    def call(pg, s_=s):
        return lib.tree_attn_decode_paged(ctypes.byref(s_), ctypes.byref(pg) if pg is not None else None,
                                          vp(0x1000), vp(0x2000), vp(0x3000), vp(0x4000), vp(0x5000),
                                          vp(0x6000), 1, vp(0), 0, None, vp(0))
    ok = dict(block_table=0x8000, max_pages_per_seq=64, page_size=64, num_pages=100, reserved=0)
    assert call(None) == -1
    assert call(ta.TaPagedKV(**{**ok, "block_table": 0})) == -1
    assert call(ta.TaPagedKV(**{**ok, "block_table": 0x8002})) == -2
    assert call(ta.TaPagedKV(**{**ok, "page_size": 24})) == -3
    assert call(ta.TaPagedKV(**{**ok, "page_size": 8})) == -3
    assert call(ta.TaPagedKV(**{**ok, "page_size": 2048})) == -3
    assert call(ta.TaPagedKV(**{**ok, "max_pages_per_seq": 63})) == -3   # 63*64 < 4096
    assert call(ta.TaPagedKV(**{**ok, "num_pages": 0})) == -3
    assert call(ta.TaPagedKV(**{**ok, "reserved": 1})) == -3


def test_fp8_needs_scales_before_any_cuda_call(ta):
    s = shape(ta, kv_dtype=2)
    assert _decode_raw(ta, s) == -1                                            # no options
    assert _decode_raw(ta, s, opts=ta.TaOptions(0, 0, None, None, None, None)) == -1
    assert _decode_raw(ta, s, opts=ta.TaOptions(1, 0, None, None, 0x100, 0x200)) == -4  # FMA: no FP8


def test_pick_splits_paged_small_pages_share_blocks(ta):
    """16-token pages let one block serve several KV heads (one copy per page
    brings all of them), so the heuristic spreads the row over more slices."""
    bf16 = shape(ta)                      # B1, 32/8 heads, d128, 131072 tokens
    fp8 = shape(ta, kv_dtype=2)
    for s in (bf16, fp8):
        for ps in (0, 64, 256, 1024):
            assert ta.tree_attn_pick_splits(s, None, 152, page_size=ps) == 19
    assert ta.tree_attn_pick_splits(bf16, None, 152, page_size=16) == 38   # 2 heads per block
    assert ta.tree_attn_pick_splits(bf16, None, 152, page_size=32) == 19
    # 4 heads per block would need 76 splits (a combine launch): 2 heads, 38 splits
    assert ta.tree_attn_pick_splits(fp8, None, 152, page_size=16) == 38
    assert ta.tree_attn_pick_splits(fp8, None, 152, page_size=32) == 19    # one head per block
    # B4, 64/8 heads: 4 heads per block keeps 19 splits (152 blocks)
    big = shape(ta, kv_dtype=2, batch=4, num_q_heads=64, max_seqlen=262144)
    assert ta.tree_attn_pick_splits(big, None, 152, page_size=16) == 19
    # head-major pools ([page][head][token][d]): FP8 still shares blocks, BF16 does not
    hnd8 = shape(ta, kv_dtype=2, kv_stride_b=8 * 16 * 128, kv_stride_h=16 * 128, kv_stride_t=128)
    assert ta.tree_attn_pick_splits(hnd8, None, 152, page_size=16) == 38
    hnd16 = shape(ta, kv_stride_b=8 * 16 * 128, kv_stride_h=16 * 128, kv_stride_t=128)
    assert ta.tree_attn_pick_splits(hnd16, None, 152, page_size=16) == 19
    # heads per block must divide the KV heads: 2 KV heads cap it at 2
    two = shape(ta, kv_dtype=2, num_q_heads=8, num_kv_heads=2)
    assert ta.tree_attn_pick_splits(two, None, 152, page_size=16) > ta.tree_attn_pick_splits(two, None, 152)
    for bad in (8, 24, 2048):
        with pytest.raises(ta.TreeAttnError):
            ta.tree_attn_pick_splits(fp8, None, 152, page_size=bad)


def test_pick_splits_paged_wide_groups(ta):
    """With 9..16 columns per KV head (two n-tiles) a block serves several KV
    heads only where that needs no more splits than one head per block."""
    # 8B-shaped, 4 queries per row: 16 columns per KV head; sharing would need 38 splits
    for kv in (1, 2):
        nq4 = shape(ta, kv_dtype=kv, num_q_heads=32 * 4)
        assert ta.tree_attn_pick_splits(nq4, None, 152, page_size=16) == 19
    # 70B-shaped B4, 2 queries: shared blocks keep 19 splits, so they stay
    for kv in (1, 2):
        big = shape(ta, kv_dtype=kv, batch=4, num_q_heads=64 * 2, max_seqlen=262144)
        assert ta.tree_attn_pick_splits(big, None, 152, page_size=16) == 19
    # 8 columns (one n-tile) still shares: 2 heads per block, 38 splits
    nq2 = shape(ta, num_q_heads=32 * 2)
    assert ta.tree_attn_pick_splits(nq2, None, 152, page_size=16) == 38


def test_cluster_merge_arguments(ta):
    s = shape(ta)
    f32 = shape(ta, q_dtype=0, kv_dtype=0)
    cl = ta.TA_FLAG_CLUSTER_MERGE
    assert _decode_raw(ta, s, P=9, ws=0x7000, wsb=1 << 30, opts=ta.TaOptions(0, cl, None, None, None, None)) == -5
    assert _decode_raw(ta, f32, P=4, ws=0x7000, wsb=1 << 30, opts=ta.TaOptions(1, cl, None, None, None, None)) == -3
    assert ta.tree_attn_launch_count(s, 8) == 1


def test_binding_shape_cache_validates_every_new_layout(ta):
    """The binding caches a validated descriptor per (shapes, strides, dtypes,
    scale); a call whose layout differs in any of them is validated afresh."""
    import torch
    from softmax_tree_reduction_gb300 import _binding as b
    q = torch.zeros(2, 8, 128, dtype=torch.bfloat16)
    k = torch.zeros(2, 2, 64, 128, dtype=torch.bfloat16)
    sl = torch.zeros(2, dtype=torch.int32)
    first = b._dense_shape(q, k, k.clone(), sl, None)
    assert b._dense_shape(q, k, k.clone(), sl, None) is first      # same layout: cached
    assert first[0].num_q_heads == 8 and first[0].num_kv_heads == 2 and first[0].max_seqlen == 64
    assert b._dense_shape(q, k, k.clone(), sl, 0.5) is not first   # the scale is part of the key
    with pytest.raises(ValueError):                                # V strided differently from K
        b._dense_shape(q, k, k.transpose(1, 2).contiguous().transpose(1, 2), sl, None)
    with pytest.raises(ValueError):                                # V of another dtype
        b._dense_shape(q, k, k.float(), sl, None)
    with pytest.raises(ValueError):                                # q with the same shape, not contiguous
        b._dense_shape(torch.zeros(2, 128, 8, dtype=torch.bfloat16).transpose(1, 2), k, k, sl, None)
    with pytest.raises(ValueError):                                # lengths must be int32
        b._dense_shape(q, k, k, sl.long(), None)
    # a token-major view is a new key with its strides in the descriptor
    kt = torch.zeros(2, 64, 2, 128, dtype=torch.bfloat16).transpose(1, 2)
    d = b._dense_shape(q, kt, kt, sl, None)[0]
    assert (d.kv_stride_b, d.kv_stride_h, d.kv_stride_t) == (64 * 2 * 128, 128, 2 * 128)


def _header_constants():
    """#define'd integer constants and enum values of the header, evaluated."""
    text = open(HEADER).read()
    consts = {}
    for name, expr in re.findall(r"^#define\s+(TA_\w+)\s+(.+?)\s*(?:/\*.*)?$", text, flags=re.M):
        expr = re.sub(r"(\d+)[uU]\b", r"\1", expr)
        if re.fullmatch(r"[\d\s()<>+\-*x]+", expr):
            consts[name] = int(eval(expr))
    for name, val in re.findall(r"^\s*(TA_\w+)\s*=\s*(-?\d+)", text, flags=re.M):
        consts[name] = int(val)
    return consts


def test_binding_constants_match_the_header(ta):
    """The Python binding's copies of the header's constants (scratch size,
    split limit, flag bits, status codes, dtype codes) equal the header's."""
    h = _header_constants()
    for name in ("TA_NOALLOC_SCRATCH_BYTES", "TA_MAX_SPLITS", "TA_FLAG_DETERMINISTIC", "TA_FLAG_DIAG_STALL",
                 "TA_FLAG_DIAG_MISHINT", "TA_FLAG_CLUSTER_MERGE", "TA_OK", "TA_ERR_DEVICE_DATA",
                 "TA_ERR_DEVICE_TIMEOUT", "TA_F32", "TA_BF16", "TA_E4M3"):
        assert name in h, name
        assert getattr(ta, name) == h[name], (name, getattr(ta, name), h[name])
    assert h["TA_NOALLOC_SCRATCH_BYTES"] == 8 << 20


def test_tc05_kernel_choice_and_limits(ta):
    """The tcgen05 kernels take BF16 q at head_dim 128 with up to 64 columns per
    KV head over a BF16 cache and up to 32 over an E4M3 cache (the automatic
    choice above 16 columns for both); they are refused
    (before any CUDA call) for other dtypes, head_dim 64, more columns, or
    together with the cluster merge."""
    wide = shape(ta, num_q_heads=256, num_kv_heads=8)       # 32 columns per KV head
    assert ta.tree_attn_launch_count(wide, 19, kernel="tc05") == 1
    assert ta.tree_attn_launch_count(wide, 64, kernel="tc05") == 2
    assert ta.tree_attn_launch_count(shape(ta), 19, kernel="tc05") == 1   # 4 columns, asked for
    fp8 = shape(ta, kv_dtype=ta.TA_E4M3)
    assert ta.tree_attn_launch_count(fp8, 19, kernel="tc05") == 1
    assert ta.tree_attn_launch_count(shape(ta, kv_dtype=ta.TA_E4M3, num_q_heads=256), 19) == 1   # 32 columns
    for bad, code in ((shape(ta, q_dtype=ta.TA_F32), -4), (shape(ta, head_dim=64), -3),
                      (shape(ta, kv_dtype=ta.TA_E4M3, q_dtype=ta.TA_F32), -4),
                      (shape(ta, kv_dtype=ta.TA_E4M3, num_q_heads=512), -3)):
        with pytest.raises(ta.TreeAttnError) as ei:
            ta.tree_attn_launch_count(bad, 8, kernel="tc05")
        assert ei.value.status == code
    lib = ta.load()
    opts = ta.TaOptions(ta.TA_KERNEL["tc05"], ta.TA_FLAG_CLUSTER_MERGE, None, None, None, None)
    assert lib.tree_attn_launch_count(ctypes.byref(wide), 4, ctypes.byref(opts)) == -3
    opts = ta.TaOptions(ta.TA_KERNEL["auto"], ta.TA_FLAG_CLUSTER_MERGE, None, None, None, None)
    assert lib.tree_attn_launch_count(ctypes.byref(wide), 4, ctypes.byref(opts)) == 1   # warp-level kernel
