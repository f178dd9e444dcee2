"""ctypes binding of libtreeattn.so (include/tree_attn.h), same names as the C ABI.

Argument marshalling only: tensors are checked and turned into pointers,
outputs and workspace are allocated with torch when the caller passes none,
and the call is enqueued on torch's current CUDA stream.  Every step of the
computation runs in the library's CUDA kernels; there is no CPU fallback, and
a missing library raises immediately.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# TREE_ATTN_LIBRARY selects another build of the library (e.g. the
# bounds-checking libtreeattn_debug.so); the default is the in-tree build.
LIB_PATH = os.environ.get("TREE_ATTN_LIBRARY") or os.path.join(_HERE, "libtreeattn.so")

TA_OK = 0
TA_ERR_DEVICE_DATA = -8      # a length or page-table entry outside its range (rows are NaN)
TA_ERR_DEVICE_TIMEOUT = -9   # a bounded on-chip wait gave up (outputs are NaN)
TA_ERR_DEVICE_BOUNDS = -11   # bounds-checking build: an index outside its buffer was caught
TA_F32, TA_BF16, TA_E4M3 = 0, 1, 2
TA_KERNEL = {"auto": 0, "fma": 1, "mma": 2, "tc05": 3}
TA_MAX_SPLITS = 4096
TA_FLAG_DETERMINISTIC = 1
TA_FLAG_DIAG_STALL = 2
TA_FLAG_DIAG_MISHINT = 4
TA_FLAG_CLUSTER_MERGE = 8
TA_CLUSTER_MAX_SPLITS = 8
TA_NOALLOC_SCRATCH_BYTES = 8 << 20

_EXPORTS = ["tree_attn_status_string", "tree_attn_version", "tree_attn_check_shape",
            "tree_attn_workspace_bytes", "tree_attn_pick_splits", "tree_attn_decode",
            "tree_attn_decode_ex", "tree_attn_combine", "tree_attn_get_device_error",
            "tree_attn_decode_noalloc", "tree_attn_launch_count", "tree_attn_decode_paged",
            "tree_attn_decode_multi", "tree_attn_pick_splits_paged"]


class TaShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("max_seqlen", ctypes.c_int32), ("q_dtype", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("scale", ctypes.c_float),
                ("kv_stride_b", ctypes.c_int64), ("kv_stride_h", ctypes.c_int64),
                ("kv_stride_t", ctypes.c_int64)]


class TaOptions(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("split_start_event", ctypes.c_void_p), ("split_end_event", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p)]


class TaPagedKV(ctypes.Structure):
    _fields_ = [("block_table", ctypes.c_void_p), ("max_pages_per_seq", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class TreeAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {tree_attn_status_string(status)} (status {status})")


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libtreeattn.so once; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m softmax_tree_reduction_gb300.build`")
        lib = ctypes.CDLL(path)
        P, SP, I32, SZ = ctypes.c_void_p, ctypes.POINTER(TaShape), ctypes.c_int, ctypes.c_size_t
        lib.tree_attn_status_string.argtypes = [I32]
        lib.tree_attn_status_string.restype = ctypes.c_char_p
        lib.tree_attn_version.argtypes = []
        lib.tree_attn_version.restype = I32
        lib.tree_attn_check_shape.argtypes = [SP]
        lib.tree_attn_check_shape.restype = I32
        lib.tree_attn_workspace_bytes.argtypes = [SP, I32]
        lib.tree_attn_workspace_bytes.restype = SZ
        lib.tree_attn_pick_splits.argtypes = [SP, P, I32]
        lib.tree_attn_pick_splits.restype = I32
        lib.tree_attn_pick_splits_paged.argtypes = [SP, I32, P, I32]
        lib.tree_attn_pick_splits_paged.restype = I32
        lib.tree_attn_decode.argtypes = [SP, P, P, P, P, P, P, I32, P, SZ, P]
        lib.tree_attn_decode.restype = I32
        lib.tree_attn_decode_ex.argtypes = [SP, P, P, P, P, P, P, I32, P, SZ,
                                            ctypes.POINTER(TaOptions), P]
        lib.tree_attn_decode_ex.restype = I32
        lib.tree_attn_combine.argtypes = [SP, P, P, P, I32, P, P, P]
        lib.tree_attn_combine.restype = I32
        lib.tree_attn_decode_noalloc.argtypes = [SP, P, P, P, P, P, P, I32, P]
        lib.tree_attn_decode_noalloc.restype = I32
        lib.tree_attn_decode_paged.argtypes = [SP, ctypes.POINTER(TaPagedKV), P, P, P, P, P, P, I32, P,
                                               SZ, ctypes.POINTER(TaOptions), P]
        lib.tree_attn_decode_paged.restype = I32
        lib.tree_attn_decode_multi.argtypes = [SP, ctypes.POINTER(TaPagedKV), I32, I32, P, P, P, P, P, P,
                                               I32, P, SZ, ctypes.POINTER(TaOptions), P]
        lib.tree_attn_decode_multi.restype = I32
        lib.tree_attn_launch_count.argtypes = [SP, I32, ctypes.POINTER(TaOptions)]
        lib.tree_attn_launch_count.restype = I32
        lib.tree_attn_get_device_error.argtypes = [P]
        lib.tree_attn_get_device_error.restype = I32
        _lib = lib
        return lib


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return TA_F32
    if dt == torch.bfloat16:
        return TA_BF16
    if dt == getattr(torch, "float8_e4m3fn", None):
        return TA_E4M3
    raise TypeError(f"unsupported dtype {dt}; use float32, bfloat16 or float8_e4m3fn (caches)")


def _options(kernel, deterministic, k_scale=None, v_scale=None, events=None, diag_stall=False,
             diag_mishint=False, cluster_merge=False):
    flags = ((TA_FLAG_DETERMINISTIC if deterministic else 0) | (TA_FLAG_DIAG_STALL if diag_stall else 0)
             | (TA_FLAG_DIAG_MISHINT if diag_mishint else 0) | (TA_FLAG_CLUSTER_MERGE if cluster_merge else 0))
    o = TaOptions(TA_KERNEL[kernel], flags, None, None, None, None)
    if events is not None:
        o.split_start_event = events[0].cuda_event
        o.split_end_event = events[1].cuda_event
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        if t is not None:
            if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous float32 CUDA tensor [num_kv_heads]")
            setattr(o, name, t.data_ptr())
    return o


def _ptr(t: Optional[torch.Tensor]):
    # a plain int (or None for NULL): the argtypes declare the pointers
    return t.data_ptr() if t is not None else None


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def make_shape(q: torch.Tensor, k_cache: torch.Tensor, scale: Optional[float] = None) -> TaShape:
    """Shape descriptor for q [B, Hq, d] and a K/V cache viewed as [B, Hkv, S, d]
    (any strides with a unit channel stride)."""
    if q.dim() != 3 or k_cache.dim() != 4:
        raise ValueError("q must be [B, Hq, d] and k_cache [B, Hkv, S, d]")
    B, Hq, d = q.shape
    Bk, Hkv, S, dk = k_cache.shape
    if Bk != B or dk != d:
        raise ValueError("q and k_cache disagree on batch or head_dim")
    if k_cache.stride(3) != 1:
        raise ValueError("k_cache channels must be contiguous")
    sb, sh, st, _ = k_cache.stride()
    dense = k_cache.is_contiguous()
    return TaShape(B, Hq, Hkv, d, S, _dtype_code(q.dtype), _dtype_code(k_cache.dtype),
                   float(scale or 0.0), 0 if dense else sb, 0 if dense else sh, 0 if dense else st)


# Shape descriptors of recent dense calls, keyed by everything make_shape and
# the decode checks read (shapes, strides, dtypes, scale), each with its
# workspace size per split count.  Repeated calls of one layer skip the
# Python-side validation and the descriptor build.
_shape_cache: dict = {}
_SHAPE_CACHE_MAX = 256


def _dense_shape(q, k_cache, v_cache, seqlens, scale):
    key = (q.shape, q.stride(), q.dtype, k_cache.shape, k_cache.stride(), k_cache.dtype,
           v_cache.shape, v_cache.stride(), v_cache.dtype, seqlens.shape, seqlens.stride(), seqlens.dtype,
           scale)
    hit = _shape_cache.get(key)
    if hit is not None:
        return hit
    if v_cache.shape != k_cache.shape or v_cache.stride() != k_cache.stride():
        raise ValueError("k_cache and v_cache must have the same shape and strides")
    if v_cache.dtype != k_cache.dtype:
        raise ValueError("k_cache and v_cache must share a dtype")
    if not q.is_contiguous():
        raise ValueError("q must be contiguous")
    if seqlens.dtype != torch.int32 or not seqlens.is_contiguous():
        raise ValueError("seqlens must be a contiguous int32 tensor")
    shape = make_shape(q, k_cache, scale)
    hit = (shape, ctypes.byref(shape), {})
    if len(_shape_cache) >= _SHAPE_CACHE_MAX:
        _shape_cache.clear()
    _shape_cache[key] = hit
    return hit


def tree_attn_status_string(status: int) -> str:
    return load().tree_attn_status_string(int(status)).decode()


def tree_attn_version() -> int:
    return int(load().tree_attn_version())


def tree_attn_check_shape(shape: TaShape) -> int:
    return int(load().tree_attn_check_shape(ctypes.byref(shape)))


def _splits_arg(num_splits: int, P: int, kernel: str, cluster_merge: bool) -> int:
    """The split count passed to the library once the workspace is sized for P:
    0 when the caller left the choice to the library (it then picks the same P,
    and for short rows may merge through a thread-block cluster), else P."""
    return 0 if int(num_splits) <= 0 and kernel == "auto" and not cluster_merge else P


def tree_attn_workspace_bytes(shape: TaShape, num_splits: int) -> int:
    return int(load().tree_attn_workspace_bytes(ctypes.byref(shape), int(num_splits)))


def tree_attn_pick_splits(shape: TaShape, host_seqlens=None, num_sms: int = 0, page_size: int = 0) -> int:
    """Split-count heuristic; ``page_size`` > 0 for paged caches (small pages
    may let one block serve several KV heads, which changes the best count)."""
    arr = None
    if host_seqlens is not None:
        arr = torch.as_tensor(host_seqlens, dtype=torch.int32).cpu().contiguous()
        if arr.numel() != shape.batch:
            raise ValueError("host_seqlens must have one entry per batch row")
    r = int(load().tree_attn_pick_splits_paged(ctypes.byref(shape), int(page_size), _ptr(arr), int(num_sms)))
    if r < 0:
        raise TreeAttnError(r, "tree_attn_pick_splits")
    return r


def tree_attn_launch_count(shape: TaShape, num_splits: int, kernel: str = "auto",
                           deterministic: bool = False) -> int:
    """Kernels one tree_attn_decode call enqueues (1 when the merge is fused)."""
    opts = _options(kernel, deterministic)
    r = int(load().tree_attn_launch_count(ctypes.byref(shape), int(num_splits), ctypes.byref(opts)))
    if r < 0:
        raise TreeAttnError(r, "tree_attn_launch_count")
    return r


def _check_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")


def tree_attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     seqlens: torch.Tensor, out: Optional[torch.Tensor] = None,
                     lse: Optional[torch.Tensor] = None, num_splits: int = 0,
                     workspace: Optional[torch.Tensor] = None, kernel: str = "auto",
                     scale: Optional[float] = None, stream=None, split_events=None,
                     want_lse: bool = True, deterministic: bool = False,
                     k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                     diag_stall: bool = False, diag_mishint: bool = False, cluster_merge: bool = False):
    """Decode attention through the C ABI; returns (out [B,Hq,d] fp32, lse [B,Hq] fp32 or None).

    ``num_splits`` <= 0 uses the library's heuristic (picked on the host so the
    workspace can be sized).  ``split_events`` = (start, end) torch.cuda.Event
    pair recorded around the per-slice kernel.  ``deterministic`` selects the
    fixed chunk assignment (bitwise reproducible results for a given split count).
    ``diag_stall`` (testing only) makes every on-chip wait give up: NaN outputs and
    TA_ERR_DEVICE_TIMEOUT from tree_attn_get_device_error, after about two seconds.
    ``diag_mishint`` (testing only) makes the copy warps' length hint wrong, so their
    first copies are discarded; the results must not change.  ``cluster_merge`` runs
    each row's 2..8 blocks as a thread-block cluster merging through distributed
    shared memory (a heuristic split count is capped at 8).
    """
    lib = load()
    _check_cuda(q, k_cache, v_cache, seqlens, out, lse, workspace)
    shape, shape_ref, ws_sizes = _dense_shape(q, k_cache, v_cache, seqlens, scale)
    if out is None:
        B, Hq, d = q.shape
        out = torch.empty(B, Hq, d, dtype=torch.float32, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    P = int(num_splits)
    if P <= 0:
        pick_key = ("pick", q.device.index)  # the heuristic's count depends on the device's SMs
        P = ws_sizes.get(pick_key)
        if P is None:
            P = ws_sizes[pick_key] = tree_attn_pick_splits(shape)
        if cluster_merge:
            P = min(P, TA_CLUSTER_MAX_SPLITS)  # one cluster per row
    nbytes = ws_sizes.get(P)
    if nbytes is None:
        nbytes = ws_sizes[P] = tree_attn_workspace_bytes(shape, P)
    if nbytes and workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _stream(stream)
    if (kernel == "auto" and split_events is None and not deterministic and k_scale is None and not diag_stall
            and not diag_mishint and not cluster_merge):
        rc = lib.tree_attn_decode(shape_ref, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(seqlens), _ptr(out), _ptr(lse), _splits_arg(num_splits, P, kernel, False),
                                  _ptr(workspace),
                                  ws_bytes, st)
    else:
        if split_events is not None:
            # torch creates the CUDA event on its first record; record once so the
            # handle exists (the library's own record then replaces this one)
            torch_stream = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.current_stream()
            for ev in split_events:
                ev.record(torch_stream)
        opts = _options(kernel, deterministic, k_scale, v_scale, split_events, diag_stall, diag_mishint,
                        cluster_merge)
        rc = lib.tree_attn_decode_ex(ctypes.byref(shape), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(seqlens), _ptr(out), _ptr(lse),
                                     _splits_arg(num_splits, P, kernel, cluster_merge), _ptr(workspace),
                                     ws_bytes, ctypes.byref(opts), st)
    if rc != TA_OK:
        raise TreeAttnError(rc, "tree_attn_decode")
    return out, lse


def tree_attn_combine(partial_o: torch.Tensor, partial_m: torch.Tensor, partial_l: torch.Tensor,
                      out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                      stream=None):
    """Tree combine of partial states [B,Hq,P,d] / [B,Hq,P] (fp32) -> (out, lse)."""
    lib = load()
    _check_cuda(partial_o, partial_m, partial_l, out, lse)
    for t in (partial_o, partial_m, partial_l):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("partial states must be contiguous float32")
    B, Hq, P, d = partial_o.shape
    if partial_m.shape != (B, Hq, P) or partial_l.shape != (B, Hq, P):
        raise ValueError("partial_m / partial_l must be [B, Hq, P]")
    if out is None:
        out = torch.empty(B, Hq, d, dtype=torch.float32, device=partial_o.device)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=partial_o.device)
    shape = TaShape(B, Hq, 1, d, 1, TA_F32, TA_F32, 0.0, 0, 0, 0)
    rc = lib.tree_attn_combine(ctypes.byref(shape), _ptr(partial_o), _ptr(partial_m),
                               _ptr(partial_l), P, _ptr(out), _ptr(lse), _stream(stream))
    if rc != TA_OK:
        raise TreeAttnError(rc, "tree_attn_combine")
    return out, lse


def tree_attn_get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load().tree_attn_get_device_error(_stream(stream)))


def tree_attn_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                             seqlens: torch.Tensor, out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                             num_splits: int = 0, scale: Optional[float] = None, stream=None):
    """Decode attention that allocates nothing: for callers that cannot allocate
    device memory while decoding (for example an engine plugin whose memory is
    planned in advance).  The caller passes every output; the partial states go
    to the library's fixed per-device scratch buffer (TA_NOALLOC_SCRATCH_BYTES).
    Calls that overlap on the GPU share that buffer and must be ordered."""
    lib = load()
    _check_cuda(q, k_cache, v_cache, seqlens, out, lse)
    if v_cache.shape != k_cache.shape or v_cache.stride() != k_cache.stride():
        raise ValueError("k_cache and v_cache must have the same shape and strides")
    shape = make_shape(q, k_cache, scale)
    rc = lib.tree_attn_decode_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(seqlens), _ptr(out), _ptr(lse), int(num_splits),
                                      _stream(stream))
    if rc != TA_OK:
        raise TreeAttnError(rc, "tree_attn_decode_noalloc")
    return out, lse


def tree_attn_decode_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                           block_table: torch.Tensor, seqlens: torch.Tensor,
                           out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                           num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                           kernel: str = "auto", scale: Optional[float] = None, stream=None,
                           deterministic: bool = False, max_seqlen: Optional[int] = None,
                           k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                           cluster_merge: bool = False):
    """Decode attention over a paged KV cache through the C ABI.

    k_pages, v_pages: [num_pages, page_size, Hkv, d] views (any strides with a unit
    channel stride; a [num_pages, Hkv, page_size, d] pool is passed as a permuted view);
    block_table: int32 [B, max_pages_per_seq]; returns (out, lse).
    """
    lib = load()
    _check_cuda(q, k_pages, v_pages, block_table, seqlens, out, lse, workspace)
    if k_pages.dim() != 4 or v_pages.shape != k_pages.shape or v_pages.stride() != k_pages.stride():
        raise ValueError("k_pages and v_pages must be [num_pages, page_size, Hkv, d] with equal strides")
    if k_pages.stride(3) != 1 or not q.is_contiguous():
        raise ValueError("channels must be contiguous and q dense")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or not block_table.is_contiguous():
        raise ValueError("block_table must be a contiguous int32 [B, max_pages] tensor")
    if seqlens.dtype != torch.int32 or not seqlens.is_contiguous():
        raise ValueError("seqlens must be a contiguous int32 tensor")
    num_pages, page_size, Hkv, d = k_pages.shape
    B, Hq, dq = q.shape
    if dq != d or block_table.shape[0] != B:
        raise ValueError("q, pages and block_table disagree")
    S = int(max_seqlen) if max_seqlen is not None else block_table.shape[1] * page_size
    sp, st, sh, _ = k_pages.stride()
    shape = TaShape(B, Hq, Hkv, d, S, _dtype_code(q.dtype), _dtype_code(k_pages.dtype),
                    float(scale or 0.0), sp, sh, st)
    paged = TaPagedKV(block_table.data_ptr(), block_table.shape[1], page_size, num_pages, 0)
    if out is None:
        out = torch.empty(B, Hq, d, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    P = int(num_splits)
    if P <= 0:
        P = tree_attn_pick_splits(shape, page_size=page_size)
        if cluster_merge:
            P = min(P, TA_CLUSTER_MAX_SPLITS)  # one cluster per row
    nbytes = tree_attn_workspace_bytes(shape, P)
    if nbytes and workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    opts = _options(kernel, deterministic, k_scale, v_scale, cluster_merge=cluster_merge)
    rc = lib.tree_attn_decode_paged(ctypes.byref(shape), ctypes.byref(paged), _ptr(q), _ptr(k_pages),
                                    _ptr(v_pages), _ptr(seqlens), _ptr(out), _ptr(lse),
                                    _splits_arg(num_splits, P, kernel, cluster_merge),
                                    _ptr(workspace), ws_bytes, ctypes.byref(opts), _stream(stream))
    if rc != TA_OK:
        raise TreeAttnError(rc, "tree_attn_decode_paged")
    return out, lse


def tree_attn_decode_multi(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           seqlens: torch.Tensor, causal: bool = True,
                           block_table: Optional[torch.Tensor] = None,
                           out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                           num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                           kernel: str = "auto", scale: Optional[float] = None, stream=None,
                           deterministic: bool = False, max_seqlen: Optional[int] = None,
                           k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                           cluster_merge: bool = False):
    """Several queries per sequence through the C ABI.

    q: [B, Hq, nq, d]; query i of row b sits at position seqlens[b] - nq + i and, when
    causal, sees tokens [0, seqlens[b] - nq + i].  k_cache/v_cache: dense [B, Hkv, S, d]
    caches, or page pools [num_pages, page_size, Hkv, d] with ``block_table``.
    Returns (out [B, Hq, nq, d], lse [B, Hq, nq]).
    """
    lib = load()
    _check_cuda(q, k_cache, v_cache, seqlens, block_table, out, lse, workspace)
    if q.dim() != 4 or not q.is_contiguous():
        raise ValueError("q must be a contiguous [B, Hq, nq, d] tensor")
    if v_cache.shape != k_cache.shape or v_cache.stride() != k_cache.stride() or k_cache.stride(3) != 1:
        raise ValueError("k_cache and v_cache must share shape and strides, channels contiguous")
    if seqlens.dtype != torch.int32 or not seqlens.is_contiguous():
        raise ValueError("seqlens must be a contiguous int32 tensor")
    B, Hq, nq, d = q.shape
    paged = None
    if block_table is None:
        base = make_shape(q[:, :, 0, :], k_cache, scale)
    else:
        if block_table.dtype != torch.int32 or not block_table.is_contiguous():
            raise ValueError("block_table must be a contiguous int32 tensor")
        num_pages, page_size, Hkv, _ = k_cache.shape
        S = int(max_seqlen) if max_seqlen is not None else block_table.shape[1] * page_size
        sp, st, sh, _ = k_cache.stride()
        base = TaShape(B, Hq, Hkv, d, S, _dtype_code(q.dtype), _dtype_code(k_cache.dtype),
                       float(scale or 0.0), sp, sh, st)
        paged = TaPagedKV(block_table.data_ptr(), block_table.shape[1], page_size, num_pages, 0)
    eff = TaShape.from_buffer_copy(base)
    eff.num_q_heads = Hq * nq
    if out is None:
        out = torch.empty(B, Hq, nq, d, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, nq, dtype=torch.float32, device=q.device)
    P = int(num_splits)
    if P <= 0:
        P = tree_attn_pick_splits(eff, page_size=paged.page_size if paged is not None else 0)
        if cluster_merge:
            P = min(P, TA_CLUSTER_MAX_SPLITS)  # one cluster per row
    nbytes = tree_attn_workspace_bytes(eff, P)
    if nbytes and workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    opts = _options(kernel, deterministic, k_scale, v_scale, cluster_merge=cluster_merge)
    rc = lib.tree_attn_decode_multi(ctypes.byref(base), ctypes.byref(paged) if paged is not None else None,
                                    nq, int(bool(causal)), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(seqlens), _ptr(out), _ptr(lse),
                                    _splits_arg(num_splits, P, kernel, cluster_merge), _ptr(workspace), ws_bytes,
                                    ctypes.byref(opts), _stream(stream))
    if rc != TA_OK:
        raise TreeAttnError(rc, "tree_attn_decode_multi")
    return out, lse
