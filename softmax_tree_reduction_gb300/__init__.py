"""GB300-native split-KV decode attention with an on-chip log-sum-exp tree combine.

The computation lives in ``libtreeattn.so`` (C ABI in ``include/tree_attn.h``);
this package only binds it (``_binding``), builds it (``build``) and draws
seeded synthetic inputs (``workloads``).
"""
from ._binding import (  # noqa: F401
    LIB_PATH, TA_OK, TA_BF16, TA_E4M3, TA_ERR_DEVICE_BOUNDS, TA_ERR_DEVICE_DATA, TA_ERR_DEVICE_TIMEOUT, TA_F32, TA_FLAG_DETERMINISTIC,
    TA_FLAG_CLUSTER_MERGE, TA_FLAG_DIAG_MISHINT, TA_FLAG_DIAG_STALL, TA_KERNEL, TA_MAX_SPLITS, TA_NOALLOC_SCRATCH_BYTES, TaOptions, TaPagedKV, TaShape, TreeAttnError, load,
    make_shape, tree_attn_check_shape, tree_attn_combine, tree_attn_decode, tree_attn_decode_multi, tree_attn_decode_noalloc, tree_attn_decode_paged,
    tree_attn_get_device_error, tree_attn_launch_count, tree_attn_pick_splits, tree_attn_status_string,
    tree_attn_version, tree_attn_workspace_bytes)
