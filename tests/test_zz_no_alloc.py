"""tree_attn_decode_noalloc: decode attention for callers that cannot allocate
device memory at decode time (for example an inference-engine plugin whose
memory is planned before serving starts).  Its partial states live in the
library's fixed per-device scratch buffer instead of a caller workspace.

Checked through the C ABI against tree_attn_decode on the same inputs, with the
parity tolerance used for BF16 KV caches (|out| 2e-3, |lse| 1e-3), on two calls
in a row (the buffer keeps the previous call's contents).  This file is named to
be collected last.
"""
import numpy as np
import pytest
import torch

import softmax_tree_reduction_gb300 as ta
from softmax_tree_reduction_gb300 import workloads

pytestmark = pytest.mark.gpu


def _inputs(seed, N=16384, B=2):
    w = workloads.Workload("noalloc", B, 32, 8, 128, N, torch.bfloat16, torch.bfloat16, seed=seed,
                           seqlen=None, ragged_range=(1, N), k_scale=0.5)
    inp = workloads.make_inputs(w, seqlens=[N, N // 3 + 5][:B])
    return {k: inp[k].cuda() for k in ("q", "k", "v", "seqlens")}


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    ta.load()
    for seed, P in ((11, 19), (12, 0)):          # explicit split count, then the heuristic
        d = _inputs(seed)
        ref_out, ref_lse = ta.tree_attn_decode(d["q"], d["k"], d["v"], d["seqlens"],
                                               num_splits=P if P else 0)
        out = torch.empty_like(ref_out)
        lse = torch.empty_like(ref_lse)
        for _ in range(2):
            out.fill_(float("nan"))
            lse.fill_(float("nan"))
            ta.tree_attn_decode_noalloc(d["q"], d["k"], d["v"], d["seqlens"], out, lse, num_splits=P)
            torch.cuda.synchronize()
            assert torch.isfinite(out).all() and torch.isfinite(lse).all()
            assert (out - ref_out).abs().max().item() <= 2e-3
            assert (lse - ref_lse).abs().max().item() <= 1e-3
    assert ta.tree_attn_get_device_error() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    ta.load()
    d = _inputs(13, N=4096, B=1)
    shape = ta.make_shape(d["q"], d["k"])
    P = 4096                                       # 32 heads x 4096 slices x 130 floats > 8 MiB
    assert ta.tree_attn_workspace_bytes(shape, P) > ta.TA_NOALLOC_SCRATCH_BYTES
    out = torch.empty(1, 32, 128, device="cuda")
    with pytest.raises(ta.TreeAttnError) as ei:
        ta.tree_attn_decode_noalloc(d["q"], d["k"], d["v"], d["seqlens"], out, None, num_splits=P)
    assert ei.value.status == -10
