"""tree_attn_decode_noalloc: decode attention for callers that cannot allocate
device memory at decode time (for example an inference-engine plugin whose
memory is planned before serving starts).  Its partial states live in the
library's fixed per-device scratch buffer instead of a caller workspace.

Checked through the C ABI against the float64 oracle and against
tree_attn_decode on the same inputs, with the parity tolerance used for BF16 KV
caches (|out| 2e-3, |lse| 1e-3), on two calls in a row (the buffer keeps the
previous call's contents): with the row merge inside the split kernel (19
splits), with the separate combine kernel (64 splits), with the heuristic, with
one split (no scratch used), and at the largest split count whose partial
states fit the buffer; one split more is refused.  This file is named to be
collected last.
"""
import numpy as np
import pytest
import torch

import oracle
import softmax_tree_reduction_gb300 as ta
from softmax_tree_reduction_gb300 import workloads

pytestmark = pytest.mark.gpu


def _inputs(seed, N=16384, B=2):
    w = workloads.Workload("noalloc", B, 32, 8, 128, N, torch.bfloat16, torch.bfloat16, seed=seed,
                           seqlen=None, ragged_range=(1, N), k_scale=0.5)
    inp = workloads.make_inputs(w, seqlens=[N, N // 3 + 5][:B])
    ref = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    return {k: inp[k].cuda() for k in ("q", "k", "v", "seqlens")}, ref


def _close(out, lse, ref_out, ref_lse):
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy()
    ro = ref_out.double().cpu().numpy() if isinstance(ref_out, torch.Tensor) else ref_out
    rl = ref_lse.double().cpu().numpy() if isinstance(ref_lse, torch.Tensor) else ref_lse
    assert np.isfinite(o).all() and np.isfinite(l).all()
    assert np.max(np.abs(o - ro)) <= 2e-3
    assert np.max(np.abs(l - rl)) <= 1e-3


def _two_calls(d, ref, P):
    """Two no-allocation calls in a row, each checked against the oracle and
    against tree_attn_decode with the same split count."""
    ref_out, ref_lse = ta.tree_attn_decode(d["q"], d["k"], d["v"], d["seqlens"], num_splits=P)
    out = torch.empty_like(ref_out)
    lse = torch.empty_like(ref_lse)
    for _ in range(2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        ta.tree_attn_decode_noalloc(d["q"], d["k"], d["v"], d["seqlens"], out, lse, num_splits=P)
        torch.cuda.synchronize()
        _close(out, lse, ref_out, ref_lse)
        _close(out, lse, *ref)


@pytest.mark.parametrize("P", [19, 64, 0, 1])
def test_noalloc_matches_decode_and_oracle_on_two_calls_in_a_row(P):
    ta.load()
    d, ref = _inputs(11 + P)
    shape = ta.make_shape(d["q"], d["k"])
    if P == 64:   # more splits than the row merge takes: the combine kernel reads the scratch
        assert ta.tree_attn_launch_count(shape, P) == 2
    _two_calls(d, ref, P)
    assert ta.tree_attn_get_device_error() == 0


def test_noalloc_at_the_scratch_limit():
    """The largest split count whose partial states fit the buffer runs and is
    correct; one more is refused with TA_ERR_SCRATCH_LIMIT, nothing enqueued."""
    ta.load()
    d, ref = _inputs(13, N=16384, B=1)
    shape = ta.make_shape(d["q"], d["k"])
    P = 1
    while ta.tree_attn_workspace_bytes(shape, P + 1) <= ta.TA_NOALLOC_SCRATCH_BYTES:
        P += 1
    assert 400 < P < ta.TA_MAX_SPLITS   # about 500 slices of 32 heads x 130 floats
    _two_calls(d, ref, P)
    out = torch.full((1, 32, 128), 7.0, device="cuda")
    with pytest.raises(ta.TreeAttnError) as ei:
        ta.tree_attn_decode_noalloc(d["q"], d["k"], d["v"], d["seqlens"], out, None, num_splits=P + 1)
    assert ei.value.status == -10
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
    assert ta.tree_attn_get_device_error() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    ta.load()
    d, _ = _inputs(14, N=4096, B=1)
    shape = ta.make_shape(d["q"], d["k"])
    P = 4096                                       # 32 heads x 4096 slices x 130 floats > 8 MiB
    assert ta.tree_attn_workspace_bytes(shape, P) > ta.TA_NOALLOC_SCRATCH_BYTES
    out = torch.empty(1, 32, 128, device="cuda")
    with pytest.raises(ta.TreeAttnError) as ei:
        ta.tree_attn_decode_noalloc(d["q"], d["k"], d["v"], d["seqlens"], out, None, num_splits=P)
    assert ei.value.status == -10
