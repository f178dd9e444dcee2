"""The merge the library picks when the split count is left to it: rows whose
slices would be short merge through a thread-block cluster (as with
TA_FLAG_CLUSTER_MERGE), longer rows through the last-arriving block.  Under
the deterministic flag the automatic call is bitwise equal to the explicit
call of the merge it should pick (with 8 or more splits the two merges cut
the rows differently), and every result is checked against the float64
oracle."""
import numpy as np
import pytest
import torch

import oracle
import softmax_tree_reduction_gb300 as ta
from softmax_tree_reduction_gb300 import workloads

pytestmark = pytest.mark.gpu


def _inputs(B, Hq, Hkv, S, fp8=False, seed=0):
    w = workloads.Workload("auto", B, Hq, Hkv, 128, S, torch.bfloat16, torch.bfloat16, seed=seed,
                           seqlen=S, k_scale=0.5, spike_logit=8.0)
    inp = workloads.make_inputs(w)
    if fp8:
        inp["k"], inp["ks"] = workloads.quantize_e4m3(inp["k"])
        inp["v"], inp["vs"] = workloads.quantize_e4m3(inp["v"])
    return inp


def _ref(inp, fp8):
    if fp8:
        return oracle.attention_e4m3(inp["q"], inp["k"], inp["v"], inp["ks"], inp["vs"], inp["seqlens"])
    return oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])


def _check(out, lse, ref_o, ref_l, what):
    o, l = out.double().cpu().numpy(), lse.double().cpu().numpy()
    assert np.max(np.abs(o - ref_o)) <= 2e-3, (what, np.max(np.abs(o - ref_o)))
    assert np.max(np.abs(l - ref_l)) <= 1e-3, what


def _runs(inp, fp8):
    dev = {k: v.cuda() for k, v in inp.items()}
    sc = dict(k_scale=dev["ks"], v_scale=dev["vs"]) if fp8 else {}
    args = (dev["q"], dev["k"], dev["v"], dev["seqlens"])
    P = ta.tree_attn_pick_splits(ta.make_shape(dev["q"], dev["k"]))
    auto = ta.tree_attn_decode(*args, num_splits=0, deterministic=True, **sc)
    ticket = ta.tree_attn_decode(*args, num_splits=P, deterministic=True, **sc)
    cluster = ta.tree_attn_decode(*args, num_splits=min(P, 8), cluster_merge=True, deterministic=True, **sc)
    fast = ta.tree_attn_decode(*args, **sc)  # default call: balanced slices
    torch.cuda.synchronize()
    assert ta.tree_attn_get_device_error() == 0
    return P, auto, ticket, cluster, fast


def _same(a, b):
    return torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,S", [(1, 32, 8, 1024), (1, 32, 8, 4096), (4, 64, 8, 2048)])
def test_short_rows_merge_through_a_cluster(fp8, B, Hq, Hkv, S):
    inp = _inputs(B, Hq, Hkv, S, fp8, seed=S + B)
    ref_o, ref_l = _ref(inp, fp8)
    P, auto, ticket, cluster, fast = _runs(inp, fp8)
    assert 2 <= min(P, 8) and -(-S // min(P, 8)) <= 640
    assert _same(auto, cluster)
    for name, r in (("auto", auto), ("ticket", ticket), ("default", fast)):
        _check(*r, ref_o, ref_l, f"{name} fp8={fp8} S={S}")


@pytest.mark.parametrize("fp8,S", [(False, 8192), (True, 16384)])
def test_longer_rows_keep_the_last_block_merge(fp8, S):
    inp = _inputs(1, 32, 8, S, fp8, seed=S)
    ref_o, ref_l = _ref(inp, fp8)
    P, auto, ticket, cluster, fast = _runs(inp, fp8)
    assert -(-S // min(P, 8)) > 768
    assert _same(auto, ticket)
    for name, r in (("auto", auto), ("cluster", cluster), ("default", fast)):
        _check(*r, ref_o, ref_l, f"{name} fp8={fp8} S={S}")


def test_paged_and_no_allocation_calls_take_the_same_choice():
    inp = _inputs(1, 32, 8, 4096, seed=11)
    ref_o, ref_l = _ref(inp, False)
    kp, vp, bt = workloads.page_pool(inp["k"], inp["v"], inp["seqlens"], 64, seed=4)
    q, sl = inp["q"].cuda(), inp["seqlens"].cuda()
    kp, vp, bt = kp.cuda(), vp.cuda(), bt.cuda()
    shape = ta.make_shape(q, inp["k"].cuda())
    Pc = min(ta.tree_attn_pick_splits(shape, page_size=64), 8)
    auto = ta.tree_attn_decode_paged(q, kp, vp, bt, sl, num_splits=0, deterministic=True, max_seqlen=4096)
    cl = ta.tree_attn_decode_paged(q, kp, vp, bt, sl, num_splits=Pc, cluster_merge=True, deterministic=True,
                                   max_seqlen=4096)
    torch.cuda.synchronize()
    assert _same(auto, cl)
    _check(*auto, ref_o, ref_l, "paged auto")
    out = torch.empty(1, 32, 128, device="cuda")
    lse = torch.empty(1, 32, device="cuda")
    ta.tree_attn_decode_noalloc(q, inp["k"].cuda(), inp["v"].cuda(), sl, out, lse, num_splits=0)
    torch.cuda.synchronize()
    _check(out, lse, ref_o, ref_l, "no-allocation auto")
    assert ta.tree_attn_get_device_error() == 0


def test_graph_capture_of_an_automatic_cluster_step():
    inp = _inputs(1, 32, 8, 2048, seed=12)
    ref_o, ref_l = _ref(inp, False)
    dev = {k: v.cuda() for k, v in inp.items()}
    out = torch.empty(1, 32, 128, device="cuda")
    lse = torch.empty(1, 32, device="cuda")
    P = ta.tree_attn_pick_splits(ta.make_shape(dev["q"], dev["k"]))
    ws = torch.empty(max(16, ta.tree_attn_workspace_bytes(ta.make_shape(dev["q"], dev["k"]), P)),
                     dtype=torch.uint8, device="cuda")
    ta.tree_attn_decode(dev["q"], dev["k"], dev["v"], dev["seqlens"], out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
            ta.tree_attn_decode(dev["q"], dev["k"], dev["v"], dev["seqlens"], out=out, lse=lse, workspace=ws)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    _check(out, lse, ref_o, ref_l, "graph replay")
    assert ta.tree_attn_get_device_error() == 0
