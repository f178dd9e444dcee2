"""More than 16 columns per KV head on BF16 caches, on both tensor-core
kernels: the tcgen05 kernel (the automatic choice; accumulators in tensor
memory) and the warp-level mma kernel (column groups of 16).  Multi-query-
attention layouts (many query heads on one KV head) and GQA with many draft
tokens, against the float64 oracle: ragged rows with NaN padding, fused and
launched merges, paged caches, causal multi-query, the cluster merge (mma
kernel) and the deterministic flag.  The tcgen05 kernel is also run on small
groups (1-16 columns) and through the failure-path diagnostics."""
import numpy as np
import pytest
import torch

import oracle
import softmax_tree_reduction_gb300 as ta
from softmax_tree_reduction_gb300 import workloads

pytestmark = pytest.mark.gpu


def _inputs(G, Hkv, lens, S, seed, nq=None):
    w = workloads.Workload("wide", len(lens), Hkv * G, Hkv, 128, S, torch.bfloat16, torch.bfloat16, seed=seed,
                           seqlen=None, ragged_range=(0, 1), pad_nan=True, k_scale=0.5, spike_logit=10.0)
    inp = workloads.make_inputs(w, seqlens=lens)
    if nq is not None:
        g = torch.Generator().manual_seed(seed + 1)
        inp["q"] = torch.randn(len(lens), Hkv * G, nq, 128, generator=g).to(torch.bfloat16)
    return inp


def _check(out, lse, ref_o, ref_l, what):
    o, l = out.double().cpu().numpy(), lse.double().cpu().numpy()
    assert np.isfinite(o).all(), what
    assert np.max(np.abs(o - ref_o)) <= 2e-3, (what, np.max(np.abs(o - ref_o)))
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin), what
    if fin.any():
        assert np.max(np.abs(l[fin] - ref_l[fin])) <= 1e-3, what


@pytest.mark.parametrize("kern", ["auto", "mma"])
@pytest.mark.parametrize("G,Hkv", [(24, 2), (32, 1), (48, 1), (64, 2)])
def test_wide_groups_dense(G, Hkv, kern):
    inp = _inputs(G, Hkv, [0, 5, 129, 1000, 2900], 3072, seed=G)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    q, k, v, sl = (inp[x].cuda() for x in ("q", "k", "v", "seqlens"))
    for P in (0, 1, 5, 19, 41):
        out, lse = ta.tree_attn_decode(q, k, v, sl, num_splits=P, kernel=kern)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"G={G} P={P} {kern}")
    o1, l1 = ta.tree_attn_decode(q, k, v, sl, num_splits=7, deterministic=True, kernel=kern)
    o2, l2 = ta.tree_attn_decode(q, k, v, sl, num_splits=7, deterministic=True, kernel=kern)
    out, lse = ta.tree_attn_decode(q, k, v, sl, num_splits=6, cluster_merge=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    _check(out, lse, ref_o, ref_l, f"G={G} cluster")
    assert ta.tree_attn_get_device_error() == 0


@pytest.mark.parametrize("kern", ["auto", "mma"])
@pytest.mark.parametrize("page_size", [16, 32, 128, 256])
def test_wide_groups_paged(page_size, kern):
    inp = _inputs(32, 2, [2000, 33, 700], 2048, seed=page_size)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    kp, vp, bt = workloads.page_pool(inp["k"], inp["v"], inp["seqlens"], page_size, seed=5)
    for P in (0, 9):
        out, lse = ta.tree_attn_decode_paged(inp["q"].cuda(), kp.cuda(), vp.cuda(), bt.cuda(), inp["seqlens"].cuda(),
                                             num_splits=P, max_seqlen=2048, kernel=kern)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"paged {page_size} P={P} {kern}")


@pytest.mark.parametrize("kern", ["auto", "mma"])
@pytest.mark.parametrize("G,nq", [(8, 4), (16, 4), (4, 16), (6, 3)])
@pytest.mark.parametrize("causal", [True, False])
def test_wide_multi_query(G, nq, causal, kern):
    inp = _inputs(G, 2, [1500, 4, 300], 1536, seed=G + nq, nq=nq)
    ref_o, ref_l = oracle.attention_multi(inp["q"], inp["k"], inp["v"], inp["seqlens"], causal=causal)
    q, k, v, sl = (inp[x].cuda() for x in ("q", "k", "v", "seqlens"))
    for P in (1, 11):
        out, lse = ta.tree_attn_decode_multi(q, k, v, sl, causal=causal, num_splits=P, kernel=kern)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"G={G} nq={nq} causal={causal} P={P} {kern}")


@pytest.mark.parametrize("G", [1, 4, 8, 13, 16, 40])
def test_tc05_any_group_size(G):
    """The tcgen05 kernel asked for explicitly, on groups of 1 to 64 columns:
    ragged rows with NaN padding, planted spikes, one and several splits."""
    inp = _inputs(G, 2, [0, 1, 17, 128, 129, 2900], 3072, seed=100 + G)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    q, k, v, sl = (inp[x].cuda() for x in ("q", "k", "v", "seqlens"))
    for P in (1, 3, 8, 64):
        out, lse = ta.tree_attn_decode(q, k, v, sl, num_splits=P, kernel="tc05")
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"tc05 G={G} P={P}")
    o = out.cpu()
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse.cpu()[0]))
    assert ta.tree_attn_get_device_error() == 0


def test_tc05_rescale_on_growing_logits():
    """Logits that grow along the sequence make the lazy reference maximum move
    many times (each move rescales O in tensor memory)."""
    G, N = 32, 4096
    w = workloads.Workload("grow", 1, G, 1, 128, N, torch.bfloat16, torch.bfloat16, seed=7, seqlen=N)
    inp = workloads.make_inputs(w)
    ramp = torch.linspace(0.0, 6.0, N).view(1, 1, N, 1)
    inp["k"] = (inp["k"].float() * (0.25 + ramp)).to(torch.bfloat16)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    q, k, v, sl = (inp[x].cuda() for x in ("q", "k", "v", "seqlens"))
    for P in (1, 2, 5):
        out, lse = ta.tree_attn_decode(q, k, v, sl, num_splits=P, kernel="tc05", deterministic=True)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"growing logits P={P}")


@pytest.mark.parametrize("P", [1, 5])
def test_tc05_stalled_waits_report_timeout(P):
    """Failure path of the tcgen05 kernel: no tile is published, every wait
    gives up, outputs are NaN, the timeout is reported, the TMEM is freed and
    the next call is correct."""
    inp = _inputs(32, 2, [1000, 333], 1024, seed=3)
    q, k, v, sl = (inp[x].cuda() for x in ("q", "k", "v", "seqlens"))
    assert ta.tree_attn_get_device_error() == 0
    out, lse = ta.tree_attn_decode(q, k, v, sl, num_splits=P, kernel="tc05", diag_stall=True)
    assert ta.tree_attn_get_device_error() == ta.TA_ERR_DEVICE_TIMEOUT
    assert torch.isnan(out).all() and torch.isnan(lse).all()
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    out, lse = ta.tree_attn_decode(q, k, v, sl, num_splits=P, kernel="tc05")
    torch.cuda.synchronize()
    assert ta.tree_attn_get_device_error() == 0
    _check(out, lse, ref_o, ref_l, "after the stall")


@pytest.mark.parametrize("P", [1, 5, 19])
def test_tc05_wrong_length_hint_changes_nothing(P):
    inp = _inputs(48, 2, [1000, 333], 1024, seed=4)
    q, k, v, sl = (inp[x].cuda() for x in ("q", "k", "v", "seqlens"))
    o1, l1 = ta.tree_attn_decode(q, k, v, sl, num_splits=P, kernel="tc05", deterministic=True)
    o2, l2 = ta.tree_attn_decode(q, k, v, sl, num_splits=P, kernel="tc05", deterministic=True, diag_mishint=True)
    torch.cuda.synchronize()
    assert ta.tree_attn_get_device_error() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_tc05_bad_seqlen_sets_error_word_and_nan_rows():
    """A length outside [0, max_seqlen] on the tcgen05 path: that row is NaN,
    the others are correct, and the error word reports it."""
    inp = _inputs(32, 2, [1000, 333, 2000], 2048, seed=8)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    q, k, v, sl = (inp[x].cuda() for x in ("q", "k", "v", "seqlens"))
    bad = sl.clone()
    bad[1] = 2048 + 7
    assert ta.tree_attn_get_device_error() == 0
    for P in (1, 4):
        out, lse = ta.tree_attn_decode(q, k, v, bad, num_splits=P, kernel="tc05")
        assert ta.tree_attn_get_device_error() == ta.TA_ERR_DEVICE_DATA
        o = out.cpu()
        assert torch.isnan(o[1]).all() and torch.isfinite(o[0]).all() and torch.isfinite(o[2]).all()
        keep = [0, 2]
        _check(out[keep], lse[keep], ref_o[keep], ref_l[keep], f"good rows P={P}")


def test_tc05_bad_page_entry_poisons_only_its_row():
    inp = _inputs(48, 2, [700, 1500], 1536, seed=9)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    kp, vp, bt = workloads.page_pool(inp["k"], inp["v"], inp["seqlens"], 64, seed=3)
    bt = bt.clone()
    bt[1, 5] = kp.shape[0] + 3        # a page past the pool for a valid token of row 1
    out, lse = ta.tree_attn_decode_paged(inp["q"].cuda(), kp.cuda(), vp.cuda(), bt.cuda(), inp["seqlens"].cuda(),
                                         num_splits=3, max_seqlen=1536, kernel="tc05")
    assert ta.tree_attn_get_device_error() == ta.TA_ERR_DEVICE_DATA
    o = out.cpu()
    assert torch.isnan(o[1]).all()
    _check(out[:1], lse[:1], ref_o[:1], ref_l[:1], "row 0")
