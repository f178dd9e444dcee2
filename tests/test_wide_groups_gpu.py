"""More than 16 columns per KV head on the BF16 tensor-core path (column
groups of 16): multi-query-attention layouts (many query heads on one KV
head) and GQA with many draft tokens, against the float64 oracle: ragged rows
with NaN padding, fused and launched merges, paged caches, causal multi-query,
the cluster merge and the deterministic flag."""
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


@pytest.mark.parametrize("G,Hkv", [(24, 2), (32, 1), (48, 1), (64, 2)])
def test_wide_groups_dense(G, Hkv):
    inp = _inputs(G, Hkv, [0, 5, 129, 1000, 2900], 3072, seed=G)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    q, k, v, sl = (inp[x].cuda() for x in ("q", "k", "v", "seqlens"))
    for P in (0, 1, 5, 19, 41):
        out, lse = ta.tree_attn_decode(q, k, v, sl, num_splits=P)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"G={G} P={P}")
    o1, l1 = ta.tree_attn_decode(q, k, v, sl, num_splits=7, deterministic=True)
    o2, l2 = ta.tree_attn_decode(q, k, v, sl, num_splits=7, deterministic=True)
    out, lse = ta.tree_attn_decode(q, k, v, sl, num_splits=6, cluster_merge=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    _check(out, lse, ref_o, ref_l, f"G={G} cluster")
    assert ta.tree_attn_get_device_error() == 0


@pytest.mark.parametrize("page_size", [16, 128])
def test_wide_groups_paged(page_size):
    inp = _inputs(32, 2, [2000, 33, 700], 2048, seed=page_size)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    kp, vp, bt = workloads.page_pool(inp["k"], inp["v"], inp["seqlens"], page_size, seed=5)
    for P in (0, 9):
        out, lse = ta.tree_attn_decode_paged(inp["q"].cuda(), kp.cuda(), vp.cuda(), bt.cuda(), inp["seqlens"].cuda(),
                                             num_splits=P, max_seqlen=2048)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"paged {page_size} P={P}")


@pytest.mark.parametrize("G,nq", [(8, 4), (16, 4), (4, 16)])
@pytest.mark.parametrize("causal", [True, False])
def test_wide_multi_query(G, nq, causal):
    inp = _inputs(G, 2, [1500, 4, 300], 1536, seed=G + nq, nq=nq)
    ref_o, ref_l = oracle.attention_multi(inp["q"], inp["k"], inp["v"], inp["seqlens"], causal=causal)
    q, k, v, sl = (inp[x].cuda() for x in ("q", "k", "v", "seqlens"))
    for P in (1, 11):
        out, lse = ta.tree_attn_decode_multi(q, k, v, sl, causal=causal, num_splits=P)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"G={G} nq={nq} causal={causal} P={P}")
