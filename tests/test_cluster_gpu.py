"""Row merge through a thread-block cluster's distributed shared memory
(TA_FLAG_CLUSTER_MERGE): a row's 2..8 blocks form one cluster.  Against the
float64 oracles: both tensor-core families, ragged rows with NaN padding,
several group sizes and split counts, paged caches (blocks serving several
KV heads), several queries per row, the deterministic flag, and the
diagnostic paths (stalled waits, a wrong length hint)."""
import numpy as np
import pytest
import torch

import oracle
import softmax_tree_reduction_gb300 as ta
from softmax_tree_reduction_gb300 import workloads

pytestmark = pytest.mark.gpu


def _inputs(G, lens, S, Hkv=2, fp8=False, seed=0, nq=None):
    w = workloads.Workload("cl", len(lens), Hkv * G, Hkv, 128, S, torch.bfloat16, torch.bfloat16, seed=seed,
                           seqlen=None, ragged_range=(0, 1), pad_nan=True, k_scale=0.5, spike_logit=8.0)
    inp = workloads.make_inputs(w, seqlens=lens)
    if nq is not None:
        g = torch.Generator().manual_seed(seed + 1)
        inp["q"] = torch.randn(len(lens), Hkv * G, nq, 128, generator=g).to(torch.bfloat16)
    if fp8:
        inp["k"], inp["ks"] = workloads.quantize_e4m3(inp["k"])
        inp["v"], inp["vs"] = workloads.quantize_e4m3(inp["v"])
    return inp


def _ref(inp, fp8, causal=True):
    if fp8:
        return oracle.attention_e4m3(inp["q"], inp["k"], inp["v"], inp["ks"], inp["vs"], inp["seqlens"],
                                     causal=causal)
    if inp["q"].dim() == 4:
        return oracle.attention_multi(inp["q"], inp["k"], inp["v"], inp["seqlens"], causal=causal)
    return oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])


def _scales(inp, fp8):
    return dict(k_scale=inp["ks"].cuda(), v_scale=inp["vs"].cuda()) if fp8 else {}


def _check(out, lse, ref_o, ref_l, what):
    o, l = out.double().cpu().numpy(), lse.double().cpu().numpy()
    assert np.isfinite(o).all(), what
    assert np.max(np.abs(o - ref_o)) <= 2e-3, (what, np.max(np.abs(o - ref_o)))
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin), what
    if fin.any():
        assert np.max(np.abs(l[fin] - ref_l[fin])) <= 1e-3, what


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("G", [1, 4, 8, 16])
def test_cluster_merge_dense(fp8, G):
    inp = _inputs(G, [0, 1, 130, 1000, 3000], 3072, fp8=fp8, seed=G)
    ref_o, ref_l = _ref(inp, fp8)
    q, k, v, sl = (inp[x].cuda() for x in ("q", "k", "v", "seqlens"))
    for P in (0, 2, 3, 5, 8):
        out, lse = ta.tree_attn_decode(q, k, v, sl, num_splits=P, cluster_merge=True, **_scales(inp, fp8))
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"fp8={fp8} G={G} P={P}")
    o1, l1 = ta.tree_attn_decode(q, k, v, sl, num_splits=8, cluster_merge=True, deterministic=True, **_scales(inp, fp8))
    o2, l2 = ta.tree_attn_decode(q, k, v, sl, num_splits=8, cluster_merge=True, deterministic=True, **_scales(inp, fp8))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert ta.tree_attn_get_device_error() == 0


@pytest.mark.parametrize("fp8,page_size", [(False, 16), (False, 64), (True, 16), (True, 256)])
def test_cluster_merge_paged_eight_kv_heads(fp8, page_size):
    inp = _inputs(4, [2000, 17, 0, 900], 2048, Hkv=8, fp8=fp8, seed=page_size)
    ref_o, ref_l = _ref(inp, fp8)
    kp, vp, bt = workloads.page_pool(inp["k"], inp["v"], inp["seqlens"], page_size, seed=3)
    args = (inp["q"].cuda(), kp.cuda(), vp.cuda(), bt.cuda(), inp["seqlens"].cuda())
    for P in (2, 8):
        out, lse = ta.tree_attn_decode_paged(*args, num_splits=P, max_seqlen=2048, cluster_merge=True,
                                             **_scales(inp, fp8))
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"paged {page_size} fp8={fp8} P={P}")
    assert ta.tree_attn_get_device_error() == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_cluster_merge_multi_query(fp8):
    inp = _inputs(4, [1500, 3, 700], 1536, fp8=fp8, seed=7, nq=4)
    ref_o, ref_l = _ref(inp, fp8, causal=True)
    out, lse = ta.tree_attn_decode_multi(inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(), inp["seqlens"].cuda(),
                                         causal=True, num_splits=6, cluster_merge=True, **_scales(inp, fp8))
    torch.cuda.synchronize()
    _check(out, lse, ref_o, ref_l, f"multi fp8={fp8}")


@pytest.mark.parametrize("fp8", [False, True])
def test_cluster_merge_diagnostic_paths(fp8):
    inp = _inputs(4, [1000, 333], 1024, fp8=fp8, seed=11)
    q, k, v, sl = (inp[x].cuda() for x in ("q", "k", "v", "seqlens"))
    kw = _scales(inp, fp8)
    o1, l1 = ta.tree_attn_decode(q, k, v, sl, num_splits=5, cluster_merge=True, deterministic=True, **kw)
    o2, l2 = ta.tree_attn_decode(q, k, v, sl, num_splits=5, cluster_merge=True, deterministic=True,
                                 diag_mishint=True, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert ta.tree_attn_get_device_error() == 0
    out, lse = ta.tree_attn_decode(q, k, v, sl, num_splits=5, cluster_merge=True, diag_stall=True, **kw)
    assert ta.tree_attn_get_device_error() == ta.TA_ERR_DEVICE_TIMEOUT
    assert torch.isnan(out).all() and torch.isnan(lse).all()
    out, lse = ta.tree_attn_decode(q, k, v, sl, num_splits=5, cluster_merge=True, **kw)
    torch.cuda.synchronize()
    assert ta.tree_attn_get_device_error() == 0
    _check(out, lse, *_ref(inp, fp8), "after a stalled call")
