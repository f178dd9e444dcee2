"""FP8 (E4M3) caches on the tcgen05 kernel (the automatic choice above 16
columns per KV head, and `kernel = tc05` for any group up to 32 columns),
against the float64 oracle over the same codes and scales: ragged rows with
NaN padding, every column count up to 32, several queries per sequence with
and without causality, paged caches, skewed and growing logits (the lazy
reference maximum moves), q at the edges of the E4M3 two-term split, and the
fixed (bitwise reproducible) chunk assignment.  The warp-level FP8 kernel
stays reachable with `kernel = mma`."""
import numpy as np
import pytest
import torch

import oracle
import softmax_tree_reduction_gb300 as ta
from softmax_tree_reduction_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL_OUT, TOL_LSE = 2e-3, 1e-3


def _inputs(lens, S, Hkv=2, G=4, seed=0, k_scale=0.5, spike=None, nq=None):
    w = workloads.Workload("fp8tc", len(lens), Hkv * G, Hkv, 128, S, torch.bfloat16, torch.bfloat16,
                           seed=seed, seqlen=None, ragged_range=(0, 1), pad_nan=True,
                           k_scale=k_scale, spike_logit=spike)
    inp = workloads.make_inputs(w, seqlens=lens)
    inp["k8"], inp["ks"] = workloads.quantize_e4m3(inp["k"])
    inp["v8"], inp["vs"] = workloads.quantize_e4m3(inp["v"])
    if nq is not None:
        g = torch.Generator().manual_seed(seed + 1)
        inp["q"] = torch.randn(len(lens), Hkv * G, nq, 128, generator=g).to(torch.bfloat16)
    return inp


def _ref(inp, causal=True):
    return oracle.attention_e4m3(inp["q"], inp["k8"], inp["v8"], inp["ks"], inp["vs"], inp["seqlens"],
                                 causal=causal)


def _dev(inp):
    return (inp["q"].cuda(), inp["k8"].cuda(), inp["v8"].cuda(), inp["seqlens"].cuda(),
            dict(k_scale=inp["ks"].cuda(), v_scale=inp["vs"].cuda()))


def _check(out, lse, ref_o, ref_l, what):
    o, l = out.double().cpu().numpy(), lse.double().cpu().numpy()
    assert np.isfinite(o).all(), what
    err = np.max(np.abs(o - ref_o))
    assert err <= TOL_OUT, (what, err)
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin), what
    if fin.any():
        assert np.max(np.abs(l[fin] - ref_l[fin])) <= TOL_LSE, what


@pytest.mark.parametrize("G", [1, 3, 4, 8, 9, 12, 16, 17, 24, 32])
def test_fp8_tc05_dense_ragged(G):
    lens = [0, 1, 15, 16, 127, 128, 129, 1000, 3001]
    inp = _inputs(lens, 3072, G=G, seed=100 + G)
    ref_o, ref_l = _ref(inp)
    q, k8, v8, sl, sc = _dev(inp)
    for P in (1, 2, 5, 19, 64):
        out, lse = ta.tree_attn_decode(q, k8, v8, sl, num_splits=P, kernel="tc05", **sc)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"tc05 G={G} P={P}")
    if G > 16:  # the automatic choice, heuristic split
        out, lse = ta.tree_attn_decode(q, k8, v8, sl, **sc)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"auto G={G}")
    if G <= 16:  # the warp-level kernel on the same inputs
        out, lse = ta.tree_attn_decode(q, k8, v8, sl, num_splits=5, kernel="mma", **sc)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"mma G={G}")
    assert ta.tree_attn_get_device_error() == 0


@pytest.mark.parametrize("G,nq", [(4, 4), (8, 2), (3, 5), (1, 16), (4, 8), (8, 4), (2, 16)])
@pytest.mark.parametrize("causal", [True, False])
def test_fp8_tc05_multi_query(G, nq, causal):
    inp = _inputs([0, 3, 300, 1700], 1792, G=G, seed=10 * G + nq, nq=nq)
    ref_o, ref_l = _ref(inp, causal=causal)
    q, k8, v8, sl, sc = _dev(inp)
    for P in (0, 1, 11):
        out, lse = ta.tree_attn_decode_multi(q, k8, v8, sl, causal=causal, num_splits=P, kernel="tc05", **sc)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"G={G} nq={nq} causal={causal} P={P}")
    assert ta.tree_attn_get_device_error() == 0


@pytest.mark.parametrize("page_size", [16, 32, 128, 256])
def test_fp8_tc05_paged(page_size):
    lens = [2000, 5, 700, 1024]
    inp = _inputs(lens, 2048, Hkv=4, G=16, seed=page_size)
    ref_o, ref_l = _ref(inp)
    kp, vp, bt = workloads.page_pool(inp["k8"], inp["v8"], inp["seqlens"], page_size, seed=7)
    q, _, _, sl, sc = _dev(inp)
    for P in (0, 1, 3, 40):
        out, lse = ta.tree_attn_decode_paged(q, kp.cuda(), vp.cuda(), bt.cuda(), sl, num_splits=P,
                                             max_seqlen=2048, kernel="tc05", **sc)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"paged {page_size} P={P}")
    assert ta.tree_attn_get_device_error() == 0


def test_fp8_tc05_spiked_logits_and_small_scales():
    inp = _inputs([5000, 4096, 77], 5120, G=16, seed=11, k_scale=1e-3, spike=30.0)
    ref_o, ref_l = _ref(inp)
    q, k8, v8, sl, sc = _dev(inp)
    for P in (1, 7, 40):
        out, lse = ta.tree_attn_decode(q, k8, v8, sl, num_splits=P, kernel="tc05", **sc)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"spiked P={P}")


def test_fp8_tc05_growing_logits():
    """Logits growing along the sequence move the reference maximum many times."""
    G, N = 16, 4096
    w = workloads.Workload("grow8", 1, G, 1, 128, N, torch.bfloat16, torch.bfloat16, seed=8, seqlen=N)
    inp = workloads.make_inputs(w)
    ramp = torch.linspace(0.0, 6.0, N).view(1, 1, N, 1)
    inp["k8"], inp["ks"] = workloads.quantize_e4m3((inp["k"].float() * (0.25 + ramp)).to(torch.bfloat16))
    inp["v8"], inp["vs"] = workloads.quantize_e4m3(inp["v"])
    ref_o, ref_l = _ref(inp)
    q, k8, v8, sl, sc = _dev(inp)
    for P in (1, 2, 5):
        out, lse = ta.tree_attn_decode(q, k8, v8, sl, num_splits=P, kernel="tc05", deterministic=True, **sc)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"growing logits P={P}")


def test_fp8_tc05_query_scales():
    """q at the edges of its two-term E4M3 form: large (logits of order 100),
    tiny (the scale brings it up by 2^40), one head all zero, one head with a
    single non-zero channel, and a head mixing magnitudes 2^12 apart."""
    inp = _inputs([2048, 700, 1500], 2048, G=12, seed=21)
    q = inp["q"].float()
    q[0] *= 40.0
    q[1] *= 2.0 ** -40
    q[2, 3].zero_()
    q[2, 5].zero_()
    q[2, 5, 17] = 3.0
    q[2, 7, :64] *= 2.0 ** 12
    inp["q"] = q.to(torch.bfloat16)
    ref_o, ref_l = _ref(inp)
    q, k8, v8, sl, sc = _dev(inp)
    for P in (1, 6):
        out, lse = ta.tree_attn_decode(q, k8, v8, sl, num_splits=P, kernel="tc05", **sc)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"q scales P={P}")


def test_fp8_tc05_deterministic_bitwise():
    inp = _inputs([4000, 3333], 4096, G=16, seed=9)
    q, k8, v8, sl, sc = _dev(inp)
    o1, l1 = ta.tree_attn_decode(q, k8, v8, sl, num_splits=13, deterministic=True, kernel="tc05", **sc)
    o2, l2 = ta.tree_attn_decode(q, k8, v8, sl, num_splits=13, deterministic=True, kernel="tc05", **sc)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert ta.tree_attn_get_device_error() == 0


def test_fp8_tc05_refusals():
    inp = _inputs([100], 128, G=4, seed=1)
    q, k8, v8, sl, sc = _dev(inp)
    with pytest.raises(ta.TreeAttnError):
        ta.tree_attn_decode(q, k8, v8, sl, num_splits=2, kernel="tc05", cluster_merge=True, **sc)
    big = _inputs([100], 128, G=40, Hkv=1, seed=2)
    qb, kb, vb, slb, scb = _dev(big)
    with pytest.raises(ta.TreeAttnError):
        ta.tree_attn_decode(qb, kb, vb, slb, num_splits=1, **scb)     # 40 columns: no FP8 kernel
    assert ta.tree_attn_get_device_error() == 0
