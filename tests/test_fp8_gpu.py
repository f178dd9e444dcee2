"""FP8 (E4M3) KV caches with one scale per KV head, on the GPU, against the
float64 oracle over the same codes and scales: ragged rows with NaN padding,
several split counts, strided and paged caches, several queries per sequence
(one or two n-tiles of columns), skewed logits, and the fixed (bitwise
reproducible) chunk assignment."""
import numpy as np
import pytest
import torch

import oracle
import softmax_tree_reduction_gb300 as ta
from softmax_tree_reduction_gb300 import workloads

pytestmark = pytest.mark.gpu

# The cache values are exact in both paths (the codes and their scales are the
# inputs); what differs is the kernel's f16/f32 arithmetic, as for BF16 caches.
TOL_OUT, TOL_LSE = 2e-3, 1e-3


def _inputs(lens, S, Hkv=2, G=4, seed=0, k_scale=0.5, spike=None, nq=None):
    w = workloads.Workload("fp8", len(lens), Hkv * G, Hkv, 128, S, torch.bfloat16, torch.bfloat16,
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
    return oracle.attention_e4m3(inp["q"], inp["k8"], inp["v8"], inp["ks"], inp["vs"],
                                 inp["seqlens"], causal=causal)


def _dev(inp):
    return (inp["q"].cuda(), inp["k8"].cuda(), inp["v8"].cuda(), inp["seqlens"].cuda(),
            inp["ks"].cuda(), inp["vs"].cuda())


def _check(out, lse, ref_o, ref_l, what):
    o, l = out.double().cpu().numpy(), lse.double().cpu().numpy()
    assert np.isfinite(o).all(), what
    err = np.max(np.abs(o - ref_o))
    assert err <= TOL_OUT, (what, err)
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin), what
    if fin.any():
        assert np.max(np.abs(l[fin] - ref_l[fin])) <= TOL_LSE, what


@pytest.mark.parametrize("G", [1, 2, 4, 8, 12, 16])
def test_fp8_dense_ragged(G):
    lens = [0, 1, 15, 16, 127, 128, 129, 1000, 3001]
    inp = _inputs(lens, 3072, G=G, seed=G)
    ref_o, ref_l = _ref(inp)
    q, k8, v8, sl, ks, vs = _dev(inp)
    for P in (1, 2, 5, 19, 64):
        out, lse = ta.tree_attn_decode(q, k8, v8, sl, num_splits=P, k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"G={G} P={P}")
    out, lse = ta.tree_attn_decode(q, k8, v8, sl, k_scale=ks, v_scale=vs)   # heuristic split
    torch.cuda.synchronize()
    _check(out, lse, ref_o, ref_l, f"G={G} auto")
    assert ta.tree_attn_get_device_error() == 0


def test_fp8_spiked_logits_and_small_scales():
    # a planted logit of 30 against a tiny K scale: the online maximum moves
    # late and the per-head scales span orders of magnitude
    inp = _inputs([5000, 4096, 77], 5120, G=4, seed=11, k_scale=1e-3, spike=30.0)
    ref_o, ref_l = _ref(inp)
    q, k8, v8, sl, ks, vs = _dev(inp)
    for P in (1, 7, 40):
        out, lse = ta.tree_attn_decode(q, k8, v8, sl, num_splits=P, k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"spiked P={P}")


def test_fp8_large_query_and_zero_query():
    inp = _inputs([2048, 700], 2048, G=4, seed=21)
    inp["q"] = (inp["q"].float() * 40.0).to(torch.bfloat16)   # logits of order 100
    inp["q"][1, 3].zero_()                                    # uniform softmax for one head
    ref_o, ref_l = _ref(inp)
    q, k8, v8, sl, ks, vs = _dev(inp)
    out, lse = ta.tree_attn_decode(q, k8, v8, sl, num_splits=6, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    _check(out, lse, ref_o, ref_l, "large q")


def test_fp8_strided_cache():
    inp = _inputs([900, 1500], 2048, G=4, seed=5)
    big_k = torch.zeros(2, 2, 4096, 128, dtype=torch.float8_e4m3fn)
    big_v = torch.zeros_like(big_k)
    big_k[:, :, 1024:3072] = inp["k8"]
    big_v[:, :, 1024:3072] = inp["v8"]
    ref_o, ref_l = _ref(inp)
    q, _, _, sl, ks, vs = _dev(inp)
    kd, vd = big_k.cuda(), big_v.cuda()
    out, lse = ta.tree_attn_decode(q, kd[:, :, 1024:3072], vd[:, :, 1024:3072], sl, num_splits=4,
                                   k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    _check(out, lse, ref_o, ref_l, "strided")


@pytest.mark.parametrize("page_size", [16, 64, 256])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_fp8_paged(page_size, layout):
    inp = _inputs([1000, 33, 2500, 0], 2560, G=4, seed=page_size)
    kp, vp, bt = workloads.page_pool(inp["k8"], inp["v8"], inp["seqlens"], page_size,
                                     layout=layout, seed=2)
    ref_o, ref_l = _ref(inp)
    q, _, _, sl, ks, vs = _dev(inp)
    for P in (1, 9):
        out, lse = ta.tree_attn_decode_paged(q, kp.cuda(), vp.cuda(), bt.cuda(), sl, num_splits=P,
                                             max_seqlen=2560, k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"paged {page_size} {layout} P={P}")


@pytest.mark.parametrize("G,nq", [(1, 2), (4, 2), (2, 4), (1, 8), (8, 1), (8, 2), (4, 4), (3, 5), (1, 16)])
@pytest.mark.parametrize("causal", [True, False])
def test_fp8_multi_query(G, nq, causal):
    inp = _inputs([0, 3, 300, 1700], 1792, G=G, seed=10 * G + nq, nq=nq)
    ref_o, ref_l = _ref(inp, causal=causal)
    q, k8, v8, sl, ks, vs = _dev(inp)
    for P in (1, 11):
        out, lse = ta.tree_attn_decode_multi(q, k8, v8, sl, causal=causal, num_splits=P,
                                             k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"G={G} nq={nq} causal={causal} P={P}")


def test_fp8_deterministic_bitwise():
    inp = _inputs([4000, 3333], 4096, G=4, seed=9)
    q, k8, v8, sl, ks, vs = _dev(inp)
    o1, l1 = ta.tree_attn_decode(q, k8, v8, sl, num_splits=13, deterministic=True, k_scale=ks,
                                 v_scale=vs)
    o2, l2 = ta.tree_attn_decode(q, k8, v8, sl, num_splits=13, deterministic=True, k_scale=ks,
                                 v_scale=vs)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fp8_argument_errors():
    inp = _inputs([100], 128, G=4, seed=1)
    q, k8, v8, sl, ks, vs = _dev(inp)
    with pytest.raises(ta.TreeAttnError):
        ta.tree_attn_decode(q, k8, v8, sl, num_splits=1)                 # no scales
    with pytest.raises(ta.TreeAttnError):
        ta.tree_attn_decode(q, k8, v8, sl, num_splits=1, kernel="fma", k_scale=ks, v_scale=vs)
    with pytest.raises(ValueError):
        ta.tree_attn_decode(q, k8, v8, sl, num_splits=1, k_scale=ks.double(), v_scale=vs)
    assert ta.tree_attn_get_device_error() == 0


@pytest.mark.parametrize("page_size", [16, 32])
def test_fp8_paged_multi_query_eight_kv_heads(page_size):
    """16 columns per KV head (two n-tiles) with blocks serving several KV heads
    of 16/32-token pages, causal over the last 4 positions."""
    lens = [2000, 5, 700]
    w = workloads.Workload("fp8mq", len(lens), 32, 8, 128, 2048, torch.bfloat16, torch.bfloat16, seed=page_size,
                           seqlen=None, ragged_range=(0, 1), pad_nan=True, k_scale=0.5)
    inp = workloads.make_inputs(w, seqlens=lens)
    g = torch.Generator().manual_seed(5)
    q = torch.randn(len(lens), 32, 4, 128, generator=g).to(torch.bfloat16)
    k8, ks = workloads.quantize_e4m3(inp["k"])
    v8, vs = workloads.quantize_e4m3(inp["v"])
    ref_o, ref_l = oracle.attention_e4m3(q, k8, v8, ks, vs, inp["seqlens"], causal=True)
    kp, vp, bt = workloads.page_pool(k8, v8, inp["seqlens"], page_size, seed=4)
    for P in (0, 3, 40):
        out, lse = ta.tree_attn_decode_multi(q.cuda(), kp.cuda(), vp.cuda(), inp["seqlens"].cuda(), causal=True,
                                             block_table=bt.cuda(), num_splits=P, max_seqlen=2048,
                                             k_scale=ks.cuda(), v_scale=vs.cuda())
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, f"paged {page_size} P={P}")
    assert ta.tree_attn_get_device_error() == 0


def _full_fp8(w, sweep, page_size=0):
    """Full-size workload with its caches rounded to E4M3 (the bench's --fp8
    configuration): every output row against the oracle over the whole input."""
    inp = workloads.make_inputs(w)
    k8, ks = workloads.quantize_e4m3(inp["k"])
    v8, vs = workloads.quantize_e4m3(inp["v"])
    ref_o, ref_l = oracle.attention_e4m3(inp["q"], k8, v8, ks, vs, inp["seqlens"], scale=w.softmax_scale)
    q, sl = inp["q"].cuda(), inp["seqlens"].cuda()
    kw = dict(k_scale=ks.cuda(), v_scale=vs.cuda())
    if page_size:
        kp, vp, bt = workloads.page_pool(k8, v8, inp["seqlens"], page_size, seed=1)
        args = (q, kp.cuda(), vp.cuda(), bt.cuda(), sl)
        call = lambda P: ta.tree_attn_decode_paged(*args, num_splits=P, max_seqlen=w.max_seqlen, **kw)
    else:
        k8d, v8d = k8.cuda(), v8.cuda()
        call = lambda P: ta.tree_attn_decode(q, k8d, v8d, sl, num_splits=P, **kw)
    for P in [0] + list(sweep):
        out, lse = call(P)
        torch.cuda.synchronize()
        o, l = out.double().cpu().numpy(), lse.double().cpu().numpy()
        assert np.isfinite(o).all() and np.isfinite(l).all(), P
        assert np.max(np.abs(o - ref_o)) <= TOL_OUT, (w.name, P)
        assert np.max(np.abs(l - ref_l)) <= TOL_LSE, (w.name, P)
    assert ta.tree_attn_get_device_error() == 0


@pytest.mark.slow
def test_full_llama31_8b_fp8():
    _full_fp8(workloads.LLAMA31_8B, [8, 19, 64])


@pytest.mark.slow
def test_full_llama31_8b_fp8_paged16():
    _full_fp8(workloads.LLAMA31_8B, [19, 38], page_size=16)


@pytest.mark.slow
def test_full_llama3_70b_fp8():
    _full_fp8(workloads.LLAMA3_70B, [19, 64])
