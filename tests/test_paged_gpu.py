"""Paged KV cache (block tables) on the GPU, against the float64 oracle on the
gathered cache and, with the deterministic flag, bitwise against the dense path
(when the paged call streams the same tiles: with 16-token pages the BF16
tensor-core kernel lets a block serve two KV heads, which changes the tile
size, so there it is compared with itself bitwise and with the dense path
within tolerance)."""
import numpy as np
import pytest
import torch

import oracle
import softmax_tree_reduction_gb300 as ta
from softmax_tree_reduction_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = {torch.float32: (1e-4, 1e-4), torch.bfloat16: (2e-3, 1e-3)}


def _case(kv, d, G, lens, S, seed):
    w = workloads.Workload("paged", len(lens), 2 * G, 2, d, S, kv, kv, seed=seed, seqlen=None,
                           ragged_range=(0, 1), pad_nan=True, k_scale=0.5)
    return workloads.make_inputs(w, seqlens=lens)


def _dense_gpu(inp, **kw):
    o, l = ta.tree_attn_decode(inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(),
                               inp["seqlens"].cuda(), **kw)
    torch.cuda.synchronize()
    return o.cpu(), l.cpu()


@pytest.mark.parametrize("page_size", [16, 64, 256])
@pytest.mark.parametrize("kern,kv,d,G", [("mma", torch.bfloat16, 128, 4), ("mma", torch.bfloat16, 64, 8),
                                         ("fma", torch.bfloat16, 128, 4), ("fma", torch.float32, 64, 1)])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_paged_matches_oracle_and_dense(page_size, kern, kv, d, G, layout):
    lens = [0, 1, 15, 300, 1024, 2500]
    S = 2560
    inp = _case(kv, d, G, lens, S, seed=page_size + G)
    kp, vp, bt = workloads.page_pool(inp["k"], inp["v"], inp["seqlens"], page_size, layout=layout,
                                     seed=page_size)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    q, sl = inp["q"].cuda(), inp["seqlens"].cuda()
    kpd, vpd, btd = kp.cuda(), vp.cuda(), bt.cuda()
    to, tl = TOL[kv]
    for P in (1, 5, 19):
        o, l = ta.tree_attn_decode_paged(q, kpd, vpd, btd, sl, num_splits=P, kernel=kern, max_seqlen=S)
        torch.cuda.synchronize()
        o64, l64 = o.double().cpu().numpy(), l.double().cpu().numpy()
        assert np.isfinite(o64).all()
        assert np.max(np.abs(o64 - ref_o)) <= to
        fin = np.isfinite(ref_l)
        assert np.array_equal(np.isfinite(l64), fin)
        assert np.max(np.abs(l64[fin] - ref_l[fin])) <= tl
        od, ld = _dense_gpu(inp, num_splits=P, kernel=kern, deterministic=True)
        op, lp = ta.tree_attn_decode_paged(q, kpd, vpd, btd, sl, num_splits=P, kernel=kern,
                                           deterministic=True, max_seqlen=S)
        torch.cuda.synchronize()
        if kern == "mma" and d == 128 and page_size == 16:   # two KV heads per block
            op2, lp2 = ta.tree_attn_decode_paged(q, kpd, vpd, btd, sl, num_splits=P, kernel=kern,
                                                 deterministic=True, max_seqlen=S)
            torch.cuda.synchronize()
            assert torch.equal(op, op2) and torch.equal(lp, lp2)
            assert (op.cpu() - od).abs().max() <= to and (lp.cpu() - ld)[torch.isfinite(ld)].abs().max() <= tl
        else:  # same tiles in the same order as the dense path: bitwise equal
            assert torch.equal(op.cpu(), od) and torch.equal(lp.cpu(), ld)
    assert ta.tree_attn_get_device_error() == 0


def test_paged_long_rows_balanced():
    """Long rows exercise the run-time chunk claims through the page table."""
    lens = [20000, 16384]
    inp = _case(torch.bfloat16, 128, 4, lens, 20480, seed=3)
    kp, vp, bt = workloads.page_pool(inp["k"], inp["v"], inp["seqlens"], 64, seed=1)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    o, l = ta.tree_attn_decode_paged(inp["q"].cuda(), kp.cuda(), vp.cuda(), bt.cuda(),
                                     inp["seqlens"].cuda(), num_splits=19, max_seqlen=20480)
    torch.cuda.synchronize()
    assert np.max(np.abs(o.double().cpu().numpy() - ref_o)) <= 2e-3
    assert np.max(np.abs(l.double().cpu().numpy() - ref_l)) <= 1e-3


@pytest.mark.parametrize("bad_entry", ["past_pool", "negative"])
def test_bad_page_entry_poisons_only_its_row(bad_entry):
    lens = [500, 700, 300]
    inp = _case(torch.bfloat16, 128, 4, lens, 1024, seed=5)
    kp, vp, bt = workloads.page_pool(inp["k"], inp["v"], inp["seqlens"], 64, seed=2)
    # a valid page of row 1 now points outside the pool
    bt[1, 3] = kp.shape[0] + 7 if bad_entry == "past_pool" else -1
    assert ta.tree_attn_get_device_error() == 0
    o, l = ta.tree_attn_decode_paged(inp["q"].cuda(), kp.cuda(), vp.cuda(), bt.cuda(),
                                     inp["seqlens"].cuda(), num_splits=1, max_seqlen=1024)
    assert ta.tree_attn_get_device_error() == -8
    o = o.cpu()
    assert torch.isnan(o[1]).all() and torch.isfinite(o[0]).all() and torch.isfinite(o[2]).all()


@pytest.mark.parametrize("fp8,page_size", [(False, 16), (False, 32), (True, 16), (True, 32), (True, 64)])
def test_paged_eight_kv_heads(fp8, page_size):
    """Eight KV heads: 16-token pages put 2 (BF16) or 4 (FP8) heads in a block,
    32-token FP8 pages 2; split counts on both sides of the fused-merge limit."""
    lens = [3000, 17, 0, 1234]
    w = workloads.Workload("paged8", len(lens), 32, 8, 128, 3072, torch.bfloat16, torch.bfloat16, seed=page_size,
                           seqlen=None, ragged_range=(0, 1), pad_nan=True, k_scale=0.5, spike_logit=9.0)
    inp = workloads.make_inputs(w, seqlens=lens)
    k, v, kw = inp["k"], inp["v"], {}
    if fp8:
        k, ks = workloads.quantize_e4m3(k)
        v, vs = workloads.quantize_e4m3(v)
        ref_o, ref_l = oracle.attention_e4m3(inp["q"], k, v, ks, vs, inp["seqlens"])
        kw = dict(k_scale=ks.cuda(), v_scale=vs.cuda())
    else:
        ref_o, ref_l = oracle.attention(inp["q"], k, v, inp["seqlens"])
    kp, vp, bt = workloads.page_pool(k, v, inp["seqlens"], page_size, seed=7)
    args = (inp["q"].cuda(), kp.cuda(), vp.cuda(), bt.cuda(), inp["seqlens"].cuda())
    fin = np.isfinite(ref_l)
    for P in (0, 1, 7, 40, 41, 76):
        o, l = ta.tree_attn_decode_paged(*args, num_splits=P, max_seqlen=3072, **kw)
        torch.cuda.synchronize()
        o64, l64 = o.double().cpu().numpy(), l.double().cpu().numpy()
        assert np.isfinite(o64).all(), P
        assert np.max(np.abs(o64 - ref_o)) <= 2e-3, P
        assert np.array_equal(np.isfinite(l64), fin), P
        assert np.max(np.abs(l64[fin] - ref_l[fin])) <= 1e-3, P
    o1, l1 = ta.tree_attn_decode_paged(*args, num_splits=19, deterministic=True, max_seqlen=3072, **kw)
    o2, l2 = ta.tree_attn_decode_paged(*args, num_splits=19, deterministic=True, max_seqlen=3072, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert ta.tree_attn_get_device_error() == 0


@pytest.mark.slow
@pytest.mark.parametrize("page_size", [16, 256])
def test_full_llama31_8b_paged(page_size):
    """The 131072-token 8B-shaped layer from a shuffled page pool (the bench's
    --paged configuration): every output row against the oracle over the whole
    input."""
    w = workloads.LLAMA31_8B
    inp = workloads.make_inputs(w)
    kp, vp, bt = workloads.page_pool(inp["k"], inp["v"], inp["seqlens"], page_size, seed=w.seed)
    args = (inp["q"].cuda(), kp.cuda(), vp.cuda(), bt.cuda(), inp["seqlens"].cuda())
    ro, rl = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"], w.softmax_scale)
    for P in (0, 19, 38):
        o, l = ta.tree_attn_decode_paged(*args, num_splits=P, max_seqlen=w.max_seqlen)
        torch.cuda.synchronize()
        o64 = o.double().cpu().numpy()
        l64 = l.double().cpu().numpy()
        assert np.isfinite(o64).all() and np.isfinite(l64).all(), (page_size, P)
        assert np.max(np.abs(o64 - ro)) <= 2e-3, (page_size, P)
        assert np.max(np.abs(l64 - rl)) <= 1e-3, (page_size, P)
    assert ta.tree_attn_get_device_error() == 0
