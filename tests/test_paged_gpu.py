"""Paged KV cache (block tables) on the GPU, against the float64 oracle on the
gathered cache and, with the deterministic flag, bitwise against the dense path."""
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
        # same tiles in the same order as the dense path: bitwise equal
        od, ld = _dense_gpu(inp, num_splits=P, kernel=kern, deterministic=True)
        op, lp = ta.tree_attn_decode_paged(q, kpd, vpd, btd, sl, num_splits=P, kernel=kern,
                                           deterministic=True, max_seqlen=S)
        torch.cuda.synchronize()
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
