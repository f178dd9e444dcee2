"""Multi-query decode (several queries per sequence) on the GPU against the
float64 oracle: causal over the last nq positions or not, rows shorter than nq,
one and two n-tiles of (head, query) columns, dense and paged caches."""
import numpy as np
import pytest
import torch

import oracle
import softmax_tree_reduction_gb300 as ta
from softmax_tree_reduction_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = {torch.float32: (1e-4, 1e-4), torch.bfloat16: (2e-3, 1e-3)}


def _inputs(kv, d, Hkv, G, nq, lens, S, seed):
    w = workloads.Workload("mq", len(lens), Hkv * G, Hkv, d, S, kv, kv, seed=seed, seqlen=None,
                           ragged_range=(0, 1), pad_nan=True, k_scale=0.5)
    inp = workloads.make_inputs(w, seqlens=lens)
    g = torch.Generator().manual_seed(seed + 1)
    inp["qm"] = torch.randn(len(lens), Hkv * G, nq, d, generator=g).to(kv)
    return inp


def _check(out, lse, ref_o, ref_l, kv, what):
    to, tl = TOL[kv]
    o, l = out.double().cpu().numpy(), lse.double().cpu().numpy()
    assert np.isfinite(o).all(), what
    assert np.max(np.abs(o - ref_o)) <= to, (what, np.max(np.abs(o - ref_o)))
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin), what
    if fin.any():
        assert np.max(np.abs(l[fin] - ref_l[fin])) <= tl, what


CASES = []
for kv in (torch.bfloat16, torch.float32):
    for G, nq in ((1, 1), (4, 1), (3, 1), (4, 2), (1, 3), (2, 4), (8, 2), (4, 3), (1, 8), (4, 4)):
        kerns = []
        if kv == torch.bfloat16 and G * nq <= 16:
            kerns.append("mma")
        if (G * nq) & (G * nq - 1) == 0 and G * nq <= 16:
            kerns.append("fma")
        for kern in kerns:
            CASES.append((kv, G, nq, kern))


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{'bf16' if c[0] == torch.bfloat16 else 'f32'}-G{c[1]}-nq{c[2]}-{c[3]}")
@pytest.mark.parametrize("causal", [True, False])
def test_multi_query_matches_oracle(case, causal):
    kv, G, nq, kern = case
    lens = [0, 2, 17, 300, 1500]
    inp = _inputs(kv, 128 if kv == torch.bfloat16 else 64, 2, G, nq, lens, 1536, seed=G * 10 + nq)
    ref_o, ref_l = oracle.attention_multi(inp["qm"], inp["k"], inp["v"], inp["seqlens"], causal=causal)
    dev = [inp[k].cuda() for k in ("qm", "k", "v", "seqlens")]
    for P in (1, 4, 19):
        out, lse = ta.tree_attn_decode_multi(*dev, causal=causal, num_splits=P, kernel=kern)
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l, kv, f"{case} causal={causal} P={P}")
    assert ta.tree_attn_get_device_error() == 0


def test_single_query_multi_equals_decode():
    inp = _inputs(torch.bfloat16, 128, 2, 4, 1, [1000, 700], 1024, seed=77)
    q1 = inp["qm"][:, :, 0, :].contiguous().cuda()
    k, v, sl = inp["k"].cuda(), inp["v"].cuda(), inp["seqlens"].cuda()
    o1, l1 = ta.tree_attn_decode(q1, k, v, sl, num_splits=5, deterministic=True)
    om, lm = ta.tree_attn_decode_multi(inp["qm"].cuda(), k, v, sl, num_splits=5, deterministic=True)
    torch.cuda.synchronize()
    assert torch.equal(om[:, :, 0], o1) and torch.equal(lm[:, :, 0], l1)


@pytest.mark.parametrize("page_size", [16, 128])
def test_multi_query_paged(page_size):
    inp = _inputs(torch.bfloat16, 128, 2, 4, 4, [900, 33, 2000], 2048, seed=page_size)
    kp, vp, bt = workloads.page_pool(inp["k"], inp["v"], inp["seqlens"], page_size, seed=3)
    ref_o, ref_l = oracle.attention_multi(inp["qm"], inp["k"], inp["v"], inp["seqlens"], causal=True)
    out, lse = ta.tree_attn_decode_multi(inp["qm"].cuda(), kp.cuda(), vp.cuda(), inp["seqlens"].cuda(),
                                         causal=True, block_table=bt.cuda(), num_splits=7,
                                         max_seqlen=2048)
    torch.cuda.synchronize()
    _check(out, lse, ref_o, ref_l, torch.bfloat16, f"paged {page_size}")


def test_multi_query_argument_errors():
    inp = _inputs(torch.bfloat16, 128, 2, 8, 16, [100], 128, seed=1)   # G*nq = 128 > 64
    with pytest.raises(ta.TreeAttnError):
        ta.tree_attn_decode_multi(inp["qm"].cuda(), inp["k"].cuda(), inp["v"].cuda(),
                                  inp["seqlens"].cuda())
