"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerances (written here, applied element by element):
  FP32 KV cache:  max |out - oracle| <= 1e-4,  max |lse - oracle| <= 1e-4
  BF16 KV cache:  max |out - oracle| <= 2e-3,  max |lse - oracle| <= 1e-3
The same bounds hold between any two split counts of one input.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import softmax_tree_reduction_gb300 as ta
from softmax_tree_reduction_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = {torch.float32: (1e-4, 1e-4), torch.bfloat16: (2e-3, 1e-3)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ta.load()


def to_dev(inp):
    return {k: (v.cuda() if k in ("q", "k", "v", "seqlens") else v) for k, v in inp.items()}


def decode(d, **kw):
    out, lse = ta.tree_attn_decode(d["q"], d["k"], d["v"], d["seqlens"], **kw)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def assert_close(out, lse, ref_out, ref_lse, kv_dtype, what=""):
    to, tl = TOL[kv_dtype]
    assert np.isfinite(out).all(), f"{what}: non-finite output"
    eo = np.max(np.abs(out - ref_out)) if out.size else 0.0
    # -inf lse (empty rows) must match exactly; compare the finite ones numerically
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: lse finiteness differs"
    assert np.all(lse[~fin] == ref_lse[~fin])
    el = np.max(np.abs(lse[fin] - ref_lse[fin])) if fin.any() else 0.0
    assert eo <= to, f"{what}: max|out err| = {eo:.3g} > {to}"
    assert el <= tl, f"{what}: max|lse err| = {el:.3g} > {tl}"
    return eo, el


# ----------------------------------------------------------------- tiny exact
@pytest.mark.parametrize("P", [8, 1, 2, 3, 5, 16, 33, 64])
def test_tiny_exact_fp32(P):
    w = workloads.TINY_EXACT
    inp = workloads.make_inputs(w)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"], 1.0 / 8.0)
    out, lse = decode(to_dev(inp), num_splits=P)
    assert_close(out, lse, ref_o, ref_l, torch.float32, f"P={P}")


# ------------------------------------------------- every kernel instantiation
CASES = []
for kv in (torch.bfloat16, torch.float32):
    for qd in (torch.bfloat16, torch.float32):
        for d in (64, 128):
            for G in (1, 2, 4, 8, 16):
                kernels = ["fma"]
                if kv == torch.bfloat16 and qd == torch.bfloat16 and G <= 8:
                    kernels.append("mma")
                for kern in kernels:
                    CASES.append((kv, qd, d, G, kern))


def _case_id(c):
    kv, qd, d, G, kern = c
    n = {torch.bfloat16: "bf16", torch.float32: "f32"}
    return f"kv{n[kv]}-q{n[qd]}-d{d}-G{G}-{kern}"


@pytest.mark.parametrize("case", CASES, ids=_case_id)
def test_kernel_instances_ragged(case):
    kv, qd, d, G, kern = case
    Hkv = 2
    lens = [0, 1, 15, 64, 65, 1000, 2049]
    w = workloads.Workload("ragged-small", len(lens), Hkv * G, Hkv, d, 2100, kv, qd, seed=CASES.index(case),
                           seqlen=None, ragged_range=(0, 1), pad_nan=True)
    inp = workloads.make_inputs(w, seqlens=lens)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    dev = to_dev(inp)
    for P in (1, 3, 8):
        out, lse = decode(dev, num_splits=P, kernel=kern)
        assert_close(out, lse, ref_o, ref_l, kv, f"{_case_id(case)} P={P}")
    # the empty row: out = 0, lse = -inf
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))


# ------------------------------------------------------------- combine only
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("P", [1, 2, 7, 64, 1000])
def test_combine_of_oracle_partials(d, P):
    B, Hq, Hkv, S = 2, 4, 2, 3000
    w = workloads.Workload("combine", B, Hq, Hkv, d, S, torch.bfloat16, torch.bfloat16, seed=P,
                           seqlen=None, ragged_range=(0, 1), k_scale=2.0)
    inp = workloads.make_inputs(w, seqlens=[3000, 1234])
    rng = np.random.default_rng(P)
    starts = np.zeros((B, P), dtype=np.int64)
    ends = np.zeros((B, P), dtype=np.int64)
    for b in range(B):
        n = int(inp["seqlens"][b])
        cuts = np.sort(rng.integers(0, n + 1, size=P - 1))
        e = np.concatenate([[0], cuts, [n]])
        starts[b], ends[b] = e[:-1], e[1:]
    po, pl, pm = oracle.partials(inp["q"], inp["k"], inp["v"], inp["seqlens"], starts, ends)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    out, lse = ta.tree_attn_combine(dev(po), dev(pm), dev(pl))
    torch.cuda.synchronize()
    assert_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l,
                 torch.float32, f"combine P={P}")


def test_combine_all_empty_rows():
    po = torch.zeros(1, 2, 5, 128, device="cuda")
    pm = torch.full((1, 2, 5), -math.inf, device="cuda")
    pl = torch.zeros(1, 2, 5, device="cuda")
    out, lse = ta.tree_attn_combine(po, pm, pl)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


# ------------------------------------- split invariance, determinism, layout
def _llama_like(N=16384, B=1, seed=0, kv=torch.bfloat16, G=4):
    w = workloads.Workload("llama-like", B, 8 * G, 8, 128, N, kv, kv, seed=seed, seqlen=N, k_scale=0.5)
    return workloads.make_inputs(w)


def test_split_invariance_and_oracle():
    inp = _llama_like()
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    dev = to_dev(inp)
    results = {}
    for kern in ("mma", "fma"):
        for P in (1, 2, 4, 8, 16, 19, 32, 64, 128, 256):
            out, lse = decode(dev, num_splits=P, kernel=kern)
            assert_close(out, lse, ref_o, ref_l, torch.bfloat16, f"{kern} P={P}")
            results[(kern, P)] = (out, lse)
    base_o, base_l = results[("mma", 1)]
    for key, (o, l) in results.items():
        assert np.max(np.abs(o - base_o)) <= 2e-3, key
        assert np.max(np.abs(l - base_l)) <= 1e-3, key


def test_heuristic_split_count_runs():
    inp = _llama_like()
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    out, lse = decode(to_dev(inp), num_splits=0)
    assert_close(out, lse, ref_o, ref_l, torch.bfloat16, "heuristic")


@pytest.mark.parametrize("kern,P", [("mma", 1), ("mma", 19), ("fma", 19), ("mma", 256), ("fma", 3)])
def test_bitwise_determinism(kern, P):
    """With the deterministic flag the chunk assignment is fixed: bitwise equal runs."""
    dev = to_dev(_llama_like(seed=3))
    a = decode(dev, num_splits=P, kernel=kern, deterministic=True)
    b = decode(dev, num_splits=P, kernel=kern, deterministic=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("kern", ["mma", "fma"])
def test_balanced_and_deterministic_schedules_agree(kern):
    """Run-time chunk balancing only reorders the merge: results agree to rounding."""
    inp = _llama_like(seed=4)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    dev = to_dev(inp)
    d_o, d_l = decode(dev, num_splits=19, kernel=kern, deterministic=True)
    for _ in range(3):
        o, l = decode(dev, num_splits=19, kernel=kern)
        assert np.max(np.abs(o - d_o)) <= 1e-5 and np.max(np.abs(l - d_l)) <= 1e-5
        assert_close(o, l, ref_o, ref_l, torch.bfloat16, f"{kern} balanced")


def test_token_major_layout_matches_dense():
    """K/V stored [B, S, Hkv, d] (token-major) and passed with strides."""
    inp = _llama_like(N=5000, B=2, seed=5)
    dev = to_dev(inp)
    out_d, lse_d = decode(dev, num_splits=7, deterministic=True)
    km = dev["k"].permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)   # [B,Hkv,S,d] view
    vm = dev["v"].permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    assert not km.is_contiguous()
    out_t, lse_t = ta.tree_attn_decode(dev["q"], km, vm, dev["seqlens"], num_splits=7,
                                       deterministic=True)
    torch.cuda.synchronize()
    assert np.array_equal(out_t.double().cpu().numpy(), out_d)
    assert np.array_equal(lse_t.double().cpu().numpy(), lse_d)


def test_lse_optional_and_outputs_fully_overwritten():
    inp = _llama_like(N=3000, seed=6)
    dev = to_dev(inp)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    for P in (1, 5):
        guard = 64
        buf = torch.full((32 * 128 + 2 * guard,), 12345.0, device="cuda")
        out = buf[guard:guard + 32 * 128].view(1, 32, 128)
        o, l = ta.tree_attn_decode(dev["q"], dev["k"], dev["v"], dev["seqlens"], out=out,
                                   num_splits=P, want_lse=False)
        torch.cuda.synchronize()
        assert l is None
        assert torch.all(buf[:guard] == 12345.0) and torch.all(buf[-guard:] == 12345.0)
        assert np.max(np.abs(out.double().cpu().numpy() - ref_o)) <= 2e-3


def test_bad_seqlen_sets_error_word_and_nan_rows():
    inp = _llama_like(N=2048, B=3, seed=7)
    dev = to_dev(inp)
    assert ta.tree_attn_get_device_error() == 0
    bad = dev["seqlens"].clone()
    bad[1] = 2048 + 5          # beyond max_seqlen: the kernel reads nothing of row 1
    for P in (1, 4):
        out, lse = ta.tree_attn_decode(dev["q"], dev["k"], dev["v"], bad, num_splits=P)
        assert ta.tree_attn_get_device_error() == -8
        o = out.cpu()
        assert torch.isnan(o[1]).all() and torch.isfinite(o[0]).all() and torch.isfinite(o[2]).all()
    out, lse = ta.tree_attn_decode(dev["q"], dev["k"], dev["v"], dev["seqlens"], num_splits=4)
    assert ta.tree_attn_get_device_error() == 0
    assert torch.isfinite(out).all()


def test_split_events_bracket_the_split_kernel():
    dev = to_dev(_llama_like(seed=8))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ta.tree_attn_decode(dev["q"], dev["k"], dev["v"], dev["seqlens"], num_splits=19,
                        split_events=(e0, e1))
    torch.cuda.synchronize()
    assert e0.elapsed_time(e1) > 0


# ------------------------------------------------------------ full-size workloads
def _check_full(w, sweep):
    """Full-size workload at the heuristic's split count and every swept one:
    every output row (all batch rows, all query heads) against the float64
    oracle over the whole input, element by element, and against the
    heuristic's result."""
    inp = workloads.make_inputs(w)
    dev = to_dev(inp)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"], w.softmax_scale)
    P0 = ta.tree_attn_pick_splits(ta.make_shape(dev["q"], dev["k"]))
    base = None
    for P in [0] + list(sweep):
        out, lse = decode(dev, num_splits=P)
        assert np.isfinite(out).all() and np.isfinite(lse).all(), f"P={P}"
        assert_close(out, lse, ref_o, ref_l, w.kv_dtype, f"{w.name} P={P or P0}")
        if base is None:
            base = (out, lse)
        else:
            assert np.max(np.abs(out - base[0])) <= 2e-3, f"P={P} vs heuristic P={P0}"
            assert np.max(np.abs(lse - base[1])) <= 1e-3, f"P={P} vs heuristic P={P0}"
    del dev
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_full_llama31_8b():
    _check_full(workloads.LLAMA31_8B, [1, 8, 64, 256])


@pytest.mark.slow
def test_full_batched_ragged_with_spikes():
    _check_full(workloads.BATCHED_RAGGED, [16, 64, 256])


@pytest.mark.slow
def test_full_llama3_70b():
    _check_full(workloads.LLAMA3_70B, [8, 64, 256])


@pytest.mark.slow
def test_full_million_token():
    _check_full(workloads.MILLION_TOKEN, [64, 512, 2048])


@pytest.mark.parametrize("P", [40, 41, 64, 1024, 4096])
def test_fused_and_launched_combine_paths(P):
    """Up to 40 splits merge in the row's last block; more go to the combine kernel.
    Many slices here are empty (more blocks than chunks)."""
    inp = _llama_like(N=16384, G=8, seed=9)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    dev = to_dev(inp)
    assert ta.tree_attn_launch_count(ta.make_shape(dev["q"], dev["k"]), P) == (1 if P <= 40 else 2)
    out, lse = decode(dev, num_splits=P)
    assert_close(out, lse, ref_o, ref_l, torch.bfloat16, f"P={P}")


def test_cuda_graph_capture_and_replay():
    """tree_attn_decode enqueues only kernels on the caller's stream, so a
    sequence of calls can be captured once and replayed."""
    inp = _llama_like(N=8192, seed=12)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    dev = to_dev(inp)
    out = torch.empty(1, 32, 128, device="cuda")
    lse = torch.empty(1, 32, device="cuda")
    shape = ta.make_shape(dev["q"], dev["k"])
    ws = torch.empty(ta.tree_attn_workspace_bytes(shape, 19), dtype=torch.uint8, device="cuda")
    ta.tree_attn_decode(dev["q"], dev["k"], dev["v"], dev["seqlens"], out=out, lse=lse, num_splits=19,
                        workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
            ta.tree_attn_decode(dev["q"], dev["k"], dev["v"], dev["seqlens"], out=out, lse=lse,
                                num_splits=19, workspace=ws)
    for _ in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l,
                     torch.bfloat16, "graph replay")
    assert ta.tree_attn_get_device_error() == 0
