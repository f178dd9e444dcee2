"""Pins of the float64 oracle to things other than itself (CPU only).

Each pin is independent of the oracle's code path:
  * brute force without max-subtraction on tiny inputs (pure Python, math.fsum);
  * a library special case: torch's scaled_dot_product_attention / logsumexp in float64;
  * hand-derived closed forms (tests/golden/closed_forms.json);
  * associativity / commutativity of the merge operator over many tree shapes
    ('The Tree Reduction Merge Operator': "associative and commutative ... trees of
    arbitrary depth, branching factor");
  * invariants: identical keys, one dominant logit, a single token, token
    permutation, shift of m, bounds on lse and on out, the empty state.
"""
import json
import math
import os
import random

import numpy as np
import pytest
import torch

import oracle
from softmax_tree_reduction_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def _rand_case(B, Hq, Hkv, d, S, seqlens, dtype, seed, k_scale=1.0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, d, generator=g).to(dtype)
    k = (torch.randn(B, Hkv, S, d, generator=g) * k_scale).to(dtype)
    v = torch.randn(B, Hkv, S, d, generator=g).to(dtype)
    return q, k, v, np.asarray(seqlens, dtype=np.int32)


def brute_force(q, k, v, seqlens, scale):
    """Softmax attention as sum(exp(s) v)/sum(exp(s)) with no max subtraction,
    every element widened by torch, sums by math.fsum (tiny inputs only)."""
    qd = q.to(torch.float64).tolist()
    kd = k.to(torch.float64).tolist()
    vd = v.to(torch.float64).tolist()
    B, Hq, d = len(qd), len(qd[0]), len(qd[0][0])
    Hkv = len(kd[0])
    G = Hq // Hkv
    out = np.zeros((B, Hq, d))
    lse = np.zeros((B, Hq))
    for b in range(B):
        for h in range(Hq):
            g = h // G
            n = int(seqlens[b])
            if n == 0:
                lse[b, h] = -math.inf
                continue
            w = [math.exp(scale * math.fsum(qd[b][h][i] * kd[b][g][t][i] for i in range(d)))
                 for t in range(n)]
            z = math.fsum(w)
            for i in range(d):
                out[b, h, i] = math.fsum(w[t] * vd[b][g][t][i] for t in range(n)) / z
            lse[b, h] = math.log(z)
    return out, lse


def sdpa_reference(q, k, v, seqlens, scale):
    """torch scaled_dot_product_attention in float64, GQA by repeating each KV head
    over its group of query heads, one batch row at a time (ragged lengths)."""
    B, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, d))
    lse = np.zeros((B, Hq))
    for b in range(B):
        n = int(seqlens[b])
        if n == 0:
            lse[b] = -np.inf
            continue
        qb = q[b].to(torch.float64)[:, None, :]                       # [Hq, 1, d]
        kb = k[b, :, :n].to(torch.float64).repeat_interleave(G, dim=0)  # [Hq, n, d]
        vb = v[b, :, :n].to(torch.float64).repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, scale=scale)
        out[b] = o[:, 0, :].numpy()
        lse[b] = torch.logsumexp(scale * (qb @ kb.transpose(1, 2))[:, 0, :], dim=-1).numpy()
    return out, lse


# ---------------------------------------------------------------------------
# Battery used both directly and by the mutation tests.
# ---------------------------------------------------------------------------

def check_brute_force(lib_handle=None):
    rng = random.Random(1)
    for trial in range(12):
        Hkv = rng.choice([1, 2])
        G = rng.choice([1, 2, 3])
        B = rng.choice([1, 2])
        d = rng.choice([1, 3, 8])
        S = rng.choice([1, 5, 16])
        seqlens = [rng.randint(0 if trial % 4 == 0 else 1, S) for _ in range(B)]
        dtype = torch.float32 if trial % 2 else torch.bfloat16
        q, k, v, sl = _rand_case(B, Hkv * G, Hkv, d, S, seqlens, dtype, seed=100 + trial)
        scale = 1.0 / math.sqrt(d)
        out, lse = oracle.attention(q, k, v, sl, scale, lib_handle=lib_handle)
        bo, bl = brute_force(q, k, v, sl, scale)
        np.testing.assert_allclose(out, bo, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-12)


def check_sdpa(lib_handle=None):
    for seed, (B, Hq, Hkv, d, S, dtype) in enumerate([
            (2, 8, 2, 64, 700, torch.float32), (3, 4, 4, 32, 300, torch.bfloat16),
            (1, 6, 3, 128, 257, torch.bfloat16)]):
        g = np.random.default_rng(seed)
        seqlens = g.integers(1, S + 1, size=B)
        q, k, v, sl = _rand_case(B, Hq, Hkv, d, S, seqlens, dtype, seed=200 + seed)
        scale = 1.0 / math.sqrt(d)
        out, lse = oracle.attention(q, k, v, sl, scale, lib_handle=lib_handle)
        ro, rl = sdpa_reference(q, k, v, sl, scale)
        np.testing.assert_allclose(out, ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, rl, rtol=1e-13, atol=1e-12)


def check_golden(lib_handle=None):
    doc = json.load(open(GOLDEN))
    for case in doc["attention_cases"]:
        dt = torch.float32 if case["dtype"] == "f32" else torch.bfloat16
        q = torch.tensor(case["q"], dtype=torch.float64).to(dt)
        k = torch.tensor(case["k"], dtype=torch.float64).to(dt)
        v = torch.tensor(case["v"], dtype=torch.float64).to(dt)
        # every fixture value is exactly representable in its dtype
        assert torch.equal(q.to(torch.float64), torch.tensor(case["q"], dtype=torch.float64))
        out, lse = oracle.attention(q, k, v, case["seqlens"], case["scale"], lib_handle=lib_handle)
        exp_lse = np.array([[float(x) for x in row] for row in case["lse"]])
        np.testing.assert_allclose(out, np.array(case["out"]), rtol=0, atol=1e-13, err_msg=case["name"])
        np.testing.assert_allclose(lse, exp_lse, rtol=0, atol=1e-13, err_msg=case["name"])


def check_tree_shapes(lib_handle=None):
    """One chunk == P chunks merged along any tree (associativity, commutativity)."""
    B, Hq, Hkv, d, S = 2, 4, 2, 16, 1500
    q, k, v, sl = _rand_case(B, Hq, Hkv, d, S, [1500, 1100], torch.bfloat16, seed=7, k_scale=2.0)
    out, lse = oracle.attention(q, k, v, sl, lib_handle=lib_handle)
    rng = np.random.default_rng(3)
    for P in (1, 2, 3, 7, 8, 64, 1000):
        # random cut points, including empty slices
        starts = np.zeros((B, P), dtype=np.int64)
        ends = np.zeros((B, P), dtype=np.int64)
        for b in range(B):
            cuts = np.sort(rng.integers(0, int(sl[b]) + 1, size=P - 1))
            edges = np.concatenate([[0], cuts, [int(sl[b])]])
            starts[b], ends[b] = edges[:-1], edges[1:]
        po, pl, pm = oracle.partials(q, k, v, sl, starts, ends, lib_handle=lib_handle)
        shapes = [("left", 2, 0), ("right", 2, 0), ("balanced", 2, 0), ("balanced", 3, 0),
                  ("balanced", 8, 0), ("random", 2, 11), ("random", 2, 12)]
        for shape, arity, seed in shapes:
            o2, l2 = oracle.combine(po, pl, pm, shape=shape, k=arity, seed=seed)
            np.testing.assert_allclose(o2, out, rtol=0, atol=1e-12, err_msg=f"P={P} {shape}/{arity}")
            np.testing.assert_allclose(l2, lse, rtol=1e-13, atol=1e-12, err_msg=f"P={P} {shape}/{arity}")


def check_permutation_and_linearity(lib_handle=None):
    """Reordering tokens (K and V rows together) leaves the result unchanged;
    out is linear in V for fixed K."""
    B, Hq, Hkv, d, S = 1, 4, 2, 8, 64
    q, k, v, sl = _rand_case(B, Hq, Hkv, d, S, [64], torch.float32, seed=5)
    out, lse = oracle.attention(q, k, v, sl, lib_handle=lib_handle)
    perm = torch.randperm(S, generator=torch.Generator().manual_seed(9))
    o2, l2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], sl, lib_handle=lib_handle)
    np.testing.assert_allclose(o2, out, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, lse, rtol=0, atol=1e-13)
    v2 = torch.randn(v.shape, generator=torch.Generator().manual_seed(10))
    oa, _ = oracle.attention(q, k, v2, sl, lib_handle=lib_handle)
    ob, _ = oracle.attention(q, k, v + v2, sl, lib_handle=lib_handle)
    # v + v2 is rounded to float32, so compare against the rounded sum's pieces loosely
    np.testing.assert_allclose(ob, out + oa, rtol=0, atol=1e-6)


BATTERY = [check_brute_force, check_sdpa, check_golden, check_tree_shapes,
           check_permutation_and_linearity]


@pytest.mark.parametrize("check", BATTERY, ids=lambda f: f.__name__)
def test_battery(check):
    check()


# ---------------------------------------------------------------------------
# Closed forms and invariants on larger inputs
# ---------------------------------------------------------------------------

def test_identical_keys_give_mean_of_v():
    B, Hq, Hkv, d, S = 2, 4, 2, 32, 900
    q, k, v, sl = _rand_case(B, Hq, Hkv, d, S, [900, 17], torch.float32, seed=21)
    k[:] = k[:, :, :1, :]                   # every key equals the first one
    out, lse = oracle.attention(q, k, v, sl)
    scale = 1.0 / math.sqrt(d)
    for b in range(B):
        n = int(sl[b])
        for h in range(Hq):
            g = h // (Hq // Hkv)
            vv = v[b, g, :n].to(torch.float64).numpy()
            mean = np.array([math.fsum(vv[:, i]) / n for i in range(d)])
            s = scale * math.fsum(float(x) * float(y) for x, y in
                                  zip(q[b, h].double(), k[b, g, 0].double()))
            np.testing.assert_allclose(out[b, h], mean, rtol=0, atol=1e-13)
            assert abs(lse[b, h] - (s + math.log(n))) < 1e-12


def test_dominant_logit_returns_its_value_row():
    B, Hq, Hkv, d, S = 1, 2, 2, 64, 256
    q, k, v, sl = _rand_case(B, Hq, Hkv, d, S, [256], torch.float32, seed=22)
    scale = 1.0 / math.sqrt(d)
    target = 60.0
    for h in range(Hq):
        qh = q[0, h].double()
        key = (target / scale) * qh / float(qh @ qh)
        k[0, h, 123] = key.float()
    out, lse = oracle.attention(q, k, v, sl)
    for h in range(Hq):
        s = scale * (k[0, h, :256].double() @ q[0, h].double()).numpy()
        gap = s[123] - np.max(np.delete(s, 123))
        assert gap > 40
        bound = 255 * math.exp(-gap) * 2 * float(v.abs().max())
        np.testing.assert_allclose(out[0, h], v[0, h, 123].double().numpy(), rtol=0, atol=bound + 1e-13)
        assert abs(lse[0, h] - s[123]) < 255 * math.exp(-gap) + 1e-12


def test_single_token_is_exact():
    q, k, v, sl = _rand_case(3, 4, 2, 16, 8, [1, 1, 1], torch.bfloat16, seed=23)
    out, lse = oracle.attention(q, k, v, sl)
    scale = 0.25
    for b in range(3):
        for h in range(4):
            g = h // 2
            np.testing.assert_array_equal(out[b, h], v[b, g, 0].double().numpy())
            s = scale * math.fsum(float(x) * float(y) for x, y in zip(q[b, h].double(), k[b, g, 0].double()))
            assert abs(lse[b, h] - s) < 1e-13


def test_empty_sequence_and_identity_state():
    q, k, v, sl = _rand_case(2, 2, 1, 8, 4, [0, 3], torch.float32, seed=24)
    out, lse = oracle.attention(q, k, v, sl)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(out[1])) and np.all(np.isfinite(lse[1]))
    # merging with the identity state changes nothing; two empties stay empty
    po, pl, pm = oracle.partials(q, k, v, sl, [[0], [0]], [[4], [4]])
    s = (po[:, :, 0], pl[:, :, 0], pm[:, :, 0])
    e = oracle.empty_state(pl.shape[:2], 8)
    for a, b in ((s, e), (e, s)):
        o2, l2, m2 = oracle.merge(a, b)
        np.testing.assert_array_equal(o2, s[0])
        np.testing.assert_array_equal(l2, s[1])
        np.testing.assert_array_equal(m2, s[2])
    o3, l3, m3 = oracle.merge(e, e)
    assert np.all(o3 == 0) and np.all(l3 == 0) and np.all(np.isneginf(m3))


def test_shift_of_m_shifts_lse_only():
    q, k, v, sl = _rand_case(1, 4, 2, 16, 300, [300], torch.float32, seed=25)
    st, en = oracle.even_bounds(sl, 5)
    po, pl, pm = oracle.partials(q, k, v, sl, st, en)
    o1, l1 = oracle.combine(po, pl, pm)
    o2, l2 = oracle.combine(po, pl, pm + 17.25)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-14)
    np.testing.assert_allclose(l2, l1 + 17.25, rtol=0, atol=1e-12)


def test_bounds_on_lse_and_out():
    q, k, v, sl = _rand_case(2, 8, 2, 64, 2000, [2000, 333], torch.bfloat16, seed=26, k_scale=3.0)
    out, lse = oracle.attention(q, k, v, sl)
    scale = 1.0 / 8.0
    for b in range(2):
        n = int(sl[b])
        for h in range(8):
            g = h // 4
            s = scale * (k[b, g, :n].double() @ q[b, h].double()).numpy()
            assert s.max() - 1e-12 <= lse[b, h] <= s.max() + math.log(n) + 1e-12
            vv = v[b, g, :n].double().numpy()
            assert np.all(out[b, h] >= vv.min(axis=0) - 1e-12)
            assert np.all(out[b, h] <= vv.max(axis=0) + 1e-12)


def test_merge_closed_form():
    doc = json.load(open(GOLDEN))
    for case in doc["merge_cases"]:
        a = (np.array(case["a"]["o"]), np.array(case["a"]["l"]), np.array(case["a"]["m"]))
        b = (np.array(case["b"]["o"]), np.array(case["b"]["l"]), np.array(case["b"]["m"]))
        for x, y in ((a, b), (b, a)):       # commutative
            o, l, m = oracle.merge(x, y)
            np.testing.assert_allclose(o, case["merged"]["o"], rtol=0, atol=1e-15)
            assert abs(l - case["merged"]["l"]) < 1e-15 and m == case["merged"]["m"]
            out, lse = oracle.normalize((o, l, m))
            np.testing.assert_allclose(out, case["out"], rtol=0, atol=1e-15)
            assert abs(lse - case["lse"]) < 1e-15


def test_planted_spike_reaches_its_logit():
    """The ragged workload's planted key gives every head of its group a logit of ~12."""
    w = workloads.custom(2, 8, 2, 128, 512, seqlens=None, spike_logit=12.0, pad_nan=True, seed=3)
    inp = workloads.make_inputs(w)
    q, k, sl, pos = inp["q"], inp["k"], inp["seqlens"], inp["spike_pos"]
    for b in range(2):
        n = int(sl[b])
        assert torch.isnan(k[b, :, n:]).all() if n < 512 else True
        for g in range(2):
            t = int(pos[b, g])
            assert 0 <= t < n
            for h in range(g * 4, g * 4 + 4):
                s = w.softmax_scale * float(k[b, g, t].double() @ q[b, h].double())
                assert abs(s - 12.0) < 0.2     # key rounded to bf16


def test_oracle_handles_nan_padding_beyond_lengths():
    w = workloads.custom(2, 4, 2, 16, 64, seqlens=None, pad_nan=True, seed=4)
    inp = workloads.make_inputs(w)
    out, lse = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    assert np.isfinite(out).all() and np.isfinite(lse).all()
