"""Pins of the oracle's multi-query decode (several queries per sequence, causal
over the last nq positions), independent of its code path."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.test_oracle_pins import _rand_case, brute_force


def _q(B, Hq, nq, d, dtype, seed):
    return torch.randn(B, Hq, nq, d, generator=torch.Generator().manual_seed(seed)).to(dtype)


def test_single_query_equals_definition():
    q, k, v, sl = _rand_case(2, 8, 2, 32, 300, [300, 77], torch.bfloat16, seed=31)
    o1, l1 = oracle.attention(q, k, v, sl)
    for causal in (True, False):
        om, lm = oracle.attention_multi(q[:, :, None, :], k, v, sl, causal=causal)
        np.testing.assert_array_equal(om[:, :, 0], o1)
        np.testing.assert_array_equal(lm[:, :, 0], l1)


@pytest.mark.parametrize("causal", [True, False])
def test_multi_query_brute_force(causal):
    """Each query against brute force over its own token range."""
    rng = np.random.default_rng(3)
    for trial in range(6):
        B, Hkv, G, nq, d, S = 2, rng.integers(1, 3), rng.integers(1, 3), rng.integers(1, 5), 4, 12
        Hq = Hkv * G
        sl = rng.integers(0, S + 1, size=B)
        q = _q(B, Hq, nq, d, torch.float32, 40 + trial)
        _, k, v, _ = _rand_case(B, Hq, Hkv, d, S, sl, torch.float32, seed=50 + trial)
        om, lm = oracle.attention_multi(q, k, v, sl, causal=causal)
        for i in range(nq):
            n_i = [max(0, int(n) - nq + 1 + i) if causal else int(n) for n in sl]
            bo, bl = brute_force(q[:, :, i, :], k, v, n_i, 1.0 / math.sqrt(d))
            np.testing.assert_allclose(om[:, :, i], bo, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lm[:, :, i], bl, rtol=0, atol=1e-12)


def test_multi_query_against_sdpa_with_causal_mask():
    B, Hq, Hkv, nq, d, S = 2, 8, 2, 4, 64, 500
    sl = [500, 333]
    q = _q(B, Hq, nq, d, torch.bfloat16, 7)
    _, k, v, _ = _rand_case(B, Hq, Hkv, d, S, sl, torch.bfloat16, seed=8)
    om, lm = oracle.attention_multi(q, k, v, sl, causal=True)
    G = Hq // Hkv
    for b in range(B):
        n = sl[b]
        qb = q[b].double()                                              # [Hq, nq, d]
        kb = k[b, :, :n].double().repeat_interleave(G, dim=0)          # [Hq, n, d]
        vb = v[b, :, :n].double().repeat_interleave(G, dim=0)
        pos = torch.arange(n)[None, :]
        qpos = (n - nq + torch.arange(nq))[:, None]
        mask = pos <= qpos                                              # [nq, n]
        ref = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask,
                                                               scale=1 / math.sqrt(d))
        np.testing.assert_allclose(om[b], ref.numpy(), rtol=0, atol=1e-12)
        sc = (qb @ kb.transpose(1, 2)) / math.sqrt(d)
        ref_l = torch.logsumexp(sc.masked_fill(~mask, -math.inf), dim=-1)
        np.testing.assert_allclose(lm[b], ref_l.numpy(), rtol=1e-13, atol=1e-12)


def test_short_rows_give_empty_queries():
    q = _q(1, 2, 4, 8, torch.float32, 9)
    _, k, v, _ = _rand_case(1, 2, 1, 8, 4, [2], torch.float32, seed=10)
    om, lm = oracle.attention_multi(q, k, v, [2], causal=True)
    # N = 2, nq = 4: queries 0 and 1 see max(0, 2-4+1+i) = 0 tokens, query 2 one, query 3 two
    assert np.all(om[0, :, :2] == 0) and np.all(np.isneginf(lm[0, :, :2]))
    np.testing.assert_array_equal(om[0, :, 2], np.broadcast_to(v[0, 0, 0].double().numpy(), (2, 8)))
