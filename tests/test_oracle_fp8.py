"""Pins of the oracle's FP8 E4M3 path: the decoder against torch's float8_e4m3fn
(all 256 codes), and attention over a quantized cache against torch SDPA in
float64 on the exactly dequantized cache."""
import math

import numpy as np
import torch

import oracle
from softmax_tree_reduction_gb300 import workloads


def test_e4m3_decoder_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    np.testing.assert_array_equal(mine[~nan], ref[~nan])
    # a few values by hand: 0x38 = 1.0, 0x7e = 448, 0x01 = 2^-9 (smallest subnormal), 0xb0 = -0.5
    assert oracle.e4m3_to_double(0x38) == 1.0 and oracle.e4m3_to_double(0x7E) == 448.0
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9 and oracle.e4m3_to_double(0xB0) == -0.5


def test_fp8_attention_matches_sdpa_on_dequantized_cache():
    B, Hq, Hkv, d, S = 2, 8, 2, 128, 300
    g = torch.Generator().manual_seed(3)
    q = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, S, d, generator=g) * 2.0
    v = torch.randn(B, Hkv, S, d, generator=g)
    k8, ks = workloads.quantize_e4m3(k)
    v8, vs = workloads.quantize_e4m3(v)
    sl = [300, 123]
    out, lse = oracle.attention_e4m3(q, k8, v8, ks, vs, sl)
    kd = k8.to(torch.float64) * ks.double().view(1, -1, 1, 1)
    vd = v8.to(torch.float64) * vs.double().view(1, -1, 1, 1)
    G = Hq // Hkv
    for b in range(B):
        n = sl[b]
        qb = q[b].double()[:, None, :]
        kb = kd[b, :, :n].repeat_interleave(G, dim=0)
        vb = vd[b, :, :n].repeat_interleave(G, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, scale=1 / math.sqrt(d))
        np.testing.assert_allclose(out[b], ref[:, 0].numpy(), rtol=0, atol=1e-12)
        rl = torch.logsumexp((qb @ kb.transpose(1, 2))[:, 0] / math.sqrt(d), dim=-1)
        np.testing.assert_allclose(lse[b], rl.numpy(), rtol=1e-13, atol=1e-12)


def test_fp8_with_unit_scales_equals_the_float_definition():
    """Codes whose values are exact floats: the FP8 path equals the definition on those floats."""
    B, Hq, Hkv, d, S = 1, 4, 1, 16, 40
    g = torch.Generator().manual_seed(4)
    codes = torch.randint(0, 126, (2, B, Hkv, S, d), generator=g, dtype=torch.uint8)
    codes[:, :, :, :, ::2] |= 0x80                       # negative values too
    k8, v8 = codes[0], codes[1]
    kf = k8.view(torch.float8_e4m3fn).float()
    vf = v8.view(torch.float8_e4m3fn).float()
    q = torch.randn(B, Hq, d, generator=g) * 0.05
    o1, l1 = oracle.attention_e4m3(q, k8, v8, [1.0], [1.0], [S])
    o2, l2 = oracle.attention(q, kf, vf, [S])
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)
