"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that
the pin battery catches every one of them.

Each mutant is the oracle's C source with one textual change (a dropped term, a
wrong sign or index, a swapped operand), compiled to a temporary library.  The
merge operator's mutants replace ``oracle.merge`` for the duration of a check.
"""
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from tests import test_oracle_multi as multi
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "tree_attn_oracle.c")

C_MUTANTS = {
    "gqa_index_modulo": ("const int g = h / G;", "const int g = h % Hkv;"),
    "dropped_scale": ("s[t] = scale * acc;", "s[t] = acc;"),
    "value_from_keys": ("o[i] += w * widen(v, kv_dtype, kvoff + t * d + i);",
                        "o[i] += w * widen(k, kv_dtype, kvoff + t * d + i);"),
    "exp_sign_flipped": ("double w = exp(s[t] - M);", "double w = exp(M - s[t]);"),
    "lse_missing_max": ("lse[bh] = M + log(L);", "lse[bh] = log(L);"),
    "not_normalised": ("o[i] = o[i] / L;", "o[i] = o[i];"),
    "first_token_dropped": ("double w = exp(s[t] - M);\n            L += w;",
                            "double w = exp(s[t] - M);\n            if (t == 0) continue;\n            L += w;"),
    "bf16_widen_shift": ("((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    "query_head_zero": ("widen(q, q_dtype, qoff + i) * widen(k, kv_dtype, kvoff + t * d + i)",
                        "widen(q, q_dtype, (int64_t)b * Hq * d + i) * widen(k, kv_dtype, kvoff + t * d + i)"),
    "partial_no_max_shift": ("double e = exp(s[t] - m);", "double e = exp(s[t]);"),
    "partial_l_counts_tokens": ("l += e;", "l += 1.0;"),
    "partial_value_from_keys": ("o[i] += e * widen(v, kv_dtype, kvoff + (t0 + t) * d + i);",
                                "o[i] += e * widen(k, kv_dtype, kvoff + (t0 + t) * d + i);"),
}


def _build_mutant(name, old, new, tmpdir):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    path = os.path.join(tmpdir, f"mut_{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    so = os.path.join(tmpdir, f"libmut_{name}.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", path, "-o", so, "-lm"], check=True,
                   capture_output=True)
    return oracle._load(so)


def _battery_fails(lib_handle):
    for check in pins.BATTERY:
        try:
            with np.errstate(all="ignore"):
                check(lib_handle=lib_handle)
        except (AssertionError, ValueError, FloatingPointError):
            return check.__name__
    return None


@pytest.fixture(scope="module")
def tmpdir():
    with tempfile.TemporaryDirectory() as d:
        yield d


def test_unmutated_copy_passes(tmpdir):
    lib = _build_mutant("none", "#include <math.h>", "#include <math.h>", tmpdir)
    assert _battery_fails(lib) is None


@pytest.mark.parametrize("name", sorted(C_MUTANTS))
def test_c_mutant_is_caught(name, tmpdir):
    old, new = C_MUTANTS[name]
    lib = _build_mutant(name, old, new, tmpdir)
    caught_by = _battery_fails(lib)
    assert caught_by is not None, f"mutant {name} survived every pin"


def _merge_beta_uses_a(a, b):
    o_a, l_a, m_a = a
    o_b, l_b, m_b = b
    m_new = np.maximum(m_a, m_b)
    m_ref = np.where(np.isneginf(m_new), 0.0, m_new)
    alpha = np.exp(m_a - m_ref)
    beta = np.exp(m_a - m_ref)
    return alpha[..., None] * o_a + beta[..., None] * o_b, alpha * l_a + beta * l_b, m_new


def _merge_min_instead_of_max(a, b):
    o_a, l_a, m_a = a
    o_b, l_b, m_b = b
    m_new = np.minimum(m_a, m_b)
    m_ref = np.where(np.isneginf(m_new), 0.0, m_new)
    alpha = np.exp(np.where(np.isneginf(m_a), -np.inf, m_a - m_ref))
    beta = np.exp(np.where(np.isneginf(m_b), -np.inf, m_b - m_ref))
    return alpha[..., None] * o_a + beta[..., None] * o_b, alpha * l_a + beta * l_b, m_new


def _merge_l_not_rescaled(a, b):
    o_a, l_a, m_a = a
    o_b, l_b, m_b = b
    m_new = np.maximum(m_a, m_b)
    m_ref = np.where(np.isneginf(m_new), 0.0, m_new)
    alpha = np.exp(m_a - m_ref)
    beta = np.exp(m_b - m_ref)
    return alpha[..., None] * o_a + beta[..., None] * o_b, l_a + l_b, m_new


@pytest.mark.parametrize("mutant", [_merge_beta_uses_a, _merge_min_instead_of_max, _merge_l_not_rescaled],
                         ids=lambda f: f.__name__)
def test_merge_mutant_is_caught(mutant, monkeypatch):
    monkeypatch.setattr(oracle, "merge", mutant)
    caught = None
    for check in (pins.check_tree_shapes, pins.test_merge_closed_form):
        try:
            with np.errstate(all="ignore"):
                check()
        except AssertionError:
            caught = check.__name__
            break
    assert caught is not None


MULTI_MUTANTS = {
    "causal_off_by_one": ("n = n - nq + 1 + i;", "n = n - nq + i;"),
    "causal_reversed": ("n = n - nq + 1 + i;", "n = n - i;"),
    "query_row_from_head": ("const int64_t qoff = w * d;", "const int64_t qoff = bh * nq * d;"),
    "kv_head_from_query": ("const int g = h / G;\n        int64_t n = seqlens[b];",
                           "const int g = (h + i) / G % Hkv;\n        int64_t n = seqlens[b];"),
}


def _multi_battery_fails(lib_handle):
    import oracle as orc
    real = orc.lib
    orc_lib = lambda: lib_handle
    try:
        orc.lib = orc_lib
        for check in (multi.test_single_query_equals_definition,
                      lambda: multi.test_multi_query_brute_force(True),
                      multi.test_multi_query_against_sdpa_with_causal_mask):
            try:
                with np.errstate(all="ignore"):
                    check()
            except (AssertionError, ValueError):
                return True
        return False
    finally:
        orc.lib = real


@pytest.mark.parametrize("name", sorted(MULTI_MUTANTS))
def test_multi_query_mutant_is_caught(name, tmpdir):
    old, new = MULTI_MUTANTS[name]
    src = open(SRC).read()
    start = src.index("int oracle_attention_multi_f64")
    assert src.count(old, start) >= 1, name
    mutated = src[:start] + src[start:].replace(old, new, 1)
    path = os.path.join(tmpdir, f"mmut_{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    so = os.path.join(tmpdir, f"libmmut_{name}.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", path, "-o", so, "-lm"], check=True,
                   capture_output=True)
    assert _multi_battery_fails(oracle._load(so)), f"mutant {name} survived"


FP8_MUTANTS = {
    "exponent_bias_8": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "subnormal_as_normal": ("v = ldexp((double)m / 8.0, -6);", "v = ldexp(1.0 + (double)m / 8.0, -6);"),
    "no_nan_code": ("if (e == 0xF && m == 0x7)\n        return NAN;", "if (0)\n        return NAN;"),
    "k_scale_dropped": ("(ks * oracle_e4m3_to_double(k8[kvoff + t * d + c]))",
                        "(oracle_e4m3_to_double(k8[kvoff + t * d + c]))"),
    "v_scale_from_k": ("const double ks = (double)k_scale[g], vs = (double)v_scale[g];",
                       "const double ks = (double)k_scale[g], vs = (double)k_scale[g];"),
}


@pytest.mark.parametrize("name", sorted(FP8_MUTANTS))
def test_fp8_mutant_is_caught(name, tmpdir):
    from tests import test_oracle_fp8 as fp8
    old, new = FP8_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = os.path.join(tmpdir, f"fmut_{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(tmpdir, f"libfmut_{name}.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", path, "-o", so, "-lm"], check=True,
                   capture_output=True)
    handle = oracle._load(so)
    real = oracle.lib
    oracle.lib = lambda: handle
    try:
        failed = False
        for check in (fp8.test_e4m3_decoder_matches_torch_for_every_code,
                      fp8.test_fp8_attention_matches_sdpa_on_dequantized_cache):
            try:
                with np.errstate(all="ignore"):
                    check()
            except (AssertionError, ValueError):
                failed = True
                break
        assert failed, f"mutant {name} survived"
    finally:
        oracle.lib = real
