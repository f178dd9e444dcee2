"""Float64 CPU oracle for Tree Attention's decode path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference leg of ``bench.py`` may import this package.  It
shares no code with the CUDA library and never imports it; the two meet only
through the seeded inputs of ``softmax_tree_reduction_gb300.workloads``.

What it restates (web pages on Tree Attention, arXiv:2408.04093):

* ``attention`` -- the exact result: softmax over the whole KV sequence taken
  with the global maximum logit ("Tree Attention Guide", section "Core
  Innovation 2", the Softmax(S)_j equation), written out in C
  (``tree_attn_oracle.c``) as a two-pass double-precision loop.
* ``attention_multi`` -- several queries per sequence (multi-query decode):
  query i of a row of N tokens sits at position N - nq + i and, when causal,
  attends to tokens [0, N - nq + i]; each query is the definition above over
  its token range (a reading: the pages describe one query per step).
* ``attention_e4m3`` -- the same over an FP8 E4M3 cache with one scale per KV
  head (an extension the pages do not describe): the cache is widened exactly
  from the E4M3 definition and multiplied by its scale, then the definition
  above applies.
* ``partials`` -- the local partial attention state (o, l, m) of one KV slice
  ("Core Innovation 1", item 2 "Local Independent Partial Attention").
* ``merge`` -- the merge operator (+) of two states ("The Tree Reduction Merge
  Operator": m = max(m_A, m_B), alpha = exp(m_A - m), beta = exp(m_B - m),
  l = alpha l_A + beta l_B, o = alpha o_A + beta o_B).
* ``tree_reduce`` -- (+) applied along a tree of any shape; the page states the
  operator is associative and commutative, so every shape must agree.
* ``normalize`` -- the root step O = o / l, plus lse = m + ln l.

Readings where the pages are silent: the empty state (o=0, l=0, m=-inf) is the
identity of (+) (a merge whose new maximum is -inf yields the empty state
instead of NaN); lse is in natural-log units; an empty sequence normalises to
out = 0, lse = -inf; query head h reads KV head h // (Hq // Hkv).
"""
from __future__ import annotations

import ctypes
import os
import random
import subprocess
import sys
import threading
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tree_attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the C oracle with gcc (OpenMP when available); return the .so path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", src, "-o", out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(out + ".tmp", out)
    return out


def _load(path: str | None = None):
    lib = ctypes.CDLL(path or build())
    p = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_attention_f64.argtypes = [i32, i32, i32, i32, i64, p, i32, p, p, i32, p, dbl, p, p, i32]
    lib.oracle_attention_f64.restype = i32
    lib.oracle_partials_f64.argtypes = [i32, i32, i32, i32, i64, p, i32, p, p, i32, p, dbl,
                                        i32, p, p, p, p, p, i32]
    lib.oracle_partials_f64.restype = i32
    lib.oracle_attention_multi_f64.argtypes = [i32, i32, i32, i32, i64, i32, i32, p, i32, p, p, i32, p,
                                               dbl, p, p, i32]
    lib.oracle_attention_multi_f64.restype = i32
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_double.restype = dbl
    lib.oracle_attention_e4m3_f64.argtypes = [i32, i32, i32, i32, i64, i32, i32, p, i32, p, p, p, p, p,
                                              dbl, p, p, i32]
    lib.oracle_attention_e4m3_f64.restype = i32
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = i32
    return lib


def lib():
    """The loaded C oracle (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load()
        return _lib


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def _as_raw(x):
    """(contiguous numpy array of the stored bits, dtype code) for a torch tensor
    or numpy array holding float32 or bfloat16 values."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16), BF16
        if x.dtype == torch.float32:
            return x.numpy(), F32
        raise TypeError(f"oracle takes float32 or bfloat16 tensors, got {x.dtype}")
    a = np.ascontiguousarray(x)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"oracle takes float32 arrays or uint16 bfloat16 bit patterns, got {a.dtype}")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def attention(q, k, v, seqlens, scale: float | None = None, threads: int = 0, lib_handle=None):
    """Exact decode attention in float64.

    q: [B, Hq, d]; k, v: [B, Hkv, S, d] (float32 or bfloat16); seqlens: [B] ints.
    Returns (out [B, Hq, d] float64, lse [B, Hq] float64).
    """
    qa, qt = _as_raw(q)
    ka, kt = _as_raw(k)
    va, vt = _as_raw(v)
    if kt != vt:
        raise TypeError("k and v must share a dtype")
    B, Hq, d = qa.shape
    _, Hkv, S, d2 = ka.shape
    if d2 != d or va.shape != ka.shape or ka.shape[0] != B:
        raise ValueError("shape mismatch")
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32).reshape(B))
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((B, Hq, d), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    L = lib_handle or lib()
    rc = L.oracle_attention_f64(B, Hq, Hkv, d, S, _ptr(qa), qt, _ptr(ka), _ptr(va), kt, _ptr(sl),
                                float(scale), _ptr(out), _ptr(lse), int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attention_f64 failed with code {rc}")
    return out, lse


def attention_multi(q, k, v, seqlens, causal: bool = True, scale: float | None = None,
                    threads: int = 0, lib_handle=None):
    """Several queries per sequence: q [B, Hq, nq, d]; query i of row b sits at
    position N_b - nq + i and, when causal, sees tokens [0, N_b - nq + i].
    Returns (out [B, Hq, nq, d], lse [B, Hq, nq]) in float64."""
    qa, qt = _as_raw(q)
    ka, kt = _as_raw(k)
    va, vt = _as_raw(v)
    B, Hq, nq, d = qa.shape
    _, Hkv, S, _ = ka.shape
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32).reshape(B))
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((B, Hq, nq, d), dtype=np.float64)
    lse = np.zeros((B, Hq, nq), dtype=np.float64)
    L = lib_handle or lib()
    rc = L.oracle_attention_multi_f64(B, Hq, Hkv, d, S, nq, int(bool(causal)), _ptr(qa), qt, _ptr(ka),
                                      _ptr(va), kt, _ptr(sl), float(scale), _ptr(out), _ptr(lse),
                                      int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attention_multi_f64 failed with code {rc}")
    return out, lse


def e4m3_to_double(code: int, lib_handle=None) -> float:
    """One FP8 E4M3 code widened from the format's definition."""
    return float((lib_handle or lib()).oracle_e4m3_to_double(int(code) & 0xFF))


def attention_e4m3(q, k8, v8, k_scale, v_scale, seqlens, causal: bool = True,
                   scale: float | None = None, threads: int = 0, lib_handle=None):
    """Decode attention over an FP8 E4M3 cache with one scale per KV head.

    q: [B, Hq, d] or [B, Hq, nq, d] (float32 / bfloat16); k8, v8: uint8 codes
    [B, Hkv, S, d] (or torch float8_e4m3fn); k_scale, v_scale: [Hkv] floats.
    K = k_scale[g] * e4m3(k8), V likewise.  Returns float64 (out, lse) shaped like q.
    """
    try:
        import torch
        if isinstance(k8, torch.Tensor):
            k8 = k8.detach().cpu().contiguous().view(torch.uint8).numpy()
            v8 = v8.detach().cpu().contiguous().view(torch.uint8).numpy()
    except ImportError:  # pragma: no cover
        pass
    qa, qt = _as_raw(q)
    single = qa.ndim == 3
    if single:
        qa = qa[:, :, None, :]
    B, Hq, nq, d = qa.shape
    ka = np.ascontiguousarray(k8, dtype=np.uint8)
    va = np.ascontiguousarray(v8, dtype=np.uint8)
    _, Hkv, S, _ = ka.shape
    ks = np.ascontiguousarray(np.asarray(k_scale, dtype=np.float32).reshape(Hkv))
    vs = np.ascontiguousarray(np.asarray(v_scale, dtype=np.float32).reshape(Hkv))
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32).reshape(B))
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((B, Hq, nq, d), dtype=np.float64)
    lse = np.zeros((B, Hq, nq), dtype=np.float64)
    qa = np.ascontiguousarray(qa)
    L = lib_handle or lib()
    rc = L.oracle_attention_e4m3_f64(B, Hq, Hkv, d, S, nq, int(bool(causal)), _ptr(qa), qt, _ptr(ka),
                                     _ptr(va), _ptr(ks), _ptr(vs), _ptr(sl), float(scale), _ptr(out),
                                     _ptr(lse), int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attention_e4m3_f64 failed with code {rc}")
    if single:
        return out[:, :, 0], lse[:, :, 0]
    return out, lse


def partials(q, k, v, seqlens, starts, ends, scale: float | None = None, threads: int = 0,
             lib_handle=None):
    """Partial states (o, l, m) of P KV slices per batch row.

    starts, ends: [B, P] token bounds (clipped to [0, seqlens[b])).
    Returns (o [B, Hq, P, d], l [B, Hq, P], m [B, Hq, P]) in float64.
    """
    qa, qt = _as_raw(q)
    ka, kt = _as_raw(k)
    va, vt = _as_raw(v)
    B, Hq, d = qa.shape
    _, Hkv, S, _ = ka.shape
    st = np.ascontiguousarray(np.asarray(starts, dtype=np.int64))
    en = np.ascontiguousarray(np.asarray(ends, dtype=np.int64))
    if st.ndim != 2 or st.shape != en.shape or st.shape[0] != B:
        raise ValueError("starts/ends must be [B, P]")
    P = st.shape[1]
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32).reshape(B))
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    po = np.zeros((B, Hq, P, d), dtype=np.float64)
    pm = np.zeros((B, Hq, P), dtype=np.float64)
    pl = np.zeros((B, Hq, P), dtype=np.float64)
    L = lib_handle or lib()
    rc = L.oracle_partials_f64(B, Hq, Hkv, d, S, _ptr(qa), qt, _ptr(ka), _ptr(va), kt, _ptr(sl),
                               float(scale), P, _ptr(st), _ptr(en), _ptr(po), _ptr(pm), _ptr(pl),
                               int(threads))
    if rc != 0:
        raise ValueError(f"oracle_partials_f64 failed with code {rc}")
    return po, pl, pm


# ---------------------------------------------------------------------------
# The merge operator and trees of merges (numpy float64, vectorised over any
# leading batch axes: o [..., d], l [...], m [...]).
# ---------------------------------------------------------------------------

def empty_state(shape: Sequence[int], d: int):
    """The identity state (o = 0, l = 0, m = -inf)."""
    return (np.zeros(tuple(shape) + (d,)), np.zeros(tuple(shape)), np.full(tuple(shape), -np.inf))


def merge(a, b):
    """(o, l, m) (+) (o, l, m): the page's four steps, with the empty state as identity."""
    o_a, l_a, m_a = a
    o_b, l_b, m_b = b
    m_new = np.maximum(m_a, m_b)
    # Where both inputs are empty, m_new = -inf and m_a - m_new is NaN; the
    # result there is the empty state, so use a finite stand-in maximum.
    m_ref = np.where(np.isneginf(m_new), 0.0, m_new)
    alpha = np.exp(m_a - m_ref)
    beta = np.exp(m_b - m_ref)
    l_new = alpha * l_a + beta * l_b
    o_new = alpha[..., None] * o_a + beta[..., None] * o_b
    return o_new, l_new, m_new


def normalize(state):
    """Root step: out = o / l, lse = m + ln l (out = 0, lse = -inf for the empty state)."""
    o, l, m = state
    empty = l == 0
    safe_l = np.where(empty, 1.0, l)
    out = np.where(empty[..., None], 0.0, o / safe_l[..., None])
    lse = np.where(empty, -np.inf, m + np.log(safe_l))
    return out, lse


def _split_states(po, pl, pm):
    P = pm.shape[-1]
    return [(po[..., p, :], pl[..., p], pm[..., p]) for p in range(P)]


def tree_reduce(states, shape="balanced", k: int = 2, seed: int = 0):
    """Merge a list of states along a tree.

    shape:
      "left"      ((s0 + s1) + s2) + ...
      "right"     s0 + (s1 + (s2 + ...))
      "balanced"  balanced k-ary tree, children in order
      "random"    random binary tree over a random permutation of the leaves
    """
    if not states:
        raise ValueError("no states")
    states = list(states)
    if shape == "left":
        acc = states[0]
        for s in states[1:]:
            acc = merge(acc, s)
        return acc
    if shape == "right":
        acc = states[-1]
        for s in reversed(states[:-1]):
            acc = merge(s, acc)
        return acc
    if shape == "balanced":
        if k < 2:
            raise ValueError("arity must be >= 2")
        level = states
        while len(level) > 1:
            nxt = []
            for i in range(0, len(level), k):
                group = level[i:i + k]
                acc = group[0]
                for s in group[1:]:
                    acc = merge(acc, s)
                nxt.append(acc)
            level = nxt
        return level[0]
    if shape == "random":
        rng = random.Random(seed)
        pool = states[:]
        rng.shuffle(pool)
        while len(pool) > 1:
            i = rng.randrange(len(pool) - 1)
            a, b = pool[i], pool[i + 1]
            if rng.random() < 0.5:
                a, b = b, a
            pool[i:i + 2] = [merge(a, b)]
        return pool[0]
    raise ValueError(f"unknown tree shape {shape!r}")


def combine(po, pl, pm, shape="balanced", k: int = 2, seed: int = 0):
    """Merge P partial states per (b, h) along a tree and normalise.

    po [..., P, d], pl [..., P], pm [..., P] -> (out [..., d], lse [...]).
    """
    return normalize(tree_reduce(_split_states(np.asarray(po, dtype=np.float64),
                                               np.asarray(pl, dtype=np.float64),
                                               np.asarray(pm, dtype=np.float64)),
                                 shape=shape, k=k, seed=seed))


def even_bounds(seqlens, P: int):
    """[B, P] starts/ends that cut each sequence into P contiguous, nearly equal slices
    (a convenience for tests; any cut is valid input to ``partials``)."""
    sl = np.asarray(seqlens, dtype=np.int64).reshape(-1)
    starts = np.zeros((sl.size, P), dtype=np.int64)
    ends = np.zeros((sl.size, P), dtype=np.int64)
    for b, n in enumerate(sl):
        c = -(-int(n) // P) if n > 0 else 0
        for p in range(P):
            starts[b, p] = min(p * c, n)
            ends[b, p] = min((p + 1) * c, n)
    return starts, ends


__all__ = ["attention", "attention_multi", "attention_e4m3", "e4m3_to_double", "partials", "merge", "normalize", "tree_reduce", "combine", "empty_state",
           "even_bounds", "build", "lib", "max_threads", "F32", "BF16"]

if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
