"""Seeded synthetic decode-attention inputs.

This module only draws inputs.  It holds none of the attention arithmetic, so
both the CUDA library's tests and the float64 oracle can take their inputs
from here without sharing any of the method.

Every tensor is drawn on the host with ``torch.Generator('cpu')`` in a fixed
order (seqlens, then q, then K per (b, kv-head), then V per (b, kv-head), then
the planted spikes), as float32 N(0, 1), scaled and then rounded to the stored
dtype.  The same bytes go to the GPU and to the oracle.

Layouts: q [B, Hq, d]; K, V [B, Hkv, S, d] (S = cache capacity); seqlens [B]
int32.  Cache rows at positions >= seqlens[b] are filled with NaN when
``pad_nan`` is set, so that any read of an invalid row shows up in the output.

The workloads are the shapes of the Tree Attention pages' decode setting
(single query per head over a long KV cache; Llama-shaped GQA layers); no
model weights or datasets are involved.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    max_seqlen: int                 # cache capacity S
    kv_dtype: torch.dtype
    q_dtype: torch.dtype
    seed: int = 0
    seqlen: Optional[int] = None    # every row's length; None => ragged
    ragged_range: Optional[tuple] = None  # inclusive [lo, hi] for ragged rows
    k_scale: float = 1.0
    spike_logit: Optional[float] = None   # planted per-(b, kv-head) logit
    pad_nan: bool = False
    scale: Optional[float] = None   # None => 1/sqrt(head_dim)
    description: str = ""

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.head_dim)

    def kv_bytes(self, seqlens) -> int:
        """Algorithmic bytes: every valid K and V element read once."""
        es = torch.empty((), dtype=self.kv_dtype).element_size()
        return int(2 * int(np.sum(np.asarray(seqlens, dtype=np.int64))) * self.num_kv_heads
                   * self.head_dim * es)


# The five decode workloads (sizes as named in the benchmark plan).
TINY_EXACT = Workload(
    "tiny_exact", 1, 1, 1, 64, 4096, torch.float32, torch.float32, seed=0, seqlen=4096,
    description="B1 Hq1 Hkv1 d64 N4096 fp32, q,K,V ~ N(0,1), scale 1/8, 8 splits")
LLAMA31_8B = Workload(
    "llama3.1-8b-decode-layer", 1, 32, 8, 128, 131072, torch.bfloat16, torch.bfloat16, seed=0,
    seqlen=131072, k_scale=0.5,
    description="B1 Hq32 Hkv8 (GQA 4:1) d128 bf16 KV, 131072 tokens, K ~ 0.5 N(0,1)")
BATCHED_RAGGED = Workload(
    "batched-ragged-decode", 16, 32, 8, 128, 65536, torch.bfloat16, torch.bfloat16, seed=0,
    ragged_range=(8192, 65536), spike_logit=12.0, pad_nan=True,
    description="B16 Hq32 Hkv8 d128 bf16 KV, seqlens ~ U[8192, 65536], planted +12 logit per "
                "(b, kv-head), NaN beyond each row's length")
LLAMA3_70B = Workload(
    "llama3-70b-decode-layer", 4, 64, 8, 128, 262144, torch.bfloat16, torch.bfloat16, seed=0,
    seqlen=262144,
    description="B4 Hq64 Hkv8 (GQA 8:1) d128 bf16 KV, 262144 tokens per row")
MILLION_TOKEN = Workload(
    "million-token-decode-layer", 1, 32, 8, 128, 1048576, torch.bfloat16, torch.bfloat16, seed=0,
    seqlen=1048576,
    description="B1 Hq32 Hkv8 d128 bf16 KV, 1048576 tokens (4 GiB K+V)")

WORKLOADS = {w.name: w for w in (TINY_EXACT, LLAMA31_8B, BATCHED_RAGGED, LLAMA3_70B, MILLION_TOKEN)}


def custom(batch, num_q_heads, num_kv_heads, head_dim, max_seqlen, kv_dtype=torch.bfloat16,
           q_dtype=None, seed=0, seqlens=None, k_scale=1.0, spike_logit=None, pad_nan=False,
           scale=None, name="custom") -> Workload:
    """A small workload for tests; ``seqlens`` may be an int (all rows) or None
    (ragged over [1, max_seqlen])."""
    q_dtype = q_dtype or kv_dtype
    if isinstance(seqlens, int) or seqlens is None:
        return Workload(name, batch, num_q_heads, num_kv_heads, head_dim, max_seqlen, kv_dtype,
                        q_dtype, seed=seed, seqlen=seqlens,
                        ragged_range=None if seqlens is not None else (1, max_seqlen),
                        k_scale=k_scale, spike_logit=spike_logit, pad_nan=pad_nan, scale=scale)
    raise TypeError("seqlens must be an int or None; use make_inputs(..., seqlens=...) for lists")


def _nan_of(dtype):
    return torch.tensor(float("nan"), dtype=dtype)


def make_inputs(w: Workload, seqlens=None, device="cpu", pin: bool = False):
    """Draw the inputs of workload ``w``.

    Returns a dict with q [B,Hq,d], k, v [B,Hkv,S,d] in their stored dtypes,
    seqlens [B] int32 (host tensor) and, when spikes are planted, the spike
    positions [B, Hkv].  ``seqlens`` overrides the workload's lengths.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed))
    B, Hq, Hkv, d, S = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_seqlen
    if seqlens is not None:
        sl = torch.as_tensor(seqlens, dtype=torch.int32).reshape(B).clone()
    elif w.seqlen is not None:
        sl = torch.full((B,), int(w.seqlen), dtype=torch.int32)
    else:
        lo, hi = w.ragged_range
        sl = torch.randint(int(lo), int(hi) + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    if int(sl.min()) < 0 or int(sl.max()) > S:
        raise ValueError("seqlens outside [0, max_seqlen]")

    q = torch.randn(B, Hq, d, generator=g, dtype=torch.float32).to(w.q_dtype)
    k = torch.empty(B, Hkv, S, d, dtype=w.kv_dtype, pin_memory=pin)
    v = torch.empty(B, Hkv, S, d, dtype=w.kv_dtype, pin_memory=pin)
    for dst, mult in ((k, w.k_scale), (v, 1.0)):
        for b in range(B):
            for h in range(Hkv):
                x = torch.randn(S, d, generator=g, dtype=torch.float32)
                if mult != 1.0:
                    x.mul_(mult)
                dst[b, h].copy_(x)
    if w.pad_nan:
        for b in range(B):
            n = int(sl[b])
            if n < S:
                k[b, :, n:, :] = _nan_of(w.kv_dtype)
                v[b, :, n:, :] = _nan_of(w.kv_dtype)

    out = {"q": q, "k": k, "v": v, "seqlens": sl}
    if w.spike_logit is not None:
        out["spike_pos"] = plant_spikes(q, k, sl, w.group, w.softmax_scale, w.spike_logit, g)
    if device != "cpu":
        out = {key: (t.to(device) if key in ("q", "k", "v", "seqlens") else t)
               for key, t in out.items()}
    return out


def plant_spikes(q, k, seqlens, group, scale, logit, gen):
    """Overwrite one key per (b, kv-head) so that every query head of the group
    sees logit ``logit`` there.

    The key is the minimum-norm solution of scale * Q_g k = logit * 1, where
    Q_g holds the group's (stored, rounded) query rows, then rounded to the
    cache dtype.  Positions are drawn uniformly in [0, seqlens[b]).
    Returns the positions [B, Hkv] (int64).
    """
    B, Hkv = k.shape[0], k.shape[1]
    pos = torch.zeros(B, Hkv, dtype=torch.int64)
    qd = q.to(torch.float64).numpy()
    for b in range(B):
        n = int(seqlens[b])
        for h in range(Hkv):
            t = int(torch.randint(0, max(n, 1), (1,), generator=gen))
            pos[b, h] = t
            if n == 0:
                continue
            Qg = qd[b, h * group:(h + 1) * group, :]          # [G, d]
            rhs = np.full(group, logit / scale)
            key = Qg.T @ np.linalg.solve(Qg @ Qg.T, rhs)       # min-norm solution
            k[b, h, t, :] = torch.from_numpy(key).to(k.dtype)
    return pos


def seqlens_of(w: Workload, seed: Optional[int] = None):
    """The row lengths ``make_inputs`` would draw, without drawing the tensors."""
    if w.seqlen is not None:
        return np.full(w.batch, w.seqlen, dtype=np.int64)
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed if seed is None else seed))
    lo, hi = w.ragged_range
    return torch.randint(int(lo), int(hi) + 1, (w.batch,), generator=g,
                         dtype=torch.int64).numpy()


def page_pool(k, v, seqlens, page_size, layout="NHD", extra_pages=3, seed=0, shuffle=True):
    """Scatter dense caches [B, Hkv, S, d] into shuffled page pools (``shuffle``
    False: each row's pages in order, one after another, as a fresh allocator
    would hand them out).

    Returns (k_pool, v_pool, block_table): pools of shape [num_pages, page_size,
    Hkv, d] ("NHD") or [num_pages, Hkv, page_size, d] ("HND", returned as a
    permuted [num_pages, page_size, Hkv, d] view); unused slots, junk pages and
    block-table entries past each row's pages are NaN / -1.  Pure data movement.
    """
    B, Hkv, S, d = k.shape
    sl = [int(x) for x in seqlens]
    pages = [(n + page_size - 1) // page_size for n in sl]
    max_pages = max(1, (S + page_size - 1) // page_size)
    num_pages = sum(pages) + extra_pages
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g) if shuffle else torch.arange(num_pages)
    shape = (num_pages, page_size, Hkv, d) if layout == "NHD" else (num_pages, Hkv, page_size, d)
    kp = torch.full(shape, float("nan"), dtype=k.dtype)
    vp = torch.full(shape, float("nan"), dtype=v.dtype)
    bt = torch.full((B, max_pages), -1, dtype=torch.int32)
    nxt = 0
    for b in range(B):
        for lp in range(pages[b]):
            phys = int(perm[nxt])
            nxt += 1
            bt[b, lp] = phys
            t0 = lp * page_size
            n = min(page_size, sl[b] - t0)
            src_k = k[b, :, t0:t0 + n, :]        # [Hkv, n, d]
            src_v = v[b, :, t0:t0 + n, :]
            if layout == "NHD":
                kp[phys, :n] = src_k.transpose(0, 1)
                vp[phys, :n] = src_v.transpose(0, 1)
            else:
                kp[phys, :, :n] = src_k
                vp[phys, :, :n] = src_v
    if layout == "HND":
        kp = kp.permute(0, 2, 1, 3)
        vp = vp.permute(0, 2, 1, 3)
    return kp, vp, bt


E4M3_MAX = 448.0


def quantize_e4m3(x, per_head_dim=1):
    """Round a [B, Hkv, S, d] cache to FP8 E4M3 with one scale per KV head
    (scale = max|x| over that head / 448, so the head's largest element maps
    to the largest finite code).  NaN elements (padding) stay NaN.  Returns
    (codes as torch.float8_e4m3fn, scales [Hkv] float32).  Data preparation only."""
    xf = x.float()
    finite = torch.nan_to_num(xf.abs(), nan=0.0)
    amax = finite.amax(dim=tuple(i for i in range(xf.dim()) if i != per_head_dim))
    scales = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).float()
    shape = [1] * xf.dim()
    shape[per_head_dim] = -1
    codes = (xf / scales.view(shape)).to(torch.float8_e4m3fn)
    return codes, scales
