"""Paths that normal inputs rarely take, forced by diagnostic flags (no fault,
no hang):

* the failure path of the bounded on-chip waits: the copy warps publish no
  tile, every compute warp's wait gives up after its time limit, the call still
  completes, its outputs are NaN, tree_attn_get_device_error reports the
  timeout, and the next call on the same context is correct again;
* a wrong length hint: the first copies, issued before the row length is read,
  are discarded and the real tiles streamed after them; results are unchanged
  (bitwise, with the deterministic flag)."""
import numpy as np
import pytest
import torch

import oracle
import softmax_tree_reduction_gb300 as ta
from softmax_tree_reduction_gb300 import workloads

pytestmark = pytest.mark.gpu


def _inputs(kv, d, fp8=False):
    w = workloads.Workload("stall", 2, 8, 2, d, 1024, kv, kv, seed=3, seqlen=None, ragged_range=(0, 1),
                           pad_nan=True, k_scale=0.5)
    inp = workloads.make_inputs(w, seqlens=[1000, 333])
    if fp8:
        inp["k"], inp["ks"] = workloads.quantize_e4m3(inp["k"])
        inp["v"], inp["vs"] = workloads.quantize_e4m3(inp["v"])
    return inp


def _kernel(family):
    return {"fp8": "mma", "fp8tc05": "tc05"}.get(family, family)


@pytest.mark.parametrize("family", ["mma", "fma", "fp8", "fp8tc05"])
@pytest.mark.parametrize("P", [1, 5])
def test_stalled_waits_report_timeout_and_leave_the_device_usable(family, P):
    fp8 = family.startswith("fp8")
    kv = torch.float32 if family == "fma" else torch.bfloat16
    inp = _inputs(kv, 128 if family != "fma" else 64, fp8=fp8)
    q, k, v, sl = (inp[x].cuda() for x in ("q", "k", "v", "seqlens"))
    kw = dict(k_scale=inp["ks"].cuda(), v_scale=inp["vs"].cuda()) if fp8 else {}
    kern = _kernel(family)
    assert ta.tree_attn_get_device_error() == 0
    out, lse = ta.tree_attn_decode(q, k, v, sl, num_splits=P, kernel=kern, diag_stall=True, **kw)
    assert ta.tree_attn_get_device_error() == ta.TA_ERR_DEVICE_TIMEOUT
    assert torch.isnan(out).all() and torch.isnan(lse).all()
    assert ta.tree_attn_get_device_error() == 0          # the word was read and cleared
    # the context and the scheduling counters are usable again
    out, lse = ta.tree_attn_decode(q, k, v, sl, num_splits=P, kernel=kern, **kw)
    torch.cuda.synchronize()
    assert ta.tree_attn_get_device_error() == 0
    if fp8:
        ref_o, ref_l = oracle.attention_e4m3(inp["q"], inp["k"], inp["v"], inp["ks"], inp["vs"], inp["seqlens"])
    else:
        ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    tol = 1e-4 if kv == torch.float32 else 2e-3
    assert np.max(np.abs(out.double().cpu().numpy() - ref_o)) <= tol
    assert np.max(np.abs(lse.double().cpu().numpy() - ref_l)) <= max(tol, 1e-3)


@pytest.mark.parametrize("family", ["mma", "fma", "fp8", "fp8tc05"])
@pytest.mark.parametrize("P", [1, 5, 19])
def test_wrong_length_hint_changes_nothing(family, P):
    fp8 = family.startswith("fp8")
    kv = torch.float32 if family == "fma" else torch.bfloat16
    inp = _inputs(kv, 128 if family != "fma" else 64, fp8=fp8)
    q, k, v, sl = (inp[x].cuda() for x in ("q", "k", "v", "seqlens"))
    kw = dict(k_scale=inp["ks"].cuda(), v_scale=inp["vs"].cuda()) if fp8 else {}
    kern = _kernel(family)
    o1, l1 = ta.tree_attn_decode(q, k, v, sl, num_splits=P, kernel=kern, deterministic=True, **kw)
    o2, l2 = ta.tree_attn_decode(q, k, v, sl, num_splits=P, kernel=kern, deterministic=True, diag_mishint=True, **kw)
    o3, l3 = ta.tree_attn_decode(q, k, v, sl, num_splits=P, kernel=kern, diag_mishint=True, **kw)
    torch.cuda.synchronize()
    assert ta.tree_attn_get_device_error() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    if fp8:
        ref_o, ref_l = oracle.attention_e4m3(inp["q"], inp["k"], inp["v"], inp["ks"], inp["vs"], inp["seqlens"])
    else:
        ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    tol = 1e-4 if kv == torch.float32 else 2e-3
    assert np.max(np.abs(o3.double().cpu().numpy() - ref_o)) <= tol
    assert np.max(np.abs(l3.double().cpu().numpy() - ref_l)) <= max(tol, 1e-3)


def test_timeout_on_one_stream_leaves_calls_on_another_stream_intact():
    """A call on stream A gives up its waits (diagnostic stall, about two
    seconds) while calls on a second non-blocking stream B run back to back.
    Reading the timeout from A must not disturb B: every B call's output, each
    in a buffer of its own, matches the oracle, also the ones in flight while
    A's error is read and cleared.  (Clearing the library's scheduling counters
    at that moment would break the B call whose row tickets are mid-count.)
    B's first round is enqueued while A stalls, so its calls are in flight
    when A's error word is read and cleared, whether the GPU runs them beside
    A's blocks or after them."""
    import threading

    w = workloads.Workload("busy", 1, 32, 8, 128, 131072, torch.bfloat16, torch.bfloat16, seed=21,
                           seqlen=131072, k_scale=0.5)
    inp = workloads.make_inputs(w)
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    q, k, v, sl = (inp[x].cuda() for x in ("q", "k", "v", "seqlens"))
    stall = _inputs(torch.bfloat16, 128)
    sq, sk, sv, ssl = (stall[x].cuda() for x in ("q", "k", "v", "seqlens"))
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    n = 64
    outs = torch.empty(n, 1, 32, 128, device="cuda")
    lses = torch.empty(n, 1, 32, device="cuda")
    shape = ta.make_shape(q, k)
    ws = torch.empty(ta.tree_attn_workspace_bytes(shape, 8), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    assert ta.tree_attn_get_device_error() == 0

    ta.tree_attn_decode(sq, sk, sv, ssl, num_splits=5, kernel="mma", diag_stall=True, stream=sa)
    result = {}
    reader = threading.Thread(target=lambda: result.update(rc=ta.tree_attn_get_device_error(sa)))
    reader.start()
    rounds, after = 0, 0
    started_during = reader.is_alive()
    while True:
        with torch.cuda.stream(sb):
            outs.fill_(float("nan"))
            lses.fill_(float("nan"))
        for i in range(n):
            ta.tree_attn_decode(q, k, v, sl, out=outs[i], lse=lses[i], num_splits=8, workspace=ws, stream=sb)
        sb.synchronize()
        o = outs.double().cpu().numpy()
        l = lses.double().cpu().numpy()
        assert np.isfinite(o).all() and np.isfinite(l).all(), f"round {rounds}"
        assert np.max(np.abs(o - ref_o[None])) <= 2e-3, f"round {rounds}"
        assert np.max(np.abs(l - ref_l[None])) <= 1e-3, f"round {rounds}"
        rounds += 1
        if not reader.is_alive():
            after += 1
            if after >= 2:
                break
    reader.join()
    assert result["rc"] == ta.TA_ERR_DEVICE_TIMEOUT
    assert started_during   # the first round was enqueued before A's error was read
    assert ta.tree_attn_get_device_error() == 0
