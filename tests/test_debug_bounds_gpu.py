"""The bounds-checking build and buffer canaries: stand-ins for a memory
checker on the GPU.

* The library built with TA_DEBUG_BOUNDS checks the indices its kernels
  compute -- q reads, block-table reads, every write of out, lse and the
  partial states, the shared-memory destinations of the TMA copies and of the
  tcgen05 kernel's P writes -- against their buffers; an index outside skips
  the access and sets TA_ERR_DEVICE_BOUNDS.  The ragged-row, paged, wide-group,
  FP8 (both kernel families), multi-query, cluster-merge and automatic-merge
  suites are rerun against that build, and after every test the device error
  word must be clear.
* Canary regions around lse and the workspace (and out) must come back
  untouched from every kernel family, fused and launched merges alike."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import softmax_tree_reduction_gb300 as ta
from softmax_tree_reduction_gb300 import workloads

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_suites_run_clean_on_the_bounds_checking_build():
    from softmax_tree_reduction_gb300 import build
    lib = build.build(debug=True)
    env = dict(os.environ, TREE_ATTN_LIBRARY=lib, TREE_ATTN_CHECK_ERRORS="1")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "gpu",
           "tests/test_parity_gpu.py::test_kernel_instances_ragged", "tests/test_parity_gpu.py::test_fused_and_launched_combine_paths",
           "tests/test_paged_gpu.py", "tests/test_wide_groups_gpu.py", "tests/test_fp8_gpu.py",
           "tests/test_fp8_tc05_gpu.py", "tests/test_multi_query_gpu.py", "tests/test_cluster_gpu.py",
           "tests/test_auto_merge_gpu.py", "-k", "not full and not stalled"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = (r.stdout + r.stderr)[-4000:]
    assert r.returncode == 0, tail
    assert " passed" in tail and "failed" not in tail, tail


GUARD = 4096  # bytes of canary on each side (keeps the payload 16-byte aligned)


@pytest.mark.parametrize("kern,G,P", [("mma", 4, 1), ("mma", 4, 7), ("mma", 4, 64), ("fma", 4, 7),
                                      ("tc05", 40, 1), ("tc05", 40, 5), ("tc05", 40, 48), ("mma", 40, 9)])
def test_lse_out_and_workspace_canaries(kern, G, P):
    B, Hkv, N = 2, 2, 3000
    w = workloads.Workload("canary", B, G * Hkv, Hkv, 128, N, torch.bfloat16, torch.bfloat16, seed=G + P,
                           seqlen=None, ragged_range=(0, 1), pad_nan=True, k_scale=0.5)
    inp = workloads.make_inputs(w, seqlens=[N, 1111])
    ref_o, ref_l = oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"])
    q, k, v, sl = (inp[x].cuda() for x in ("q", "k", "v", "seqlens"))
    Hq = G * Hkv
    shape = ta.make_shape(q, k)
    nbytes = ta.tree_attn_workspace_bytes(shape, P)
    wsbuf = torch.full((nbytes + 2 * GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    ws = wsbuf[GUARD:GUARD + nbytes] if nbytes else None
    g4 = GUARD // 4
    lsebuf = torch.full((B * Hq + 2 * g4,), 777.0, device="cuda")
    outbuf = torch.full((B * Hq * 128 + 2 * g4,), 777.0, device="cuda")
    lse = lsebuf[g4:g4 + B * Hq].view(B, Hq)
    out = outbuf[g4:g4 + B * Hq * 128].view(B, Hq, 128)
    ta.tree_attn_decode(q, k, v, sl, out=out, lse=lse, num_splits=P, workspace=ws, kernel=kern)
    torch.cuda.synchronize()
    assert ta.tree_attn_get_device_error() == 0
    assert torch.all(wsbuf[:GUARD] == 0xA5) and torch.all(wsbuf[GUARD + nbytes:] == 0xA5)
    assert torch.all(lsebuf[:g4] == 777.0) and torch.all(lsebuf[g4 + B * Hq:] == 777.0)
    assert torch.all(outbuf[:g4] == 777.0) and torch.all(outbuf[g4 + B * Hq * 128:] == 777.0)
    assert np.max(np.abs(out.double().cpu().numpy() - ref_o)) <= 2e-3
    assert np.max(np.abs(lse.double().cpu().numpy() - ref_l)) <= 1e-3


@pytest.mark.parametrize("kern,G,P", [("tc05", 24, 1), ("tc05", 24, 5), ("tc05", 12, 48), ("mma", 12, 7),
                                      ("auto", 4, 0)])
def test_fp8_and_automatic_merge_canaries(kern, G, P):
    """The same canaries around the FP8 kernels' outputs and workspace, and
    around a call whose split count and merge the library picks (short rows:
    the cluster merge)."""
    B, Hkv, N = 2, 2, 2048
    w = workloads.Workload("canary8", B, G * Hkv, Hkv, 128, N, torch.bfloat16, torch.bfloat16, seed=G + P,
                           seqlen=None, ragged_range=(0, 1), pad_nan=True, k_scale=0.5)
    inp = workloads.make_inputs(w, seqlens=[N, 777])
    k8, ks = workloads.quantize_e4m3(inp["k"])
    v8, vs = workloads.quantize_e4m3(inp["v"])
    ref_o, ref_l = oracle.attention_e4m3(inp["q"], k8, v8, ks, vs, inp["seqlens"])
    q, sl = inp["q"].cuda(), inp["seqlens"].cuda()
    k8d, v8d = k8.cuda(), v8.cuda()
    Hq = G * Hkv
    shape = ta.make_shape(q, k8d)
    nbytes = ta.tree_attn_workspace_bytes(shape, P if P > 0 else ta.tree_attn_pick_splits(shape))
    wsbuf = torch.full((nbytes + 2 * GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    ws = wsbuf[GUARD:GUARD + nbytes] if nbytes else None
    g4 = GUARD // 4
    lsebuf = torch.full((B * Hq + 2 * g4,), 777.0, device="cuda")
    outbuf = torch.full((B * Hq * 128 + 2 * g4,), 777.0, device="cuda")
    lse = lsebuf[g4:g4 + B * Hq].view(B, Hq)
    out = outbuf[g4:g4 + B * Hq * 128].view(B, Hq, 128)
    ta.tree_attn_decode(q, k8d, v8d, sl, out=out, lse=lse, num_splits=P, workspace=ws, kernel=kern,
                        k_scale=ks.cuda(), v_scale=vs.cuda())
    torch.cuda.synchronize()
    assert ta.tree_attn_get_device_error() == 0
    assert torch.all(wsbuf[:GUARD] == 0xA5) and torch.all(wsbuf[GUARD + nbytes:] == 0xA5)
    assert torch.all(lsebuf[:g4] == 777.0) and torch.all(lsebuf[g4 + B * Hq:] == 777.0)
    assert torch.all(outbuf[:g4] == 777.0) and torch.all(outbuf[g4 + B * Hq * 128:] == 777.0)
    assert np.max(np.abs(out.double().cpu().numpy() - ref_o)) <= 2e-3
    assert np.max(np.abs(lse.double().cpu().numpy() - ref_l)) <= 1e-3
