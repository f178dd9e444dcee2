"""Write ``closed_forms.json``: hand-derived expected values for tiny decode-attention cases.

The pages on Tree Attention print no worked numerical example, so these cases
are derived by hand from the definitions they give (exact softmax with the
global maximum; the partial state (o, l, m); the merge operator), with the
derivation stored next to each case.  Values are evaluated with Python's
``math`` module only: nothing here calls the oracle or the CUDA library.

Run from the repository root:  python tests/golden/make_closed_forms.py
"""
import json
import math
import os

e = math.e
e2 = math.exp(2.0)
cases = [
    dict(name="two_tokens_logits_0_and_1",
         derivation="s = scale*q.K^T = [0, 1]; softmax weights 1/(1+e), e/(1+e); out = w0*v0 + w1*v1; "
                    "lse = ln(1+e)",
         dtype="f32", B=1, Hq=1, Hkv=1, d=2, S=2, seqlens=[2], scale=1.0,
         q=[[[1.0, 0.0]]], k=[[[[0.0, 5.0], [1.0, -2.0]]]], v=[[[[1.0, 0.0], [0.0, 1.0]]]],
         out=[[[1 / (1 + e), e / (1 + e)]]], lse=[[math.log(1 + e)]]),
    dict(name="four_equal_logits_mean_of_v",
         derivation="every logit equals scale*q.k = 0.5*(0.5*2+0.5*2) = 1, so out is the mean of the V rows "
                    "and lse = 1 + ln 4",
         dtype="bf16", B=1, Hq=1, Hkv=1, d=2, S=4, seqlens=[4], scale=0.5,
         q=[[[0.5, 0.5]]], k=[[[[2.0, 2.0]] * 4]],
         v=[[[[1.0, 2.0], [3.0, 4.0], [5.0, 6.0], [7.0, 8.0]]]],
         out=[[[4.0, 5.0]]], lse=[[1.0 + math.log(4.0)]]),
    dict(name="gqa_two_groups",
         derivation="Hq=4, Hkv=2: heads 0,1 read KV head 0 (all keys zero: uniform weights, out = mean V0 = "
                    "[0.5,0.5], lse = ln 2); head 2 reads KV head 1 with logits [2, 0]: out = (e^2 v0 + v1)/(e^2+1), "
                    "lse = ln(e^2+1); head 3 has q = 0: out = mean V1 = [1,-1], lse = ln 2",
         dtype="f32", B=1, Hq=4, Hkv=2, d=2, S=2, seqlens=[2], scale=1.0,
         q=[[[1.0, 1.0], [-3.0, 7.0], [2.0, 0.0], [0.0, 0.0]]],
         k=[[[[0.0, 0.0], [0.0, 0.0]], [[1.0, 0.0], [0.0, 0.0]]]],
         v=[[[[1.0, 0.0], [0.0, 1.0]], [[2.0, 0.0], [0.0, -2.0]]]],
         out=[[[0.5, 0.5], [0.5, 0.5], [2 * e2 / (e2 + 1), -2 / (e2 + 1)], [1.0, -1.0]]],
         lse=[[math.log(2.0), math.log(2.0), math.log(e2 + 1), math.log(2.0)]]),
    dict(name="dominant_logit",
         derivation="logits [0, 50]: out = (v0 + e^50 v1)/(1 + e^50), lse = 50 + ln(1 + e^-50)",
         dtype="f32", B=1, Hq=1, Hkv=1, d=2, S=2, seqlens=[2], scale=1.0,
         q=[[[1.0, 0.0]]], k=[[[[0.0, 0.0], [50.0, 0.0]]]], v=[[[[3.0, -1.0], [-7.0, 9.0]]]],
         out=[[[(3.0 + math.exp(50) * -7.0) / (1 + math.exp(50)),
                (-1.0 + math.exp(50) * 9.0) / (1 + math.exp(50))]]],
         lse=[[50.0 + math.log1p(math.exp(-50.0))]]),
    dict(name="ragged_batch_empty_and_single",
         derivation="row 0 has length 0: out = 0, lse = -inf (empty state); row 1 has length 1: out = v0, "
                    "lse = s0 = scale*q.k0 = 0.25*(1*2 + 2*3) = 2",
         dtype="f32", B=2, Hq=1, Hkv=1, d=2, S=2, seqlens=[0, 1], scale=0.25,
         q=[[[1.0, 1.0]], [[1.0, 2.0]]],
         k=[[[[9.0, 9.0], [9.0, 9.0]]], [[[2.0, 3.0], [100.0, 100.0]]]],
         v=[[[[9.0, 9.0], [9.0, 9.0]]], [[[-1.5, 0.25], [100.0, 100.0]]]],
         out=[[[0.0, 0.0]], [[-1.5, 0.25]]], lse=[["-inf"], [2.0]]),
]
merge_cases = [
    dict(name="merge_two_states",
         derivation="A = (o=[2,0], l=2, m=1), B = (o=[0,3], l=3, m=0): m = 1, alpha = 1, beta = e^-1, "
                    "l = 2 + 3/e, o = [2, 3/e]; out = o/l, lse = 1 + ln(2 + 3/e)",
         a=dict(o=[2.0, 0.0], l=2.0, m=1.0), b=dict(o=[0.0, 3.0], l=3.0, m=0.0),
         merged=dict(o=[2.0, 3 / e], l=2 + 3 / e, m=1.0),
         out=[2 / (2 + 3 / e), (3 / e) / (2 + 3 / e)], lse=1 + math.log(2 + 3 / e)),
]
doc = {
    "source": "Hand-derived closed forms. Definition of exact decode attention: 'Tree Attention Guide: "
              "Topology-Aware LLM Decoding', section 'Core Innovation 2: Mathematical Formulation of Online "
              "Softmax on Trees' (the Softmax(S)_j equation with the global maximum). Partial state and merge: same "
              "page, 'Local Independent Partial Attention' and 'The Tree Reduction Merge Operator'. The pages print "
              "no worked numerical example; each expected value is derived by hand (derivation per case) and "
              "evaluated with Python's math module.",
    "attention_cases": cases,
    "merge_cases": merge_cases,
}
with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "closed_forms.json"), "w") as f:
    json.dump(doc, f, indent=1)
