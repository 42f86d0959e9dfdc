"""Writes tests/golden/tiny_oracle.json from the fp64 oracle alone.

The pages print no worked example for this path, so this fixture is a
regression pin of the oracle itself (it is not an independent pin): the small
tiny-GQA workload (batch 1, 2 q heads / 1 kv head, head_dim 64, prompt 64,
8 decode steps, seed 0), its prefill and decode outputs summarised by sums and
a few sampled values.  Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from gqa_attention_preallocated_qa_gb300.configs import TINY  # noqa: E402
from gqa_attention_preallocated_qa_gb300.inputs import bf16_bits_to_f64 as f  # noqa: E402
from oracle import oracle  # noqa: E402


def compute():
    w = TINY
    inp = w.inputs()
    lay = oracle.OracleLayer(oracle.Geometry(w.B, w.Hq, w.Hkv, w.D, w.cap, w.theta, w.eps))
    _, out = lay.prefill(w.prompt_lens, f(inp.q), f(inp.k), f(inp.v), f(inp.wq), f(inp.wk))
    res = {"prefill_sum": float(out.sum()), "prefill_abs_sum": float(abs(out).sum()),
           "prefill_samples": [float(out[t, h, d]) for t, h, d in ((0, 0, 0), (17, 1, 5),
                                                                  (63, 0, 63), (63, 1, 31))],
           "decode": []}
    for s in range(w.steps):
        _, o = lay.decode(f(inp.dq[s]), f(inp.dk[s]), f(inp.dv[s]), f(inp.wq), f(inp.wk))
        res["decode"].append({"sum": float(o.sum()), "first": float(o[0, 0, 0]),
                              "last": float(o[0, 1, 63])})
    res["final_len"] = int(lay.lens[0])
    return res


if __name__ == "__main__":
    doc = {"what": "fp64 oracle on the tiny GQA workload (seed 0); regression pin of the oracle",
           "written_by": "tests/golden/make_golden.py (calls only oracle/)", "values": compute()}
    with open(os.path.join(HERE, "tiny_oracle.json"), "w") as fh:
        json.dump(doc, fh, indent=1)
