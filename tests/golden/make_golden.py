"""Write the stored expected values under tests/golden/ by calling only the
CPU oracle (never the CUDA path).

    python tests/golden/make_golden.py

The pages print no worked numeric example for the verification path, so the
fixtures here are (a) oracle outputs for the seeded tiny greedy workload and a
small ragged stochastic batch, with a hash of the generated inputs so that a
change of generator is detected, and (b) nothing copied from the pages.
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workloads as W  # noqa: E402


def digest(*arrays):
    h = hashlib.sha256()
    for a in arrays:
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def tiny_greedy():
    vb = W.tiny_greedy()
    res = oracle.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                               vb.draft_ids)
    return {
        "workload": "tiny greedy verify: B=4, k=4, V=1024, fp32 N(0,2), seed 1000",
        "input_sha256": digest(vb.logits, vb.cu_rows, vb.draft_ids),
        "accepted_len": res.accepted_len.tolist(),
        "out_tokens": res.out_tokens.tolist(),
        "next_token": res.next_token.tolist(),
        "row_argmax": res.rows["row_argmax"].tolist(),
        "row_lse": [float(x) for x in res.rows["row_lse"]],
    }


def small_stochastic():
    vb, p = W.stochastic(seed=3001, B=6, k=3, V=4096)
    res = oracle.verify_sample(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                               vb.draft_ids, p)
    return {
        "workload": "stochastic verify: B=6, k=3, V=4096, bf16 N(0,3), seed 3001",
        "input_sha256": digest(vb.logits, vb.cu_rows, vb.draft_ids, p.temperature, p.top_k,
                               p.top_p, p.min_p, p.seed),
        "accepted_len": res.accepted_len.tolist(),
        "out_tokens": res.out_tokens.tolist(),
        "row_token": res.rows["row_token"].tolist(),
    }


if __name__ == "__main__":
    for name, fn in [("tiny_greedy.json", tiny_greedy), ("small_stochastic.json", small_stochastic)]:
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(fn(), f, indent=1)
            f.write("\n")
        print("wrote", name)
