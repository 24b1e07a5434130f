"""Writes the stored fixtures under tests/golden/.

* two_keys_closed_form.json: a two-key attention example whose result is
  derived by hand (no code path computes it; the numbers below are the closed
  form evaluated with ``math``).  One query at position 1, q = (2, 0, 0...),
  keys k0 = (1, 0, ...), k1 = (0, 1, ...), values v0 = (1, 2, ...),
  v1 = (3, 4, ...), scale 1/2: scores s0 = 1, s1 = 0, so
  O = (v0 + e^-1 v1) / (1 + e^-1) = ((e + 3) / (e + 1), (2e + 4) / (e + 1))
  and LSE = ln(e^1 + e^0) = ln(e + 1).  All inputs are exact in bf16.

* tiny_mixed_oracle.json: the CPU oracle's LSE and per-row sums of O on the
  tiny mixed workload (3 requests, 4 heads, head_dim 64), a regression
  fixture written by calling only the oracle package.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import math
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)


def two_keys():
    e = math.e
    return {
        "description": "one query at position 1 over two keys; closed form derived by hand",
        "q": [2.0, 0.0], "k0": [1.0, 0.0], "k1": [0.0, 1.0],
        "v0": [1.0, 2.0], "v1": [3.0, 4.0], "scale": 0.5,
        "expected_o": [(e + 3) / (e + 1), (2 * e + 4) / (e + 1)],
        "expected_lse": math.log(e + 1),
    }


def tiny_mixed(seed=1):
    import oracle
    from paged_kv_attention_25_gb300 import workloads as wl
    b = wl.tiny_mixed(seed)
    kp, vp = b.pool_arrays()
    oracle.append(kp, vp, b.block_tables, b.cu_q_lens, b.q_positions, b.k_new, b.v_new)
    O, L = oracle.paged_attn(b.q, kp, vp, b.block_tables, b.ctx_lens, b.cu_q_lens, b.q_positions, b.scale)
    return {"description": "CPU oracle on the tiny mixed workload (seeded)", "seed": seed,
            "lse": L.tolist(), "o_row_sums": O.sum(axis=2).tolist()}


if __name__ == "__main__":
    with open(os.path.join(HERE, "two_keys_closed_form.json"), "w") as f:
        json.dump(two_keys(), f, indent=1)
    with open(os.path.join(HERE, "tiny_mixed_oracle.json"), "w") as f:
        json.dump(tiny_mixed(), f, indent=1)
