"""Writes tests/golden/tiny_oracle.json: the CPU oracle's result on the
seeded tiny workload (4 heads, latent 192 / value 128 / rotary 64 at offset
128, bs=16, pasts {20,5} with {1,7} new tokens, one slot -1).

The file locks the oracle's arithmetic: any later change to the oracle that
moves a bit shows up as a diff of this file, which must then be justified
by the passage of the operator definition it follows. It calls only the
oracle and the seeded input generator.

Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import pa_oracle as O  # noqa: E402
from paged_latent_attention_cache_gb300 import workloads as W  # noqa: E402


def tiny_oracle():
    w = W.tiny()
    p = W.oracle_params(w)
    cache, out, _ = O.run_operator_bits(
        W.to_bits(w.query), W.to_bits(w.key), W.to_bits(w.key_cache),
        W.to_bits(w.cos_cache), W.to_bits(w.sin_cache), w.cumseq.numpy(), w.past.numpy(),
        w.block_table.numpy(), w.slot_mapping.numpy(), p)
    rows = sorted(int(s) for s in w.slot_mapping.tolist() if s >= 0)
    flat = cache.reshape(-1, w.head_size)
    return {
        "workload": "tiny (seed 1)",
        "source": "paged_attention.rs module doc: write phase then read phase",
        "written_rows": {str(r): " ".join(format(int(v), "04x") for v in flat[r])
                         for r in rows},
        "output_bf16_hex": [" ".join(format(int(v), "04x") for v in row) for row in out],
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_oracle.json"), "w") as f:
        json.dump(tiny_oracle(), f, indent=1)
        f.write("\n")
