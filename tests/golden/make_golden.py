"""Writes tests/golden/tiny_oracle_digest.txt from the CPU oracle only.

The digest is a regression pin on the oracle: SHA-256 of the codes and scales
it produces for the seeded tiny workload (N=64, H=8, heads_per_group=8) and
of the paged cache it produces for a small insert case. Re-run only when a
change to the oracle's arithmetic is justified by a reading of the pages,
and name that reading in the commit message.
"""
import hashlib
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads as W  # noqa: E402


def main():
    inp = W.inverse_inputs(W.TINY)
    codes, scales = oracle.inv_rope_fp8_quant(inp["x"], inp["positions"], inp["cos_sin_cache"], 8)
    inv = hashlib.sha256(codes.tobytes() + scales.tobytes()).hexdigest()
    ins_spec = W.InsertSpec("small-insert", 256, 4096, 8, 64, seed=0)
    ii = W.insert_inputs(ins_spec)
    cache = oracle.rope_fp8_quant_insert(ii["kv"], ii["positions"], ii["cos_sin_cache"],
                                         ii["slot_mapping"], ii["k_cache"], ii["block_size"])
    ins = hashlib.sha256(cache.tobytes()).hexdigest()
    with open(os.path.join(HERE, "tiny_oracle_digest.txt"), "w") as f:
        f.write("# written by tests/golden/make_golden.py (CPU oracle only)\n")
        f.write(f"inverse {inv}  tiny N=64 H=8 hpg=8 seed 0 eps 1e-10\n")
        f.write(f"insert {ins}  N=256 8 blocks x 64 slots seed 0 eps 1e-10\n")


if __name__ == "__main__":
    main()
