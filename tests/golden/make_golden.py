"""Write oracle_small.json: a small fixed case and the oracle's answer for it.

Calls only the oracle (and numpy for the inputs).  Rerun after a justified
change to the oracle's arithmetic:  python tests/golden/make_golden.py
"""
import json
import math
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def case():
    rng = np.random.default_rng(2024)
    B, Hq, Hkv, D, bs = 2, 4, 2, 64, 4
    lens = np.array([5, 11], dtype=np.int32)
    num_blocks = 6
    max_blocks = 3
    table = np.full((B, max_blocks), -1, dtype=np.int32)
    perm = rng.permutation(num_blocks)
    p = 0
    for b in range(B):
        n = -(-int(lens[b]) // bs)
        table[b, :n] = perm[p:p + n]
        p += n
    # values on a 1/64 grid in [-2, 2]: exact in float32 and in bfloat16
    q = (rng.integers(-128, 129, size=(B, Hq, D)) / 64.0).astype(np.float32)
    k = (rng.integers(-128, 129, size=(num_blocks, bs, Hkv, D)) / 64.0).astype(np.float32)
    v = (rng.integers(-128, 129, size=(num_blocks, bs, Hkv, D)) / 64.0).astype(np.float32)
    return q, k, v, table, lens, 1.0 / math.sqrt(D)


def main():
    q, k, v, table, lens, scale = case()
    out, rc = oracle.decode_f64(q, k, v, table, lens, scale)
    assert rc == 0
    doc = {
        "what": "paged GQA decode, float64 oracle answer for a small fixed case; values are "
                "multiples of 1/64 in [-2, 2], exact in float32 and bfloat16",
        "written_by": "tests/golden/make_golden.py (oracle only)",
        "B": 2, "Hq": 4, "Hkv": 2, "D": 64, "block_size": 4, "num_blocks": 6,
        "scale": scale,
        "q": q.ravel().tolist(), "k_pool": k.ravel().tolist(), "v_pool": v.ravel().tolist(),
        "block_table": table.ravel().tolist(), "seq_lens": lens.tolist(),
        "out": [float(x) for x in out.ravel()],
    }
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(doc, f)
        f.write("\n")


if __name__ == "__main__":
    main()
