"""Stored fixtures: the oracle's answer on a fixed small case (regression) and
the numbers the pages print for KV accounting."""
import json
import os

import numpy as np

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def load_small():
    with open(os.path.join(HERE, "golden", "oracle_small.json")) as f:
        doc = json.load(f)
    B, Hq, Hkv, D, bs, nb = (doc[k] for k in ("B", "Hq", "Hkv", "D", "block_size", "num_blocks"))
    q = np.array(doc["q"], dtype=np.float32).reshape(B, Hq, D)
    k = np.array(doc["k_pool"], dtype=np.float32).reshape(nb, bs, Hkv, D)
    v = np.array(doc["v_pool"], dtype=np.float32).reshape(nb, bs, Hkv, D)
    t = np.array(doc["block_table"], dtype=np.int32).reshape(B, -1)
    L = np.array(doc["seq_lens"], dtype=np.int32)
    out = np.array(doc["out"], dtype=np.float64).reshape(B, Hq, D)
    return q, k, v, t, L, doc["scale"], out


def test_oracle_reproduces_stored_answer():
    q, k, v, t, L, scale, want = load_small()
    got, rc = oracle.decode_f64(q, k, v, t, L, scale)
    assert rc == 0
    assert np.array_equal(got, want)
