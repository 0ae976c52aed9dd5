"""Stored fixtures: the oracle's answer on a fixed small case (regression) and
the GQA cache reduction the pages print, which the byte accounting follows."""
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


def test_page_numbers_pin_host_accounting():
    from paged_gqa_decode_04_gb300 import accounting as acc

    with open(os.path.join(HERE, "golden", "pages_numbers.json")) as f:
        entries = {e["id"]: e for e in json.load(f)["entries"]}
    e = entries["gqa_reduction_factor"]
    assert acc.gqa_reduction_factor(e["query_heads"], e["kv_heads"]) == e["reduction_factor"]
    # the same factor shows up in the algorithmic KV bytes of a step
    lens = [100, 2000, 37]
    mha = acc.algorithmic_bytes(lens, 40, 40, 128, 16, 2) - 2 * 3 * 40 * 128 * 2
    gqa = acc.algorithmic_bytes(lens, 40, 8, 128, 16, 2) - 2 * 3 * 40 * 128 * 2
    pages_words = 4 * (3 + sum(-(-L // 16) for L in lens))
    assert (mha - pages_words) == e["reduction_factor"] * (gqa - pages_words)
