"""Exact reference of the KV write path: storing new tokens' K/V rows into
their slots and copying blocks (copy-on-write).

TEST INFRASTRUCTURE ONLY.  Byte semantics on numpy arrays (float32, or
bfloat16 held as uint16 bits): slot s of a [num_blocks, bs, Hkv, D] pool is
pool[s // bs, s % bs]; a block copy replaces pool[dst] by pool[src].  The
pages: blocks allocated when needed ("The Ultimate Guide to LLM Inference
Optimization - Part 2", "Paged Attention"), modified shared blocks copied
("Modern LLM Inference ...", section 8.2, "Prefix Sharing (Copy-on-Write)").
"""
import numpy as np


def append(k_pool, v_pool, k_new, v_new, slots):
    k, v = k_pool.copy(), v_pool.copy()
    bs = k.shape[1]
    for i, s in enumerate(np.asarray(slots).tolist()):
        k[s // bs, s % bs] = k_new[i]
        v[s // bs, s % bs] = v_new[i]
    return k, v


def copy_blocks(k_pool, v_pool, src, dst):
    k, v = k_pool.copy(), v_pool.copy()
    for s, d in zip(np.asarray(src).tolist(), np.asarray(dst).tolist()):
        k[d] = k[s]
        v[d] = v[s]
    return k, v
