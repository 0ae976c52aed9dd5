"""Exact reference of the KV write path: storing new tokens' K/V rows into
their slots and copying blocks (copy-on-write).

TEST INFRASTRUCTURE ONLY.  Byte semantics on numpy arrays (float32, or
bfloat16 held as uint16 bits, 8-bit codes as uint8): slot s of a
[num_blocks, bs, Hkv, D] pool is pool[s // bs, s % bs]; a block copy replaces
pool[dst] by pool[src], and with per-block scales its scale rows too.  The
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


def copy_blocks(k_pool, v_pool, src, dst, k_scale=None, v_scale=None):
    """Block dst[i] becomes a copy of block src[i].  With per-block scale
    tables ([num_blocks, Hkv], 8-bit pages) the destination scale rows are
    copied too and (k, v, k_scale, v_scale) is returned."""
    k, v = k_pool.copy(), v_pool.copy()
    ks = None if k_scale is None else np.array(k_scale, copy=True)
    vs = None if v_scale is None else np.array(v_scale, copy=True)
    for s, d in zip(np.asarray(src).tolist(), np.asarray(dst).tolist()):
        k[d] = k[s]
        v[d] = v[s]
        if ks is not None:
            ks[d] = ks[s]
            vs[d] = vs[s]
    return (k, v) if ks is None else (k, v, ks, vs)
