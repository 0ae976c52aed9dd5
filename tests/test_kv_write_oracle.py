"""Pins of the KV write reference (oracle/kv_write.py) on the CPU.

The expected pools below are written out by hand, entry by entry, from the
slot rule of the paged cache: slot s of a [num_blocks, block_size, Hkv, D]
pool is row s % block_size of block s // block_size ("The Ultimate Guide to
LLM Inference Optimization - Part 2", section "Paged Attention": fixed-size
blocks addressed through a table), and a block copy replaces a whole
destination block, K and V, by its source ("Modern LLM Inference ...",
section 8.2, "Prefix Sharing (Copy-on-Write)").  Nothing here recomputes
them with the reference's own indexing.

A second part plants plausible mistakes in a copy of the reference (swapped
quotient and remainder, K written into V, a reversed copy pair, ...) and
checks that the pins catch every one.
"""
import os
import types

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kv_write.py")


def _pool(nblocks, base):
    """[nblocks, 4 slots, 2 heads, 1] with entry base + 100 block + 10 slot + head."""
    x = np.zeros((nblocks, 4, 2, 1), dtype=np.int64)
    for b in range(nblocks):
        for s in range(4):
            for h in range(2):
                x[b, s, h, 0] = base + 100 * b + 10 * s + h
    return x


# append: slots 6, 1, 9 of a 3-block pool of 4-slot blocks are
# (block 1, row 2), (block 0, row 1), (block 2, row 1)
APPEND_SLOTS = [6, 1, 9]
APPEND_K_NEW = np.array([[[-1], [-2]], [[-3], [-4]], [[-5], [-6]]], dtype=np.int64)
APPEND_V_NEW = np.array([[[-11], [-12]], [[-13], [-14]], [[-15], [-16]]], dtype=np.int64)
APPEND_K_WANT = np.array([
    [[0, 1], [-3, -4], [20, 21], [30, 31]],
    [[100, 101], [110, 111], [-1, -2], [130, 131]],
    [[200, 201], [-5, -6], [220, 221], [230, 231]],
], dtype=np.int64)[..., None]
APPEND_V_WANT = np.array([
    [[1000, 1001], [-13, -14], [1020, 1021], [1030, 1031]],
    [[1100, 1101], [1110, 1111], [-11, -12], [1130, 1131]],
    [[1200, 1201], [-15, -16], [1220, 1221], [1230, 1231]],
], dtype=np.int64)[..., None]

# copy_blocks: pairs (3 -> 0) and (1 -> 2) of a 4-block pool; blocks 1 and 3
# keep their contents
COPY_SRC, COPY_DST = [3, 1], [0, 2]
COPY_K_WANT = np.array([
    [[300, 301], [310, 311], [320, 321], [330, 331]],
    [[100, 101], [110, 111], [120, 121], [130, 131]],
    [[100, 101], [110, 111], [120, 121], [130, 131]],
    [[300, 301], [310, 311], [320, 321], [330, 331]],
], dtype=np.int64)[..., None]
COPY_V_WANT = COPY_K_WANT + 1000


def pin_append(mod):
    k0, v0 = _pool(3, 0), _pool(3, 1000)
    k_keep, v_keep = k0.copy(), v0.copy()
    k, v = mod.append(k0, v0, APPEND_K_NEW, APPEND_V_NEW, np.array(APPEND_SLOTS))
    assert np.array_equal(k, APPEND_K_WANT), "K pool after append"
    assert np.array_equal(v, APPEND_V_WANT), "V pool after append"
    # the inputs are left as they were (the reference returns new pools)
    assert np.array_equal(k0, k_keep) and np.array_equal(v0, v_keep), "inputs modified"


def pin_append_bf16_bits(mod):
    # bfloat16 pools are held as uint16 bit patterns: bits are moved, not values
    k0 = np.full((2, 4, 1, 2), 0x3F80, dtype=np.uint16)      # 1.0
    v0 = np.full((2, 4, 1, 2), 0x7FC0, dtype=np.uint16)      # NaN
    kn = np.array([[[0x8001, 0xFF80]]], dtype=np.uint16)     # denormal, -inf
    vn = np.array([[[0x0000, 0x8000]]], dtype=np.uint16)     # +0, -0
    k, v = mod.append(k0, v0, kn, vn, np.array([5]))         # block 1, row 1
    assert k.dtype == np.uint16 and v.dtype == np.uint16
    assert k[1, 1, 0].tolist() == [0x8001, 0xFF80] and v[1, 1, 0].tolist() == [0x0000, 0x8000]
    assert int((k != 0x3F80).sum()) == 2 and int((v != 0x7FC0).sum()) == 2


def pin_copy_blocks(mod):
    k0, v0 = _pool(4, 0), _pool(4, 1000)
    k_keep, v_keep = k0.copy(), v0.copy()
    k, v = mod.copy_blocks(k0, v0, np.array(COPY_SRC), np.array(COPY_DST))
    assert np.array_equal(k, COPY_K_WANT), "K pool after copy"
    assert np.array_equal(v, COPY_V_WANT), "V pool after copy"
    assert np.array_equal(k0, k_keep) and np.array_equal(v0, v_keep), "inputs modified"


def pin_copy_blocks_scale_rows(mod):
    # 8-bit pages with a scale per block and KV head: the copies 3 -> 0 and
    # 1 -> 2 carry the scale rows, blocks 1 and 3 keep theirs
    k0, v0 = _pool(4, 0), _pool(4, 1000)
    ks = np.array([[0.5, 1.5], [2.5, 3.5], [4.5, 5.5], [6.5, 7.5]], dtype=np.float32)
    vs = ks + 10
    k, v, ks2, vs2 = mod.copy_blocks(k0, v0, np.array(COPY_SRC), np.array(COPY_DST), ks, vs)
    assert np.array_equal(k, COPY_K_WANT) and np.array_equal(v, COPY_V_WANT)
    assert ks2.tolist() == [[6.5, 7.5], [2.5, 3.5], [2.5, 3.5], [6.5, 7.5]]
    assert vs2.tolist() == [[16.5, 17.5], [12.5, 13.5], [12.5, 13.5], [16.5, 17.5]]
    assert ks.tolist()[0] == [0.5, 1.5], "input scales modified"


def pin_empty_calls(mod):
    k0, v0 = _pool(2, 0), _pool(2, 1000)
    k, v = mod.append(k0, v0, np.zeros((0, 2, 1), np.int64), np.zeros((0, 2, 1), np.int64),
                      np.zeros(0, np.int32))
    assert np.array_equal(k, k0) and np.array_equal(v, v0)
    k, v = mod.copy_blocks(k0, v0, np.zeros(0, np.int32), np.zeros(0, np.int32))
    assert np.array_equal(k, k0) and np.array_equal(v, v0)


PINS = [pin_append, pin_append_bf16_bits, pin_copy_blocks, pin_copy_blocks_scale_rows,
        pin_empty_calls]


def _load(src, name="kv_write_under_test"):
    mod = types.ModuleType(name)
    exec(compile(src, SRC, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_reference_passes_pin(pin):
    import oracle.kv_write as kv_write

    pin(kv_write)


MUTANTS = {
    "quotient_remainder_swapped_k": ("k[s // bs, s % bs]", "k[s % bs, s // bs]"),
    "quotient_remainder_swapped_v": ("v[s // bs, s % bs]", "v[s % bs, s // bs]"),
    "block_size_from_head_axis": ("bs = k.shape[1]", "bs = k.shape[2]"),
    "k_row_written_into_v": ("= v_new[i]", "= k_new[i]"),
    "v_row_written_into_k": ("= k_new[i]", "= v_new[i]"),
    "first_row_for_every_token": ("= k_new[i]", "= k_new[0]"),
    "copy_pair_reversed": ("k[d] = k[s]", "k[s] = k[d]"),
    "copy_skips_v": ("v[d] = v[s]", "pass"),
    "copy_v_from_k": ("v[d] = v[s]", "v[d] = k[s]"),
    "in_place_update": ("k, v = k_pool.copy(), v_pool.copy()", "k, v = k_pool, v_pool"),
    "scale_rows_not_copied": ("            ks[d] = ks[s]\n", "            pass\n"),
    "v_scale_row_from_k": ("vs[d] = vs[s]", "vs[d] = ks[s]"),
    "scale_copied_in_place": ("ks = None if k_scale is None else np.array(k_scale, copy=True)",
                              "ks = k_scale"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert old in src, "mutation site missing: %r" % old
    mod = _load(src.replace(old, new))
    caught = []
    for pin in PINS:
        try:
            pin(mod)
        except Exception:  # a failed assertion or a crash both count as caught
            caught.append(pin.__name__)
    assert caught, "mutant %s survived every pin" % name
