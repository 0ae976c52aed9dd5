"""Pins for the float64 oracle: facts fixed by the pages and by the mathematics.

Each ``pin_*`` takes an oracle object (with ``decode_f64``) and raises
AssertionError when the oracle disagrees with something that does not depend
on the oracle itself: a second dense formulation (brute force on tiny inputs),
closed forms, exact special cases, and invariances the pages state.  The same
pins are run against deliberately broken copies of the oracle in
``test_oracle_mutants.py`` to show each plausible mistake is caught.

Sources:
  * Attention(Q,K,V) = softmax(Q K^T / sqrt(d)) V -- "Modern LLM Inference -
    Workloads, Bottlenecks, and Optimization Techniques", section "Why
    Cross-Layer Attention Shares K/V but Not Q".
  * N query heads share K KV heads, one group per KV head, and the cache shrinks
    by N/K -- same notes, section 4.1 "Grouped-Query Attention".
  * Contiguous grouping: query layout [batch, seq, groups, per-group heads, dim]
    with a singleton KV-head axis -- itinai.com page on variable-length batches
    and GQA.
  * A continuous logical sequence over scattered physical blocks -- "Advanced
    Optimizations: MQA, GQA, and PagedAttention", section "PagedAttention: The
    OS Analogy"; blocks of e.g. 16 tokens and a block table -- "The Ultimate
    Guide to LLM Inference Optimization - Part 2", section "Paged Attention".
  * Several sequences pointing at the same blocks (prefix sharing) -- "Modern
    LLM Inference ...", section 8.2 "Prefix Sharing (Copy-on-Write)".
  * FlashAttention computes the exact softmax -- same notes, "Linear Attention
    vs. FlashAttention (Online Softmax)".
"""
import math

import numpy as np
import torch

from oracle.brute import bf16_bits_to_f64, brute_decode, brute_decode_ex


# ----------------------------------------------------------------------------- inputs
def bf16_bits(a):
    """float array -> uint16 bfloat16 bits (round to nearest even, via torch)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def paged_case(rng, B, Hq, Hkv, D, bs, lens, dtype="f32", spare=3, max_blocks=None):
    """Random q / pools with a random physical block permutation."""
    lens = np.asarray(lens, dtype=np.int32)
    nb = [-(-int(L) // bs) for L in lens]
    used = sum(nb)
    num_blocks = used + spare
    max_blocks = max_blocks if max_blocks is not None else max(1, max(nb) if nb else 1)
    perm = rng.permutation(num_blocks)
    table = np.full((B, max_blocks), -1, dtype=np.int32)
    p = 0
    for b in range(B):
        table[b, :nb[b]] = perm[p:p + nb[b]]
        p += nb[b]
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    k = rng.standard_normal((num_blocks, bs, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((num_blocks, bs, Hkv, D)).astype(np.float32)
    if dtype == "bf16":
        q, k, v = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    return q, k, v, table, lens


def as_f64(a):
    return bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def contiguous_layout(q, k, v, table, lens, bs_new=None):
    """The same logical caches laid out in order: sequence b's tokens in
    consecutive physical blocks, starting at block 0, optionally re-blocked."""
    B = q.shape[0]
    _, bs, Hkv, D = k.shape
    bs_new = bs_new or bs
    nb_new = [-(-int(L) // bs_new) for L in lens]
    total = max(1, sum(nb_new))
    kk = np.zeros((total, bs_new, Hkv, D), dtype=k.dtype)
    vv = np.zeros((total, bs_new, Hkv, D), dtype=v.dtype)
    tt = np.full((B, max(1, max(nb_new) if nb_new else 1)), -1, dtype=np.int32)
    p = 0
    for b in range(B):
        for t in range(int(lens[b])):
            src_blk, src_slot = table[b, t // bs], t % bs
            dst_blk, dst_slot = p + t // bs_new, t % bs_new
            kk[dst_blk, dst_slot] = k[src_blk, src_slot]
            vv[dst_blk, dst_slot] = v[src_blk, src_slot]
        tt[b, :nb_new[b]] = np.arange(p, p + nb_new[b])
        p += nb_new[b]
    return q, kk, vv, tt, lens


# ----------------------------------------------------------------------------- pins
def pin_brute_force(orc):
    """Dense numpy formulation agrees to 1e-12 on tiny random inputs."""
    rng = np.random.default_rng(7)
    cases = [
        (3, 4, 2, 8, 4, [5, 1, 9], "f32"),
        (2, 4, 4, 16, 2, [3, 8], "f32"),          # MHA
        (2, 6, 1, 8, 3, [7, 4], "bf16"),          # MQA, odd block size
        (4, 8, 2, 16, 16, [1, 7, 16, 33], "bf16"),
        (1, 2, 1, 4, 5, [40], "f32"),
    ]
    for B, Hq, Hkv, D, bs, lens, dt in cases:
        q, k, v, t, L = paged_case(rng, B, Hq, Hkv, D, bs, lens, dt)
        scale = 1.0 / math.sqrt(D)
        out, rc = orc.decode_f64(q, k, v, t, L, scale)
        ref = brute_decode(q, k, v, t, L, scale)
        assert rc == 0
        assert np.abs(out - ref).max() <= 1e-12, (B, Hq, Hkv, D, bs, lens, dt)


def pin_paged_equals_contiguous(orc):
    """Scattered blocks give exactly the result of the same tokens laid out in
    order, and of the same tokens re-blocked with another block size."""
    rng = np.random.default_rng(11)
    q, k, v, t, L = paged_case(rng, 5, 8, 2, 16, 4, [13, 1, 4, 22, 9], "bf16")
    out, _ = orc.decode_f64(q, k, v, t, L, 0.25)
    for bs_new in (4, 1, 7, 32):
        out2, _ = orc.decode_f64(*contiguous_layout(q, k, v, t, L, bs_new), 0.25)
        assert np.array_equal(out, out2), bs_new


def pin_gqa_equals_repeated_mha(orc):
    """GQA equals MHA whose KV head h holds the GQA KV head h // G."""
    rng = np.random.default_rng(13)
    for Hq, Hkv in ((8, 2), (6, 3), (5, 1)):
        G = Hq // Hkv
        q, k, v, t, L = paged_case(rng, 3, Hq, Hkv, 8, 4, [6, 11, 3], "f32")
        out, _ = orc.decode_f64(q, k, v, t, L, 0.4)
        k_mha = np.repeat(k, G, axis=2)
        v_mha = np.repeat(v, G, axis=2)
        out_mha, _ = orc.decode_f64(q, k_mha, v_mha, t, L, 0.4)
        assert np.array_equal(out, out_mha), (Hq, Hkv)


def pin_length_one_returns_v_row(orc):
    """With one cached token the softmax weight is 1: out[b,h] is exactly the V
    row of KV head h // G (this fixes the head grouping on its own)."""
    rng = np.random.default_rng(17)
    B, Hq, Hkv, D, bs = 3, 12, 3, 8, 4
    q, k, v, t, L = paged_case(rng, B, Hq, Hkv, D, bs, [1, 1, 1], "bf16")
    out, rc = orc.decode_f64(q, k, v, t, L, 0.3)
    assert rc == 0
    vf = as_f64(v)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(out[b, h], vf[t[b, 0], 0, h // G]), (b, h)


def pin_identical_keys_mean_of_v(orc):
    """Equal logits give uniform weights: identical keys, or scale 0, return the
    plain mean of the V rows."""
    rng = np.random.default_rng(19)
    B, Hq, Hkv, D, bs = 2, 4, 2, 8, 4
    q, k, v, t, L = paged_case(rng, B, Hq, Hkv, D, bs, [10, 5], "f32")
    k[:] = k[0, 0, 0]
    vf = as_f64(v)
    out, _ = orc.decode_f64(q, k, v, t, L, 0.5)
    q2, k2, v2, t2, L2 = paged_case(rng, B, Hq, Hkv, D, bs, [10, 5], "f32")
    out0, _ = orc.decode_f64(q2, k2, v2, t2, L2, 0.0)
    v2f = as_f64(v2)
    G = Hq // Hkv
    for b in range(B):
        n = int(L[b])
        for h in range(Hq):
            rows = np.stack([vf[t[b, i // bs], i % bs, h // G] for i in range(n)])
            assert np.abs(out[b, h] - rows.mean(axis=0)).max() <= 1e-12
            rows2 = np.stack([v2f[t2[b, i // bs], i % bs, h // G] for i in range(n)])
            assert np.abs(out0[b, h] - rows2.mean(axis=0)).max() <= 1e-12


def pin_hard_one_hot_large_logits(orc):
    """A key aligned with q and all others orthogonal to it: the output is that
    key's V row within exp(-margin).  Logits near 900 overflow exp() unless the
    maximum is subtracted first, so this also pins the range handling."""
    rng = np.random.default_rng(23)
    D, bs, L = 16, 4, 11
    q = np.zeros((1, 1, D), dtype=np.float32)
    q[0, 0, 0] = 3.0
    k = rng.standard_normal((4, bs, 1, D)).astype(np.float32)
    k[..., 0] = 0.0                      # every key orthogonal to q ...
    j = 6
    t = np.array([[2, 0, 3]], dtype=np.int32)
    k[t[0, j // bs], j % bs, 0, :] = 0.0
    k[t[0, j // bs], j % bs, 0, 0] = 600.0  # ... except key j: logit 0.5*3*600 = 900
    v = rng.standard_normal((4, bs, 1, D)).astype(np.float32)
    out, _ = orc.decode_f64(q, k, v, t, np.array([L], np.int32), 0.5)
    assert np.all(np.isfinite(out))
    want = v[t[0, j // bs], j % bs, 0].astype(np.float64)
    assert np.abs(out[0, 0] - want).max() <= 1e-12


def pin_closed_form_three_tokens(orc):
    """Logits 0, 1, 2 (q = e0, keys 0, 1, 2 times e0, scale 1) give weights
    1 : e : e^2, so out = (v0 + e v1 + e^2 v2) / (1 + e + e^2)."""
    D, bs = 2, 2
    q = np.array([[[1.0, 0.0]]], dtype=np.float32)
    k = np.zeros((3, bs, 1, D), dtype=np.float32)
    v = np.zeros((3, bs, 1, D), dtype=np.float32)
    t = np.array([[2, 0]], dtype=np.int32)          # logical block 0 -> physical 2, 1 -> 0
    vals = [(0.5, -1.0), (2.0, 0.25), (-3.0, 4.0)]
    for i, a in enumerate([0.0, 1.0, 2.0]):
        blk, slot = t[0, i // bs], i % bs
        k[blk, slot, 0, 0] = a
        v[blk, slot, 0] = vals[i]
    out, _ = orc.decode_f64(q, k, v, t, np.array([3], np.int32), 1.0)
    e = math.e
    z = 1.0 + e + e * e
    want = [(vals[0][d] + e * vals[1][d] + e * e * vals[2][d]) / z for d in range(D)]
    assert np.abs(out[0, 0] - np.array(want)).max() <= 1e-15


def pin_scale_two_tokens(orc):
    """Two tokens with logit gap `scale * delta`: out = v0 + (v1 - v0) *
    1 / (1 + exp(-scale * delta)).  A dropped, squared or inverted scale fails."""
    D, bs = 3, 1
    q = np.array([[[2.0, 1.0, -1.0]]], dtype=np.float32)
    k = np.array([[[[0.5, 0.0, 1.0]]], [[[1.0, 2.0, 0.0]]]], dtype=np.float32)  # [2,1,1,3]
    v = np.array([[[[1.0, -2.0, 0.5]]], [[[3.0, 1.0, -0.5]]]], dtype=np.float32)
    t = np.array([[0, 1]], dtype=np.int32)
    for scale in (0.37, 1.9, 0.0):
        out, _ = orc.decode_f64(q, k, v, t, np.array([2], np.int32), scale)
        s0 = 2 * 0.5 + 1 * 0.0 + (-1) * 1.0
        s1 = 2 * 1.0 + 1 * 2.0 + (-1) * 0.0
        w1 = 1.0 / (1.0 + math.exp(-scale * (s1 - s0)))
        want = v[0, 0, 0].astype(np.float64) + (v[1, 0, 0] - v[0, 0, 0]).astype(np.float64) * w1
        assert np.abs(out[0, 0] - want).max() <= 1e-15, scale


def pin_prefix_sharing_aliases(orc):
    """Two table rows that point at the same physical blocks, with the same q
    and length, give bit-identical rows; a row sharing only a prefix differs."""
    rng = np.random.default_rng(29)
    q, k, v, t, L = paged_case(rng, 3, 4, 2, 8, 4, [14, 3, 9], "bf16", max_blocks=4)
    t[1] = t[0]
    L[1] = L[0]
    q[1] = q[0]
    t[2, :3] = t[0, :3]                  # shares three blocks, then stops at 9 tokens
    q[2] = q[0]
    out, _ = orc.decode_f64(q, k, v, t, L, 0.35)
    assert np.array_equal(out[0], out[1])
    assert not np.array_equal(out[0], out[2])


def pin_shift_invariance(orc):
    """Adding one vector u to every key of a KV head adds scale*<q,u> to all of a
    query head's logits, which the softmax removes."""
    rng = np.random.default_rng(31)
    q, k, v, t, L = paged_case(rng, 2, 6, 2, 8, 4, [9, 17], "f32")
    out, _ = orc.decode_f64(q, k, v, t, L, 0.3)
    u = rng.standard_normal((1, 1, 2, 8)).astype(np.float32)
    k2 = (k.astype(np.float64) + u).astype(np.float32)
    # the float32 rounding of k + u perturbs logits by ~1e-7 relative; compare loosely
    out2, _ = orc.decode_f64(q, k2, v, t, L, 0.3)
    assert np.abs(out - out2).max() <= 1e-5


def pin_edge_statuses(orc):
    """L = 0 gives zeros; a bad block id or an over-long length gives NaN rows
    and a non-zero status; unused blocks and tail slots are never read."""
    rng = np.random.default_rng(37)
    q, k, v, t, L = paged_case(rng, 3, 4, 2, 8, 4, [0, 6, 5], "f32", max_blocks=3)
    out, rc = orc.decode_f64(q, k, v, t, L, 0.3)
    assert rc == 0 and np.array_equal(out[0], np.zeros_like(out[0]))
    # poison everything the definition does not touch
    used = set(t[1, :2]) | set(t[2, :2])
    kp, vp = k.copy(), v.copy()
    for blk in range(k.shape[0]):
        if blk not in used:
            kp[blk] = np.nan
            vp[blk] = np.nan
    kp[t[1, 1], 2:] = np.nan
    vp[t[1, 1], 2:] = np.nan
    kp[t[2, 1], 1:] = np.nan
    vp[t[2, 1], 1:] = np.nan
    t2 = t.copy()
    t2[1:, 2] = 12345                    # entries past the last block are ignored
    out_p, rc = orc.decode_f64(q, kp, vp, t2, L, 0.3)
    assert rc == 0 and np.array_equal(out, out_p)
    t3 = t.copy()
    t3[1, 1] = k.shape[0]                # out of range
    out_b, rc = orc.decode_f64(q, k, v, t3, L, 0.3)
    assert rc == 2 and np.all(np.isnan(out_b[1])) and np.array_equal(out_b[2], out[2])
    L4 = L.copy()
    L4[2] = 3 * 4 + 1                    # longer than max_blocks * block_size
    out_l, rc = orc.decode_f64(q, k, v, t, L4, 0.3)
    assert rc == 3 and np.all(np.isnan(out_l[2])) and np.array_equal(out_l[1], out[1])


def pin_bf16_widening(orc):
    """bfloat16 bit patterns decode exactly (value = the float32 whose top 16
    bits they are): 1.0, -2.0, 1 + 2^-7, the largest finite, the smallest
    subnormal, -0."""
    pats = np.array([0x3F80, 0xC000, 0x3F81, 0x7F7F, 0x0001, 0x8000, 0x4049, 0xBE80],
                    dtype=np.uint16)
    want = np.array([1.0, -2.0, 1.0 + 2.0 ** -7, (2 - 2.0 ** -7) * 2.0 ** 127, 2.0 ** -133,
                     -0.0, 3.140625, -0.25])
    D = pats.size
    q = np.zeros((1, 1, D), dtype=np.uint16)
    k = np.zeros((1, 1, 1, D), dtype=np.uint16)
    v = pats.reshape(1, 1, 1, D)
    out, _ = orc.decode_f64(q, k, v, np.array([[0]], np.int32), np.array([1], np.int32), 1.0)
    assert np.array_equal(out[0, 0], want)


def pin_rows_match_full(orc):
    """The selected-rows entry point returns the same rows as the full one."""
    rng = np.random.default_rng(41)
    q, k, v, t, L = paged_case(rng, 4, 8, 2, 16, 4, [3, 17, 1, 8], "bf16")
    out, _ = orc.decode_f64(q, k, v, t, L, 0.25)
    rows = np.array([[0, 0], [3, 7], [1, 5], [2, 2]])
    sub, _ = orc.decode_rows_f64(q, k, v, t, L, 0.25, rows)
    for i, (b, h) in enumerate(rows):
        assert np.array_equal(sub[i], out[b, h])


# ----------------------------------------------------------------- extension pins
# Several query tokens per sequence (speculative verification, "Modern LLM
# Inference ...", section 7.1) and local attention over the most recent W
# tokens (same notes, section 4.4 "Local Attention").
def _ex_case(rng, B, q_len, Hq, Hkv, D, bs, lens, dtype="f32", max_blocks=None):
    q, k, v, t, L = paged_case(rng, B, Hq * q_len, Hkv * q_len, D, bs, lens, dtype,
                               max_blocks=max_blocks)
    # reuse the generator's shapes, then reshape q to [B, q_len, Hq, D]
    q = q.reshape(B, q_len, Hq, D)
    k = k[:, :, :Hkv].copy()
    v = v[:, :, :Hkv].copy()
    return q, k, v, t, L


def pin_ex_reduces_to_single_query(orc):
    """q_len = 1 and no window is exactly the single-query decode."""
    rng = np.random.default_rng(43)
    q, k, v, t, L = paged_case(rng, 3, 8, 2, 16, 4, [9, 1, 14], "bf16")
    a, _ = orc.decode_f64(q, k, v, t, L, 0.3)
    b, _ = orc.decode_ex_f64(q[:, None], k, v, t, L, 0.3, 0)
    assert np.array_equal(a, b[:, 0])


def pin_ex_brute_force(orc):
    """Dense masked formulation, several query counts and windows."""
    rng = np.random.default_rng(47)
    for q_len, window, dt in ((3, 0, "f32"), (4, 5, "bf16"), (2, 1, "f32"), (5, 100, "f32"),
                              (1, 3, "bf16")):
        q, k, v, t, L = _ex_case(rng, 3, q_len, 4, 2, 8, 4, [9, 17, 6], dt)
        out, rc = orc.decode_ex_f64(q, k, v, t, L, 0.35, window)
        ref = brute_decode_ex(q, k, v, t, L, 0.35, window)
        assert rc == 0 and np.abs(out - ref).max() <= 1e-12, (q_len, window, dt)


def pin_ex_causal_prefix(orc):
    """Query i of a q_len call equals a single-query call on the sequence cut
    right after query i's own token."""
    rng = np.random.default_rng(53)
    q_len = 4
    q, k, v, t, L = _ex_case(rng, 2, q_len, 6, 3, 8, 4, [11, 7], "bf16")
    out, _ = orc.decode_ex_f64(q, k, v, t, L, 0.25, 0)
    for i in range(q_len):
        cut = L - q_len + i + 1
        one, _ = orc.decode_f64(q[:, i], k, v, t, cut, 0.25)
        assert np.array_equal(out[:, i], one), i


def pin_ex_window_is_recent_tokens(orc):
    """A window of W equals attention over a sequence holding only the W most
    recent tokens; W = 1 returns the query token's own V row."""
    rng = np.random.default_rng(59)
    q, k, v, t, L = _ex_case(rng, 2, 1, 4, 2, 8, 4, [13, 6], "bf16")
    for W in (1, 3, 6, 20):
        out, _ = orc.decode_ex_f64(q, k, v, t, L, 0.4, W)
        for b in range(2):
            n = min(W, int(L[b]))
            lo = int(L[b]) - n
            kk = np.zeros((1, n, 2, 8), dtype=k.dtype)
            vv = np.zeros_like(kk)
            for j in range(n):
                tok = lo + j
                kk[0, j] = k[t[b, tok // 4], tok % 4]
                vv[0, j] = v[t[b, tok // 4], tok % 4]
            one, _ = orc.decode_f64(q[b:b + 1, 0], kk, vv, np.zeros((1, 1), np.int32),
                                    np.array([n], np.int32), 0.4)
            assert np.array_equal(out[b, 0], one[0]), (W, b)
        if W == 1:
            vf = as_f64(v)
            for b in range(2):
                tok = int(L[b]) - 1
                for h in range(4):
                    assert np.array_equal(out[b, 0, h], vf[t[b, tok // 4], tok % 4, h // 2])


def pin_ex_blocks_before_window_unread(orc):
    """Blocks older than the window may be discarded (table entry -1): the
    result does not change; discarding a block the window still needs is an
    error.  Sequence 0: L 17, two queries at positions 15 and 16, window 5, so
    tokens 11..16 are read (blocks 2, 3, 4 of 4-token blocks)."""
    rng = np.random.default_rng(61)
    q, k, v, t, L = _ex_case(rng, 2, 2, 4, 2, 8, 4, [17, 9], "f32")
    a, rc = orc.decode_ex_f64(q, k, v, t, L, 0.3, 5)
    t2 = t.copy()
    t2[0, :2] = -1                     # tokens 0..7: outside every window of sequence 0
    b, rc2 = orc.decode_ex_f64(q, k, v, t2, L, 0.3, 5)
    assert rc == rc2 == 0 and np.array_equal(a, b)
    t3 = t.copy()
    t3[0, 2] = -1                      # tokens 8..11: token 11 is still in a window
    _, rc3 = orc.decode_ex_f64(q, k, v, t3, L, 0.3, 5)
    assert rc3 == 2


def pin_ex_empty_rows_are_zero(orc):
    """A query whose position is before the sequence start (L < q_len) has an
    empty range and gives zeros; the others are unaffected."""
    rng = np.random.default_rng(67)
    q, k, v, t, L = _ex_case(rng, 1, 4, 4, 2, 8, 4, [2], "f32")
    out, rc = orc.decode_ex_f64(q, k, v, t, L, 0.3, 0)
    assert rc == 0
    assert np.array_equal(out[0, :2], np.zeros_like(out[0, :2]))
    ref = brute_decode_ex(q, k, v, t, L, 0.3, 0)
    assert np.abs(out - ref).max() <= 1e-12


# ----------------------------------------------------------------- 8-bit K/V pins
# K/V stored as 8-bit floats (1 sign, 4 exponent bits with bias 7, 3 mantissa
# bits) with one scale per KV head: quantized KV pages ("Modern LLM Inference
# ...", section 6, quantization; "The Ultimate Guide ... Part 2", "KV Cache
# Compression").
E4M3_CASES = [(0x38, 1.0), (0x40, 2.0), (0x30, 0.5), (0x39, 1.125), (0x7E, 448.0),
              (0xFE, -448.0), (0x08, 2.0 ** -6), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9),
              (0xB8, -1.0), (0x00, 0.0), (0x5A, 20.0), (0x5C, 24.0)]


def _kv8_case(rng, B, Hq, Hkv, D, bs, lens):
    q, k, v, t, L = paged_case(rng, B, Hq, Hkv, D, bs, lens, "f32")
    k8 = rng.integers(0, 256, size=k.shape).astype(np.uint8)
    v8 = rng.integers(0, 256, size=v.shape).astype(np.uint8)
    k8[(k8 & 0x7F) == 0x7F] = 0x38          # no NaN codes
    v8[(v8 & 0x7F) == 0x7F] = 0x30
    ks = rng.uniform(0.01, 0.1, size=Hkv).astype(np.float32)   # keep logits moderate
    vs = rng.uniform(0.5, 2.0, size=Hkv).astype(np.float32)
    return q, k8, v8, ks, vs, t, L


def pin_kv8_e4m3_values(orc):
    """One cached token: the output is v_scale times the e4m3 value, for codes
    with known values (normal, subnormal, largest, signed zero)."""
    D = len(E4M3_CASES)
    q = np.zeros((1, 1, D), dtype=np.float32)
    k8 = np.zeros((1, 1, 1, D), dtype=np.uint8)
    v8 = np.array([c for c, _ in E4M3_CASES], dtype=np.uint8).reshape(1, 1, 1, D)
    for vs in (1.0, 0.75):
        out, rc = orc.decode_kv8_f64(q, k8, v8, np.ones(1, np.float32),
                                     np.full(1, vs, np.float32), np.zeros((1, 1), np.int32),
                                     np.ones(1, np.int32), 1.0)
        assert rc == 0
        assert np.array_equal(out[0, 0], vs * np.array([x for _, x in E4M3_CASES]))


def pin_kv8_brute_force(orc):
    """Against the dense formulation fed by torch's own e4m3 decoding."""
    from oracle.brute import brute_decode_kv8
    rng = np.random.default_rng(71)
    for lens, q_len, window in (([9, 17, 3], 1, 0), ([12, 5, 30], 3, 0), ([20, 8, 14], 2, 6)):
        q, k8, v8, ks, vs, t, L = _kv8_case(rng, 3, 4 * q_len, 2, 8, 4, lens)
        q = q.reshape(3, q_len, 4, 8)
        out, rc = orc.decode_kv8_f64(q, k8, v8, ks, vs, t, L, 0.3, window)
        ref = brute_decode_kv8(q, k8, v8, ks, vs, t, L, 0.3, window)
        assert rc == 0 and np.abs(out - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def pin_kv8_equals_wide_pages(orc):
    """With unit scales, 8-bit pages give exactly the result of bfloat16 pages
    holding the same values (every finite e4m3 value is a bfloat16 value)."""
    from oracle.brute import e4m3_to_f64
    rng = np.random.default_rng(73)
    q, k8, v8, _, _, t, L = _kv8_case(rng, 2, 4, 2, 8, 4, [11, 6])
    qb = bf16_bits(q)
    one = np.ones(2, np.float32)
    a, _ = orc.decode_kv8_f64(qb, k8, v8, one, one, t, L, 0.05)
    kb = bf16_bits(e4m3_to_f64(k8).astype(np.float32))
    vb = bf16_bits(e4m3_to_f64(v8).astype(np.float32))
    b, _ = orc.decode_f64(qb, kb, vb, t, L, 0.05)
    assert np.array_equal(a, b)


def pin_kv8_scales(orc):
    """A V scale s multiplies the output by s; a K scale s acts like a logit
    scale times s."""
    rng = np.random.default_rng(79)
    q, k8, v8, ks, vs, t, L = _kv8_case(rng, 2, 4, 2, 8, 4, [9, 13])
    one = np.ones(2, np.float32)
    base, _ = orc.decode_kv8_f64(q, k8, v8, one, one, t, L, 0.02)
    v2, _ = orc.decode_kv8_f64(q, k8, v8, one, np.array([3.0, 0.5], np.float32), t, L, 0.02)
    assert np.abs(v2[:, :2] - 3.0 * base[:, :2]).max() <= 1e-12 * np.abs(base).max()
    assert np.abs(v2[:, 2:] - 0.5 * base[:, 2:]).max() <= 1e-12 * np.abs(base).max()
    k2, _ = orc.decode_kv8_f64(q, k8, v8, np.full(2, 2.0, np.float32), one, t, L, 0.02)
    s2, _ = orc.decode_kv8_f64(q, k8, v8, one, one, t, L, 0.04)
    assert np.abs(k2 - s2).max() <= 1e-12 * np.abs(s2).max()


# ------------------------------------------- int8 codes and per-block scales
# The same quantized pages with signed 8-bit integer codes, and with a scale
# per physical block and KV head instead of one per KV head: a block's scale is
# fixed when the block is written, so a cache filled token by token can give
# each block its own range ("Modern LLM Inference ...", section 6, int8 / fp8
# quantization; "The Ultimate Guide ... Part 2", "KV Cache Compression").
INT8_CASES = [(0x80, -128.0), (0xFF, -1.0), (0x00, 0.0), (0x01, 1.0), (0x7F, 127.0),
              (0x9C, -100.0), (0x64, 100.0), (0xC0, -64.0), (0x2A, 42.0)]


def _q8_case(rng, code, B, Hq, Hkv, D, bs, lens, per_block):
    q, k, v, t, L = paged_case(rng, B, Hq, Hkv, D, bs, lens, "f32")
    k8 = rng.integers(0, 256, size=k.shape).astype(np.uint8)
    v8 = rng.integers(0, 256, size=v.shape).astype(np.uint8)
    if code == "e4m3":
        k8[(k8 & 0x7F) == 0x7F] = 0x38          # no NaN codes
        v8[(v8 & 0x7F) == 0x7F] = 0x30
    shape = (k.shape[0], Hkv) if per_block else (Hkv,)
    lo, hi = (0.01, 0.1) if code == "e4m3" else (0.0005, 0.005)   # moderate logits
    ks = rng.uniform(lo, hi, size=shape).astype(np.float32)
    vs = rng.uniform(0.5, 2.0, size=shape).astype(np.float32)
    return q, k8, v8, ks, vs, t, L


def pin_q8_int8_values(orc):
    """One cached token: the output is the V scale times the signed integer
    code, with the scale taken from the row of the block the token sits in."""
    D = len(INT8_CASES)
    q = np.zeros((1, 1, D), dtype=np.float32)
    k8 = np.zeros((3, 1, 1, D), dtype=np.uint8)
    v8 = np.zeros((3, 1, 1, D), dtype=np.uint8)
    v8[2, 0, 0] = [c for c, _ in INT8_CASES]
    want = np.array([x for _, x in INT8_CASES])
    table = np.array([[2]], np.int32)
    one = np.ones(1, np.int32)
    out, rc = orc.decode_q8_f64(q, k8, v8, "int8", np.ones(1, np.float32),
                                np.full(1, 0.75, np.float32), table, one, 1.0)
    assert rc == 0 and np.array_equal(out[0, 0], 0.75 * want)
    vs = np.array([[9.0], [5.0], [0.25]], np.float32)           # block 2 -> 0.25
    out, rc = orc.decode_q8_f64(q, k8, v8, "int8", np.ones((3, 1), np.float32), vs, table, one,
                                1.0)
    assert rc == 0 and np.array_equal(out[0, 0], 0.25 * want)


def pin_q8_block_scale_closed_form(orc):
    """Four tokens in two 2-token blocks stored at physical blocks 3 and 1.
    Every K code is 1 and q = 1, so token t has logit ks[block(t)]; V codes
    are 1, 2, 3, 4.  With K scales (2.0 at block 3, 0.5 at block 1) and V
    scales (0.25 at block 3, 3.0 at block 1):
        out = (e^2 * 0.25 * (1 + 2) + e^0.5 * 3.0 * (3 + 4)) / (2 e^2 + 2 e^0.5)."""
    for code, one_code, v_codes in (("int8", 1, [1, 2, 3, 4]),
                                    ("e4m3", 0x38, [0x38, 0x40, 0x44, 0x48])):  # 1, 2, 3, 4
        k8 = np.zeros((4, 2, 1, 1), dtype=np.uint8)
        v8 = np.zeros((4, 2, 1, 1), dtype=np.uint8)
        k8[3, :, 0, 0] = one_code
        k8[1, :, 0, 0] = one_code
        v8[3, :, 0, 0] = v_codes[:2]
        v8[1, :, 0, 0] = v_codes[2:]
        ks = np.array([[5.0], [0.5], [7.0], [2.0]], np.float32)
        vs = np.array([[9.0], [3.0], [11.0], [0.25]], np.float32)
        q = np.ones((1, 1, 1), dtype=np.float32)
        out, rc = orc.decode_q8_f64(q, k8, v8, code, ks, vs, np.array([[3, 1]], np.int32),
                                    np.array([4], np.int32), 1.0)
        e2, e05 = math.exp(2.0), math.exp(0.5)
        want = (e2 * 0.25 * (1 + 2) + e05 * 3.0 * (3 + 4)) / (2 * e2 + 2 * e05)
        assert rc == 0 and abs(out[0, 0, 0] - want) <= 1e-12 * want, (code, out[0, 0, 0], want)


def pin_q8_brute_force(orc):
    """Against the dense formulation on pages dequantised outside the oracle
    (torch's e4m3 decoding, numpy's int8 view), both scale forms, several
    query tokens and windows."""
    from oracle.brute import brute_decode_q8
    rng = np.random.default_rng(83)
    for code in ("e4m3", "int8"):
        for per_block in (False, True):
            for lens, q_len, window in (([9, 17, 3], 1, 0), ([12, 5, 30], 3, 0),
                                        ([20, 8, 14], 2, 6)):
                q, k8, v8, ks, vs, t, L = _q8_case(rng, code, 3, 4 * q_len, 2, 8, 4, lens,
                                                   per_block)
                q = q.reshape(3, q_len, 4, 8)
                out, rc = orc.decode_q8_f64(q, k8, v8, code, ks, vs, t, L, 0.3, window)
                ref = brute_decode_q8(q, k8, v8, code, ks, vs, t, L, 0.3, window)
                assert rc == 0
                assert np.abs(out - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max()), (
                    code, per_block, q_len, window)


def pin_q8_uniform_block_scales(orc):
    """A per-block table whose every row holds the per-head scales gives
    exactly the per-head result."""
    rng = np.random.default_rng(89)
    for code in ("e4m3", "int8"):
        q, k8, v8, ks, vs, t, L = _q8_case(rng, code, 2, 8, 2, 8, 4, [13, 7], False)
        a, _ = orc.decode_q8_f64(q, k8, v8, code, ks, vs, t, L, 0.5)
        nb = k8.shape[0]
        b, _ = orc.decode_q8_f64(q, k8, v8, code, np.tile(ks, (nb, 1)), np.tile(vs, (nb, 1)), t,
                                 L, 0.5)
        assert np.array_equal(a, b)


def pin_q8_block_permutation(orc):
    """Moving physical blocks together with their scale rows (and renumbering
    the table) leaves the output unchanged, bit for bit."""
    rng = np.random.default_rng(97)
    for code in ("e4m3", "int8"):
        q, k8, v8, ks, vs, t, L = _q8_case(rng, code, 3, 4, 2, 8, 4, [10, 3, 15], True)
        a, _ = orc.decode_q8_f64(q, k8, v8, code, ks, vs, t, L, 0.5)
        nb = k8.shape[0]
        perm = rng.permutation(nb)                     # new block i holds old block perm[i]
        inv = np.argsort(perm)
        t2 = np.where(t >= 0, inv[np.maximum(t, 0)], -1).astype(np.int32)
        b, _ = orc.decode_q8_f64(q, k8[perm], v8[perm], code, ks[perm], vs[perm], t2, L, 0.5)
        assert np.array_equal(a, b)


PINS = [
    pin_brute_force,
    pin_paged_equals_contiguous,
    pin_gqa_equals_repeated_mha,
    pin_length_one_returns_v_row,
    pin_identical_keys_mean_of_v,
    pin_hard_one_hot_large_logits,
    pin_closed_form_three_tokens,
    pin_scale_two_tokens,
    pin_prefix_sharing_aliases,
    pin_shift_invariance,
    pin_edge_statuses,
    pin_bf16_widening,
    pin_rows_match_full,
    pin_ex_reduces_to_single_query,
    pin_ex_brute_force,
    pin_ex_causal_prefix,
    pin_ex_window_is_recent_tokens,
    pin_ex_blocks_before_window_unread,
    pin_ex_empty_rows_are_zero,
    pin_kv8_e4m3_values,
    pin_kv8_brute_force,
    pin_kv8_equals_wide_pages,
    pin_kv8_scales,
    pin_q8_int8_values,
    pin_q8_block_scale_closed_form,
    pin_q8_brute_force,
    pin_q8_uniform_block_scales,
    pin_q8_block_permutation,
]
