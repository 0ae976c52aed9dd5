"""Host model of the split-KV work partition the kernels use (CPU only).

Restates, in Python, the rules of partition.cuh and the merge kernel's
enumeration of the pieces of a run, and checks on random length mixes that
  * every (sequence, KV head, tile) lands in exactly one CTA span;
  * the spans differ in size by at most one tile (balance);
  * the pieces a CTA writes as partials are exactly the pieces the merge
    enumerates, in the same slots, with no slot written twice;
  * runs inside one span are written whole and never merged.
"""
import numpy as np
import pytest

T = 64


def tiles(L, max_tokens):
    return (L + T - 1) // T if 0 <= L <= max_tokens else 0


def span_begin(c, N, P):
    return (c * N) // P


def span_owner(x, N, P):
    return ((x + 1) * P - 1) // N


def decode_pieces(lens, hkv, P, max_tokens):
    """What the decode CTAs write: {(b, kvh): [(cta, kind, slot, tiles)]}."""
    n = [tiles(L, max_tokens) for L in lens]
    base = np.concatenate([[0], np.cumsum([hkv * x for x in n])]).astype(np.int64)
    N = int(base[-1])
    out = {}
    seen = np.zeros(N, dtype=np.int64)
    for c in range(P):
        r0, r1 = span_begin(c, N, P), span_begin(c + 1, N, P)
        for x in range(r0, r1):
            seen[x] += 1
        for b in range(len(lens)):
            for kvh in range(hkv):
                t0 = int(base[b]) + kvh * n[b]
                t1 = t0 + n[b]
                s0, s1 = max(t0, r0), min(t1, r1)
                if s0 >= s1:
                    continue
                partial = s0 != t0 or s1 != t1
                slot = (1 if s0 != r0 else 0) if partial else None
                out.setdefault((b, kvh), []).append((c, "partial" if partial else "whole", slot,
                                                     s1 - s0))
    return out, seen, base, N


def merge_reads(lens, hkv, P, base, N, max_tokens):
    """What the merge kernel reads: {(b, kvh): [(cta, slot)]} for split runs."""
    reads = {}
    for b, L in enumerate(lens):
        nb = tiles(L, max_tokens)
        if nb == 0:
            continue
        for kvh in range(hkv):
            t0 = int(base[b]) + kvh * nb
            c0, c1 = span_owner(t0, N, P), span_owner(t0 + nb - 1, N, P)
            if c0 == c1:
                continue
            lst = []
            for c in range(c0, c1 + 1):
                sb = span_begin(c, N, P)
                if sb == span_begin(c + 1, N, P):
                    continue
                lst.append((c, 1 if sb < t0 else 0))
            reads[(b, kvh)] = lst
    return reads


@pytest.mark.parametrize("seed", range(12))
def test_partition_covers_balances_and_merges(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 12))
    hkv = int(rng.choice([1, 2, 8]))
    max_tokens = 2048
    lens = rng.integers(0, max_tokens + 1, size=B)
    lens[rng.random(B) < 0.2] = 0
    if seed % 3 == 0:
        lens[0] = max_tokens + 5          # invalid: owns no tiles
    P = int(rng.choice([1, 2, 3, 7, 152, 1000]))
    pieces, seen, base, N = decode_pieces(list(lens), hkv, P, max_tokens)
    assert np.all(seen == 1)
    if N:
        sizes = [span_begin(c + 1, N, P) - span_begin(c, N, P) for c in range(P)]
        assert max(sizes) - min(sizes) <= 1
    reads = merge_reads(list(lens), hkv, P, base, N, max_tokens)
    slots_written = set()
    for key, lst in pieces.items():
        whole = [p for p in lst if p[1] == "whole"]
        if whole:
            assert len(lst) == 1 and key not in reads
            continue
        written = sorted((c, s) for c, _, s, _ in lst)
        assert written == sorted(reads[key]), key
        for cs in written:
            assert cs not in slots_written
            slots_written.add(cs)


def spans_in_use(N, P, min_tiles):
    """The kernel's rule: fewer spans only when asked (min_tiles > 1)."""
    if min_tiles <= 1:
        return P
    return max(1, min(P, -(-N // min_tiles)))


@pytest.mark.parametrize("N,P,mt,want", [(6, 152, 4, 2), (12, 152, 1, 152), (1000, 152, 4, 152),
                                         (0, 152, 4, 1), (7, 3, 4, 2)])
def test_spans_in_use(N, P, mt, want):
    assert spans_in_use(N, P, mt) == want
