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


def layout(lens, hkv, max_tokens, W):
    """Tiles per unit of each sequence, its first virtual slot and the virtual
    total: each run (sequence, KV head) is W cost slots, then its tiles."""
    n = [tiles(L, max_tokens) for L in lens]
    v = [hkv * (x + W) if x > 0 else 0 for x in n]
    base = np.concatenate([[0], np.cumsum(v)]).astype(np.int64)
    return n, base, int(base[-1])


def run_tiles(n, base, b, kvh, W):
    """Virtual indices [t0, t1) of the real tiles of run (b, kvh)."""
    t0 = int(base[b]) + kvh * (n[b] + W) + W
    return t0, t0 + n[b]


def decode_pieces(lens, hkv, P, max_tokens, W=0):
    """What the decode CTAs write: {(b, kvh): [(cta, kind, slot, tiles)]}."""
    n, base, N = layout(lens, hkv, max_tokens, W)
    out = {}
    seen = np.zeros(N, dtype=np.int64)
    real = np.zeros(N, dtype=bool)
    span_real = []
    for c in range(P):
        r0, r1 = span_begin(c, N, P), span_begin(c + 1, N, P)
        cnt = 0
        for b in range(len(lens)):
            if n[b] == 0:
                continue
            for kvh in range(hkv):
                t0, t1 = run_tiles(n, base, b, kvh, W)
                real[t0:t1] = True
                s0, s1 = max(t0, r0), min(t1, r1)
                if s0 >= s1:
                    continue
                seen[s0:s1] += 1
                cnt += s1 - s0
                partial = s0 != t0 or s1 != t1
                slot = (1 if s0 != r0 else 0) if partial else None
                out.setdefault((b, kvh), []).append((c, "partial" if partial else "whole", slot,
                                                     s1 - s0))
        span_real.append(cnt)
    return out, seen, real, base, N, span_real


def merge_reads(lens, hkv, P, base, N, max_tokens, W=0):
    """What the merge reads: {(b, kvh): [(cta, slot)]} for split runs."""
    n = [tiles(L, max_tokens) for L in lens]
    reads = {}
    for b in range(len(lens)):
        if n[b] == 0:
            continue
        for kvh in range(hkv):
            t0, t1 = run_tiles(n, base, b, kvh, W)
            c0, c1 = span_owner(t0, N, P), span_owner(t1 - 1, N, P)
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


@pytest.mark.parametrize("W", [0, 3])
@pytest.mark.parametrize("seed", range(12))
def test_partition_covers_balances_and_merges(seed, W):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 12))
    hkv = int(rng.choice([1, 2, 8]))
    max_tokens = 2048
    lens = rng.integers(0, max_tokens + 1, size=B)
    lens[rng.random(B) < 0.2] = 0
    if seed % 3 == 0:
        lens[0] = max_tokens + 5          # invalid: owns no tiles
    P = int(rng.choice([1, 2, 3, 7, 152, 1000]))
    pieces, seen, real, base, N, span_real = decode_pieces(list(lens), hkv, P, max_tokens, W)
    assert np.all(seen[real] == 1) and np.all(seen[~real] == 0)   # cost slots hold no work
    if N:
        sizes = [span_begin(c + 1, N, P) - span_begin(c, N, P) for c in range(P)]
        assert max(sizes) - min(sizes) <= 1
        # a span's size is its real tiles plus the cost slots it holds
        for c in range(P):
            r0, r1 = span_begin(c, N, P), span_begin(c + 1, N, P)
            assert span_real[c] == int(real[r0:r1].sum())
    reads = merge_reads(list(lens), hkv, P, base, N, max_tokens, W)
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


def test_run_cost_moves_tiles_away_from_run_starts():
    """Three sequences of 10 tiles, two spans.  Without a run cost they split
    15 / 15 tiles.  With W = 4 the virtual total is 3 * 14 = 42 and span 0 =
    slots [0, 21) holds the starts of runs 0 and 1 (8 cost slots, 13 tiles),
    span 1 = [21, 42) the start of run 2 (4 cost slots, 17 tiles)."""
    lens, hkv, P = [64 * 10] * 3, 1, 2
    for W, want in ((0, [15, 15]), (4, [13, 17])):
        _, _, _, _, _, span_real = decode_pieces(lens, hkv, P, 4096, W)
        assert span_real == want


def spans_in_use(N, P, min_tiles):
    """The kernel's rule: fewer spans only when asked (min_tiles > 1)."""
    if min_tiles <= 1:
        return P
    return max(1, min(P, -(-N // min_tiles)))


@pytest.mark.parametrize("N,P,mt,want", [(6, 152, 4, 2), (12, 152, 1, 152), (1000, 152, 4, 152),
                                         (0, 152, 4, 1), (7, 3, 4, 2)])
def test_spans_in_use(N, P, mt, want):
    assert spans_in_use(N, P, mt) == want
