"""Byte and token accounting for paged decode attention (host side).

The roofline of decode attention is HBM bandwidth: every cached K/V byte of
every sequence is read once per step ("Modern LLM Inference ...", section 3:
decode attention has arithmetic intensity about 1 whatever the batch, and
"Advanced Optimizations: MQA, GQA, and PagedAttention": moving KV tensors
dominates).  Algorithmic bytes of one step:

    sum_b L_b * Hkv * D * elt * 2        K and V of the valid tokens
  + 2 * B * Hq * D * elt                 q in, out back
  + 4 * (B + sum_b ceil(L_b / bs))       seq_lens and the table entries used

Tail slots of the last block, unused table entries, the rest of the pool and
the split-KV workspace are not counted.
"""
import numpy as np

ELT = {"f32": 4, "bf16": 2, "fp8": 1, "i8": 1}      # K/V element bytes
Q_ELT = {"f32": 4, "bf16": 2, "fp8": 2, "i8": 2}    # q / out element bytes (bf16 with 8-bit pages)


def kv_bytes_per_token(hkv, d, elt):
    """K plus V bytes one cached token holds for one layer."""
    return 2 * hkv * d * elt


def gqa_reduction_factor(hq, hkv):
    """Cache shrink of GQA against MHA with the same query heads: N / K."""
    return kv_bytes_per_token(hq, 1, 1) / kv_bytes_per_token(hkv, 1, 1)


def algorithmic_bytes(lens, hq, hkv, d, block_size, elt, q_elt=None, block_scales=False):
    """elt: K/V element bytes; q_elt: q / out element bytes (default elt);
    block_scales: 8-bit pages with a K and a V float32 scale per block and KV
    head, read once for every block used (8 * Hkv bytes per block)."""
    q_elt = elt if q_elt is None else q_elt
    lens = np.asarray(lens, dtype=np.int64)
    pages = int(np.sum((lens + block_size - 1) // block_size))
    B = int(lens.size)
    return (int(lens.sum()) * kv_bytes_per_token(hkv, d, elt) + 2 * B * hq * d * q_elt
            + 4 * (B + pages) + (8 * hkv * pages if block_scales else 0))


def flops(lens, hq, d):
    """Multiply-adds of q.k and p.v, two flops each."""
    return 4 * int(np.sum(lens)) * hq * d


def tokens_read(L, q_len=1, window=0):
    """Cached tokens a call reads for one sequence: from the earliest token any
    of its q_len queries attends to (window W: max(0, L - q_len - W + 1)) to the
    end."""
    L = int(L)
    lo = max(0, L - q_len - window + 1) if window > 0 else 0
    return max(0, L - lo)


def algorithmic_bytes_ex(lens, hq, hkv, d, block_size, elt, q_len=1, window=0, q_elt=None,
                         block_scales=False):
    """Algorithmic bytes of a multi-token / windowed call: K/V of the tokens
    read, q and out for q_len tokens per sequence, the table words of the
    blocks read and seq_lens (and the per-block scales of the blocks read)."""
    q_elt = elt if q_elt is None else q_elt
    lens = np.asarray(lens, dtype=np.int64)
    kv = 0
    words = 0
    for L in lens.tolist():
        n = tokens_read(L, q_len, window)
        kv += n * kv_bytes_per_token(hkv, d, elt)
        if n:
            lo = L - n
            words += (L - 1) // block_size - lo // block_size + 1
    B = int(lens.size)
    return (kv + 2 * B * q_len * hq * d * q_elt + 4 * (B + words)
            + (8 * hkv * words if block_scales else 0))
