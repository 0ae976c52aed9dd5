"""Dense numpy brute force for tiny inputs; pins the C oracle.

TEST INFRASTRUCTURE ONLY.  A second, independent formulation of the same
textbook result: materialise every sequence's logical K and V with fancy
indexing, repeat each KV head over its query-head group, and evaluate
softmax(q K^T * scale) V as dense matrix products (Attention(Q,K,V) equation in
"Modern LLM Inference - Workloads, Bottlenecks, and Optimization Techniques",
section "Why Cross-Layer Attention Shares K/V but Not Q"; group sharing per its
section 4.1).  Sizes are meant to be tiny (L <= a few hundred).
"""
import numpy as np


def bf16_bits_to_f64(bits):
    """uint16 bfloat16 bit patterns -> float64, exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


def to_f64(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


def brute_decode(q, k_pool, v_pool, block_table, seq_lens, scale):
    q = to_f64(q)
    k_pool = to_f64(k_pool)
    v_pool = to_f64(v_pool)
    B, Hq, D = q.shape
    _, bs, Hkv, _ = k_pool.shape
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(seq_lens[b])
        if L == 0:
            continue
        t = np.arange(L)
        phys = np.asarray(block_table[b])[t // bs]
        K = k_pool[phys, t % bs]            # [L, Hkv, D]
        V = v_pool[phys, t % bs]
        K = np.repeat(K, G, axis=1)         # [L, Hq, D]: query head h reads KV head h // G
        V = np.repeat(V, G, axis=1)
        S = np.einsum("hd,lhd->hl", q[b], K) * scale   # [Hq, L]
        S = S - S.max(axis=1, keepdims=True)
        P = np.exp(S)
        P = P / P.sum(axis=1, keepdims=True)
        out[b] = np.einsum("hl,lhd->hd", P, V)
    return out


def brute_decode_ex(q, k_pool, v_pool, block_table, seq_lens, scale, window=0):
    """q [B, q_len, Hq, D]: dense scores over every cached token with a mask
    that keeps, for query i at position p = L - q_len + i, the positions
    max(0, p - window + 1) <= t <= p (no lower bound when window <= 0)."""
    q = to_f64(q)
    k_pool = to_f64(k_pool)
    v_pool = to_f64(v_pool)
    B, q_len, Hq, D = q.shape
    _, bs, Hkv, _ = k_pool.shape
    G = Hq // Hkv
    out = np.zeros((B, q_len, Hq, D))
    for b in range(B):
        L = int(seq_lens[b])
        if L == 0:
            continue
        t = np.arange(L)
        phys = np.asarray(block_table[b])[t // bs]
        K = np.repeat(k_pool[phys, t % bs], G, axis=1)      # [L, Hq, D]
        V = np.repeat(v_pool[phys, t % bs], G, axis=1)
        S = np.einsum("ihd,lhd->ihl", q[b], K) * scale       # [q_len, Hq, L]
        pos = L - q_len + np.arange(q_len)                    # [q_len]
        keep = t[None, :] <= pos[:, None]
        if window > 0:
            keep &= t[None, :] >= pos[:, None] - window + 1
        for i in range(q_len):
            if not keep[i].any():
                continue
            s = np.where(keep[i][None, :], S[i], -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            P = np.exp(s)
            P = P / P.sum(axis=1, keepdims=True)
            out[b, i] = np.einsum("hl,lhd->hd", P, V)
    return out


def e4m3_to_f64(bits):
    """uint8 e4m3 bit patterns -> float64, through torch's float8_e4m3fn type
    (an implementation independent of the C oracle's decoder)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def brute_decode_kv8(q, k8, v8, k_scale, v_scale, block_table, seq_lens, scale, window=0):
    """Dequantise the 8-bit pages (value = per-head scale x e4m3) and run the
    dense masked formulation."""
    k = e4m3_to_f64(k8) * np.asarray(k_scale, dtype=np.float64)[None, None, :, None]
    v = e4m3_to_f64(v8) * np.asarray(v_scale, dtype=np.float64)[None, None, :, None]
    q = np.asarray(q)
    if q.ndim == 3:
        return brute_decode_ex(q[:, None], k, v, block_table, seq_lens, scale, window)[:, 0]
    return brute_decode_ex(q, k, v, block_table, seq_lens, scale, window)


def int8_to_f64(bits):
    """uint8 bytes read as two's-complement int8 codes -> float64."""
    return np.ascontiguousarray(bits, dtype=np.uint8).view(np.int8).astype(np.float64)


def brute_decode_q8(q, k8, v8, code, k_scale, v_scale, block_table, seq_lens, scale,
                    window=0):
    """Dequantise 8-bit pages (value = scale x code value; the scale per KV
    head [Hkv] or per physical block and KV head [num_blocks, Hkv]) into
    dense float64 pools and run the dense masked formulation."""
    dec = e4m3_to_f64 if code == "e4m3" else int8_to_f64
    ks = np.asarray(k_scale, dtype=np.float64)
    vs = np.asarray(v_scale, dtype=np.float64)
    # broadcast the scales over [num_blocks, bs, Hkv, D]
    ks = ks[None, None, :, None] if ks.ndim == 1 else ks[:, None, :, None]
    vs = vs[None, None, :, None] if vs.ndim == 1 else vs[:, None, :, None]
    k = dec(k8) * ks
    v = dec(v8) * vs
    q = np.asarray(q)
    if q.ndim == 3:
        return brute_decode_ex(q[:, None], k, v, block_table, seq_lens, scale, window)[:, 0]
    return brute_decode_ex(q, k, v, block_table, seq_lens, scale, window)
