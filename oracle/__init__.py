"""Float64 CPU oracle for paged grouped-query decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports this module;
only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It
shares no code with the CUDA library.

``decode_f64`` wraps the C oracle (oracle.c) through ctypes.  Inputs are numpy
arrays in their stored type: float32, or bfloat16 held as uint16 bit patterns;
the C code widens them exactly to double.  ``brute`` is an independent dense
numpy formulation used only to pin the C oracle on tiny inputs.
"""
import ctypes

import numpy as np

from . import build as _build

F32 = 0
BF16 = 1
FP8_E4M3 = 2
INT8 = 3
STATUS = {0: "ok", 1: "bad arguments", 2: "block id out of range", 3: "sequence length out of range"}


def _prep(q, k_pool, v_pool, block_table, seq_lens):
    q = np.ascontiguousarray(q)
    k_pool = np.ascontiguousarray(k_pool)
    v_pool = np.ascontiguousarray(v_pool)
    if q.dtype == np.float32:
        dtype = F32
    elif q.dtype == np.uint16:
        dtype = BF16
    else:
        raise TypeError("q must be float32 or uint16 (bfloat16 bits), got %s" % q.dtype)
    if k_pool.dtype != q.dtype or v_pool.dtype != q.dtype:
        raise TypeError("q, k_pool and v_pool must share one dtype")
    if q.ndim != 3 or k_pool.ndim != 4 or k_pool.shape != v_pool.shape:
        raise ValueError("q must be [B,Hq,D]; pools [num_blocks,block_size,Hkv,D]")
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, D = q.shape
    num_blocks, block_size, Hkv, D2 = k_pool.shape
    if D2 != D:
        raise ValueError("head_dim mismatch")
    if block_table.ndim != 2 or block_table.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("block_table must be [B,max_blocks], seq_lens [B]")
    dims = (B, Hq, Hkv, D, block_size, num_blocks, block_table.shape[1])
    return q, k_pool, v_pool, block_table, seq_lens, dtype, dims


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path):
        lib = ctypes.CDLL(path)
        argt = ([ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 + [ctypes.c_int64, ctypes.c_int,
                                                              ctypes.c_double])
        lib.oracle_decode_f64.argtypes = argt + [ctypes.c_void_p]
        lib.oracle_decode_f64.restype = ctypes.c_int
        lib.oracle_decode_rows_f64.argtypes = argt + [ctypes.c_void_p, ctypes.c_int64,
                                                      ctypes.c_void_p]
        lib.oracle_decode_rows_f64.restype = ctypes.c_int
        lib.oracle_decode_ex_f64.argtypes = ([ctypes.c_void_p] * 5 + [ctypes.c_int] * 7 +
                                             [ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_double, ctypes.c_void_p])
        lib.oracle_decode_ex_f64.restype = ctypes.c_int
        lib.oracle_decode_kv8_f64.argtypes = ([ctypes.c_void_p, ctypes.c_int] +
                                              [ctypes.c_void_p] * 6 + [ctypes.c_int] * 6 +
                                              [ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_double, ctypes.c_void_p])
        lib.oracle_decode_kv8_f64.restype = ctypes.c_int
        lib.oracle_decode_q8_f64.argtypes = ([ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p] + [ctypes.c_int] * 6 +
                                             [ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_double, ctypes.c_void_p])
        lib.oracle_decode_q8_f64.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_num_threads.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def num_threads(self):
        return int(self.lib.oracle_num_threads())

    def set_num_threads(self, n):
        """Rows computed at once from now on (the arithmetic of a row does not
        change); returns the count in effect."""
        return int(self.lib.oracle_set_num_threads(int(n)))

    def decode_f64(self, q, k_pool, v_pool, block_table, seq_lens, scale):
        """All rows.  Returns (out[B,Hq,D] float64, status)."""
        q, k_pool, v_pool, bt, sl, dtype, dims = _prep(q, k_pool, v_pool, block_table, seq_lens)
        B, Hq, Hkv, D, bs, nb, mb = dims
        out = np.empty((B, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_decode_f64(q.ctypes.data, k_pool.ctypes.data, v_pool.ctypes.data,
                                        bt.ctypes.data, sl.ctypes.data, dtype, B, Hq, Hkv, D,
                                        bs, nb, mb, float(scale), out.ctypes.data)
        if rc == 1:
            raise ValueError("oracle rejected the arguments")
        return out, int(rc)

    def decode_rows_f64(self, q, k_pool, v_pool, block_table, seq_lens, scale, rows):
        """Selected (b, h) rows; rows is [n, 2].  Returns (out[n, D] float64, status)."""
        q, k_pool, v_pool, bt, sl, dtype, dims = _prep(q, k_pool, v_pool, block_table, seq_lens)
        B, Hq, Hkv, D, bs, nb, mb = dims
        rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
        out = np.empty((rows.shape[0], D), dtype=np.float64)
        rc = self.lib.oracle_decode_rows_f64(q.ctypes.data, k_pool.ctypes.data,
                                             v_pool.ctypes.data, bt.ctypes.data, sl.ctypes.data,
                                             dtype, B, Hq, Hkv, D, bs, nb, mb, float(scale),
                                             rows.ctypes.data, rows.shape[0], out.ctypes.data)
        if rc == 1:
            raise ValueError("oracle rejected the arguments")
        return out, int(rc)


    def decode_ex_f64(self, q, k_pool, v_pool, block_table, seq_lens, scale, window=0):
        """q [B, q_len, Hq, D]: several query tokens per sequence (the last
        q_len cached tokens), causal, optional window.  Returns (out, status)."""
        q = np.ascontiguousarray(q)
        if q.ndim != 4:
            raise ValueError("q must be [B, q_len, Hq, D]")
        B, q_len, Hq, D = q.shape
        flat = q.reshape(B, q_len * Hq, D)
        _, k_pool, v_pool, bt, sl, dtype, dims = _prep(flat, k_pool, v_pool, block_table,
                                                       seq_lens)
        _, _, Hkv, _, bs, nb, mb = dims
        if Hq % Hkv:
            raise ValueError("oracle rejected the arguments")
        out = np.empty((B, q_len, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_decode_ex_f64(q.ctypes.data, k_pool.ctypes.data, v_pool.ctypes.data,
                                           bt.ctypes.data, sl.ctypes.data, dtype, B, q_len, Hq,
                                           Hkv, D, bs, nb, mb, int(window), float(scale),
                                           out.ctypes.data)
        if rc == 1:
            raise ValueError("oracle rejected the arguments")
        return out, int(rc)


    def decode_kv8_f64(self, q, k8, v8, k_scale, v_scale, block_table, seq_lens, scale,
                       window=0):
        """8-bit (e4m3) K/V pages with one scale per KV head.  q is
        [B, q_len, Hq, D] (or [B, Hq, D]) float32 or bfloat16 bits; k8 / v8 are
        uint8 [num_blocks, bs, Hkv, D]; k_scale / v_scale float32 [Hkv].
        Returns (out with q's shape, float64; status)."""
        q = np.ascontiguousarray(q)
        squeeze = q.ndim == 3
        if squeeze:
            q = q[:, None]
        if q.dtype == np.float32:
            q_dtype = F32
        elif q.dtype == np.uint16:
            q_dtype = BF16
        else:
            raise TypeError("q must be float32 or bfloat16 bits")
        k8 = np.ascontiguousarray(k8, dtype=np.uint8)
        v8 = np.ascontiguousarray(v8, dtype=np.uint8)
        ks = np.ascontiguousarray(k_scale, dtype=np.float32)
        vs = np.ascontiguousarray(v_scale, dtype=np.float32)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, q_len, Hq, D = q.shape
        nb, bs, Hkv, D2 = k8.shape
        if D2 != D or v8.shape != k8.shape or ks.shape != (Hkv,) or vs.shape != (Hkv,):
            raise ValueError("shape mismatch")
        out = np.empty((B, q_len, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_decode_kv8_f64(q.ctypes.data, q_dtype, k8.ctypes.data,
                                            v8.ctypes.data, ks.ctypes.data, vs.ctypes.data,
                                            bt.ctypes.data, sl.ctypes.data, B, q_len, Hq, Hkv,
                                            D, bs, nb, bt.shape[1], int(window), float(scale),
                                            out.ctypes.data)
        if rc == 1:
            raise ValueError("oracle rejected the arguments")
        return (out[:, 0] if squeeze else out), int(rc)

    def decode_q8_f64(self, q, k8, v8, code, k_scale, v_scale, block_table, seq_lens, scale,
                      window=0):
        """8-bit K/V pages of `code` "e4m3" or "int8" (signed).  k_scale /
        v_scale float32 [Hkv] (one scale per KV head) or [num_blocks, Hkv] (one
        per physical block and KV head).  q is [B, q_len, Hq, D] (or [B, Hq,
        D]) float32 or bfloat16 bits.  Returns (out with q's shape, float64;
        status)."""
        q = np.ascontiguousarray(q)
        squeeze = q.ndim == 3
        if squeeze:
            q = q[:, None]
        if q.dtype == np.float32:
            q_dtype = F32
        elif q.dtype == np.uint16:
            q_dtype = BF16
        else:
            raise TypeError("q must be float32 or bfloat16 bits")
        codes = {"e4m3": FP8_E4M3, "int8": INT8}
        if code not in codes:
            raise ValueError("code must be 'e4m3' or 'int8'")
        k8 = np.ascontiguousarray(k8).view(np.uint8)
        v8 = np.ascontiguousarray(v8).view(np.uint8)
        ks = np.ascontiguousarray(k_scale, dtype=np.float32)
        vs = np.ascontiguousarray(v_scale, dtype=np.float32)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, q_len, Hq, D = q.shape
        nb, bs, Hkv, D2 = k8.shape
        if ks.shape == (Hkv,) and vs.shape == (Hkv,):
            per_block = 0
        elif ks.shape == (nb, Hkv) and vs.shape == (nb, Hkv):
            per_block = 1
        else:
            raise ValueError("scales must be [Hkv] or [num_blocks, Hkv]")
        if D2 != D or v8.shape != k8.shape:
            raise ValueError("shape mismatch")
        out = np.empty((B, q_len, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_decode_q8_f64(q.ctypes.data, q_dtype, k8.ctypes.data,
                                           v8.ctypes.data, codes[code], ks.ctypes.data,
                                           vs.ctypes.data, per_block, bt.ctypes.data,
                                           sl.ctypes.data, B, q_len, Hq, Hkv, D, bs, nb,
                                           bt.shape[1], int(window), float(scale),
                                           out.ctypes.data)
        if rc == 1:
            raise ValueError("oracle rejected the arguments")
        return (out[:, 0] if squeeze else out), int(rc)


_default = None


def default():
    """The oracle built from oracle.c beside this file (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def num_threads():
    return default().num_threads()


def set_num_threads(n):
    return default().set_num_threads(n)


def decode_f64(q, k_pool, v_pool, block_table, seq_lens, scale):
    return default().decode_f64(q, k_pool, v_pool, block_table, seq_lens, scale)


def decode_ex_f64(q, k_pool, v_pool, block_table, seq_lens, scale, window=0):
    return default().decode_ex_f64(q, k_pool, v_pool, block_table, seq_lens, scale, window)


def decode_kv8_f64(q, k8, v8, k_scale, v_scale, block_table, seq_lens, scale, window=0):
    return default().decode_kv8_f64(q, k8, v8, k_scale, v_scale, block_table, seq_lens, scale,
                                    window)


def decode_q8_f64(q, k8, v8, code, k_scale, v_scale, block_table, seq_lens, scale, window=0):
    return default().decode_q8_f64(q, k8, v8, code, k_scale, v_scale, block_table, seq_lens,
                                   scale, window)


def decode_rows_f64(q, k_pool, v_pool, block_table, seq_lens, scale, rows):
    return default().decode_rows_f64(q, k_pool, v_pool, block_table, seq_lens, scale, rows)
