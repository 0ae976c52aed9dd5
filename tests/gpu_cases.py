"""Helpers for the GPU parity tests: run the CUDA path, run the oracle, compare."""
import numpy as np
import torch

import gen
import oracle
import paged_gqa_decode_04_gb300 as pgd

# Tolerances against the float64 oracle (bf16 KV with fp32 accumulation; fp32 KV).
BF16_MAX, BF16_MEAN = 1e-2, 1e-3
F32_MAX, F32_MEAN = 1e-5, 1e-5


def tol(dtype):
    """float32 pools: 1e-5; bfloat16 and 8-bit pages (bf16 out, fp32 accumulation)."""
    return (F32_MAX, F32_MEAN) if dtype in ("f32", torch.float32) else (BF16_MAX, BF16_MEAN)


def run_cuda(w, num_splits=0, stream=None, check_error=True):
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool, w.k_scale, w.v_scale)
    try:
        out = pgd.paged_gqa_decode(pool, w.q, w.block_table, w.seq_lens, w.scale,
                                   num_splits=num_splits, stream=stream)
        status = pgd.paged_gqa_get_error(pool, stream)
    finally:
        pool.close()
    if check_error:
        assert status == 0, pgd.strerror(status)
    return out, status


def host(t):
    return gen.to_numpy_bits(t)


def run_oracle(w, table=None, lens=None, q=None, window=None):
    """Oracle answer for workload w (8-bit pages included); q [B, q_len, Hq, D]
    and window select the multi-token / windowed form."""
    table = w.table_np if table is None else table
    lens = w.lens_np if lens is None else lens
    qq = w.q if q is None else q
    if w.dtype in ("fp8", "i8"):
        # 8-bit pages: e4m3 or int8 codes, scales per KV head or per block and KV head
        return oracle.decode_q8_f64(host(qq), host(w.k_pool), host(w.v_pool),
                                    "e4m3" if w.dtype == "fp8" else "int8",
                                    w.k_scale.cpu().numpy(), w.v_scale.cpu().numpy(), table,
                                    lens, w.scale, window or 0)
    if q is not None or window:
        return oracle.decode_ex_f64(host(qq), host(w.k_pool), host(w.v_pool), table, lens,
                                    w.scale, window or 0)
    return oracle.decode_f64(host(w.q), host(w.k_pool), host(w.v_pool), table, lens, w.scale)


def errors(got, want):
    g = got.detach().float().cpu().numpy().astype(np.float64)
    e = np.abs(g - want)
    return g, float(e.max()), float(e.mean())


# 8-bit pages: an output is (float32 scale) x (e4m3 or int8 code) arithmetic,
# not a bfloat16 value, so rounding it to the bfloat16 output adds up to half
# an ulp, 2^-8 |out| (a one-token sequence returns a scaled V row of up to ~7);
# bfloat16 pages return their bfloat16 rows exactly there.
FP8_REL = 2.0 ** -8


def assert_close(got, want, dtype, what=""):
    g, emax, emean = errors(got, want)
    tmax, tmean = tol(dtype)
    assert np.isfinite(g).all(), "%s: non-finite output" % what
    if dtype in ("fp8", "i8", torch.float8_e4m3fn, torch.int8):
        excess = float((np.abs(g - want) - (tmax + FP8_REL * np.abs(want))).max())
        assert excess <= 0 and emean <= tmean, "%s: max %.3g (over the bound by %.3g) mean %.3g" % (
            what, emax, excess, emean)
        return emax, emean
    assert emax <= tmax and emean <= tmean, "%s: max %.3g mean %.3g" % (what, emax, emean)
    return emax, emean
