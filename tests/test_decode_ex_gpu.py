"""Several query tokens per sequence (speculative verification) and local
attention windows, on the GPU against the float64 oracle (GPU only)."""
import numpy as np
import pytest
import torch

import gen
import oracle
import paged_gqa_decode_04_gb300 as pgd
from gpu_cases import assert_close, host

pytestmark = pytest.mark.gpu
DEV = "cuda"


def make_q(w, q_len, seed=5):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return torch.randn((w.B, q_len, w.Hq, w.D), generator=g, device=DEV).to(torch.bfloat16)


def run_ex(w, q, window, num_splits=0, table=None):
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool, w.k_scale, w.v_scale)
    try:
        bt = w.block_table if table is None else table
        out = pgd.paged_gqa_decode_ex(pool, q, bt, w.seq_lens, w.scale, window=window,
                                      num_splits=num_splits)
        st = pgd.paged_gqa_get_error(pool)
    finally:
        pool.close()
    assert st == 0, pgd.strerror(st)
    return out


def oracle_ex(w, q, window, table=None):
    from gpu_cases import run_oracle
    return run_oracle(w, table=table, q=q, window=window)


CASES = [
    # recipe, overrides, q_len, window
    ("llama3_8b", dict(B=6, lens=("uniform", 1, 700), max_len=768), 4, 0),      # 16 rows / head
    ("llama3_8b", dict(B=6, lens=("uniform", 1, 700), max_len=768), 1, 100),
    ("llama3_8b", dict(B=6, lens=("uniform", 50, 900), max_len=1024), 3, 37),
    ("llama3_8b", dict(B=4, lens=[5, 2, 130, 64], max_len=256), 8, 0),          # 32 rows / head
    ("long_70b", dict(B=2, lens=("uniform", 2000, 4000), max_len=4096), 2, 1000),
    ("mha_13b_b8", dict(B=2, lens=[300, 77], max_len=512), 5, 64),
    ("mqa_13b_b8", dict(B=2, lens=[300, 77], max_len=512), 1, 20),
    ("sweep_bs8", dict(B=8, lens=("lognormal", 100.0, 1.0, 1, 400), max_len=512), 2, 16),
    ("sweep_bs128", dict(B=8, lens=("lognormal", 300.0, 1.0, 1, 900), max_len=1024), 2, 200),
    ("llama3_8b_fp8", dict(B=6, lens=("uniform", 50, 900), max_len=1024), 4, 0),
    ("llama3_8b_fp8", dict(B=6, lens=("uniform", 50, 900), max_len=1024), 2, 100),
    ("llama3_8b", dict(B=4, D=64, lens=[5, 100, 260, 64], max_len=320), 3, 50),   # head_dim 64
    ("llama3_8b", dict(B=3, Hq=16, Hkv=4, lens=[90, 200, 17], max_len=256), 4, 0),  # 4 heads/unit
    ("llama3_8b_fp8", dict(B=3, Hq=16, Hkv=4, lens=[90, 300, 17], max_len=320), 2, 64),
    ("llama3_8b", dict(B=3, lens=[700, 33, 300], max_len=768), 16, 0),           # 64 rows / head
    ("long_70b", dict(B=2, lens=[3000, 1000], max_len=4096), 8, 100),           # 64 rows, window
    ("llama3_8b_fp8", dict(B=6, block_size=8, lens=("lognormal", 200.0, 1.0, 1, 900),
                           max_len=1024), 3, 40),                                # 8-token blocks
    ("mqa_13b_b8", dict(B=2, block_size=128, lens=[900, 300], max_len=1024), 1, 100),
    ("mha_13b_b8", dict(B=3, lens=[1000, 5, 260], max_len=1024), 2, 0),
    # int8 pages and per-block scales: causal and window bounds inside tiles
    # whose blocks carry different scales
    ("llama3_8b_i8", dict(B=6, lens=("uniform", 50, 900), max_len=1024), 4, 0),
    ("llama3_8b_i8_pb", dict(B=6, lens=("uniform", 50, 900), max_len=1024), 3, 40),
    ("llama3_8b_fp8_pb", dict(B=6, block_size=8, lens=("lognormal", 200.0, 1.0, 1, 900),
                              max_len=1024), 2, 100),
    ("long_70b_i8_pb", dict(B=2, lens=[3000, 1000], max_len=4096), 8, 100),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_multi_query_and_window_match_oracle(case):
    recipe, over, q_len, window = CASES[case]
    w = gen.make(recipe, device=DEV, poison=True, **over)
    q = make_q(w, q_len)
    out = run_ex(w, q, window)
    want, rc = oracle_ex(w, q, window)
    assert rc == 0
    assert_close(out, want, "bf16", "q_len %d window %d" % (q_len, window))


@pytest.mark.parametrize("splits", [1, 3, 29, 1000])
def test_split_invariance_with_window(splits):
    w = gen.make("llama3_8b", device=DEV, B=5, lens=("uniform", 100, 1500), max_len=1536,
                 poison=True)
    q = make_q(w, 3)
    want, _ = oracle_ex(w, q, 150)
    out = run_ex(w, q, 150, num_splits=splits)
    assert_close(out, want, "bf16", "splits %d" % splits)


def test_single_query_no_window_equals_decode():
    w = gen.make("llama3_8b", device=DEV, B=7, lens=("uniform", 1, 900), max_len=1024)
    q = w.q[:, None].contiguous()
    ex = run_ex(w, q, 0)
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool)
    plain = pgd.paged_gqa_decode(pool, w.q, w.block_table, w.seq_lens, w.scale)
    pool.close()
    assert torch.equal(ex[:, 0], plain)


def test_discarded_blocks_before_window_are_not_read():
    """Blocks wholly before every query's window get table entry -1 (a local-
    attention cache may release them): same result, no error."""
    w = gen.make("llama3_8b", device=DEV, B=4, lens=[600, 333, 90, 1000], max_len=1024,
                 poison=True)
    q_len, window = 2, 64
    q = make_q(w, q_len)
    base = run_ex(w, q, window)
    table = w.table_np.copy()
    for b, L in enumerate(w.lens_np):
        lo = max(0, int(L) - q_len - window + 1)
        table[b, :lo // w.block_size] = -1
    out = run_ex(w, q, window, table=torch.from_numpy(table).to(DEV))
    assert torch.equal(out, base)
    want, rc = oracle_ex(w, q, window, table=table)
    assert rc == 0
    assert_close(out, want, "bf16")


def test_short_sequences_give_zero_rows():
    """q_len larger than the sequence: queries before its start attend to
    nothing and return zeros; the rest match the oracle."""
    w = gen.make("llama3_8b", device=DEV, B=3, lens=[2, 1, 9], max_len=64)
    q = make_q(w, 4)
    out = run_ex(w, q, 0)
    assert torch.count_nonzero(out[0, :2]) == 0 and torch.count_nonzero(out[1, :3]) == 0
    want, _ = oracle_ex(w, q, 0)
    assert_close(out, want, "bf16")


def test_f32_rejects_extensions():
    w = gen.make("tiny", device=DEV)
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool)
    with pytest.raises(pgd.PagedGQAError) as e:
        pgd.paged_gqa_decode_ex(pool, w.q[:, None].contiguous(), w.block_table, w.seq_lens,
                                w.scale, window=4)
    assert e.value.status == pgd._lib.PGD_ERR_UNSUPPORTED
    pool.close()


def test_stale_shared_memory_never_reaches_windowed_outputs():
    """Pages wholly before a window are not fetched, so their rows in the stage
    hold whatever an earlier kernel left there; their V rows must be zeroed
    even when a warp's token slice ends before the tile's last valid token
    (several token groups per tile: 8-bit pages at 4 KV heads per unit, and
    MQA).  A decode over an all-NaN pool first leaves NaN in every SM's
    stages."""
    filler = gen.make("llama3_8b", device=DEV, B=64, lens=[4096] * 64, max_len=4096)
    filler.k_pool.fill_(float("nan"))
    filler.v_pool.fill_(float("nan"))
    fp = pgd.PagedKVPool(filler.k_pool, filler.v_pool)
    cases = [("llama3_8b_fp8", dict(B=3, Hq=16, Hkv=4, lens=[90, 300, 17], max_len=320), 2, 64),
             ("mqa_13b_b8", dict(B=2, lens=[300, 77], max_len=512), 1, 20),
             ("llama3_8b", dict(B=3, Hq=16, Hkv=4, lens=[90, 300, 40], max_len=320), 1, 33)]
    try:
        for recipe, over, q_len, window in cases:
            pgd.paged_gqa_decode(fp, filler.q, filler.block_table, filler.seq_lens, 0.1)
            torch.cuda.synchronize()
            w = gen.make(recipe, device=DEV, poison=True, **over)
            q = make_q(w, q_len)
            out = run_ex(w, q, window)
            want, rc = oracle_ex(w, q, window)
            assert rc == 0
            assert_close(out, want, "bf16", "%s after a NaN filler" % recipe)
    finally:
        fp.close()
