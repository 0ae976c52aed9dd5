"""Every workload at its full size, in the launch configuration the benchmark
times (automatic split count), checked row by row against the float64 oracle
(GPU only).  The oracle passes over a whole Llama-3-8B-shaped batch in well
under a second on the host cores, so every output row is compared."""
import pytest

import gen
from gpu_cases import assert_close, run_cuda, run_oracle

pytestmark = pytest.mark.gpu

FULL = ["llama3_8b", "long_70b", "mha_13b_b1", "mha_13b_b8", "mqa_13b_b1", "mqa_13b_b8",
        "sweep_bs8", "sweep_bs16", "sweep_bs32", "sweep_bs64", "sweep_bs128"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_row(name):
    w = gen.make(name, device="cuda", poison=True)
    out, _ = run_cuda(w)
    want, rc = run_oracle(w)
    assert rc == 0
    assert_close(out, want, w.dtype, name)
    del w, out


# 8-bit pages at full size: e4m3 and int8 codes, scales per KV head and per
# block and KV head.
@pytest.mark.parametrize("name", ["llama3_8b_fp8", "long_70b_fp8", "llama3_8b_i8", "long_70b_i8",
                                  "llama3_8b_fp8_pb", "long_70b_fp8_pb", "llama3_8b_i8_pb",
                                  "long_70b_i8_pb"])
def test_full_size_8bit_every_row(name):
    w = gen.make(name, device="cuda", poison=True)
    out, _ = run_cuda(w)
    want, rc = run_oracle(w)
    assert rc == 0
    assert_close(out, want, w.dtype, name)
    del w, out


# Several query tokens and windows at full size, as `bench.py --op decode_ex`
# runs them (its query draw: a device generator seeded with seed + 7).
EX_FULL = [("llama3_8b", 4, 0), ("llama3_8b", 4, 512), ("llama3_8b", 1, 1024),
           ("long_70b", 1, 4096), ("llama3_8b_fp8", 4, 0), ("llama3_8b_i8_pb", 4, 0),
           ("llama3_8b_fp8_pb", 2, 512)]


@pytest.mark.parametrize("name,q_len,window", EX_FULL)
def test_full_size_multi_token_and_window(name, q_len, window):
    import torch

    import paged_gqa_decode_04_gb300 as pgd

    w = gen.make(name, device="cuda", poison=True)
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed + 7)
    q = torch.randn((w.B, q_len, w.Hq, w.D), generator=g, device="cuda").to(torch.bfloat16)
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool, w.k_scale, w.v_scale)
    try:
        out = pgd.paged_gqa_decode_ex(pool, q, w.block_table, w.seq_lens, w.scale,
                                      window=window)
        st = pgd.paged_gqa_get_error(pool)
    finally:
        pool.close()
    assert st == 0, pgd.strerror(st)
    want, rc = run_oracle(w, q=q, window=window)
    assert rc == 0
    assert_close(out, want, w.dtype, "%s q_len %d window %d" % (name, q_len, window))
    del w, out, q
