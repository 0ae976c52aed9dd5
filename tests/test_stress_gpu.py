"""Many consecutive decode steps on one workspace (GPU only).

The split-merge bookkeeping lives in the workspace: each run's counter must be
back at zero after every call and its flag bit must alternate, or a later call
would merge too early or wait forever.  Each merge variant runs hundreds of
back-to-back steps here; every step's output must equal the first step's, bit
for bit (the decode is deterministic), and no error may be latched.
"""
import pytest
import torch

import gen
import paged_gqa_decode_04_gb300 as pgd

pytestmark = pytest.mark.gpu

# (recipe, overrides, query tokens, window, steps).  The host's merge choice:
# separate run-merge kernel (Llama shape, 32 runs of 4 rows, about 5 spans a
# run), last arriver (8 runs of 4 rows, about 19 pieces each), shared under a
# cooperative launch (70B-like: 2 long runs of 8 rows; 24 runs of 16 rows),
# separate (40 runs of 16 rows, with and without a window)
CASES = [
    ("llama3_8b", dict(B=32, lens=("uniform", 128, 2048), max_len=2048), 1, 0, 600),
    ("llama3_8b", dict(B=8, lens=("uniform", 128, 2048), max_len=2048), 1, 0, 600),
    ("long_70b", dict(B=2, lens=[40000, 25000], max_len=40960), 1, 0, 300),
    ("llama3_8b", dict(B=24, lens=("uniform", 64, 1500), max_len=1536), 4, 0, 400),
    ("llama3_8b", dict(B=40, lens=("uniform", 64, 1500), max_len=1536), 4, 0, 400),
    ("llama3_8b", dict(B=40, lens=("uniform", 64, 1500), max_len=1536), 4, 200, 400),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_back_to_back_steps_on_one_workspace(case):
    recipe, over, q_len, window, steps = CASES[case]
    w = gen.make(recipe, device="cuda", **over)
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool)
    try:
        if q_len == 1 and window == 0:
            q = w.q
            ws = pgd.alloc_workspace(pool, w.B, w.Hq)
            call = lambda out: pgd.paged_gqa_decode(pool, q, w.block_table, w.seq_lens, w.scale,
                                                    out=out, workspace=ws)
        else:
            g = torch.Generator(device="cuda")
            g.manual_seed(31 + case)
            q = torch.randn((w.B, q_len, w.Hq, w.D), generator=g,
                            device="cuda").to(torch.bfloat16)
            ws = torch.zeros(pgd.paged_gqa_workspace_size_ex(pool, w.B, q_len, w.Hq),
                             dtype=torch.uint8, device="cuda")
            call = lambda out: pgd.paged_gqa_decode_ex(pool, q, w.block_table, w.seq_lens,
                                                       w.scale, window=window, out=out,
                                                       workspace=ws)
        first = torch.empty_like(q)
        call(first)
        out = torch.empty_like(q)
        same = torch.ones((), dtype=torch.bool, device="cuda")
        for _ in range(steps):
            call(out)
            same &= (out.view(torch.int16) == first.view(torch.int16)).all()  # stays on the GPU
        assert pgd.paged_gqa_get_error(pool) == 0
        assert bool(same), "a step differed from the first"
        # every run's count is back at zero (flag bits may be set); one counter
        # word per (sequence, KV head) here (at most 16 query rows per head)
        words = ws[:4 * w.B * w.Hkv].view(torch.int32)
        assert int((words & ((1 << 30) - 1)).abs().sum()) == 0
    finally:
        pool.close()
