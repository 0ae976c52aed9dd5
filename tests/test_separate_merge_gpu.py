"""The separate merge (decode pieces write partials, a second kernel merges
them) on its less common paths, against the float64 oracle (GPU only):

  * more spans than tiles (an explicit split count above the call's tiles):
    each span holds at most one tile and the pieces of a run are the owners of
    its tiles, found by the span arithmetic instead of as consecutive CTAs;
  * runs of more than four pieces (more spans per run), merged in several
    batches of loads;
  * several query tokens with a window, and 8-bit pages with a scale per block.

Each case first checks, from the host plan, that the call does take the
separate merge, and that two calls give the same bits."""
import pytest
import torch

import gen
import paged_gqa_decode_04_gb300 as pgd
from gpu_cases import assert_close, run_oracle

pytestmark = pytest.mark.gpu

# (name, recipe, overrides, q_len, window, num_splits)
CASES = [
    # 32 runs of 1 to 3 tiles, 100 spans: more spans than tiles
    ("sparse", "llama3_8b", dict(B=32, lens=("uniform", 1, 40), max_len=64), 1, 0, 100),
    # 32 runs over 160 spans: 5 spans a run, up to 7 pieces
    ("many_pieces", "llama3_8b", dict(B=32, lens=("uniform", 1500, 2048), max_len=2048), 1, 0, 160),
    ("window_q3", "llama3_8b", dict(B=40, lens=("uniform", 200, 1500), max_len=1536), 3, 100, 0),
    ("fp8_per_block", "llama3_8b_fp8_pb", dict(B=32, lens=("uniform", 128, 2048), max_len=2048),
     1, 0, 0),
    ("int8_q4", "llama3_8b_i8", dict(B=32, lens=("uniform", 64, 1500), max_len=1536), 4, 0, 0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_separate_merge_matches_oracle(case):
    _, recipe, over, q_len, window, num_splits = case
    w = gen.make(recipe, device="cuda", poison=True, **over)
    plan = pgd.paged_gqa_plan(w.k_pool.dtype, w.Hkv, w.D, w.B, w.Hq, q_len=q_len,
                              num_splits=num_splits, window=window)
    assert plan["merge"] == "separate", plan
    ex = q_len > 1 or window > 0
    if ex:
        g = torch.Generator(device="cuda")
        g.manual_seed(23)
        q = torch.randn((w.B, q_len, w.Hq, w.D), generator=g, device="cuda").to(torch.bfloat16)
    else:
        q = w.q
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool, w.k_scale, w.v_scale)
    try:
        outs = []
        for _ in range(2):
            if ex:
                outs.append(pgd.paged_gqa_decode_ex(pool, q, w.block_table, w.seq_lens, w.scale,
                                                    window=window, num_splits=num_splits))
            else:
                outs.append(pgd.paged_gqa_decode(pool, q, w.block_table, w.seq_lens, w.scale,
                                                 num_splits=num_splits))
        st = pgd.paged_gqa_get_error(pool)
    finally:
        pool.close()
    assert st == 0, pgd.strerror(st)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    want, rc = run_oracle(w, q=q if ex else None, window=window if ex else None)
    assert rc == 0
    assert_close(outs[0], want, w.dtype, "separate merge, %s" % case[0])
