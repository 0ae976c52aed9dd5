"""The shared split merge (every piece's warp merges a share of a long run's
rows, under a cooperative launch) against the float64 oracle (GPU only):
automatic and explicit split counts, one span per tile, a grid too large to be
resident at once (the last-arriver merge instead), and one workspace reused
across calls that share and calls that do not."""
import pytest
import torch

import gen
import paged_gqa_decode_04_gb300 as pgd
from gpu_cases import assert_close, run_oracle

pytestmark = pytest.mark.gpu

# 40 query heads on one KV head, two long sequences: 16-row merges of many pieces
MQA = dict(B=2, lens=[4096, 3000], max_len=4096)


def _decode(w, num_splits=0, workspace=None):
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool, w.k_scale, w.v_scale)
    try:
        out = pgd.paged_gqa_decode(pool, w.q, w.block_table, w.seq_lens, w.scale,
                                   num_splits=num_splits, workspace=workspace)
        st = pgd.paged_gqa_get_error(pool)
    finally:
        pool.close()
    assert st == 0, pgd.strerror(st)
    return out


@pytest.mark.parametrize("splits", [0, 16, 64, 152, 500])
def test_shared_merge_matches_oracle(splits):
    # 0 / 16 / 64: several tiles per span; 152: one tile per span (more spans
    # than tiles); 500: more CTAs than can be resident, last-arriver merge
    w = gen.make("mqa_13b_b1", device="cuda", poison=True, **MQA)
    want, rc = run_oracle(w)
    assert rc == 0
    assert_close(_decode(w, splits), want, w.dtype, "splits %d" % splits)


def test_long_runs_70b_shape_share():
    w = gen.make("long_70b", device="cuda", poison=True, B=2, lens=[40000, 23000],
                 max_len=40960)
    want, rc = run_oracle(w)
    assert rc == 0
    assert_close(_decode(w), want, w.dtype, "70B shape, 2 sequences")


def test_one_workspace_shared_and_last_arriver_calls():
    # the run counter words carry a flag bit after a shared call; a later call
    # of another shape over the same words must still count from zero
    a = gen.make("mqa_13b_b1", device="cuda", poison=True, **MQA)
    b = gen.make("llama3_8b", device="cuda", poison=True, B=6, lens=("uniform", 300, 2000),
                 max_len=2048)
    pa = pgd.PagedKVPool(a.k_pool, a.v_pool)
    pb = pgd.PagedKVPool(b.k_pool, b.v_pool)
    try:
        nbytes = max(pgd.paged_gqa_workspace_size(pa, a.B, a.Hq, 0),
                     pgd.paged_gqa_workspace_size(pb, b.B, b.Hq, 0))
    finally:
        pa.close()
        pb.close()
    ws = torch.zeros(nbytes + 256, dtype=torch.uint8, device="cuda")
    want_a, _ = run_oracle(a)
    want_b, _ = run_oracle(b)
    for w, want in ((a, want_a), (b, want_b), (a, want_a), (a, want_a), (b, want_b)):
        assert_close(_decode(w, workspace=ws), want, w.dtype, w.name)
