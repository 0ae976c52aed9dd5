"""The device's split plan, read back from the workspace after a decode.

The span scan every decode CTA runs (csrc/partition.cuh, find_span_start)
leaves in the workspace the first slot of each sequence in the virtual tile
sequence the spans cut, the total, and then the spans in use and the run cost
(CTA 0 writes them; the run-merge kernel reads the last two).  This reads that
table after real decodes and compares it with the rules written out here:

  * tiles per KV-head unit of a sequence: ceil(L / T) minus the whole tiles
    before the earliest position any of its q_len queries sees (window), none
    for L = 0 or L beyond the table;
  * units per sequence: Hkv / head group of the launch plan;
  * spans in use: the grid, or with automatic splits at most one per two
    tiles of work (at least one);
  * run cost: 3 virtual slots before each run once spans average 8 or more
    real tiles, none otherwise, and none on the float32 path.

So the CUDA scan itself is checked, not only a host restatement of it
(tests/test_partition_model.py checks the properties of the cut on CPU).
Workspace layout (the library's own, csrc/api.cpp): one counter word per
(sequence, KV head, row tile), rounded up to 256 bytes, then the B + 3 int64
entries of this table.
"""
import numpy as np
import pytest
import torch

import gen
import paged_gqa_decode_04_gb300 as pgd

pytestmark = pytest.mark.gpu

MIN_TILES_PER_CTA = 2
RUN_COST_TILES = 3
RUN_COST_MIN_TILES = 8


def tiles_of(L, max_blocks, bs, T, q_len, window):
    if L <= 0 or L > max_blocks * bs:
        return 0
    first = 0
    if window > 0:
        lo = L - q_len - window + 1
        first = lo // T if lo > 0 else 0
    return -(-L // T) - first


def expected_table(lens, max_blocks, bs, T, q_len, window, units, parts, auto, run_cost):
    n = [tiles_of(int(L), max_blocks, bs, T, q_len, window) for L in lens]
    real = units * sum(n)
    p = parts
    if auto:
        p = max(1, min(parts, -(-real // MIN_TILES_PER_CTA)))
    W = run_cost if real >= RUN_COST_MIN_TILES * p else 0
    v = [units * (x + W) if x > 0 else 0 for x in n]
    return np.concatenate([[0], np.cumsum(v), [p, W]]).astype(np.int64), W


# (recipe, overrides, q_len, window, num_splits)
CASES = [
    ("llama3_8b", {}, 1, 0, 0),                                     # run cost on
    ("llama3_8b", dict(B=40, lens=("uniform", 0, 4096)), 1, 0, 500),  # explicit splits, zeros
    ("llama3_8b", dict(B=24), 4, 512, 0),                           # several queries, window
    ("llama3_8b_fp8", dict(B=32), 1, 0, 0),                         # 8-bit pages: 32-token tiles
    ("llama3_8b", dict(B=3, lens=[5, 0, 40], max_len=64), 1, 0, 0),  # few tiles: no run cost
    ("mqa_13b_b8", {}, 1, 0, 0),                                    # one KV head, 3 row tiles
    ("long_70b", dict(B=4, lens=("uniform", 1000, 40000), max_len=40960), 1, 4096, 0),
    ("tiny", {}, 1, 0, 0),                                          # float32: no run cost
]


@pytest.mark.parametrize("recipe,over,q_len,window,num_splits", CASES,
                         ids=["%s-q%d-w%d-s%d" % (c[0], c[2], c[3], c[4]) for c in CASES])
def test_device_tile_table_matches_rules(recipe, over, q_len, window, num_splits):
    w = gen.make(recipe, device="cuda", **over)
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool, w.k_scale, w.v_scale)
    try:
        plan = pgd.paged_gqa_plan(w.k_pool.dtype, w.Hkv, w.D, w.B, w.Hq, q_len=q_len,
                                  num_splits=num_splits, window=window)
        if q_len == 1 and window == 0:
            q = w.q
            ws = pgd.alloc_workspace(pool, w.B, w.Hq, num_splits)
            pgd.paged_gqa_decode(pool, q, w.block_table, w.seq_lens, w.scale, workspace=ws,
                                 num_splits=num_splits)
        else:
            g = torch.Generator(device="cuda")
            g.manual_seed(w.seed + 11)
            q = torch.randn((w.B, q_len, w.Hq, w.D), generator=g, device="cuda").to(torch.bfloat16)
            nbytes = pgd.paged_gqa_workspace_size_ex(pool, w.B, q_len, w.Hq, num_splits)
            ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda")
            pgd.paged_gqa_decode_ex(pool, q, w.block_table, w.seq_lens, w.scale, window=window,
                                    workspace=ws, num_splits=num_splits)
        assert pgd.paged_gqa_get_error(pool) == 0
    finally:
        pool.close()
    torch.cuda.synchronize()

    f32 = w.dtype == "f32"
    rows = q_len * (w.Hq // w.Hkv)
    mtiles = -(-rows // 16)
    off = -(-(w.B * w.Hkv * mtiles * 4) // 256) * 256
    got = ws[off:off + 8 * (w.B + 3)].cpu().view(torch.int64).numpy()
    units = w.Hkv // plan["head_group"]
    want, W = expected_table(w.lens_np, w.max_blocks, w.block_size, plan["tile_tokens"],
                             1 if f32 else q_len, 0 if f32 else window, units, plan["grid"],
                             num_splits == 0 and not f32, 0 if f32 else RUN_COST_TILES)
    assert np.array_equal(got, want), (
        "device table differs (run cost %d): first at %d: %s vs %s" %
        ((W,) + ((int(np.argmax(got != want)), got[got != want][:4], want[got != want][:4])
                 if got.shape == want.shape else (-1, got.shape, want.shape))))
    # the cases above are chosen so that both run-cost regimes are met
    if recipe == "llama3_8b" and not over:
        assert W == RUN_COST_TILES
    if over.get("lens") == [5, 0, 40]:
        assert W == 0
