"""The host's launch plan (paged_gqa_plan), on CPU: head grouping, row tiles,
tile sizes, grid and split-merge choice for every workload shape, and the
statuses a decode returns for shapes it does not take.  The decode entry points
use the same planning function, so this pins the host side of every launch."""
import pytest
import torch

import paged_gqa_decode_04_gb300 as pgd
from paged_gqa_decode_04_gb300 import _lib

BF16, FP8, F32, I8 = torch.bfloat16, torch.float8_e4m3fn, torch.float32, torch.int8


def plan(dtype, hkv, d, B, Hq, **kw):
    return pgd.paged_gqa_plan(dtype, hkv, d, B, Hq, num_sms=152, **kw)


# (name, args, kwargs, expected (head_group, m_tiles, tile_tokens, grid, merge)).
# Merge: shared when a warp's merge would take many loads (long runs); separate
# (a second kernel) when runs cover 2 to 5 spans, fill the SMs and have 4+ rows
# per head; else shared with two or more row tiles per head; otherwise the last
# arriver.  Shared needs the grid resident at once (grid <= SMs).
CASES = [
    ("llama3_8b", (BF16, 8, 128, 64, 32), {}, (8, 1, 16, 152, "separate")),
    ("long_70b", (BF16, 8, 128, 8, 64), {}, (8, 1, 16, 152, "shared (cooperative)")),
    ("mha_13b_b1", (BF16, 40, 128, 1, 40), {}, (8, 1, 16, 152, "last arriver")),
    ("mqa_13b_b1", (BF16, 1, 128, 1, 40), {}, (1, 3, 128, 152, "shared (cooperative)")),
    ("mqa_13b_b8", (BF16, 1, 128, 8, 40), {}, (1, 3, 128, 152, "shared (cooperative)")),
    ("sweep B 256", (BF16, 8, 128, 256, 32), {}, (8, 1, 16, 152, "last arriver")),
    # the separate merge's edges: 152 spans over 32 runs (4.75 a run) separate,
    # over 96 runs (1.6) last arriver; 4 tokens at B 16 (9.5) shared; MHA B 8
    # (one row per head) last arriver
    ("B 32", (BF16, 8, 128, 32, 32), {}, (8, 1, 16, 152, "separate")),
    ("B 96", (BF16, 8, 128, 96, 32), {}, (8, 1, 16, 152, "last arriver")),
    ("4 query tokens, B 16", (BF16, 8, 128, 16, 32), dict(q_len=4),
     (8, 1, 16, 152, "shared (cooperative)")),
    ("mha_13b_b8", (BF16, 40, 128, 8, 40), {}, (8, 1, 16, 152, "last arriver")),
    # the separate merge's conditions at their edges: 2 runs <= P (76 runs yes,
    # 77 no), P <= 5 runs (31 yes, 30 no), runs x head group >= SMs (Hkv 2: 40
    # runs x 2 no, 76 x 2 yes), at least 4 rows per head (G 2 no)
    ("B 76", (BF16, 8, 128, 76, 32), {}, (8, 1, 16, 152, "separate")),
    ("B 77", (BF16, 8, 128, 77, 32), {}, (8, 1, 16, 152, "last arriver")),
    ("B 31", (BF16, 8, 128, 31, 32), {}, (8, 1, 16, 152, "separate")),
    ("B 30", (BF16, 8, 128, 30, 32), {}, (8, 1, 16, 152, "last arriver")),
    ("Hkv 2, B 40", (BF16, 2, 128, 40, 8), {}, (2, 1, 64, 152, "last arriver")),
    ("Hkv 2, B 76", (BF16, 2, 128, 76, 8), {}, (2, 1, 64, 152, "separate")),
    ("G 2, B 64", (BF16, 8, 128, 64, 16), {}, (8, 1, 16, 152, "last arriver")),
    ("4 query tokens, B 64", (BF16, 8, 128, 64, 32), dict(q_len=4), (8, 1, 16, 152, "separate")),
    ("4 query tokens, B 24", (BF16, 8, 128, 24, 32), dict(q_len=4),
     (8, 1, 16, 152, "shared (cooperative)")),
    # 32 / 64 rows per head (two / four row tiles): 128 / 256 runs over 152
    # spans, too short for the separate merge; with several row tiles per head
    # the shared merge beats the last arriver
    ("8 query rows x 4 tokens", (BF16, 8, 128, 64, 64), dict(q_len=4),
     (4, 2, 32, 152, "shared (cooperative)")),
    ("64 query rows", (BF16, 8, 128, 64, 128), dict(q_len=4), (2, 4, 64, 152, "shared (cooperative)")),
    ("32 rows, B 8", (BF16, 8, 128, 8, 64), dict(q_len=4), (4, 2, 32, 152, "shared (cooperative)")),
    ("8-bit llama3", (FP8, 8, 128, 64, 32), {}, (8, 1, 32, 152, "separate")),
    ("8-bit long_70b", (FP8, 8, 128, 8, 64), {}, (8, 1, 32, 152, "shared (cooperative)")),
    ("int8 llama3", (I8, 8, 128, 64, 32), {}, (8, 1, 32, 152, "separate")),
    ("int8 long_70b", (I8, 8, 128, 8, 64), {}, (8, 1, 32, 152, "shared (cooperative)")),
    ("int8 4 query tokens", (I8, 8, 128, 64, 32), dict(q_len=4), (8, 1, 32, 152, "separate")),
    ("head_dim 64", (BF16, 2, 64, 4, 8), {}, (2, 1, 64, 152, "last arriver")),
    ("Hkv 6", (BF16, 6, 128, 4, 24), {}, (2, 1, 64, 152, "last arriver")),
    ("float32 tiny", (F32, 2, 64, 4, 8), {}, (1, 1, 64, 152, "merge kernel")),
    # 500 spans over 64 runs: about 8 spans a run, past the separate merge
    ("explicit splits", (BF16, 8, 128, 64, 32), dict(num_splits=500),
     (8, 1, 16, 500, "last arriver")),
    # the shared merge needs its grid resident at once (one CTA per SM): a
    # split count above the SM count takes the last arriver instead
    ("long_70b, 152 splits", (BF16, 8, 128, 8, 64), dict(num_splits=152),
     (8, 1, 16, 152, "shared (cooperative)")),
    ("long_70b, 153 splits", (BF16, 8, 128, 8, 64), dict(num_splits=153),
     (8, 1, 16, 153, "last arriver")),
    ("mqa B 1, 1000 splits", (BF16, 1, 128, 1, 40), dict(num_splits=1000),
     (1, 3, 128, 1000, "last arriver")),
]


@pytest.mark.parametrize("name,args,kw,want", CASES, ids=[c[0] for c in CASES])
def test_plan_of_each_shape(name, args, kw, want):
    p = plan(*args, **kw)
    assert (p["head_group"], p["m_tiles"], p["tile_tokens"], p["grid"], p["merge"]) == want


def test_plan_invariants():
    for dtype in (BF16, FP8, I8):
        for hkv in (1, 2, 3, 4, 5, 6, 8, 40):
            for G in (1, 2, 4, 8, 16, 40, 64):
                for q_len in (1, 2, 4):
                    if q_len * G > 64:
                        continue
                    p = plan(dtype, hkv, 128, 16, hkv * G, q_len=q_len)
                    hg, mt, T = p["head_group"], p["m_tiles"], p["tile_tokens"]
                    assert hkv % hg == 0 and hg in (1, 2, 4, 8)
                    assert mt == (q_len * G + 15) // 16
                    assert hg * mt <= 8                       # at most 8 consumer warps
                    assert T * hg == (128 if dtype == BF16 else 256)  # 64 KB stages


@pytest.mark.parametrize("args,kw,status", [
    ((BF16, 8, 128, 4, 30), {}, _lib.PGD_ERR_SHAPE),             # Hq % Hkv
    ((BF16, 1, 128, 4, 65), {}, _lib.PGD_ERR_SHAPE),             # 65 rows per head
    ((BF16, 8, 128, 4, 32), dict(q_len=17), _lib.PGD_ERR_SHAPE),  # 68 rows per head
    ((BF16, 8, 96, 4, 32), {}, _lib.PGD_ERR_SHAPE),              # head_dim 96
    ((FP8, 8, 64, 4, 32), {}, _lib.PGD_ERR_SHAPE),               # 8-bit pages: head_dim 128
    ((I8, 8, 64, 4, 32), {}, _lib.PGD_ERR_SHAPE),
    ((F32, 2, 64, 4, 8), dict(q_len=2), _lib.PGD_ERR_UNSUPPORTED),
    ((F32, 2, 64, 4, 8), dict(window=16), _lib.PGD_ERR_UNSUPPORTED),
    ((BF16, 8, 128, -1, 32), {}, _lib.PGD_ERR_ARG),
    ((BF16, 8, 128, 4, 32), dict(num_splits=-1), _lib.PGD_ERR_ARG),
])
def test_plan_rejects_what_the_decode_rejects(args, kw, status):
    with pytest.raises(pgd.PagedGQAError) as e:
        plan(*args, **kw)
    assert e.value.status == status


def test_plan_null_output_and_bad_dtype():
    lib = _lib.load()
    assert lib.paged_gqa_plan(1, 8, 128, 152, 4, 1, 32, 0, 0, None) == _lib.PGD_ERR_ARG
    import ctypes
    out = (ctypes.c_int * 5)()
    assert lib.paged_gqa_plan(7, 8, 128, 152, 4, 1, 32, 0, 0, out) == _lib.PGD_ERR_DTYPE
