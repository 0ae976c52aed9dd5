"""CUDA path against the float64 oracle, element by element (GPU only).

Small versions of every workload shape (each spanning several tiles, CTAs and a
ragged tail), split-count invariance, poisoned pools, the degenerate cases the
method has, and device-side error reporting.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import paged_gqa_decode_04_gb300 as pgd
from gpu_cases import assert_close, errors, host, run_cuda, run_oracle, tol

pytestmark = pytest.mark.gpu
DEV = "cuda"

SMALL = {
    # name: (recipe, overrides)
    "tiny_f32": ("tiny", {}),
    "llama3_8b_small": ("llama3_8b", dict(B=8, lens=("uniform", 1, 700), max_len=1024)),
    "mha_13b_small": ("mha_13b_b8", dict(B=2, lens=[333, 64], max_len=512)),
    "mqa_13b_small": ("mqa_13b_b8", dict(B=2, lens=[517, 1], max_len=1024)),
    "long_70b_small": ("long_70b", dict(B=2, lens=("uniform", 2000, 4100), max_len=4224)),
    "sweep_bs8": ("sweep_bs8", dict(B=12, lens=("lognormal", 200.0, 1.0, 1, 900), max_len=1024)),
    "sweep_bs16": ("sweep_bs16", dict(B=12, lens=("lognormal", 200.0, 1.0, 1, 900),
                                      max_len=1024)),
    "sweep_bs32": ("sweep_bs32", dict(B=12, lens=("lognormal", 200.0, 1.0, 1, 900),
                                      max_len=1024)),
    "sweep_bs64": ("sweep_bs64", dict(B=12, lens=("lognormal", 200.0, 1.0, 1, 900),
                                      max_len=1024)),
    "sweep_bs128": ("sweep_bs128", dict(B=12, lens=("lognormal", 200.0, 1.0, 1, 900),
                                        max_len=1024)),
    "d64_bf16": ("llama3_8b", dict(B=5, D=64, lens=[1, 65, 130, 64, 300], max_len=320)),
    "group16": ("llama3_8b", dict(B=3, Hq=32, Hkv=2, lens=[90, 200, 17], max_len=256)),
    "group24": ("llama3_8b", dict(B=3, Hq=48, Hkv=2, lens=[90, 200, 17], max_len=256)),
    "group64": ("llama3_8b", dict(B=2, Hq=64, Hkv=1, lens=[150, 9], max_len=256)),
    "bs256": ("llama3_8b", dict(B=3, block_size=256, lens=[700, 256, 3], max_len=768)),
    # head-group sizes 4 and 2 with several units per sequence, and head_dim 64
    "hkv4": ("llama3_8b", dict(B=5, Hq=16, Hkv=4, lens=[1, 65, 130, 64, 300], max_len=320)),
    "hkv4_g16": ("llama3_8b", dict(B=3, Hq=64, Hkv=4, lens=[90, 200, 17], max_len=256)),
    "hkv6": ("llama3_8b", dict(B=3, Hq=24, Hkv=6, lens=[90, 200, 17], max_len=256)),
    "hkv12": ("llama3_8b", dict(B=3, Hq=48, Hkv=12, lens=[300, 20, 150], max_len=320)),
    "d64_hkv4": ("llama3_8b", dict(B=3, D=64, Hq=16, Hkv=4, lens=[70, 200, 5], max_len=256)),
    # 8-bit (e4m3) pages with per-head scales, bfloat16 q and out
    "fp8_llama3_small": ("llama3_8b_fp8", dict(B=8, lens=("uniform", 1, 700), max_len=1024)),
    "fp8_long_small": ("long_70b_fp8", dict(B=2, lens=("uniform", 2000, 4100), max_len=4224)),
    "fp8_mha": ("llama3_8b_fp8", dict(B=2, Hq=40, Hkv=40, lens=[333, 64], max_len=512)),
    "fp8_mqa": ("llama3_8b_fp8", dict(B=2, Hq=40, Hkv=1, lens=[517, 1], max_len=1024)),
    "fp8_bs8": ("llama3_8b_fp8", dict(B=12, block_size=8, lens=("lognormal", 200.0, 1.0, 1, 900),
                                      max_len=1024)),
    "fp8_bs128": ("llama3_8b_fp8", dict(B=12, block_size=128,
                                        lens=("lognormal", 200.0, 1.0, 1, 900), max_len=1024)),
    "fp8_hkv4": ("llama3_8b_fp8", dict(B=5, Hq=16, Hkv=4, lens=[1, 65, 130, 64, 300],
                                       max_len=320)),
    "fp8_hkv2_g16": ("llama3_8b_fp8", dict(B=3, Hq=32, Hkv=2, lens=[90, 200, 17], max_len=256)),
    "fp8_hkv6": ("llama3_8b_fp8", dict(B=3, Hq=24, Hkv=6, lens=[90, 300, 17], max_len=320)),
    "fp8_bs256": ("llama3_8b_fp8", dict(B=3, block_size=256, lens=[700, 256, 3], max_len=768)),
    # an odd KV head count (one head per unit) with an odd group
    "hkv5_g3": ("llama3_8b", dict(B=4, Hq=15, Hkv=5, lens=[333, 1, 48, 97], max_len=384)),
    # lengths on and next to tile and block boundaries (16-token tiles and blocks)
    "tile_edges": ("llama3_8b", dict(B=8, lens=[15, 16, 17, 31, 32, 33, 127, 128], max_len=160)),
    "fp8_tile_edges": ("llama3_8b_fp8", dict(B=8, lens=[31, 32, 33, 63, 64, 65, 255, 256],
                                             max_len=288)),
    # int8 pages (per-head scales) and 8-bit pages with a scale per block and
    # KV head (e4m3 and int8): tiles of 32 tokens span 2-4 blocks of 8-16
    # tokens, each with its own scale
    "i8_llama3_small": ("llama3_8b_i8", dict(B=8, lens=("uniform", 1, 700), max_len=1024)),
    "i8_long_small": ("long_70b_i8", dict(B=2, lens=("uniform", 2000, 4100), max_len=4224)),
    "i8_mqa": ("llama3_8b_i8", dict(B=2, Hq=40, Hkv=1, lens=[517, 1], max_len=1024)),
    "i8_hkv6": ("llama3_8b_i8", dict(B=3, Hq=24, Hkv=6, lens=[90, 300, 17], max_len=320)),
    "fp8pb_llama3_small": ("llama3_8b_fp8_pb", dict(B=8, lens=("uniform", 1, 700),
                                                    max_len=1024)),
    "fp8pb_long_small": ("long_70b_fp8_pb", dict(B=2, lens=("uniform", 2000, 4100),
                                                 max_len=4224)),
    "fp8pb_bs8": ("llama3_8b_fp8_pb", dict(B=12, block_size=8,
                                           lens=("lognormal", 200.0, 1.0, 1, 900), max_len=1024)),
    "fp8pb_bs256": ("llama3_8b_fp8_pb", dict(B=3, block_size=256, lens=[700, 256, 3],
                                             max_len=768)),
    "fp8pb_mha": ("llama3_8b_fp8_pb", dict(B=2, Hq=40, Hkv=40, lens=[333, 64], max_len=512)),
    "fp8pb_mqa": ("llama3_8b_fp8_pb", dict(B=2, Hq=40, Hkv=1, lens=[517, 1], max_len=1024)),
    "fp8pb_hkv2_g16": ("llama3_8b_fp8_pb", dict(B=3, Hq=32, Hkv=2, lens=[90, 200, 17],
                                                max_len=256)),
    "i8pb_llama3_small": ("llama3_8b_i8_pb", dict(B=8, lens=("uniform", 1, 700), max_len=1024)),
    "i8pb_long_small": ("long_70b_i8_pb", dict(B=2, lens=("uniform", 2000, 4100),
                                               max_len=4224)),
    "i8pb_bs8": ("llama3_8b_i8_pb", dict(B=12, block_size=8,
                                         lens=("lognormal", 200.0, 1.0, 1, 900), max_len=1024)),
    "i8pb_hkv4": ("llama3_8b_i8_pb", dict(B=5, Hq=16, Hkv=4, lens=[1, 65, 130, 64, 300],
                                          max_len=320)),
    "i8pb_mqa": ("llama3_8b_i8_pb", dict(B=2, Hq=40, Hkv=1, lens=[517, 1], max_len=1024)),
    "i8pb_tile_edges": ("llama3_8b_i8_pb", dict(B=8, lens=[31, 32, 33, 63, 64, 65, 255, 256],
                                                max_len=288)),
}


@pytest.mark.parametrize("case", sorted(SMALL))
def test_small_configs_match_oracle(case):
    recipe, over = SMALL[case]
    w = gen.make(recipe, device=DEV, poison=True, **over)
    out, _ = run_cuda(w)
    want, rc = run_oracle(w)
    assert rc == 0
    assert_close(out, want, w.dtype, case)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64, 152, 1000])
def test_split_count_invariance(splits):
    w = gen.make("llama3_8b", device=DEV, B=6, lens=("uniform", 1, 2000), max_len=2048,
                 poison=True)
    want, _ = run_oracle(w)
    out, _ = run_cuda(w, num_splits=splits)
    assert_close(out, want, "bf16", "splits=%d" % splits)
    ref, _ = run_cuda(w, num_splits=0)
    d = (out.float() - ref.float()).abs().max().item()
    assert d <= 2 * tol("bf16")[0]


def test_f32_split_invariance():
    w = gen.make("tiny", device=DEV)
    want, _ = run_oracle(w)
    for splits in (1, 2, 3, 5, 16, 500):
        out, _ = run_cuda(w, num_splits=splits)
        assert_close(out, want, "f32", "splits=%d" % splits)


def test_poison_never_leaks():
    """NaN in every unused block and every tail slot: output finite and equal
    to the unpoisoned run."""
    over = dict(B=10, lens=("uniform", 1, 500), max_len=512)
    clean = gen.make("llama3_8b", device=DEV, poison=False, **over)
    dirty = gen.make("llama3_8b", device=DEV, poison=True, **over)
    a, _ = run_cuda(clean)
    b, _ = run_cuda(dirty)
    assert torch.isfinite(b.float()).all()
    assert torch.equal(a, b)


def test_zero_and_one_length():
    w = gen.make("llama3_8b", device=DEV, B=4, lens=[0, 1, 0, 37], max_len=64, poison=True)
    out, _ = run_cuda(w)
    assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[2]) == 0
    # length one: the output is the V row of the KV head, exactly (bf16 in, bf16 out)
    G = w.G
    blk = int(w.table_np[1, 0])
    v_rows = w.v_pool[blk, 0]                       # [Hkv, D]
    assert torch.equal(out[1], v_rows.repeat_interleave(G, dim=0))
    want, _ = run_oracle(w)
    assert_close(out, want, "bf16")


def test_all_empty_batch():
    w = gen.make("llama3_8b", device=DEV, B=3, lens=[0, 0, 0], max_len=64, num_blocks=4)
    out, _ = run_cuda(w)
    assert torch.count_nonzero(out) == 0


def test_single_token_everywhere_mqa_mha():
    for Hkv in (1, 40):
        w = gen.make("mha_13b_b1", device=DEV, B=3, Hkv=Hkv, lens=[1, 1, 1], max_len=16)
        out, _ = run_cuda(w)
        want, _ = run_oracle(w)
        g, emax, _ = errors(out, want)
        assert emax == 0.0


def test_prefix_sharing_aliases():
    """Two sequences pointing at the same physical blocks with the same query."""
    w = gen.make("llama3_8b", device=DEV, B=4, lens=[300, 300, 120, 50], max_len=320)
    w.block_table[1] = w.block_table[0]
    w.q[1] = w.q[0]
    w.table_np[1] = w.table_np[0]
    for splits in (1, 0):
        out, _ = run_cuda(w, num_splits=splits)
        if splits == 1:
            assert torch.equal(out[0], out[1])
        want, _ = run_oracle(w)
        assert_close(out, want, "bf16")


def test_deterministic_repeat():
    w = gen.make("llama3_8b", device=DEV, B=8, lens=("uniform", 1, 900), max_len=1024)
    a, _ = run_cuda(w)
    b, _ = run_cuda(w)
    assert torch.equal(a, b)


def test_side_stream():
    w = gen.make("llama3_8b", device=DEV, B=5, lens=("uniform", 50, 400), max_len=512)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out, _ = run_cuda(w, stream=s)
    s.synchronize()
    want, _ = run_oracle(w)
    assert_close(out, want, "bf16")


def test_bad_block_id_latches_and_poisons_only_that_sequence():
    for dt in ("bf16", "f32"):
        rec = "llama3_8b" if dt == "bf16" else "tiny"
        w = gen.make(rec, device=DEV, B=4, lens=[100, 40, 70, 33], max_len=128,
                     Hq=8, Hkv=2, D=64, dtype=dt, num_blocks=None)
        w.block_table[2, 1] = w.num_blocks + 5
        out, status = run_cuda(w, check_error=False)
        assert status == pgd._lib.PGD_ERR_BLOCK_ID
        assert torch.isnan(out[2].float()).all()
        want, _ = run_oracle(w)
        for b in (0, 1, 3):
            assert_close(out[b], want[b], dt, "seq %d" % b)


def test_bad_seq_len_latches():
    w = gen.make("llama3_8b", device=DEV, B=3, lens=[100, 40, 70], max_len=128)
    w.seq_lens[1] = 128 + 1
    out, status = run_cuda(w, check_error=False)
    assert status == pgd._lib.PGD_ERR_SEQ_LEN
    assert torch.isnan(out[1].float()).all()
    w.seq_lens[1] = -3
    out, status = run_cuda(w, check_error=False)
    assert status == pgd._lib.PGD_ERR_SEQ_LEN
    want, _ = run_oracle(w, lens=np.array([100, 40, 70], np.int32))
    assert_close(out[0], want[0], "bf16")
    assert_close(out[2], want[2], "bf16")


def test_argument_errors_raise():
    w = gen.make("llama3_8b", device=DEV, B=2, lens=[10, 20], max_len=32)
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool)
    with pytest.raises(pgd.PagedGQAError) as e:
        pgd.paged_gqa_decode(pool, w.q[:, :30].contiguous(), w.block_table, w.seq_lens, w.scale)
    assert e.value.status == pgd._lib.PGD_ERR_SHAPE
    ws = torch.empty(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(pgd.PagedGQAError) as e:
        pgd.paged_gqa_decode(pool, w.q, w.block_table, w.seq_lens, w.scale, workspace=ws)
    assert e.value.status == pgd._lib.PGD_ERR_WORKSPACE
    with pytest.raises(pgd.PagedGQAError) as e:
        pgd.paged_gqa_decode(pool, w.q, w.block_table, w.seq_lens, w.scale, out=w.q)
    assert e.value.status == pgd._lib.PGD_ERR_ARG
    pool.close()


def test_workspace_size_scales_with_splits():
    w = gen.make("llama3_8b", device=DEV, B=2, lens=[10, 20], max_len=32)
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool)
    a = pgd.paged_gqa_workspace_size(pool, 64, 32, 1)
    b = pgd.paged_gqa_workspace_size(pool, 64, 32, 1000)
    assert b > a
    assert pgd.paged_gqa_auto_splits(pool) == torch.cuda.get_device_properties(0).multi_processor_count
    pool.close()


def test_golden_fixture_on_gpu():
    """The stored oracle answer (tests/golden/oracle_small.json) reproduced by
    the float32 CUDA path."""
    from test_golden import load_small

    q, k, v, t, L, scale, want = load_small()
    dev = lambda a: torch.from_numpy(a).to(DEV)
    out = pgd.decode(dev(q), dev(k), dev(v), dev(t), dev(L), scale)
    assert_close(out, want, "f32", "golden")


@pytest.mark.parametrize("splits", [1, 7, 1000])
@pytest.mark.parametrize("recipe", ["llama3_8b_fp8", "llama3_8b_i8", "llama3_8b_fp8_pb",
                                    "llama3_8b_i8_pb"])
def test_8bit_split_invariance_and_poison(recipe, splits):
    w = gen.make(recipe, device=DEV, B=6, lens=("uniform", 1, 2000), max_len=2048, poison=True)
    want, _ = run_oracle(w)
    out, _ = run_cuda(w, num_splits=splits)
    assert_close(out, want, w.dtype, "%s splits=%d" % (recipe, splits))
