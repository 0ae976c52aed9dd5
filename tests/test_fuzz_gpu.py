"""Seeded random configurations against the oracle (GPU only).

Each case draws a page type (bfloat16, 8-bit e4m3, float32), head dim, KV head
count and group size, block size, a batch whose lengths mix empty, one-token,
short and longer sequences, the number of query tokens, a window and a split
count, poisons every pool slot no sequence owns with NaN, and checks the
library's output against the float64 oracle with the tolerance of its page type.
"""
import numpy as np
import pytest
import torch

import gen
import paged_gqa_decode_04_gb300 as pgd
from gpu_cases import assert_close, run_oracle

pytestmark = pytest.mark.gpu

N_CASES = 96


def draw(case):
    rng = np.random.default_rng(7000 + case)
    dtype = str(rng.choice(["bf16"] * 5 + ["fp8"] * 2 + ["f32"]))
    D = 128 if dtype == "fp8" else int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 3, 4, 6, 8]))
    q_len = 1 if dtype == "f32" else int(rng.choice([1, 1, 2, 3, 4]))
    G = int(rng.choice([g for g in (1, 2, 3, 4, 5, 8, 16) if q_len * g <= 64]))
    bs = int(rng.choice([5, 16, 48] if dtype == "f32" else [8, 16, 32, 64, 128]))
    B = int(rng.integers(1, 10))
    lens = []
    for _ in range(B):
        u = rng.random()
        lens.append(0 if u < 0.1 else 1 if u < 0.2 else int(rng.integers(2, 65)) if u < 0.5
                    else int(rng.integers(65, 700)))
    lens[0] = max(lens[0], 1)   # at least one block in the pool
    window = 0 if dtype == "f32" or rng.random() < 0.5 else int(rng.integers(1, 300))
    splits = int(rng.choice([0, 0, 1, 3, 17, 152, 500]))
    max_len = max(lens) + int(rng.integers(0, 40))
    return dict(dtype=dtype, D=D, Hkv=Hkv, Hq=Hkv * G, q_len=q_len, block_size=bs, B=B,
                lens=lens, window=window, splits=splits, max_len=max_len)


# A second sweep over the 8-bit page types: e4m3 and int8 codes with scales
# per KV head or per block and KV head (its own seeds, so the sweep above
# keeps its draws).
N_Q8_CASES = 32


def draw_q8(case):
    c = draw(7100 - 7000 + case)
    rng = np.random.default_rng(7100 + case)
    c["dtype"] = str(rng.choice(["fp8", "i8"]))
    c["scales"] = str(rng.choice(["head", "block"]))
    c["D"] = 128
    if c["q_len"] == 1 and c["dtype"] != "f32":
        c["q_len"] = int(rng.choice([1, 1, 2, 4]))
    c["Hq"] = c["Hkv"] * max(1, min(c["Hq"] // c["Hkv"], 64 // c["q_len"]))
    if c["block_size"] not in (8, 16, 32, 64, 128):
        c["block_size"] = 16
    return c


def _run_case(c, case):
    w = gen.make("llama3_8b", device="cuda", poison=True, seed=7000 + case, B=c["B"],
                 lens=c["lens"], Hq=c["Hq"], Hkv=c["Hkv"], D=c["D"], block_size=c["block_size"],
                 dtype=c["dtype"], max_len=c["max_len"], scales=c.get("scales", "head"))
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool, w.k_scale, w.v_scale)
    try:
        if c["q_len"] == 1 and c["window"] == 0:
            out = pgd.paged_gqa_decode(pool, w.q, w.block_table, w.seq_lens, w.scale,
                                       num_splits=c["splits"])
            want, _ = run_oracle(w)
        else:
            g = torch.Generator(device="cuda")
            g.manual_seed(9000 + case)
            q = torch.randn((w.B, c["q_len"], w.Hq, w.D), generator=g,
                            device="cuda").to(torch.bfloat16)
            out = pgd.paged_gqa_decode_ex(pool, q, w.block_table, w.seq_lens, w.scale,
                                          window=c["window"], num_splits=c["splits"])
            want, _ = run_oracle(w, q=q, window=c["window"])
        assert pgd.paged_gqa_get_error(pool) == 0
        assert_close(out.view(want.shape), want, w.dtype, str(c))
    finally:
        pool.close()


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_configuration_matches_oracle(case):
    _run_case(draw(case), case)


@pytest.mark.parametrize("case", range(N_Q8_CASES))
def test_random_8bit_configuration_matches_oracle(case):
    _run_case(draw_q8(case), 100 + case)
