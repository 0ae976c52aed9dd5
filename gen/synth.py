"""Workload recipes: shapes, length mixes, block permutations and values.

Every workload is a decode step over a paged KV cache:

  q           [B, Hq, D]                       query of the one new token per sequence
  k_pool      [num_blocks, block_size, Hkv, D] physical K blocks
  v_pool      [num_blocks, block_size, Hkv, D] physical V blocks
  block_table [B, max_blocks] int32            logical block i of sequence b -> physical id
  seq_lens    [B] int32                        cached tokens of each sequence

Recipe (one fixed rule for every workload):
  * lengths, the pool size and the block permutation come from
    ``numpy.random.default_rng(seed)``;
  * the pool holds ceil(1.10 * sum_b ceil(L_b / bs)) blocks unless the recipe
    fixes it; physical ids are the first sum_b ceil(L_b / bs) entries of a
    seeded permutation of the pool, handed out in logical order (sequence by
    sequence, block by block);
  * table entries past a sequence's last block hold -1 (never read);
  * q, K and V are drawn N(0, 1) in float32 from a ``torch.Generator`` seeded
    with the same seed on the target device, then rounded to the workload's
    dtype (round-to-nearest-even for bfloat16);
  * ``poison=True`` fills every unused pool block and every slot past L_b in a
    sequence's last block with NaN, so a kernel that reads them shows it.

The shapes follow the layer shapes of the models the pages discuss (Llama-3-8B,
Llama-2-13B with MHA and MQA, a 70B long-context layer) and the block-size
trade-off of "Advanced Optimizations: MQA, GQA, and PagedAttention", section
"Optimizing Block Size"; the 16-token default block is the example of "The
Ultimate Guide to LLM Inference Optimization - Part 2", section "Paged
Attention".  No public dataset is involved.
"""
from dataclasses import dataclass, field
import math

import numpy as np
import torch

# name -> recipe.  lens: explicit list, ("uniform", lo, hi) inclusive integers, or
# ("lognormal", median, sigma, lo, hi) rounded to the nearest integer and clipped.
CONFIGS = {
    "tiny": dict(B=4, lens=[1, 7, 16, 33], Hq=8, Hkv=2, D=64, block_size=16, dtype="f32",
                 num_blocks=64, max_len=33, seed=1001),
    "llama3_8b": dict(B=64, lens=("uniform", 128, 4096), Hq=32, Hkv=8, D=128, block_size=16,
                      dtype="bf16", max_len=4096, seed=1002),
    "mha_13b_b1": dict(B=1, lens=[4096], Hq=40, Hkv=40, D=128, block_size=16, dtype="bf16",
                       max_len=4096, seed=1003),
    "mha_13b_b8": dict(B=8, lens=[4096] * 8, Hq=40, Hkv=40, D=128, block_size=16, dtype="bf16",
                       max_len=4096, seed=1003),
    "mqa_13b_b1": dict(B=1, lens=[4096], Hq=40, Hkv=1, D=128, block_size=16, dtype="bf16",
                       max_len=4096, seed=1003),
    "mqa_13b_b8": dict(B=8, lens=[4096] * 8, Hq=40, Hkv=1, D=128, block_size=16, dtype="bf16",
                       max_len=4096, seed=1003),
    "long_70b": dict(B=8, lens=("uniform", 32768, 131072), Hq=64, Hkv=8, D=128, block_size=32,
                     dtype="bf16", max_len=131072, seed=1004),
}
for _bs in (8, 16, 32, 64, 128):
    CONFIGS["sweep_bs%d" % _bs] = dict(B=256, lens=("lognormal", 600.0, 1.0, 1, 8192), Hq=32,
                                       Hkv=8, D=128, block_size=_bs, dtype="bf16", max_len=8192,
                                       seed=1005)

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.float8_e4m3fn,
                "i8": torch.int8}
Q8 = ("fp8", "i8")   # 8-bit pages
CODE_MAX = {"fp8": 448.0, "i8": 127.0}

# 8-bit (e4m3) pages: the Llama-3-8B and 70B layer shapes with K/V stored as
# e4m3 codes of N(0, 1) draws and one scale per KV head drawn from U[0.5, 1.5];
# q stays bfloat16.
CONFIGS["llama3_8b_fp8"] = dict(CONFIGS["llama3_8b"], dtype="fp8")
CONFIGS["long_70b_fp8"] = dict(CONFIGS["long_70b"], dtype="fp8")
# int8 pages with one scale per KV head: N(0, 1) draws divided by a per-head
# scale U[0.5, 1.5] * 4 / 127, rounded, clipped to [-127, 127].
CONFIGS["llama3_8b_i8"] = dict(CONFIGS["llama3_8b"], dtype="i8")
CONFIGS["long_70b_i8"] = dict(CONFIGS["long_70b"], dtype="i8")
# 8-bit pages with a scale per physical block and KV head, quantized the way a
# writer quantizes a filled block: scale = max |x| over the block's slots and
# head dimension / the code's largest value (448 for e4m3, 127 for int8),
# code = x / scale rounded to the code (nearest even for e4m3, nearest for int8).
for _base in ("llama3_8b", "long_70b"):
    for _code in Q8:
        CONFIGS["%s_%s_pb" % (_base, _code)] = dict(CONFIGS[_base], dtype=_code, scales="block")


def config_names():
    return list(CONFIGS)


@dataclass
class Workload:
    name: str
    q: torch.Tensor
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    scale: float
    B: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    max_blocks: int
    dtype: str
    seed: int
    lens_np: np.ndarray = field(repr=False)
    table_np: np.ndarray = field(repr=False)
    k_scale: torch.Tensor = None   # 8-bit pages: per-KV-head scales [Hkv] float32
    v_scale: torch.Tensor = None

    @property
    def G(self):
        return self.Hq // self.Hkv

    def pages_used(self):
        return int(sum(-(-int(L) // self.block_size) for L in self.lens_np))


def _lengths(spec, B, rng):
    if isinstance(spec, (list, tuple)) and spec and spec[0] == "uniform":
        _, lo, hi = spec
        return rng.integers(lo, hi + 1, size=B).astype(np.int64)
    if isinstance(spec, (list, tuple)) and spec and spec[0] == "lognormal":
        _, median, sigma, lo, hi = spec
        x = np.rint(np.exp(rng.normal(math.log(median), sigma, size=B)))
        return np.clip(x, lo, hi).astype(np.int64)
    lens = np.asarray(spec, dtype=np.int64)
    if lens.shape != (B,):
        raise ValueError("explicit lens must have B entries")
    return lens


def _randn(shape, gen, device, dtype, chunk_elems=1 << 27):
    """N(0,1) float32 draws rounded to `dtype`, generated in slices of dim 0."""
    out = torch.empty(shape, dtype=dtype, device=device)
    if out.numel() == 0:
        return out
    per_row = out[0].numel() if out.dim() > 0 else 1
    rows = max(1, chunk_elems // max(per_row, 1))
    for r0 in range(0, shape[0], rows):
        r1 = min(shape[0], r0 + rows)
        out[r0:r1] = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=gen, device=device,
                                 dtype=torch.float32).to(dtype)
    return out


def _quantized(shape, gen, device, code, scales, chunk_elems=1 << 27):
    """8-bit pages of N(0, 1) draws: (codes [num_blocks, bs, Hkv, D], scales
    [Hkv] or [num_blocks, Hkv] float32), made in slices of blocks."""
    nb, bs, hkv, d = shape
    codes = torch.empty(shape, dtype=TORCH_DTYPES[code], device=device)
    if scales == "block":
        sc = torch.empty((nb, hkv), dtype=torch.float32, device=device)
    else:  # per head: fixed before the data, values beyond 4 * U scale saturate
        sc = ((0.5 + torch.rand((hkv,), generator=gen, device=device)) * 4.0 / CODE_MAX[code]
              ).to(torch.float32)
    rows = max(1, chunk_elems // (bs * hkv * d))
    for r0 in range(0, nb, rows):
        r1 = min(nb, r0 + rows)
        x = torch.randn((r1 - r0, bs, hkv, d), generator=gen, device=device, dtype=torch.float32)
        if scales == "block":
            amax = x.abs().amax(dim=(1, 3))                       # [blocks, Hkv]
            s = (amax / CODE_MAX[code]).clamp_min(1e-30)
            sc[r0:r1] = s
        else:
            s = sc[None, :].expand(r1 - r0, hkv)
        y = x / s[:, None, :, None]
        if code == "i8":
            codes[r0:r1] = torch.round(y).clamp_(-127, 127).to(torch.int8)
        else:
            codes[r0:r1] = y.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
    return codes, sc


def make(name="tiny", device="cpu", poison=False, seed=None, **over):
    """Build a workload from the recipe `name`, with optional field overrides.

    Overrides may replace any recipe field (B, lens, Hq, Hkv, D, block_size,
    dtype, num_blocks, max_len, seed).  ``max_blocks`` defaults to
    ceil(max_len / block_size).
    """
    spec = dict(CONFIGS[name])
    spec.update(over)
    if seed is not None:
        spec["seed"] = seed
    B, Hq, Hkv, D, bs = spec["B"], spec["Hq"], spec["Hkv"], spec["D"], spec["block_size"]
    rng = np.random.default_rng(spec["seed"])
    lens = _lengths(spec["lens"], B, rng)
    max_len = int(spec.get("max_len", int(lens.max()) if B else 0))
    max_blocks = int(spec.get("max_blocks", -(-max_len // bs)))
    nb = [-(-int(L) // bs) for L in lens]
    used = int(sum(nb))
    num_blocks = int(spec.get("num_blocks") or math.ceil(1.10 * used))
    if num_blocks < used:
        raise ValueError("pool too small for the lengths")
    perm = rng.permutation(num_blocks).astype(np.int64)
    table = np.full((B, max_blocks), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        table[b, :nb[b]] = perm[pos:pos + nb[b]]
        pos += nb[b]

    tdt = TORCH_DTYPES[spec["dtype"]]
    q8 = spec["dtype"] in Q8
    scales = spec.get("scales", "head")
    gen = torch.Generator(device=device)
    gen.manual_seed(int(spec["seed"]))
    q = _randn((B, Hq, D), gen, device, torch.bfloat16 if q8 else tdt)
    k_scale = v_scale = None
    if q8 and (spec["dtype"] == "i8" or scales == "block"):
        k_pool, k_scale = _quantized((num_blocks, bs, Hkv, D), gen, device, spec["dtype"], scales)
        v_pool, v_scale = _quantized((num_blocks, bs, Hkv, D), gen, device, spec["dtype"], scales)
    else:
        k_pool = _randn((num_blocks, bs, Hkv, D), gen, device, tdt)
        v_pool = _randn((num_blocks, bs, Hkv, D), gen, device, tdt)
        if q8:
            k_scale = (0.5 + torch.rand((Hkv,), generator=gen, device=device)).to(torch.float32)
            v_scale = (0.5 + torch.rand((Hkv,), generator=gen, device=device)).to(torch.float32)
    if poison:
        # NaN where the type has one; int8 pages get the code -128, which no
        # writer above produces, and (per-block scales) NaN scale rows for
        # the unused blocks
        bad = -128 if spec["dtype"] == "i8" else float("nan")
        used_mask = np.zeros(num_blocks, dtype=bool)
        used_mask[perm[:used]] = True
        unused = torch.from_numpy(np.nonzero(~used_mask)[0]).to(device)
        if unused.numel():
            k_pool[unused] = bad
            v_pool[unused] = bad
            if k_scale is not None and k_scale.dim() == 2:
                k_scale[unused] = float("nan")
                v_scale[unused] = float("nan")
        for b in range(B):
            L = int(lens[b])
            if L % bs:
                last = int(table[b, nb[b] - 1])
                k_pool[last, L % bs:] = bad
                v_pool[last, L % bs:] = bad
    return Workload(name=name, q=q, k_pool=k_pool, v_pool=v_pool,
                    block_table=torch.from_numpy(table).to(device),
                    seq_lens=torch.from_numpy(lens.astype(np.int32)).to(device),
                    scale=1.0 / math.sqrt(D), B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=bs,
                    num_blocks=num_blocks, max_blocks=max_blocks, dtype=spec["dtype"],
                    seed=int(spec["seed"]), lens_np=lens, table_np=table, k_scale=k_scale,
                    v_scale=v_scale)


def to_numpy_bits(t):
    """A float32 or bfloat16 tensor as a host numpy array the oracle accepts
    (float32 as is, bfloat16 as its uint16 bit patterns, 8-bit e4m3 and int8
    codes as their uint8 bytes)."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.float8_e4m3fn, torch.uint8, torch.int8):
        return t.view(torch.uint8).numpy()
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError("unsupported dtype %s" % t.dtype)
