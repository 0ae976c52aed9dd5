"""KV write path on the GPU: the append and block-copy kernels against the
exact reference (bit for bit), and a whole cache lifecycle -- prompts written
token by token, prefix-sharing forks, copy-on-write on divergence, decode --
against the float64 oracle on the logical sequences (GPU only)."""
import numpy as np
import pytest
import torch

import gen
import oracle
import paged_gqa_decode_04_gb300 as pgd
from gpu_cases import assert_close
from oracle import kv_write

pytestmark = pytest.mark.gpu
DEV = "cuda"


def bits(t):
    return gen.to_numpy_bits(t)


def rand_rows(n, hkv, d, dtype, g):
    return torch.randn((n, hkv, d), generator=g, device=DEV, dtype=torch.float32).to(dtype)


FP8 = torch.float8_e4m3fn
I8 = torch.int8


def make_pool(k, v, per_block=False, unit=False):
    """8-bit pages (the rows are codes already) get random scales per KV head
    or per block and KV head, or unit per-head scales."""
    if k.dtype in (FP8, I8):
        shape = (k.shape[0], k.shape[2]) if per_block else (k.shape[2],)
        if unit:
            ones = torch.ones(shape, dtype=torch.float32, device=DEV)
            return pgd.PagedKVPool(k, v, ones, ones.clone())
        g = torch.Generator(device=DEV)
        g.manual_seed(11)
        ks = 0.5 + torch.rand(shape, generator=g, device=DEV, dtype=torch.float32)
        vs = 0.5 + torch.rand(shape, generator=g, device=DEV, dtype=torch.float32)
        return pgd.PagedKVPool(k, v, ks, vs)
    return pgd.PagedKVPool(k, v)


def rand_pages(shape, dtype, g):
    if dtype == I8:
        return torch.randint(-127, 128, shape, generator=g, device=DEV, dtype=torch.int32).to(I8)
    return torch.randn(shape, generator=g, device=DEV).to(dtype)


@pytest.mark.parametrize("dtype,per_block", [(torch.bfloat16, False), (torch.float32, False),
                                             (FP8, False), (I8, False), (FP8, True), (I8, True)])
def test_append_and_copy_match_reference(dtype, per_block):
    g = torch.Generator(device=DEV)
    g.manual_seed(3)
    nb, bs, hkv, d = 20, 16, 8, 128
    k = rand_pages((nb, bs, hkv, d), dtype, g)
    v = rand_pages((nb, bs, hkv, d), dtype, g)
    pool = make_pool(k, v, per_block)
    try:
        slots = torch.tensor([5, 16 * 3 + 7, 319, 0, 200], dtype=torch.int32, device=DEV)
        kn, vn = rand_pages((5, hkv, d), dtype, g), rand_pages((5, hkv, d), dtype, g)
        want_k, want_v = kv_write.append(bits(k), bits(v), bits(kn), bits(vn), slots.cpu().numpy())
        pgd.paged_kv_append(pool, kn, vn, slots)
        assert pgd.paged_gqa_get_error(pool) == 0
        assert np.array_equal(bits(k), want_k) and np.array_equal(bits(v), want_v)
        src = torch.tensor([3, 0, 7], dtype=torch.int32, device=DEV)
        dst = torch.tensor([11, 12, 19], dtype=torch.int32, device=DEV)
        if per_block:
            want_k, want_v, want_ks, want_vs = kv_write.copy_blocks(
                bits(k), bits(v), src.cpu().numpy(), dst.cpu().numpy(),
                pool.k_scale.cpu().numpy(), pool.v_scale.cpu().numpy())
        else:
            want_k, want_v = kv_write.copy_blocks(bits(k), bits(v), src.cpu().numpy(),
                                                  dst.cpu().numpy())
            if pool.k_scale is not None:   # per-head scales: untouched
                want_ks, want_vs = pool.k_scale.cpu().numpy(), pool.v_scale.cpu().numpy()
        pgd.paged_kv_copy_blocks(pool, src, dst)
        assert pgd.paged_gqa_get_error(pool) == 0
        assert np.array_equal(bits(k), want_k) and np.array_equal(bits(v), want_v)
        if pool.k_scale is not None:
            assert np.array_equal(pool.k_scale.cpu().numpy(), want_ks)
            assert np.array_equal(pool.v_scale.cpu().numpy(), want_vs)
        # out-of-range slot: skipped and reported
        before = bits(k)
        bad = torch.tensor([nb * bs], dtype=torch.int32, device=DEV)
        pgd.paged_kv_append(pool, kn[:1], vn[:1], bad)
        assert pgd.paged_gqa_get_error(pool) == pgd._lib.PGD_ERR_BLOCK_ID
        assert np.array_equal(bits(k), before)
    finally:
        pool.close()


@pytest.mark.parametrize("hkv,hq,d,dtype", [(2, 8, 64, torch.bfloat16),
                                            (8, 32, 128, torch.bfloat16), (8, 32, 128, FP8)])
def test_cache_lifecycle_decode_matches_oracle(hkv, hq, d, dtype):
    """Prompts appended token by token, two forks sharing a prefix, twenty
    generated tokens with copy-on-write, then one decode step; every unwritten
    slot of the pool is NaN, so a read of the wrong slot shows."""
    g = torch.Generator(device=DEV)
    g.manual_seed(11)
    nb, bs = 96, 16
    k = torch.full((nb, bs, hkv, d), float("nan"), device=DEV, dtype=dtype)
    v = torch.full_like(k, float("nan"))
    pool = make_pool(k, v, unit=True)
    m = pgd.KVBlockManager(nb, bs, max_seqs=8, max_blocks_per_seq=16)
    rows = {}                                     # seq -> list of (k_row, v_row) host bits

    def step(seqs):
        slots, copies = m.append_slots(seqs)
        if copies:
            src = torch.tensor([c[0] for c in copies], dtype=torch.int32, device=DEV)
            dst = torch.tensor([c[1] for c in copies], dtype=torch.int32, device=DEV)
            pgd.paged_kv_copy_blocks(pool, src, dst)
        kn, vn = rand_rows(len(seqs), hkv, d, dtype, g), rand_rows(len(seqs), hkv, d, dtype, g)
        pgd.paged_kv_append(pool, kn, vn, torch.from_numpy(slots).to(DEV))
        kb, vb = bits(kn), bits(vn)
        for i, s in enumerate(seqs):
            rows[s].append((kb[i], vb[i]))
        return copies

    try:
        prompts = {0: 45, 1: 32, 2: 7, 3: 70}
        for s in prompts:
            m.add_sequence(s)
            rows[s] = []
        for t in range(max(prompts.values())):
            step([s for s, n in prompts.items() if t < n])
        for parent, child in ((0, 4), (1, 5)):
            m.fork(parent, child)
            rows[child] = list(rows[parent])
        n_copies = 0
        for _ in range(20):
            n_copies += len(step(list(range(6))))
        assert n_copies == 1          # only seq 0's partly filled shared block (45 % 16 != 0)
        assert pgd.paged_gqa_get_error(pool) == 0

        seqs = list(range(6))
        table, lens = m.block_tables(seqs, 16)
        q = torch.randn((6, hq, d), generator=g, device=DEV).to(torch.bfloat16)
        out = pgd.paged_gqa_decode(pool, q, torch.from_numpy(table).to(DEV),
                                   torch.from_numpy(lens).to(DEV), 1.0 / np.sqrt(d))
        assert pgd.paged_gqa_get_error(pool) == 0
        # oracle on the logical sequences, laid out contiguously (one block each)
        L = max(len(rows[s]) for s in seqs)
        kc = np.zeros((6, L, hkv, d), dtype=np.uint8 if dtype == FP8 else np.uint16)
        vc = np.zeros_like(kc)
        for i, s in enumerate(seqs):
            assert len(rows[s]) == lens[i]
            for t, (kr, vr) in enumerate(rows[s]):
                kc[i, t], vc[i, t] = kr, vr
        one_block = np.arange(6, dtype=np.int32)[:, None]
        if dtype == FP8:
            unit = np.ones(hkv, dtype=np.float32)
            want, rc = oracle.decode_kv8_f64(bits(q), kc, vc, unit, unit, one_block, lens,
                                             1.0 / np.sqrt(d))
        else:
            want, rc = oracle.decode_f64(bits(q), kc, vc, one_block, lens, 1.0 / np.sqrt(d))
        assert rc == 0
        assert_close(out, want, "bf16", "lifecycle")
        for s in seqs:
            m.free_sequence(s)
        assert m.num_free() == nb
    finally:
        pool.close()
