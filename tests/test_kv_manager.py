"""Host block manager of the paged cache (CPU only, through the C ABI).

Blocks on demand, freed on finish ("The Ultimate Guide to LLM Inference
Optimization - Part 2", "Paged Attention"); prefix sharing with reference
counts and copy-on-write of the modified block only ("Modern LLM Inference
...", section 8.2).  A small pure-Python model of the same rules checks long
random operation sequences.
"""
import json
import os
import random

import numpy as np
import pytest

import paged_gqa_decode_04_gb300 as pgd
from paged_gqa_decode_04_gb300 import _lib

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__

    __graft_entry__.build()


def test_blocks_only_on_demand_and_returned_on_finish():
    m = pgd.KVBlockManager(num_blocks=8, block_size=4, max_seqs=2, max_blocks_per_seq=8)
    m.add_sequence(0)
    for t in range(13):
        slots, copies = m.append_slots([0])
        assert copies == []
        assert m.num_free() == 8 - (t // 4 + 1)         # a block per 4 tokens, when needed
        table, lens = m.block_tables([0])
        assert lens[0] == t + 1
        assert slots[0] == table[0, t // 4] * 4 + t % 4  # slot = block * bs + position
    m.free_sequence(0)
    assert m.num_free() == 8


def test_page_example_internal_fragmentation():
    """The pages' example: reserving 2048 slots for a 10-token reply wastes
    2038; with 16-token blocks the reply holds one block and wastes 6."""
    with open(os.path.join(HERE, "golden", "pages_numbers.json")) as f:
        ent = {e["id"]: e for e in json.load(f)["entries"]}
    e = ent["contiguous_reservation_waste"]
    bs = ent["default_block_tokens"]["block_size"]
    m = pgd.KVBlockManager(num_blocks=128, block_size=bs, max_seqs=1, max_blocks_per_seq=128)
    m.add_sequence(0)
    for _ in range(e["generated_tokens"]):
        m.append_slots([0])
    used = 128 - m.num_free()
    assert used == 1
    assert used * bs - e["generated_tokens"] == 6 < e["wasted_slots"]


def test_fifty_requests_share_one_system_prompt():
    """50 requests with the same system prompt (the example of "The Ultimate
    Guide ... Part 2", "Paged Attention"): the prompt's blocks are stored once;
    when the requests diverge only the partly filled shared block is copied."""
    bs, prompt = 16, 40                                  # 2 full blocks + 8 tokens
    m = pgd.KVBlockManager(num_blocks=256, block_size=bs, max_seqs=51, max_blocks_per_seq=16)
    m.add_sequence(0)
    for _ in range(prompt):
        m.append_slots([0])
    for c in range(1, 51):
        m.fork(0, c)
    assert 256 - m.num_free() == 3
    table, _ = m.block_tables([0])
    assert all(m.ref_count(b) == 51 for b in table[0, :3])
    slots, copies = m.append_slots(list(range(1, 51)))
    assert len(copies) == 50 and all(src == table[0, 2] for src, _ in copies)
    assert len({dst for _, dst in copies}) == 50
    assert m.ref_count(table[0, 2]) == 1                 # the parent keeps the original
    assert all(m.ref_count(b) == 51 for b in table[0, :2])   # full blocks stay shared
    t2, lens = m.block_tables(list(range(1, 51)))
    assert (lens == prompt + 1).all()
    assert (t2[:, :2] == table[0, :2]).all()
    for c in range(51):
        m.free_sequence(c)
    assert m.num_free() == 256


def test_aligned_prompt_shares_without_copies():
    bs = 8
    m = pgd.KVBlockManager(num_blocks=32, block_size=bs, max_seqs=4, max_blocks_per_seq=8)
    m.add_sequence(0)
    for _ in range(2 * bs):
        m.append_slots([0])
    m.fork(0, 1)
    slots, copies = m.append_slots([0, 1])
    assert copies == [] and slots[0] // bs != slots[1] // bs


def test_out_of_blocks_changes_nothing():
    m = pgd.KVBlockManager(num_blocks=2, block_size=2, max_seqs=3, max_blocks_per_seq=4)
    for s in range(3):
        m.add_sequence(s)
    m.append_slots([0, 1])
    before = m.block_tables([0, 1, 2]), m.num_free()
    with pytest.raises(pgd.PagedGQAError) as e:
        m.append_slots([0, 1, 2])                        # seq 2 needs a block; none left
    assert e.value.status == _lib.PGD_ERR_NO_BLOCKS
    after = m.block_tables([0, 1, 2]), m.num_free()
    assert np.array_equal(before[0][0], after[0][0]) and before[1] == after[1]


def test_errors():
    m = pgd.KVBlockManager(num_blocks=4, block_size=2, max_seqs=2, max_blocks_per_seq=1)
    with pytest.raises(pgd.PagedGQAError) as e:
        m.append_slots([0])
    assert e.value.status == _lib.PGD_ERR_NO_SEQ
    m.add_sequence(0)
    with pytest.raises(pgd.PagedGQAError) as e:
        m.add_sequence(0)
    assert e.value.status == _lib.PGD_ERR_SEQ_EXISTS
    with pytest.raises(pgd.PagedGQAError) as e:
        m.add_sequence(5)
    assert e.value.status == _lib.PGD_ERR_NO_SEQ
    m.append_slots([0])
    m.append_slots([0])
    with pytest.raises(pgd.PagedGQAError) as e:
        m.append_slots([0])                              # one block per sequence at most
    assert e.value.status == _lib.PGD_ERR_SEQ_FULL
    m.add_sequence(1)
    with pytest.raises(pgd.PagedGQAError) as e:
        m.append_slots([1, 1])
    assert e.value.status == _lib.PGD_ERR_ARG


class ModelManager:
    """The manager's rules restated in Python (LIFO free list, refcounts, CoW)."""

    def __init__(self, nb, bs, max_seqs, max_bps):
        self.free = list(range(nb - 1, -1, -1))
        self.refs = [0] * nb
        self.bs, self.max_bps = bs, max_bps
        self.seqs = {}

    def add(self, s):
        assert s not in self.seqs
        self.seqs[s] = [[], 0]

    def fork(self, p, c):
        self.seqs[c] = [list(self.seqs[p][0]), self.seqs[p][1]]
        for b in self.seqs[c][0]:
            self.refs[b] += 1

    def free_seq(self, s):
        for b in self.seqs.pop(s)[0]:
            self.refs[b] -= 1
            if self.refs[b] == 0:
                self.free.append(b)

    def append(self, seqs):
        need = 0
        for s in seqs:
            blocks, n = self.seqs[s]
            if n % self.bs == 0:
                if len(blocks) >= self.max_bps:
                    return "full"
                need += 1
            elif self.refs[blocks[-1]] > 1:
                need += 1
        if need > len(self.free):
            return "noblocks"
        slots, copies = [], []
        for s in seqs:
            blocks, n = self.seqs[s]
            if n % self.bs == 0:
                b = self.free.pop()
                self.refs[b] = 1
                blocks.append(b)
            elif self.refs[blocks[-1]] > 1:
                b = self.free.pop()
                self.refs[b] = 1
                self.refs[blocks[-1]] -= 1
                copies.append((blocks[-1], b))
                blocks[-1] = b
            slots.append(blocks[-1] * self.bs + n % self.bs)
            self.seqs[s][1] = n + 1
        return slots, copies


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_model(seed):
    rnd = random.Random(seed)
    nb, bs, ms, mbps = 40, rnd.choice([1, 2, 4, 8]), 12, 12
    m = pgd.KVBlockManager(nb, bs, ms, mbps)
    ref = ModelManager(nb, bs, ms, mbps)
    for _ in range(400):
        live = sorted(ref.seqs)
        op = rnd.random()
        if op < 0.15 and len(live) < ms:
            s = rnd.choice([x for x in range(ms) if x not in ref.seqs])
            m.add_sequence(s)
            ref.add(s)
        elif op < 0.25 and live and len(live) < ms:
            p = rnd.choice(live)
            c = rnd.choice([x for x in range(ms) if x not in ref.seqs])
            m.fork(p, c)
            ref.fork(p, c)
        elif op < 0.35 and live:
            s = rnd.choice(live)
            m.free_sequence(s)
            ref.free_seq(s)
        elif live:
            seqs = rnd.sample(live, rnd.randint(1, len(live)))
            want = ref.append(seqs)
            if want in ("full", "noblocks"):
                with pytest.raises(pgd.PagedGQAError) as e:
                    m.append_slots(seqs)
                assert e.value.status == (_lib.PGD_ERR_SEQ_FULL if want == "full"
                                          else _lib.PGD_ERR_NO_BLOCKS)
            else:
                slots, copies = m.append_slots(seqs)
                assert slots.tolist() == want[0] and copies == want[1]
        assert m.num_free() == len(ref.free)
        for b in range(nb):
            assert m.ref_count(b) == ref.refs[b]
        if ref.seqs:
            live = sorted(ref.seqs)
            table, lens = m.block_tables(live, mbps)
            for i, s in enumerate(live):
                blocks, n = ref.seqs[s]
                assert lens[i] == n
                assert table[i, :len(blocks)].tolist() == blocks
                assert (table[i, len(blocks):] == -1).all()
