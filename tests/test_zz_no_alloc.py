"""paged_gqa_decode_noalloc, the entry point for callers that cannot allocate
device memory (a plugin inside a runtime that owns all device memory, or a
path that must not let cudaMalloc / cudaFree synchronise the device).

Called through the C ABI and checked against paged_gqa_decode (the entry
point that takes a caller workspace) on two calls in a row: the second call
reuses the static scratch array the first one left behind.  This file sorts
last so that a run stopping at the first failure has run everything else."""
import ctypes

import pytest
import torch

import gen
import paged_gqa_decode_04_gb300 as pgd
from gpu_cases import BF16_MAX, BF16_MEAN
from paged_gqa_decode_04_gb300 import _lib

pytestmark = pytest.mark.gpu


def _noalloc(lib, pool, w, out, num_splits, stream):
    return lib.paged_gqa_decode_noalloc(pool.handle, w.q.data_ptr(), w.B, w.Hq,
                                        w.block_table.data_ptr(), w.block_table.shape[1],
                                        w.seq_lens.data_ptr(), ctypes.c_float(w.scale),
                                        out.data_ptr(), num_splits,
                                        ctypes.c_void_p(stream.cuda_stream))


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    import __graft_entry__

    __graft_entry__.build()
    lib = _lib.load()
    # runs longer than one span, so split runs, partials and counters are all used
    w = gen.make("llama3_8b", device="cuda", B=8, lens=("uniform", 1, 2000), max_len=2048,
                 poison=True)
    stream = torch.cuda.current_stream()
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool)
    try:
        ref = pgd.paged_gqa_decode(pool, w.q, w.block_table, w.seq_lens, w.scale)
        assert pgd.paged_gqa_get_error(pool) == 0
        outs = [torch.full_like(w.q, float("nan")) for _ in range(2)]
        taken = []
        for out in outs:
            torch.cuda.synchronize()
            before = torch.cuda.mem_get_info()[0]
            rc = _noalloc(lib, pool, w, out, 0, stream)
            assert rc == 0, pgd.strerror(rc)
            assert pgd.paged_gqa_get_error(pool) == 0   # synchronises the stream
            taken.append(before - torch.cuda.mem_get_info()[0])
            diff = (out.float() - ref.float()).abs()
            assert torch.isfinite(out.float()).all()
            assert diff.max().item() <= BF16_MAX and diff.mean().item() <= BF16_MEAN
        # The first call on a device may map the library's static array (module
        # loading); the second call takes no device memory at all.
        assert taken[1] == 0
        # the Python face gives the same bytes, and checks `out` before the call
        again = pgd.paged_gqa_decode_noalloc(pool, w.q, w.block_table, w.seq_lens, w.scale,
                                             out=torch.empty_like(w.q))
        assert torch.equal(again, outs[1])
        with pytest.raises(ValueError):
            pgd.paged_gqa_decode_noalloc(pool, w.q, w.block_table, w.seq_lens, w.scale,
                                         out=torch.empty_like(w.q)[:1])
        # a request beyond the fixed scratch is refused before anything runs
        big = torch.zeros_like(w.q)
        rc = _noalloc(lib, pool, w, big, 1 << 20, stream)
        assert rc == _lib.PGD_ERR_TOO_LARGE
        torch.cuda.synchronize()
        assert torch.count_nonzero(big) == 0
    finally:
        pool.close()
