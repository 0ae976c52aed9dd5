"""paged_gqa_decode_noalloc, the entry point for callers that cannot allocate
device memory (a plugin inside a runtime that owns all device memory, or a
path that must not let cudaMalloc / cudaFree synchronise the device).

For each page type (bfloat16, 8-bit e4m3, float32, and bfloat16 with the
separate run merge) it is called through the C
ABI twice in a row -- the second call reuses the static scratch array the
first one left behind -- and each result is checked against the float64
oracle at the parity tolerances and against paged_gqa_decode (the entry point
that takes a caller workspace).  This file sorts last so that a run stopping
at the first failure has run everything else."""
import ctypes

import pytest
import torch

import gen
import paged_gqa_decode_04_gb300 as pgd
from gpu_cases import assert_close, run_oracle, tol
from paged_gqa_decode_04_gb300 import _lib

pytestmark = pytest.mark.gpu


def _noalloc(lib, pool, w, out, num_splits, stream):
    return lib.paged_gqa_decode_noalloc(pool.handle, w.q.data_ptr(), w.B, w.Hq,
                                        w.block_table.data_ptr(), w.block_table.shape[1],
                                        w.seq_lens.data_ptr(), ctypes.c_float(w.scale),
                                        out.data_ptr(), num_splits,
                                        ctypes.c_void_p(stream.cuda_stream))


# runs longer than one span, so split runs, partials and counters are all used
CASES = {
    "bf16": dict(name="llama3_8b", B=8, lens=("uniform", 1, 2000), max_len=2048),
    "fp8": dict(name="llama3_8b_fp8", B=8, lens=("uniform", 1, 2000), max_len=2048),
    "f32": dict(name="tiny", B=6, lens=("uniform", 1, 700), max_len=704, num_blocks=None),
    # runs over 2 to 5 spans: the separate run merge, a second kernel reading
    # the same static scratch
    "bf16_separate": dict(name="llama3_8b", B=32, lens=("uniform", 128, 2048), max_len=2048),
}


@pytest.mark.parametrize("page", sorted(CASES))
def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls(page):
    import __graft_entry__

    __graft_entry__.build()
    lib = _lib.load()
    spec = dict(CASES[page])
    w = gen.make(spec.pop("name"), device="cuda", poison=True, **spec)
    want, rc = run_oracle(w)
    assert rc == 0
    tmax, tmean = tol(w.dtype)
    stream = torch.cuda.current_stream()
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool, w.k_scale, w.v_scale)
    try:
        ref = pgd.paged_gqa_decode(pool, w.q, w.block_table, w.seq_lens, w.scale)
        assert pgd.paged_gqa_get_error(pool) == 0
        assert_close(ref, want, w.dtype, "%s workspace entry point" % page)
        outs = [torch.full_like(w.q, float("nan")) for _ in range(2)]
        taken = []
        for i, out in enumerate(outs):
            torch.cuda.synchronize()
            before = torch.cuda.mem_get_info()[0]
            rc = _noalloc(lib, pool, w, out, 0, stream)
            assert rc == 0, pgd.strerror(rc)
            assert pgd.paged_gqa_get_error(pool) == 0   # synchronises the stream
            taken.append(before - torch.cuda.mem_get_info()[0])
            assert_close(out, want, w.dtype, "%s no-alloc call %d" % (page, i + 1))
            diff = (out.float() - ref.float()).abs()
            assert diff.max().item() <= tmax and diff.mean().item() <= tmean
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
        # so is an argument error (out aliasing q), with the decode's status
        rc = lib.paged_gqa_decode_noalloc(pool.handle, w.q.data_ptr(), w.B, w.Hq,
                                          w.block_table.data_ptr(), w.block_table.shape[1],
                                          w.seq_lens.data_ptr(), ctypes.c_float(w.scale),
                                          w.q.data_ptr(), 0, ctypes.c_void_p(stream.cuda_stream))
        assert rc == _lib.PGD_ERR_ARG
        torch.cuda.synchronize()
        assert torch.count_nonzero(big) == 0
        # and the scratch still serves the next call
        rc = _noalloc(lib, pool, w, outs[0], 0, stream)
        assert rc == 0 and pgd.paged_gqa_get_error(pool) == 0
        assert torch.equal(outs[0], outs[1])
    finally:
        pool.close()
