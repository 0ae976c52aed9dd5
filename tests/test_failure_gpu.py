"""Failure detection on the GPU without a fault: a bounded wait that runs out
reports PGD_ERR_TIMEOUT through the error word and leaves the context usable;
decode steps captured in a CUDA graph replay to the same result (GPU only)."""
import ctypes

import pytest
import torch

import gen
import paged_gqa_decode_04_gb300 as pgd
from gpu_cases import assert_close, run_oracle
from paged_gqa_decode_04_gb300 import _lib

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_context_survives():
    w = gen.make("llama3_8b", device="cuda", B=3, lens=[100, 37, 260], max_len=320)
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool)
    try:
        assert pgd.paged_gqa_get_error(pool) == 0
        stream = torch.cuda.current_stream()
        rc = _lib.load().paged_gqa_selftest_wait_timeout(pool.handle, 1000,
                                                         ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0
        assert pgd.paged_gqa_get_error(pool) == _lib.PGD_ERR_TIMEOUT
        assert pgd.paged_gqa_get_error(pool) == 0          # read-and-clear
        out = pgd.paged_gqa_decode(pool, w.q, w.block_table, w.seq_lens, w.scale)
        assert pgd.paged_gqa_get_error(pool) == 0
        want, _ = run_oracle(w)
        assert_close(out, want, "bf16", "after timeout")
    finally:
        pool.close()


def test_decode_replays_from_a_cuda_graph():
    """The decode call allocates nothing and never synchronises, so a step can
    be captured once and replayed (launch overhead gone for small steps)."""
    w = gen.make("llama3_8b", device="cuda", B=8, lens=("uniform", 1, 1500), max_len=1536)
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool)
    try:
        out = torch.empty_like(w.q)
        ws = pgd.alloc_workspace(pool, w.B, w.Hq)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):   # first call outside capture: kernel attributes set
            pgd.paged_gqa_decode(pool, w.q, w.block_table, w.seq_lens, w.scale, out=out,
                                 workspace=ws, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pgd.paged_gqa_decode(pool, w.q, w.block_table, w.seq_lens, w.scale, out=out,
                                 workspace=ws, stream=s)
        want, _ = run_oracle(w)
        for _ in range(3):
            out.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert_close(out, want, "bf16", "graph replay")
        assert pgd.paged_gqa_get_error(pool) == 0
    finally:
        pool.close()
