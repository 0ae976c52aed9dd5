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


# (recipe, overrides, q_len): one workload per split-merge variant the host
# picks -- last arriver (8 runs of 4 rows), shared under a cooperative launch
# (40 rows of one KV head, long runs), separate run-merge kernel (40 runs of 16
# rows, 2 to 5 spans a run: two kernels in the graph)
GRAPH_CASES = [
    ("llama3_8b", dict(B=8, lens=("uniform", 1, 1500), max_len=1536), 1),
    ("mqa_13b_b1", dict(B=2, lens=[4096, 2500], max_len=4096), 1),
    ("llama3_8b", dict(B=40, lens=("uniform", 64, 600), max_len=640), 4),
]


@pytest.mark.parametrize("case", range(len(GRAPH_CASES)))
def test_decode_replays_from_a_cuda_graph(case):
    """The decode call allocates nothing and never synchronises, so a step can
    be captured once and replayed (launch overhead gone for small steps),
    whichever merge variant (and launch kind) it uses."""
    recipe, over, q_len = GRAPH_CASES[case]
    w = gen.make(recipe, device="cuda", **over)
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool)
    try:
        if q_len == 1:
            q = w.q
            call = lambda s: pgd.paged_gqa_decode(pool, q, w.block_table, w.seq_lens, w.scale,
                                                  out=out, workspace=ws, stream=s)
            nbytes = pgd.paged_gqa_workspace_size(pool, w.B, w.Hq, 0)
        else:
            g0 = torch.Generator(device="cuda")
            g0.manual_seed(11)
            q = torch.randn((w.B, q_len, w.Hq, w.D), generator=g0, device="cuda").to(w.q.dtype)
            call = lambda s: pgd.paged_gqa_decode_ex(pool, q, w.block_table, w.seq_lens, w.scale,
                                                     out=out, workspace=ws, stream=s)
            nbytes = pgd.paged_gqa_workspace_size_ex(pool, w.B, q_len, w.Hq, 0)
        out = torch.empty_like(q)
        ws = torch.zeros(max(256, nbytes), dtype=torch.uint8, device="cuda")
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):   # first call outside capture: kernel attributes set
            call(s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            call(s)
        want, _ = run_oracle(w, q=None if q_len == 1 else q)
        for _ in range(3):
            out.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert_close(out, want, "bf16", "graph replay")
        assert pgd.paged_gqa_get_error(pool) == 0
    finally:
        pool.close()
