"""Streams, threads and graphs (GPU only).

One pool handle serves decodes issued from two host threads on two streams at
once, each with its own workspace and output, and every result equals the same
decode run alone, bit for bit.  The host-memory entry point with page-locked
buffers enqueues no copy, so it can be captured in a CUDA graph and replayed.
"""
import threading

import pytest
import torch

import gen
import paged_gqa_decode_04_gb300 as pgd

pytestmark = pytest.mark.gpu


def test_two_threads_two_streams_one_handle():
    # 48 sequences of Llama-3-8B shape; each thread decodes its own half.  With
    # 24 runs over 152 spans the host picks the last-arriver merge, which never
    # waits on another CTA, so the two grids may share the device in any way.
    w = gen.make("llama3_8b", device="cuda", B=48, lens=("uniform", 128, 2048), max_len=2048)
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool)
    try:
        halves = [slice(0, 24), slice(24, 48)]
        want = [pgd.paged_gqa_decode(pool, w.q[h].contiguous(), w.block_table[h].contiguous(),
                                     w.seq_lens[h].contiguous(), w.scale) for h in halves]
        assert pgd.paged_gqa_get_error(pool) == 0
        errors = []

        def worker(i):
            try:
                h = halves[i]
                q, bt, sl = (t[h].contiguous() for t in (w.q, w.block_table, w.seq_lens))
                s = torch.cuda.Stream()
                ws = pgd.alloc_workspace(pool, q.shape[0], w.Hq)
                outs = [torch.empty_like(q) for _ in range(2)]
                torch.cuda.synchronize()
                with torch.cuda.stream(s):
                    for it in range(40):
                        pgd.paged_gqa_decode(pool, q, bt, sl, w.scale, out=outs[it % 2],
                                             workspace=ws, stream=s)
                s.synchronize()
                for o in outs:
                    if not torch.equal(o, want[i]):
                        errors.append("thread %d: result differs from the lone decode" % i)
            except Exception as e:  # reported on the main thread
                errors.append("thread %d: %r" % (i, e))

        threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
        assert not errors, errors
        assert pgd.paged_gqa_get_error(pool) == 0
    finally:
        pool.close()


def test_host_entry_with_page_locked_buffers_replays_from_a_graph():
    w = gen.make("llama3_8b", device="cuda", B=6, lens=[900, 17, 300, 1, 64, 2000], max_len=2048)
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool)
    try:
        want = pgd.paged_gqa_decode(pool, w.q, w.block_table, w.seq_lens, w.scale).cpu()
        h_q, h_bt, h_sl = (t.cpu().pin_memory() for t in (w.q, w.block_table, w.seq_lens))
        h_out = torch.empty(w.q.shape, dtype=w.q.dtype).pin_memory()
        ws = torch.zeros(pgd.paged_gqa_workspace_size_host(pool, w.B, 1, w.Hq, h_bt.shape[1]),
                         dtype=torch.uint8, device="cuda")
        s = torch.cuda.Stream()
        call = lambda: pgd.paged_gqa_decode_host(pool, h_q, h_bt, h_sl, w.scale, out=h_out,
                                                 workspace=ws, stream=s)
        with torch.cuda.stream(s):   # first call outside capture: kernel attributes set
            call()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            call()
        for _ in range(3):
            h_out.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(h_out, want)
        assert pgd.paged_gqa_get_error(pool) == 0
    finally:
        pool.close()
