"""paged_gqa_decode_host: the step's q, block table, lengths and output in host
memory.  Page-locked buffers are used in place by the kernel; pageable or
misaligned ones are staged through the workspace.  Either way the result is
the device-memory call's, bit for bit, and within tolerance of the oracle
(GPU only).  Where the device-memory call merges split runs in a second kernel
(runs over 2 to 5 spans), the host entry writing out in place merges them
inside the decode kernel; the two merges fold alike, so the bits still agree."""
import pytest
import torch

import gen
import paged_gqa_decode_04_gb300 as pgd
from gpu_cases import assert_close, run_oracle
from paged_gqa_decode_04_gb300 import _lib

pytestmark = pytest.mark.gpu


def _host(t, pinned, offset=0):
    """CPU copy of t, page-locked or not; `offset` elements into a larger
    buffer (so the copy starts off a 16-byte boundary)."""
    t = t.cpu()
    buf = torch.empty(t.numel() + offset, dtype=t.dtype, pin_memory=pinned)
    view = buf[offset:].view(t.shape)
    view.copy_(t)
    return view


# (recipe, overrides, q_len, window)
CASES = [
    ("llama3_8b", dict(B=5, lens=[1, 300, 17, 1000, 64], max_len=1024), 1, 0),
    ("long_70b", dict(B=2, lens=[5000, 1300], max_len=8192), 1, 0),
    ("llama3_8b", dict(B=3, lens=[90, 300, 17], max_len=320), 3, 64),
    ("llama3_8b_fp8", dict(B=3, lens=[90, 300, 17], max_len=320), 1, 0),
    ("tiny", dict(), 1, 0),
    # separate merge on the device-memory call, fused when out is used in place
    ("llama3_8b", dict(B=32, lens=("uniform", 128, 2048), max_len=2048), 1, 0),
    ("llama3_8b_i8", dict(B=32, lens=("uniform", 128, 2048), max_len=2048), 4, 0),
]

# how each of (q, block_table, seq_lens, out) is held on the host
LAYOUTS = {
    "pinned": dict(pin=(True, True, True, True), off=(0, 0, 0, 0)),
    "pageable": dict(pin=(False, False, False, False), off=(0, 0, 0, 0)),
    # seq_lens 4 bytes into its buffer (aligned enough: used in place); out 2
    # bytes in (not 16-byte aligned: staged and copied back)
    "mixed": dict(pin=(True, False, True, True), off=(0, 0, 1, 1)),
}


@pytest.mark.parametrize("layout", sorted(LAYOUTS))
@pytest.mark.parametrize("case", range(len(CASES)))
def test_host_buffers_match_device_call(case, layout):
    recipe, over, q_len, window = CASES[case]
    w = gen.make(recipe, device="cuda", **over)
    if q_len > 1:
        g0 = torch.Generator(device="cuda")
        g0.manual_seed(5)
        q = torch.randn((w.B, q_len, w.Hq, w.D), generator=g0, device="cuda").to(w.q.dtype)
    else:
        q = w.q
    pin, off = LAYOUTS[layout]["pin"], LAYOUTS[layout]["off"]
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool, w.k_scale, w.v_scale)
    try:
        want_dev = pgd.paged_gqa_decode_ex(
            pool, q if q.dim() == 4 else q.unsqueeze(1), w.block_table, w.seq_lens, w.scale,
            window=window).view(q.shape)
        assert pgd.paged_gqa_get_error(pool) == 0
        h_q = _host(q, pin[0], off[0])
        h_bt = _host(w.block_table, pin[1], off[1])
        h_sl = _host(w.seq_lens, pin[2], off[2])
        h_out = _host(torch.full_like(q, float("nan")), pin[3], off[3])
        nbytes = pgd.paged_gqa_workspace_size_host(pool, w.B, q_len, w.Hq, h_bt.shape[1])
        wsb = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
        for _ in range(2):   # the workspace is reused as is
            h_out.fill_(float("nan"))
            got = pgd.paged_gqa_decode_host(pool, h_q, h_bt, h_sl, w.scale, window=window,
                                            out=h_out, workspace=wsb)
            assert got.data_ptr() == h_out.data_ptr()
            assert pgd.paged_gqa_get_error(pool) == 0
            assert torch.equal(h_out, want_dev.cpu()), "host call differs from device call"
        want, _ = run_oracle(w, q=None if q_len == 1 and not window else
                             (q if q.dim() == 4 else q.unsqueeze(1)), window=window)
        assert_close(h_out.view(want.shape), want, w.dtype, "%s %s" % (recipe, layout))
    finally:
        pool.close()


def test_host_call_rejects_small_workspace_and_accepts_empty_batch():
    w = gen.make("llama3_8b", device="cuda", B=2, lens=[40, 7], max_len=64)
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool)
    try:
        h_q, h_bt, h_sl = (t.cpu().pin_memory() for t in (w.q, w.block_table, w.seq_lens))
        need = pgd.paged_gqa_workspace_size_host(pool, w.B, 1, w.Hq, h_bt.shape[1])
        dec = pgd.paged_gqa_workspace_size_ex(pool, w.B, 1, w.Hq)
        assert need > dec      # staging room after the decode workspace
        small = torch.zeros(dec, dtype=torch.uint8, device="cuda")
        with pytest.raises(pgd.PagedGQAError) as e:
            pgd.paged_gqa_decode_host(pool, h_q, h_bt, h_sl, w.scale, workspace=small)
        assert e.value.status == _lib.PGD_ERR_WORKSPACE
        empty = pgd.paged_gqa_decode_host(pool, h_q[:0], h_bt[:0], h_sl[:0], w.scale)
        assert empty.shape[0] == 0
        assert pgd.paged_gqa_get_error(pool) == 0
    finally:
        pool.close()
