"""Paged grouped-query decode attention for GB300 (sm_103a).

Python face of libpaged_gqa.so.  The functions keep the C ABI's names and take
torch tensors for device memory; they only marshal pointers, sizes and the
current CUDA stream.  The computation -- block-table walk, TMA page staging,
q K^T, online softmax, P V and the split-KV log-sum-exp merge -- runs in the
library's kernels.
"""
import ctypes

import torch

from . import _lib
from ._lib import PagedGQAError, STATUS_NAMES, strerror  # noqa: F401
from .kv_cache import KVBlockManager, paged_kv_append, paged_kv_copy_blocks  # noqa: F401

__all__ = [
    "PagedKVPool", "PagedGQAError", "paged_kv_pool_create", "paged_kv_pool_destroy",
    "paged_gqa_workspace_size", "paged_gqa_decode", "paged_gqa_get_error",
    "paged_gqa_auto_splits", "paged_gqa_decode_ex", "paged_gqa_workspace_size_ex",
    "paged_gqa_decode_noalloc", "paged_gqa_noalloc_scratch_bytes",
    "paged_gqa_decode_host", "paged_gqa_workspace_size_host", "paged_gqa_plan",
    "strerror", "decode", "KVBlockManager", "paged_kv_append", "paged_kv_copy_blocks",
]

_DTYPES = {torch.float32: _lib.PGD_F32, torch.bfloat16: _lib.PGD_BF16}
_FP8 = (torch.float8_e4m3fn, torch.uint8)  # 8-bit e4m3 pages (uint8 = raw codes)
_Q8 = _FP8 + (torch.int8,)                  # 8-bit pages of either code


def _code_of(dtype):
    """Library dtype of a pool's torch dtype (int8 pages: int8 codes)."""
    if dtype == torch.int8:
        return _lib.PGD_INT8
    return _lib.PGD_FP8_E4M3 if dtype in _FP8 else _DTYPES[dtype]


def _check(rc, what=""):
    if rc != 0:
        raise PagedGQAError(rc, what)


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


class PagedKVPool:
    """Non-owning handle on a K/V block pool pair [num_blocks, block_size, Hkv, D].

    Keeps references to the two tensors so they outlive the handle.
    """

    def __init__(self, k_pool, v_pool, k_scale=None, v_scale=None):
        """float32 / bfloat16 pools, or 8-bit pages -- e4m3 (torch.float8_e4m3fn
        or uint8 codes) or int8 (torch.int8 codes) -- with float32 scales
        k_scale / v_scale of shape [Hkv] (one per KV head) or [num_blocks, Hkv]
        (one per physical block and KV head)."""
        lib = _lib.load()
        if not (isinstance(k_pool, torch.Tensor) and isinstance(v_pool, torch.Tensor)):
            raise TypeError("k_pool and v_pool must be torch tensors")
        if k_pool.shape != v_pool.shape or k_pool.dim() != 4:
            raise ValueError("pools must both be [num_blocks, block_size, Hkv, D]")
        fp8 = k_pool.dtype in _Q8
        if k_pool.dtype != v_pool.dtype or not (fp8 or k_pool.dtype in _DTYPES):
            raise TypeError("pools must be float32, bfloat16 or 8-bit, the same for K and V")
        if not (k_pool.is_cuda and v_pool.is_cuda):
            raise ValueError("pools must be CUDA tensors")
        if not (k_pool.is_contiguous() and v_pool.is_contiguous()):
            raise ValueError("pools must be contiguous")
        self.k_pool, self.v_pool = k_pool, v_pool
        self.num_blocks, self.block_size, self.num_kv_heads, self.head_dim = k_pool.shape
        self.dtype = k_pool.dtype
        self.q_dtype = torch.bfloat16 if fp8 else k_pool.dtype
        self.k_scale, self.v_scale = k_scale, v_scale
        self.scale_per_block = False
        h = ctypes.c_void_p()
        with torch.cuda.device(k_pool.device):
            if fp8:
                per_head, per_block = (self.num_kv_heads,), (self.num_blocks, self.num_kv_heads)
                for sc in (k_scale, v_scale):
                    if (not isinstance(sc, torch.Tensor) or sc.dtype != torch.float32 or
                            not sc.is_cuda or not sc.is_contiguous() or
                            tuple(sc.shape) not in (per_head, per_block) or
                            sc.shape != k_scale.shape):
                        raise ValueError("8-bit pools need float32 contiguous CUDA scales "
                                         "[Hkv] or [num_blocks, Hkv], the same for K and V")
                self.scale_per_block = tuple(k_scale.shape) == per_block
                _check(lib.paged_kv_pool_create_q8(
                    ctypes.byref(h), k_pool.data_ptr(), v_pool.data_ptr(),
                    _code_of(k_pool.dtype), k_scale.data_ptr(), v_scale.data_ptr(),
                    _lib.PGD_SCALE_PER_BLOCK if self.scale_per_block else _lib.PGD_SCALE_PER_HEAD,
                    self.num_blocks, self.block_size, self.num_kv_heads, self.head_dim),
                    "paged_kv_pool_create_q8")
            else:
                _check(lib.paged_kv_pool_create(ctypes.byref(h), k_pool.data_ptr(),
                                                v_pool.data_ptr(), self.num_blocks,
                                                self.block_size, self.num_kv_heads,
                                                self.head_dim, _DTYPES[self.dtype]),
                       "paged_kv_pool_create")
        self._h = h

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("pool handle destroyed")
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None and _lib._lib is not None:
            rc = _lib._lib.paged_kv_pool_destroy(self._h)
            self._h = None
            _check(rc, "paged_kv_pool_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def paged_kv_pool_create(k_pool, v_pool):
    return PagedKVPool(k_pool, v_pool)


def paged_kv_pool_destroy(pool):
    pool.close()


def paged_gqa_workspace_size(pool, B, Hq, num_splits=0):
    n = ctypes.c_size_t()
    _check(_lib.load().paged_gqa_workspace_size(pool.handle, int(B), int(Hq), int(num_splits),
                                                ctypes.byref(n)), "paged_gqa_workspace_size")
    return n.value


def paged_gqa_auto_splits(pool):
    n = ctypes.c_int()
    _check(_lib.load().paged_gqa_auto_splits(pool.handle, ctypes.byref(n)))
    return n.value


def alloc_workspace(pool, B, Hq, num_splits=0):
    """A zero-filled workspace tensor of the right size on the pool's device.

    Reusable across calls: every completed call leaves it ready for the next."""
    nbytes = paged_gqa_workspace_size(pool, B, Hq, num_splits)
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=pool.k_pool.device)


def _check_decode_args(pool, q, block_table, seq_lens, q_dims):
    """Shapes, dtypes and placement of a decode call's tensors (q has q_dims
    dimensions: [B, Hq, D] or [B, q_len, Hq, D])."""
    if q.dim() != q_dims or block_table.dim() != 2 or seq_lens.dim() != 1:
        raise ValueError("q must be [B,%sHq,D], block_table [B,max_blocks], seq_lens [B]"
                         % ("q_len," if q_dims == 4 else ""))
    if q.dtype != pool.q_dtype:
        raise TypeError("q must be %s for this pool" % pool.q_dtype)
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    if (q.shape[-1] != pool.head_dim or block_table.shape[0] != q.shape[0] or
            seq_lens.shape[0] != q.shape[0]):
        raise ValueError("shape mismatch between q, tables and pool")
    for t in (q, block_table, seq_lens):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")


def paged_gqa_decode(pool, q, block_table, seq_lens, scale, out=None, workspace=None,
                     num_splits=0, stream=None):
    """Enqueue one decode step; returns `out` ([B, Hq, D], q's dtype).

    q [B, Hq, D], block_table [B, max_blocks] int32 and seq_lens [B] int32 are
    CUDA tensors on the pool's device.  Raises PagedGQAError on an argument
    error; device-side errors are reported by paged_gqa_get_error.
    """
    lib = _lib.load()
    _check_decode_args(pool, q, block_table, seq_lens, 3)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_workspace(pool, B, Hq, num_splits)
    _check(lib.paged_gqa_decode(pool.handle, q.data_ptr(), B, Hq, block_table.data_ptr(),
                                block_table.shape[1], seq_lens.data_ptr(), float(scale),
                                out.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                int(num_splits), _stream_handle(stream)), "paged_gqa_decode")
    return out


def paged_gqa_workspace_size_ex(pool, B, q_len, Hq, num_splits=0):
    n = ctypes.c_size_t()
    _check(_lib.load().paged_gqa_workspace_size_ex(pool.handle, int(B), int(q_len), int(Hq),
                                                   int(num_splits), ctypes.byref(n)),
           "paged_gqa_workspace_size_ex")
    return n.value


def paged_gqa_decode_ex(pool, q, block_table, seq_lens, scale, window=0, out=None,
                        workspace=None, num_splits=0, stream=None):
    """Several query tokens per sequence and an optional window.

    q [B, q_len, Hq, D] (bf16): the last q_len cached tokens of each sequence,
    each attending causally to the positions before it, or only to the
    `window` most recent ones when window > 0.  Returns out [B, q_len, Hq, D].
    """
    lib = _lib.load()
    _check_decode_args(pool, q, block_table, seq_lens, 4)
    B, q_len, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = paged_gqa_workspace_size_ex(pool, B, q_len, Hq, num_splits)
        workspace = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    _check(lib.paged_gqa_decode_ex(pool.handle, q.data_ptr(), B, q_len, Hq,
                                   block_table.data_ptr(), block_table.shape[1],
                                   seq_lens.data_ptr(), int(window), float(scale),
                                   out.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                   int(num_splits), _stream_handle(stream)), "paged_gqa_decode_ex")
    return out


def paged_gqa_decode_noalloc(pool, q, block_table, seq_lens, scale, out, num_splits=0,
                             stream=None):
    """paged_gqa_decode for callers that cannot allocate device memory.

    No workspace: the split-KV scratch is the library's fixed static device
    array (paged_gqa_noalloc_scratch_bytes()), shared by every call, so calls
    that may overlap on the GPU must be serialised by the caller.  `out` must
    be given (nothing is allocated here either).  Raises PagedGQAError with
    PGD_ERR_TOO_LARGE when the request needs more scratch than the array holds.
    """
    lib = _lib.load()
    _check_decode_args(pool, q, block_table, seq_lens, 3)
    if (not isinstance(out, torch.Tensor) or out.shape != q.shape or out.dtype != q.dtype or
            not out.is_cuda or not out.is_contiguous()):
        raise ValueError("out must be a contiguous CUDA tensor shaped and typed like q")
    B, Hq, _ = q.shape
    _check(lib.paged_gqa_decode_noalloc(pool.handle, q.data_ptr(), B, Hq, block_table.data_ptr(),
                                        block_table.shape[1], seq_lens.data_ptr(), float(scale),
                                        out.data_ptr(), int(num_splits), _stream_handle(stream)),
           "paged_gqa_decode_noalloc")
    return out


def paged_gqa_noalloc_scratch_bytes():
    return int(_lib.load().paged_gqa_noalloc_scratch_bytes())


def paged_gqa_workspace_size_host(pool, B, q_len, Hq, max_blocks, num_splits=0):
    n = ctypes.c_size_t()
    _check(_lib.load().paged_gqa_workspace_size_host(pool.handle, int(B), int(q_len), int(Hq),
                                                     int(max_blocks), int(num_splits),
                                                     ctypes.byref(n)),
           "paged_gqa_workspace_size_host")
    return n.value


def paged_gqa_decode_host(pool, q, block_table, seq_lens, scale, window=0, out=None,
                          workspace=None, num_splits=0, stream=None):
    """Decode with the step's inputs and output in host memory.

    q [B, Hq, D] or [B, q_len, Hq, D], block_table [B, max_blocks] int32 and
    seq_lens [B] int32 are contiguous CPU tensors; `out` (allocated like q,
    page-locked when q is, if not given) receives the result.  Page-locked
    tensors are read and written by the kernel in place; pageable ones are
    staged through the workspace (a CUDA uint8 tensor of at least
    paged_gqa_workspace_size_host bytes, zero-filled before first use).  The
    call is asynchronous on `stream`: `out` is ready after that stream
    synchronises.
    """
    lib = _lib.load()
    if q.dim() not in (3, 4) or block_table.dim() != 2 or seq_lens.dim() != 1:
        raise ValueError("q must be [B,(q_len,)Hq,D], block_table [B,max_blocks], seq_lens [B]")
    if q.dtype != pool.q_dtype:
        raise TypeError("q must be %s for this pool" % pool.q_dtype)
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    for t in (q, block_table, seq_lens):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CPU tensors")
    B, Hq, D = q.shape[0], q.shape[-2], q.shape[-1]
    q_len = q.shape[1] if q.dim() == 4 else 1
    if D != pool.head_dim or block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("shape mismatch between q, tables and pool")
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=q.is_pinned())
    if out.is_cuda or not out.is_contiguous() or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must be a contiguous CPU tensor shaped and typed like q")
    max_blocks = block_table.shape[1]
    if workspace is None:
        nbytes = paged_gqa_workspace_size_host(pool, B, q_len, Hq, max_blocks, num_splits)
        workspace = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=pool.k_pool.device)
    _check(lib.paged_gqa_decode_host(pool.handle, q.data_ptr(), B, q_len, Hq,
                                     block_table.data_ptr(), max_blocks, seq_lens.data_ptr(),
                                     int(window), float(scale), out.data_ptr(),
                                     workspace.data_ptr(), workspace.numel(), int(num_splits),
                                     _stream_handle(stream)), "paged_gqa_decode_host")
    return out


PLAN_MERGE = {0: "last arriver", 1: "shared (cooperative)", 2: "separate", 3: "merge kernel"}


def paged_gqa_plan(dtype, num_kv_heads, head_dim, B, Hq, q_len=1, num_splits=0, window=0,
                   num_sms=None):
    """The launch plan a decode with these shapes would use (host only, no device
    needed when num_sms is given): dict with head_group, m_tiles, tile_tokens,
    grid and merge (see paged_gqa.h)."""
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    if isinstance(dtype, torch.dtype):
        dtype = _code_of(dtype)
    plan = (ctypes.c_int * 5)()
    _check(_lib.load().paged_gqa_plan(int(dtype), int(num_kv_heads), int(head_dim), int(num_sms),
                                      int(B), int(q_len), int(Hq), int(num_splits), int(window),
                                      plan), "paged_gqa_plan")
    return {"head_group": plan[0], "m_tiles": plan[1], "tile_tokens": plan[2], "grid": plan[3],
            "merge": PLAN_MERGE[plan[4]]}


def paged_gqa_get_error(pool, stream=None):
    """Synchronise the stream and return (then clear) the latched device status."""
    return int(_lib.load().paged_gqa_get_error(pool.handle, _stream_handle(stream)))


def decode(q, k_pool, v_pool, block_table, seq_lens, scale, num_splits=0, k_scale=None,
           v_scale=None):
    """One-shot convenience: build a pool handle, decode, check device errors."""
    pool = PagedKVPool(k_pool, v_pool, k_scale, v_scale)
    try:
        out = paged_gqa_decode(pool, q, block_table, seq_lens, scale, num_splits=num_splits)
        _check(paged_gqa_get_error(pool), "device")
        return out
    finally:
        pool.close()
