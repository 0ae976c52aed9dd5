"""Python face of the KV write path (include/paged_kv_manager.h).

``KVBlockManager`` wraps the C++ host block manager (on-demand block
allocation, reference counts, copy-on-write of a shared last block);
``paged_kv_append`` and ``paged_kv_copy_blocks`` wrap the device kernels that
store new tokens and copy blocks.  Argument marshalling only.
"""
import ctypes

import numpy as np
import torch

from . import _lib
from ._lib import PagedGQAError


def _check(rc, what=""):
    if rc != 0:
        raise PagedGQAError(rc, what)


def _ints(seqs):
    arr = (ctypes.c_int * len(seqs))(*[int(s) for s in seqs])
    return arr


class KVBlockManager:
    """Host-side owner of a pool's blocks: which sequence holds which blocks."""

    def __init__(self, num_blocks, block_size, max_seqs, max_blocks_per_seq):
        lib = _lib.load()
        h = ctypes.c_void_p()
        _check(lib.pgd_kvm_create(ctypes.byref(h), int(num_blocks), int(block_size),
                                  int(max_seqs), int(max_blocks_per_seq)), "pgd_kvm_create")
        self._h = h
        self.block_size = int(block_size)
        self.max_blocks_per_seq = int(max_blocks_per_seq)

    def close(self):
        if getattr(self, "_h", None) is not None and _lib._lib is not None:
            _lib._lib.pgd_kvm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_sequence(self, seq):
        _check(_lib.load().pgd_kvm_add_sequence(self._h, int(seq)), "add_sequence")

    def fork(self, parent, child):
        _check(_lib.load().pgd_kvm_fork(self._h, int(parent), int(child)), "fork")

    def free_sequence(self, seq):
        _check(_lib.load().pgd_kvm_free_sequence(self._h, int(seq)), "free_sequence")

    def append_slots(self, seqs):
        """Reserve one new token position per sequence.  Returns (slots int32
        array, [(src_block, dst_block), ...] copies to run first)."""
        n = len(seqs)
        slots = np.empty(n, dtype=np.int32)
        src = np.empty(max(n, 1), dtype=np.int32)
        dst = np.empty(max(n, 1), dtype=np.int32)
        nc = ctypes.c_int()
        p32 = ctypes.POINTER(ctypes.c_int32)
        _check(_lib.load().pgd_kvm_append_slots(
            self._h, _ints(seqs), n, slots.ctypes.data_as(p32), src.ctypes.data_as(p32),
            dst.ctypes.data_as(p32), ctypes.byref(nc)), "append_slots")
        return slots, list(zip(src[:nc.value].tolist(), dst[:nc.value].tolist()))

    def block_tables(self, seqs, max_blocks=None):
        """(table [n, max_blocks] int32 with -1 past each sequence's blocks, lens [n] int32)."""
        max_blocks = int(max_blocks or self.max_blocks_per_seq)
        n = len(seqs)
        table = np.empty((n, max_blocks), dtype=np.int32)
        lens = np.empty(n, dtype=np.int32)
        p32 = ctypes.POINTER(ctypes.c_int32)
        _check(_lib.load().pgd_kvm_block_tables(self._h, _ints(seqs), n, table.ctypes.data_as(p32),
                                                max_blocks, lens.ctypes.data_as(p32)),
               "block_tables")
        return table, lens

    def num_free(self):
        n = ctypes.c_int64()
        _check(_lib.load().pgd_kvm_num_free(self._h, ctypes.byref(n)))
        return n.value

    def ref_count(self, block):
        c = ctypes.c_int()
        _check(_lib.load().pgd_kvm_ref_count(self._h, int(block), ctypes.byref(c)))
        return c.value


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if isinstance(stream, torch.cuda.Stream)
                           else int(stream))


def paged_kv_append(pool, k_new, v_new, slot_mapping, stream=None):
    """Store n new tokens: k_new / v_new [n, Hkv, D] (pool dtype, CUDA),
    slot_mapping [n] int32 CUDA tensor of physical slots."""
    if k_new.shape != v_new.shape or k_new.dim() != 3 or k_new.dtype != pool.dtype:
        raise ValueError("k_new / v_new must be [n, Hkv, D] in the pool's dtype (8-bit codes "
                         "for 8-bit pools, already scaled)")
    if slot_mapping.dtype != torch.int32 or slot_mapping.numel() != k_new.shape[0]:
        raise ValueError("slot_mapping must be int32 with one slot per new token")
    for t in (k_new, v_new, slot_mapping):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    _check(_lib.load().paged_kv_append(pool.handle, k_new.data_ptr(), v_new.data_ptr(),
                                       slot_mapping.data_ptr(), k_new.shape[0], _stream(stream)),
           "paged_kv_append")


def paged_kv_copy_blocks(pool, src, dst, stream=None):
    """Copy whole blocks src[i] -> dst[i] (int32 CUDA tensors), K and V."""
    if src.dtype != torch.int32 or dst.dtype != torch.int32 or src.shape != dst.shape:
        raise ValueError("src and dst must be int32 tensors of one shape")
    _check(_lib.load().paged_kv_copy_blocks(pool.handle, src.data_ptr(), dst.data_ptr(),
                                            src.numel(), _stream(stream)), "paged_kv_copy_blocks")
