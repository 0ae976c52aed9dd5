"""ctypes binding of libpaged_gqa.so (the C ABI declared in include/paged_gqa.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  There is no CPU fallback; if the library is missing
the first call raises.
"""
import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpaged_gqa.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "paged_gqa.h")
HEADERS = [HEADER, os.path.join(os.path.dirname(HERE), "include", "paged_kv_manager.h")]

PGD_F32 = 0
PGD_BF16 = 1
PGD_FP8_E4M3 = 2
PGD_INT8 = 3
PGD_SCALE_PER_HEAD = 0
PGD_SCALE_PER_BLOCK = 1

STATUS_NAMES = {
    0: "PGD_OK", 1: "PGD_ERR_ARG", 2: "PGD_ERR_SHAPE", 3: "PGD_ERR_DTYPE", 4: "PGD_ERR_ALIGN",
    5: "PGD_ERR_WORKSPACE", 6: "PGD_ERR_CUDA", 7: "PGD_ERR_BLOCK_ID", 8: "PGD_ERR_SEQ_LEN",
    9: "PGD_ERR_UNSUPPORTED", 10: "PGD_ERR_TIMEOUT", 11: "PGD_ERR_TOO_LARGE",
    20: "PGD_ERR_NO_BLOCKS", 21: "PGD_ERR_NO_SEQ", 22: "PGD_ERR_SEQ_EXISTS", 23: "PGD_ERR_SEQ_FULL",
}
globals().update({v: k for k, v in STATUS_NAMES.items()})

_lib = None


class PagedGQAError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        msg = "%s: %s" % (name, strerror(status) if _lib is not None else "")
        super().__init__(("%s (%s)" % (msg, what)) if what else msg)


def load(path=LIB_PATH):
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libpaged_gqa.so not built: run `python -c \"import __graft_entry__ as "
                           "g; g.build()\"` or paged_gqa_decode_04_gb300/build.py")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.paged_kv_pool_create.argtypes = [ctypes.POINTER(vp), vp, vp, i64, i32, i32, i32, i32]
    lib.paged_kv_pool_create.restype = i32
    lib.paged_kv_pool_create_fp8.argtypes = [ctypes.POINTER(vp), vp, vp, vp, vp, i64, i32, i32,
                                             i32]
    lib.paged_kv_pool_create_fp8.restype = i32
    lib.paged_kv_pool_create_q8.argtypes = [ctypes.POINTER(vp), vp, vp, i32, vp, vp, i32, i64,
                                            i32, i32, i32]
    lib.paged_kv_pool_create_q8.restype = i32
    lib.paged_kv_pool_destroy.argtypes = [vp]
    lib.paged_kv_pool_destroy.restype = i32
    lib.paged_gqa_workspace_size.argtypes = [vp, i32, i32, i32, ctypes.POINTER(sz)]
    lib.paged_gqa_workspace_size.restype = i32
    lib.paged_gqa_decode.argtypes = [vp, vp, i32, i32, vp, i32, vp, ctypes.c_float, vp, vp, sz,
                                     i32, vp]
    lib.paged_gqa_decode.restype = i32
    lib.paged_gqa_get_error.argtypes = [vp, vp]
    lib.paged_gqa_get_error.restype = i32
    lib.paged_gqa_auto_splits.argtypes = [vp, ctypes.POINTER(i32)]
    lib.paged_gqa_auto_splits.restype = i32
    lib.paged_gqa_strerror.argtypes = [i32]
    lib.paged_gqa_strerror.restype = ctypes.c_char_p
    lib.paged_gqa_decode_ex.argtypes = [vp, vp, i32, i32, i32, vp, i32, vp, i32, ctypes.c_float,
                                        vp, vp, sz, i32, vp]
    lib.paged_gqa_decode_ex.restype = i32
    lib.paged_gqa_workspace_size_ex.argtypes = [vp, i32, i32, i32, i32, ctypes.POINTER(sz)]
    lib.paged_gqa_workspace_size_ex.restype = i32
    lib.paged_gqa_decode_noalloc.argtypes = [vp, vp, i32, i32, vp, i32, vp, ctypes.c_float, vp,
                                             i32, vp]
    lib.paged_gqa_decode_noalloc.restype = i32
    lib.paged_gqa_selftest_wait_timeout.argtypes = [vp, i64, vp]
    lib.paged_gqa_selftest_wait_timeout.restype = i32
    lib.paged_gqa_noalloc_scratch_bytes.argtypes = []
    lib.paged_gqa_noalloc_scratch_bytes.restype = sz
    lib.paged_gqa_decode_host.argtypes = [vp, vp, i32, i32, i32, vp, i32, vp, i32,
                                          ctypes.c_float, vp, vp, sz, i32, vp]
    lib.paged_gqa_decode_host.restype = i32
    lib.paged_gqa_plan.argtypes = [i32] * 9 + [ctypes.POINTER(i32)]
    lib.paged_gqa_plan.restype = i32
    lib.paged_gqa_workspace_size_host.argtypes = [vp, i32, i32, i32, i32, i32,
                                                  ctypes.POINTER(sz)]
    lib.paged_gqa_workspace_size_host.restype = i32
    # KV write path (include/paged_kv_manager.h)
    pi32 = ctypes.POINTER(ctypes.c_int32)
    pint = ctypes.POINTER(ctypes.c_int)
    lib.pgd_kvm_create.argtypes = [ctypes.POINTER(vp), i64, i32, i32, i32]
    lib.pgd_kvm_destroy.argtypes = [vp]
    lib.pgd_kvm_add_sequence.argtypes = [vp, i32]
    lib.pgd_kvm_fork.argtypes = [vp, i32, i32]
    lib.pgd_kvm_free_sequence.argtypes = [vp, i32]
    lib.pgd_kvm_append_slots.argtypes = [vp, pint, i32, pi32, pi32, pi32, pint]
    lib.pgd_kvm_block_tables.argtypes = [vp, pint, i32, pi32, i32, pi32]
    lib.pgd_kvm_num_free.argtypes = [vp, ctypes.POINTER(i64)]
    lib.pgd_kvm_ref_count.argtypes = [vp, i64, pint]
    lib.paged_kv_copy_blocks.argtypes = [vp, vp, vp, i32, vp]
    lib.paged_kv_append.argtypes = [vp, vp, vp, vp, i32, vp]
    for name in ("pgd_kvm_create", "pgd_kvm_destroy", "pgd_kvm_add_sequence", "pgd_kvm_fork",
                 "pgd_kvm_free_sequence", "pgd_kvm_append_slots", "pgd_kvm_block_tables",
                 "pgd_kvm_num_free", "pgd_kvm_ref_count", "paged_kv_copy_blocks",
                 "paged_kv_append"):
        getattr(lib, name).restype = i32
    _lib = lib
    return lib


def strerror(status):
    return load().paged_gqa_strerror(int(status)).decode()


def declared_functions(headers=None):
    """Names of the functions the headers under include/ declare."""
    names = set()
    for h in headers or HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b((?:paged|pgd)_\w+)\s*\(", text))
    return sorted(names)
