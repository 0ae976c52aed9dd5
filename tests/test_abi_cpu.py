"""The C ABI on a machine without a GPU: the library loads, exports every
function the header declares, and rejects bad arguments before touching CUDA."""
import ctypes

import pytest

import paged_gqa_decode_04_gb300 as pgd
from paged_gqa_decode_04_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    return _lib.load()


def test_exports_every_declared_function(lib):
    names = _lib.declared_functions()
    assert set(names) >= {"paged_kv_pool_create", "paged_kv_pool_destroy", "paged_gqa_decode",
                          "paged_gqa_workspace_size", "paged_gqa_get_error",
                          "paged_gqa_strerror", "paged_gqa_auto_splits"}
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_names_every_status(lib):
    for code, name in _lib.STATUS_NAMES.items():
        s = pgd.strerror(code)
        assert s and s != "unknown status", (code, name)
    assert pgd.strerror(12345) == "unknown status"


def _create(lib, k, v, nb=10, bs=16, hkv=8, d=128, dtype=1):
    h = ctypes.c_void_p()
    rc = lib.paged_kv_pool_create(ctypes.byref(h), k, v, nb, bs, hkv, d, dtype)
    return rc, h


@pytest.mark.parametrize("args,code", [
    (dict(k=None, v=None), _lib.PGD_ERR_ARG),
    (dict(k=256, v=256, nb=0), _lib.PGD_ERR_ARG),
    (dict(k=256, v=256, hkv=0), _lib.PGD_ERR_ARG),
    (dict(k=256, v=256, d=96), _lib.PGD_ERR_SHAPE),
    (dict(k=256, v=256, bs=12), _lib.PGD_ERR_SHAPE),      # bf16 needs a power of two
    (dict(k=256, v=256, bs=4), _lib.PGD_ERR_SHAPE),       # bf16 needs >= 8
    (dict(k=256, v=256, bs=2048, dtype=0), _lib.PGD_ERR_SHAPE),
    (dict(k=256, v=256, dtype=7), _lib.PGD_ERR_DTYPE),
    (dict(k=264 + 1, v=256), _lib.PGD_ERR_ALIGN),
])
def test_pool_create_rejects(lib, args, code):
    rc, h = _create(lib, **args)
    assert rc == code
    assert h.value is None


def test_null_handles_rejected(lib):
    n = ctypes.c_size_t()
    assert lib.paged_gqa_workspace_size(None, 1, 8, 0, ctypes.byref(n)) == _lib.PGD_ERR_ARG
    assert lib.paged_gqa_decode(None, None, 1, 8, None, 1, None, 1.0, None, None, 0, 0,
                                None) == _lib.PGD_ERR_ARG
    assert lib.paged_gqa_get_error(None, None) == _lib.PGD_ERR_ARG
    assert lib.paged_kv_pool_destroy(None) == _lib.PGD_OK
    k = ctypes.c_int()
    assert lib.paged_gqa_auto_splits(None, ctypes.byref(k)) == _lib.PGD_ERR_ARG
    assert lib.paged_gqa_workspace_size_host(None, 1, 1, 8, 4, 0,
                                             ctypes.byref(n)) == _lib.PGD_ERR_ARG
    assert lib.paged_gqa_decode_host(None, None, 1, 1, 8, None, 1, None, 0, 1.0, None, None, 0,
                                     0, None) == _lib.PGD_ERR_ARG


def test_python_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load(str(tmp_path / "missing.so"))


def test_fp8_pool_create_rejects(lib):
    h = ctypes.c_void_p()
    # 8-bit pages need their scales: the plain create refuses the dtype
    assert lib.paged_kv_pool_create(ctypes.byref(h), 256, 256, 10, 16, 8, 128,
                                    _lib.PGD_FP8_E4M3) == _lib.PGD_ERR_ARG
    assert lib.paged_kv_pool_create_fp8(ctypes.byref(h), 256, 256, None, None, 10, 16, 8,
                                        128) == _lib.PGD_ERR_ARG
    assert lib.paged_kv_pool_create_fp8(ctypes.byref(h), 256, 256, 256, 256, 10, 16, 8,
                                        64) == _lib.PGD_ERR_SHAPE
    assert lib.paged_kv_pool_create_fp8(ctypes.byref(h), 256, 256, 258, 256, 10, 16, 8,
                                        128) == _lib.PGD_ERR_ALIGN
    assert h.value is None


def test_q8_pool_create_rejects(lib):
    """The 8-bit pool entry of either code and scale granularity refuses bad
    arguments before any CUDA call."""
    h = ctypes.c_void_p()
    f = lib.paged_kv_pool_create_q8
    # unknown code, and a wide dtype passed as a code
    assert f(ctypes.byref(h), 256, 256, 7, 256, 256, 0, 10, 16, 8, 128) == _lib.PGD_ERR_DTYPE
    assert f(ctypes.byref(h), 256, 256, _lib.PGD_BF16, 256, 256, 0, 10, 16, 8,
             128) == _lib.PGD_ERR_DTYPE
    # unknown scale granularity
    for code in (_lib.PGD_FP8_E4M3, _lib.PGD_INT8):
        assert f(ctypes.byref(h), 256, 256, code, 256, 256, 2, 10, 16, 8, 128) == _lib.PGD_ERR_ARG
        # missing scales, head_dim 64, misaligned scales, non-power-of-two block
        for gran in (_lib.PGD_SCALE_PER_HEAD, _lib.PGD_SCALE_PER_BLOCK):
            assert f(ctypes.byref(h), 256, 256, code, None, 256, gran, 10, 16, 8,
                     128) == _lib.PGD_ERR_ARG
            assert f(ctypes.byref(h), 256, 256, code, 256, 256, gran, 10, 16, 8,
                     64) == _lib.PGD_ERR_SHAPE
            assert f(ctypes.byref(h), 256, 256, code, 258, 256, gran, 10, 16, 8,
                     128) == _lib.PGD_ERR_ALIGN
            assert f(ctypes.byref(h), 256, 256, code, 256, 256, gran, 10, 24, 8,
                     128) == _lib.PGD_ERR_SHAPE
    # int8 pages need scales too: the plain create refuses the dtype
    assert lib.paged_kv_pool_create(ctypes.byref(h), 256, 256, 10, 16, 8, 128,
                                    _lib.PGD_INT8) == _lib.PGD_ERR_ARG
    assert h.value is None


def test_binding_checks_decode_arguments_before_the_library():
    """The Python face rejects malformed tensors before any call into the
    library: wrong ranks, dtypes, shapes, then anything not a contiguous CUDA
    tensor (checked on CPU tensors here, so that last check is what passes)."""
    import types

    import torch

    import paged_gqa_decode_04_gb300 as pgd

    pool = types.SimpleNamespace(q_dtype=torch.bfloat16, head_dim=128)
    q = torch.zeros(2, 8, 128, dtype=torch.bfloat16)
    bt = torch.zeros(2, 4, dtype=torch.int32)
    sl = torch.zeros(2, dtype=torch.int32)
    check = pgd._check_decode_args
    with pytest.raises(ValueError, match="q must be"):
        check(pool, q.unsqueeze(1), bt, sl, 3)
    with pytest.raises(ValueError, match="q must be"):
        check(pool, q, bt, sl, 4)
    with pytest.raises(TypeError, match="q must be"):
        check(pool, q.float(), bt, sl, 3)
    with pytest.raises(TypeError, match="int32"):
        check(pool, q, bt.long(), sl, 3)
    with pytest.raises(ValueError, match="shape mismatch"):
        check(pool, q[..., :64], bt, sl, 3)
    with pytest.raises(ValueError, match="shape mismatch"):
        check(pool, q, bt[:1], sl, 3)
    with pytest.raises(ValueError, match="CUDA"):
        check(pool, q, bt, sl, 3)
    with pytest.raises(ValueError, match="CUDA"):
        check(pool, q.unsqueeze(1).expand(2, 3, 8, 128), bt, sl, 4)
