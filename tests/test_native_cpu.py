"""CPU-side checks of the C ABI: the library builds, loads, exports every declared
symbol, and rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from asynchronous_expert_execution_gb300 import _native as N
    return N.load()


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(moe_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_exported(lib):
    from asynchronous_expert_execution_gb300 import _native as N
    declared = _declared()
    assert declared, "no declarations found"
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(N.EXPORTS) | (declared - set(N.EXPORTS))
    assert set(N.EXPORTS) <= declared


def test_status_strings(lib):
    for code in range(9):
        assert lib.moe_async_status_string(code)


def test_host_validation_without_gpu(lib):
    from asynchronous_expert_execution_gb300 import _native as N
    # router: bad sizes are rejected on the host
    assert lib.moe_async_route(None, -1, 8, 2, None, None, None) == N.MOE_ERR_INVALID
    assert lib.moe_async_route(None, 4, 8, 9, None, None, None) == N.MOE_ERR_INVALID
    assert lib.moe_async_route(None, 4, 2000, 2, None, None, None) == N.MOE_ERR_INVALID
    assert lib.moe_async_route(None, 0, 8, 2, None, None, None) == N.MOE_OK      # empty: no-op
    # create: invalid configurations never reach CUDA
    out = ctypes.c_void_p()
    bad = [
        dict(hidden=60),             # H not a multiple of 8
        dict(inter=24),              # I not a multiple of 16
        dict(top_k=0),
        dict(top_k=9),               # K > E
        dict(num_experts=2000),
        dict(dtype=5),
        dict(max_slots=0),
    ]
    for over in bad:
        c = dict(num_layers=1, num_experts=8, top_k=2, hidden=64, inter=128, dtype=0, has_shared=0,
                 max_slots=32, bucket_capacity=0, expert_kind=1, trace_capacity=0)
        c.update(over)
        cfg = N.Config(**c)
        assert lib.moe_async_create(ctypes.byref(cfg), None, None, None, None, None, None, None,
                                    ctypes.byref(out)) == N.MOE_ERR_INVALID, over
    # SwiGLU without weights
    cfg = N.Config(1, 8, 2, 64, 128, 0, 0, 32, 0, 0, 0)
    assert lib.moe_async_create(ctypes.byref(cfg), None, None, None, None, None, None, None,
                                ctypes.byref(out)) == N.MOE_ERR_INVALID
    # calls on a null handle
    pol = N.Policy(0, 0, 0, 1)
    assert lib.moe_async_schedule_step(None, 0, ctypes.byref(pol), None) == N.MOE_ERR_INVALID
    assert lib.moe_async_enqueue(None, 0, 1, None, None, None, None, None, None, None, None) == N.MOE_ERR_INVALID
    assert lib.moe_async_destroy(None, None) == N.MOE_ERR_INVALID
    # allocation-free forward: argument and size checks come before any CUDA call
    fwd = lib.moe_async_forward_noalloc
    p = ctypes.c_void_p(256)                   # never dereferenced: every call below returns early
    assert fwd(-1, 8, 2, 64, 128, 1, p, p, p, p, p, p, p, None) == N.MOE_ERR_INVALID
    assert fwd(4, 8, 9, 64, 128, 1, p, p, p, p, p, p, p, None) == N.MOE_ERR_INVALID       # K > E
    assert fwd(4, 8, 2, 64, 128, 7, p, p, p, p, p, p, p, None) == N.MOE_ERR_INVALID       # dtype
    assert fwd(4, 8, 2, 64, 128, 1, None, p, p, p, p, p, p, None) == N.MOE_ERR_INVALID    # no x
    assert fwd(0, 8, 2, 64, 128, 1, None, None, None, None, None, None, None, None) == N.MOE_OK
    # scratch is 16 MiB of fp32 h rows: T * K * I * 4 bytes must fit
    assert fwd(1024, 8, 2, 64, 4096, 1, p, p, p, p, p, p, p, None) == N.MOE_ERR_CAPACITY   # 32 MiB


def test_product_path_has_no_oracle_import():
    """The product package must not import the oracle (tests/bench/smoke only)."""
    pkg = os.path.join(ROOT, "asynchronous_expert_execution_gb300")
    for f in os.listdir(pkg):
        if f.endswith(".py"):
            src = open(os.path.join(pkg, f)).read()
            assert not re.search(r"^\s*(from|import)\s+oracle\b", src, flags=re.M), f


def test_release_build_refuses_raw_record_writes(lib):
    """Only the bounds-checked build accepts raw records; the release library refuses before
    looking at its arguments (no handle, no GPU needed)."""
    from asynchronous_expert_execution_gb300 import _native as N
    assert lib.moe_async_debug_append_record(None, 0, 0, 0, None) == N.MOE_ERR_UNSUPPORTED


def test_bounds_checked_build_exports_every_symbol(lib):
    from asynchronous_expert_execution_gb300 import build as b
    assert os.path.exists(b.LIB_DEBUG), "build() makes the bounds-checked library too"
    dbg = ctypes.CDLL(b.LIB_DEBUG)
    for name in _declared():
        assert hasattr(dbg, name), name
    dbg.moe_async_debug_append_record.restype = ctypes.c_int
    dbg.moe_async_debug_append_record.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                                  ctypes.c_int32, ctypes.c_void_p]
    # the debug build checks its host arguments: no handle -> MOE_ERR_INVALID (not unsupported)
    assert dbg.moe_async_debug_append_record(None, 0, 0, 0, None) == 1
