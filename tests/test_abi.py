"""The C-ABI library loads and exports every symbol include/chain.h declares
(no GPU needed, no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "chain.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "typedef")))


def test_header_declares_entry_points():
    names = declared_symbols()
    for n in ("chain_fwd", "chain_bwd", "chain_bwd_workspace_size", "sp_relayout",
              "sp_relayout_inverse", "chain_check", "chain_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    import chain_gb300
    from chain_gb300 import _build
    path = _build.build()
    lib = ctypes.CDLL(path)
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings():
    import chain_gb300 as cg
    lib = cg.lib()
    for s in (0, -1, -2, -3, -4, -5, -6):
        assert lib.chain_status_string(s)
    assert b"unknown" in lib.chain_status_string(-99)


def _dense_desc(cg, ptr, shape, dtype):
    d = cg.TensorDesc()
    d.ptr = ptr
    d.dtype = dtype
    d.ndim = len(shape)
    st = 1
    for i in reversed(range(len(shape))):
        d.shape[i] = shape[i]
        d.stride[i] = st
        st *= shape[i]
    return d


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="host-side argument check only; never run with a device present")
def test_relayout_refuses_index_overflow():
    # The relayout kernel counts 16-byte vectors in 32 bits with a grid-stride
    # loop that can step up to 2^22 vectors past the end before it stops, so
    # a problem within that distance of 2^32 vectors is refused before any
    # launch.  The descriptors hold dummy addresses: the call must return on
    # the host argument check.
    import chain_gb300 as cg
    lib = cg.lib()
    n_loc = (2 ** 32 - 2 ** 22) // 16  # 128 bf16 = 16 vectors per row
    seq = _dense_desc(cg, 0x10000, (1, n_loc, 1, 128), cg.BF16)
    hm = _dense_desc(cg, 0x20000, (1, n_loc, 128), cg.BF16)
    assert lib.sp_relayout(ctypes.byref(seq), 1, 0, ctypes.byref(hm), None) == cg.ERR_ARG
    assert lib.sp_relayout_inverse(ctypes.byref(hm), 1, 0, ctypes.byref(seq), None) == cg.ERR_ARG
    # the same count over four shards of four heads (one head per group)
    n4 = (2 ** 32 - 2 ** 22) // (4 * 4 * 16)
    seq4 = _dense_desc(cg, 0x10000, (4, n4, 4, 128), cg.BF16)
    hm4 = _dense_desc(cg, 0x20000, (1, 4 * n4, 128), cg.BF16)
    assert lib.sp_relayout(ctypes.byref(seq4), 4, 3, ctypes.byref(hm4), None) == cg.ERR_ARG
