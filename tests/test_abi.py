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
