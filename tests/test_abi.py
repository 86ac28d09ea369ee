"""The C-ABI library loads and exports every entry point that include/ep.h declares (no GPU needed)."""
import ctypes
import os
import re

import pytest

from combine_get_dispatch_03_gb300 import build as B
from combine_get_dispatch_03_gb300 import ep

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ep.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ep_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def library():
    B.build()
    return ctypes.CDLL(B.LIB)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ep_get_dispatch_layout", "ep_dispatch", "ep_combine", "ep_ll_dispatch", "ep_ll_combine",
                     "ep_handle_create", "ep_handle_destroy", "ep_handle_status"):
        assert required in names


def test_every_declared_symbol_is_exported(library):
    missing = [n for n in declared_functions() if not hasattr(library, n)]
    assert not missing, missing


def test_binding_covers_the_exports():
    assert sorted(ep.EXPORTS) == declared_functions()


def test_host_only_entry_points(library):
    L = ep.lib()
    assert L.ep_ll_msg_bytes(7168, 1) == 16 + 7168 + 4 * 56 == 7408
    assert L.ep_ll_msg_bytes(7168, 0) == 16 + 2 * 7168
    for code in range(9):
        assert L.ep_status_string(code)
    # argument validation happens before any CUDA call
    h = ctypes.c_void_p()
    assert L.ep_handle_create(None, ctypes.byref(h)) == 1
    bad = ep.Config(num_ranks=3, num_max_tokens=4, hidden=128, num_experts=8, num_topk=2).c()
    assert L.ep_handle_create(ctypes.byref(bad), ctypes.byref(h)) == 1
    assert b"multiple of num_ranks" in L.ep_last_error()
    big = ep.Config(num_ranks=64, num_max_tokens=4, hidden=128, num_experts=64, num_topk=2).c()
    assert L.ep_handle_create(ctypes.byref(big), ctypes.byref(h)) == 5
    assert L.ep_dispatch(None, 0, None, 0, None, 0, None, None, None, None, None, None, None, None, None,
                         None, 0, None) == 1
