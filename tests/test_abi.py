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


BASE = dict(num_ranks=8, num_max_tokens=64, hidden=1024, num_experts=32, num_topk=4)
BAD_CONFIGS = [  # (change to BASE, expected status, words of the message)
    (dict(num_ranks=0), 5, "num_ranks"),
    (dict(num_ranks=33, num_experts=33), 5, "num_ranks"),
    (dict(num_max_tokens=-1), 1, "num_max_tokens"),
    (dict(hidden=0), 1, "hidden"),
    (dict(hidden=1020), 1, "hidden"),
    (dict(num_experts=12), 1, "multiple of num_ranks"),
    (dict(num_experts=4096), 5, "num_experts"),
    (dict(num_topk=0), 5, "num_topk"),
    (dict(num_topk=33), 5, "num_topk"),
    (dict(num_channels=0), 1, "num_channels"),
    (dict(expert_alignment=0), 1, "expert_alignment"),
    (dict(max_sms=-1), 1, "max_sms"),
    (dict(recv_capacity=-1), 1, "recv_capacity"),
    (dict(recv_capacity=2**31), 1, "recv_capacity"),
    (dict(num_ranks=32, num_experts=32, num_max_tokens=2**27), 5, "num_ranks * num_max_tokens"),
    (dict(num_ranks=1, num_experts=8, num_max_tokens=2**27, num_topk=32), 5, "num_max_tokens * num_topk"),
]


@pytest.mark.parametrize("change,code,words", BAD_CONFIGS, ids=[str(b[0]) for b in BAD_CONFIGS])
def test_config_is_rejected_before_any_cuda_call(library, change, code, words):
    L = ep.lib()
    cfg = ep.Config(**{**BASE, **change}).c()
    h = ctypes.c_void_p()
    assert L.ep_handle_create(ctypes.byref(cfg), ctypes.byref(h)) == code
    assert words.encode() in L.ep_last_error()
    assert not h.value


def _noalloc(L, R=8, T=16, maxT=16, H=1024, E=32, K=4, x=16, idx=8, fp8=0, ue8m0=0, msgs=16, out=16):
    """ep_ll_dispatch_noalloc with fake, suitably aligned addresses (the checks run before any CUDA call)."""
    a = lambda align: None if align is None else 0x10000 + (0 if align >= 16 else align)  # noqa: E731
    return L.ep_ll_dispatch_noalloc(R, T, maxT, H, E, K, a(x), a(idx), fp8, 0, ue8m0, a(msgs), a(out), a(out),
                                    None, a(out), a(out), None)


NOALLOC_BAD = [
    (dict(R=0), 5, "num_ranks"),
    (dict(E=30), 1, "multiple of num_ranks"),
    (dict(R=16, E=2048), 5, "count scratch"),
    (dict(K=0), 5, "num_topk"),
    (dict(T=17), 1, "num_tokens"),
    (dict(H=1020), 1, "hidden"),
    (dict(ue8m0=1), 1, "use_ue8m0"),
    (dict(fp8=1, H=1024 + 128), 5, "hidden % 512"),
    (dict(x=8), 1, "x"),
    (dict(idx=4), 1, "topk_idx"),
    (dict(x=None), 1, "x"),
    (dict(msgs=8), 1, "output pointer"),
    (dict(out=None), 1, "output pointer"),
]


@pytest.mark.parametrize("kw,code,words", NOALLOC_BAD, ids=[str(b[0]) for b in NOALLOC_BAD])
def test_noalloc_arguments_are_rejected_before_any_cuda_call(library, kw, code, words):
    L = ep.lib()
    assert _noalloc(L, **kw) == code
    assert words.encode() in L.ep_last_error()
