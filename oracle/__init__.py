"""CPU oracle for the expert-parallel layout / dispatch / combine path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library: the arithmetic lives in ``ep_oracle.c`` (plain C,
single-threaded, built with ``-ffp-contract=off``) and this module only
marshals numpy arrays into it.  Each wrapper names the definition it follows;
the C file carries the page citations.

Array conventions (all C-contiguous numpy arrays):
  bf16 values travel as ``np.uint16`` bit patterns, FP8 e4m3 as ``np.uint8``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libep_oracle.so")

OK = 0
CAPACITY = 1
BAD_ARG = -1
BAD_EXPERT = -2
INCONSISTENT = -3

_lib = None


def build(force: bool = False) -> str:
    """Compile ep_oracle.c into libep_oracle.so next to it (gcc, portable C)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    L = ctypes.c_int64
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_e4m3.restype = ctypes.c_uint8
    lib.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_f32.restype = ctypes.c_float
    lib.oracle_fp8_quantize_group.argtypes = [P, I, I, P, P, P]
    lib.oracle_fp8_quantize_group.restype = None
    lib.oracle_get_dispatch_layout.argtypes = [I, I, I, I, P, P, P, P, P, P]
    lib.oracle_dispatch_notify.argtypes = [I, I, I, I, I, L, P, P, P, P, P, P, P, P, P, P]
    lib.oracle_rdma_prefix.argtypes = [I, I, I, P, P, P]
    lib.oracle_dispatch.argtypes = [I, I, I, I, I, L, I, P, P, P, P, P, P, L, P, P, P, P]
    lib.oracle_combine.argtypes = [I, I, I, I, L, P, P, P, P, P, I, P, L, P, P]
    lib.oracle_ll_msg_bytes.argtypes = [I, I]
    lib.oracle_ll_msg_bytes.restype = L
    lib.oracle_ll_dispatch.argtypes = [I, I, I, I, I, I, P, P, P, I, I, I, P, P, P, P]
    lib.oracle_ll_combine.argtypes = [I, I, I, I, I, I, P, P, P, P, P, L, P]
    for name in ("oracle_get_dispatch_layout", "oracle_dispatch_notify", "oracle_rdma_prefix", "oracle_dispatch",
                 "oracle_combine", "oracle_ll_dispatch", "oracle_ll_combine"):
        getattr(lib, name).restype = I
    return lib


class use_library:
    """Run the wrappers against another build of the oracle source (the mutation tests plant a
    mistake in a copy of ep_oracle.c and check that the pins catch it)."""

    def __init__(self, path):
        self.lib = _bind(ctypes.CDLL(path))

    def __enter__(self):
        global _lib
        self.saved = _load()
        _lib = self.lib
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc, name):
    if rc < 0 and rc != INCONSISTENT:
        raise ValueError(f"{name}: oracle rejected the input (code {rc})")
    return rc


# ---------------------------------------------------------------- formats

def bf16_to_f32(b: int) -> float:
    return _load().oracle_bf16_to_f32(b)


def f32_to_bf16(f: float) -> int:
    return _load().oracle_f32_to_bf16(f)


def f32_to_e4m3(f: float) -> int:
    return _load().oracle_f32_to_e4m3(f)


def e4m3_to_f32(c: int) -> float:
    return _load().oracle_e4m3_to_f32(c)


def f32_to_e4m3_array(v: np.ndarray) -> np.ndarray:
    """Element-wise e4m3 encoding of a float32 array (loops over the C encoder)."""
    lib = _load()
    flat = np.ascontiguousarray(v, dtype=np.float32).ravel()
    return np.fromiter((lib.oracle_f32_to_e4m3(float(f)) for f in flat), dtype=np.uint8,
                       count=flat.size).reshape(np.shape(v))


def fp8_quantize_group(x_bits: np.ndarray, round_scale: bool = False):
    """One group of bf16 bits -> (e4m3 codes, scale, exponent)."""
    x = _c(x_bits, np.uint16)
    q = np.zeros(x.size, np.uint8)
    sc = np.zeros(1, np.float32)
    ex = np.zeros(1, np.int32)
    _load().oracle_fp8_quantize_group(_p(x), x.size, int(round_scale), _p(q), _p(sc), _p(ex))
    return q, float(sc[0]), int(ex[0])


# ---------------------------------------------------------------- layout

def get_dispatch_layout(topk_idx: np.ndarray, num_experts: int, with_rdma: bool = True, rank_mask=None):
    """get_dispatch_layout: counts per rank / RDMA node / expert and is_token_in_rank.
    rank_mask: optional [R] ints, nonzero = the rank neither sends nor receives."""
    R, T, K = topk_idx.shape
    idx = _c(topk_idx, np.int64)
    mask = _c(rank_mask, np.int32)
    tpr = np.zeros((R, R), np.int32)
    tprdma = np.zeros((R, (R + 7) // 8), np.int32) if with_rdma else None
    tpe = np.zeros((R, num_experts), np.int32)
    itr = np.zeros((R, T, R), np.uint8)
    _check(_load().oracle_get_dispatch_layout(R, T, K, num_experts, _p(idx), _p(mask), _p(tpr), _p(tprdma),
                                              _p(tpe), _p(itr)), "get_dispatch_layout")
    return dict(num_tokens_per_rank=tpr, num_tokens_per_rdma_rank=tprdma,
                num_tokens_per_expert=tpe, is_token_in_rank=itr)


def dispatch_notify(num_tokens_per_rank, is_token_in_rank, num_tokens_per_expert,
                    num_channels: int, expert_alignment: int, capacity: int):
    """Prefix matrices, receive rows (send_head, recv_src_idx), aligned per-expert counts."""
    R, T, _ = is_token_in_rank.shape
    E = num_tokens_per_expert.shape[1]
    C = num_channels
    tpr = _c(num_tokens_per_rank, np.int32)
    itr = _c(is_token_in_rank, np.uint8)
    tpe = _c(num_tokens_per_expert, np.int32)
    out = dict(
        rank_prefix_matrix=np.zeros((R, R), np.int32),
        channel_prefix_matrix=np.zeros((R, R, C), np.int32),
        recv_channel_prefix_matrix=np.zeros((R, R, C), np.int32),
        num_recv=np.zeros(R, np.int32),
        send_head=np.zeros((R, T, R), np.int32),
        recv_src_idx=np.full((R, capacity), -1, np.int32),
        num_recv_tokens_per_expert=np.zeros((R, E // R), np.int32),
    )
    rc = _check(_load().oracle_dispatch_notify(
        R, T, E, C, expert_alignment, capacity, _p(tpr), _p(itr), _p(tpe),
        _p(out["rank_prefix_matrix"]), _p(out["channel_prefix_matrix"]),
        _p(out["recv_channel_prefix_matrix"]), _p(out["num_recv"]), _p(out["send_head"]),
        _p(out["recv_src_idx"]), _p(out["num_recv_tokens_per_expert"])), "dispatch_notify")
    out["status"] = rc
    return out


def rdma_prefix(is_token_in_rank, num_channels: int):
    """Node-level record of whole nodes of 8 ranks (R > 8, R % 8 == 0): RDMA channel prefix
    [R][NN][C] and, per receiving rank, the RDMA rank prefix [R][NN]."""
    R, T, _ = is_token_in_rank.shape
    NN = R // 8
    out = dict(rdma_channel_prefix_matrix=np.zeros((R, NN, num_channels), np.int32),
               recv_rdma_rank_prefix_sum=np.zeros((R, NN), np.int32))
    _check(_load().oracle_rdma_prefix(R, T, num_channels, _p(_c(is_token_in_rank, np.uint8)),
                                      _p(out["rdma_channel_prefix_matrix"]), _p(out["recv_rdma_rank_prefix_sum"])),
           "rdma_prefix")
    return out


MODE_BF16, MODE_CAST_FP8, MODE_FP8_IN = 0, 1, 2


def dispatch(x, send_head, capacity: int, num_experts: int, mode: int = MODE_BF16,
             x_scales=None, topk_idx=None, topk_weights=None, tokens=None, out=None):
    """Normal dispatch of every (listed) token to its receive rows.

    x: [R][T][H] uint16 (bf16 bits) for modes 0/1, uint8 (e4m3) for mode 2.
    tokens: optional flat token ids s*T+t; only their rows are written.
    out: optional dict of preallocated outputs (recv_x, recv_x_scales,
    recv_topk_idx, recv_topk_weights) -- large ones may be lazily-zeroed.
    """
    R, T, H = x.shape
    K = topk_idx.shape[2] if topk_idx is not None else 1
    G = H // 128
    pay = np.uint16 if mode == MODE_BF16 else np.uint8
    out = dict(out or {})
    out.setdefault("recv_x", np.zeros((R, capacity, H), pay))
    if mode != MODE_BF16:
        out.setdefault("recv_x_scales", np.zeros((R, capacity, G), np.float32))
    if topk_idx is not None:
        out.setdefault("recv_topk_idx", np.full((R, capacity, K), -2, np.int64))
        if topk_weights is not None:
            out.setdefault("recv_topk_weights", np.full((R, capacity, K), np.nan, np.float32))
    xs = _c(x, np.uint8 if mode == MODE_FP8_IN else np.uint16)
    tok = _c(tokens, np.int64)
    _check(_load().oracle_dispatch(
        R, T, H, K, num_experts, capacity, mode, _p(xs), _p(_c(x_scales, np.float32)),
        _p(_c(topk_idx, np.int64)), _p(_c(topk_weights, np.float32)), _p(_c(send_head, np.int32)),
        _p(tok), 0 if tok is None else tok.size,
        _p(out["recv_x"]), _p(out.get("recv_x_scales")), _p(out.get("recv_topk_idx")),
        _p(out.get("recv_topk_weights"))), "dispatch")
    return out


def combine(y, send_head, recv_topk_weights=None, bias0=None, bias1=None, out_fp32=False,
            tokens=None, num_topk: int = 1, out=None):
    """Normal combine: fp32 sum of every receiving rank's row (+ biases).
    out: optional dict of preallocated outputs (out, combined_topk_weights) that the listed
    tokens' rows are written into."""
    R, cap, H = y.shape
    T = send_head.shape[1]
    K = recv_topk_weights.shape[2] if recv_topk_weights is not None else num_topk
    pre = out or {}
    out = pre.get("out")
    if out is None:
        out = np.zeros((R, T, H), np.float32 if out_fp32 else np.uint16)
    if out.shape != (R, T, H) or out.dtype != (np.float32 if out_fp32 else np.uint16) or not out.flags.c_contiguous:
        raise ValueError("out['out'] does not match the combine output")
    cw = pre.get("combined_topk_weights")
    if cw is None and recv_topk_weights is not None:
        cw = np.zeros((R, T, K), np.float32)
    if cw is not None and (cw.shape != (R, T, K) or cw.dtype != np.float32 or not cw.flags.c_contiguous):
        raise ValueError("out['combined_topk_weights'] does not match the weight output")
    tok = _c(tokens, np.int64)
    _check(_load().oracle_combine(
        R, T, H, K, cap, _p(_c(send_head, np.int32)), _p(_c(y, np.uint16)),
        _p(_c(recv_topk_weights, np.float32)), _p(_c(bias0, np.uint16)), _p(_c(bias1, np.uint16)),
        int(out_fp32), _p(tok), 0 if tok is None else tok.size, _p(out), _p(cw)), "combine")
    return dict(out=out, combined_topk_weights=cw)


def ll_msg_bytes(hidden: int, use_fp8: bool) -> int:
    return int(_load().oracle_ll_msg_bytes(hidden, int(use_fp8)))


def ll_dispatch(x, topk_idx, num_max_tokens: int, num_experts: int, use_fp8=True,
                round_scale=False, use_ue8m0=False, rank_mask=None):
    """Low-latency dispatch: one message per valid (token, slot), packed per local expert.
    rank_mask: optional [R] ints, nonzero = the rank neither sends nor receives."""
    R, T, H = x.shape
    K = topk_idx.shape[2]
    EL = num_experts // R
    msg = ll_msg_bytes(H, use_fp8)
    out = dict(
        msgs_by_slot=np.zeros((R, T, K, msg), np.uint8),
        slot_row=np.zeros((R, T, K), np.int32),
        packed_recv_count=np.zeros((R, EL), np.int32),
        packed_recv_layout_range=np.zeros((R, EL, R), np.int64),
    )
    rc = _check(_load().oracle_ll_dispatch(
        R, T, num_max_tokens, H, K, num_experts, _p(_c(x, np.uint16)), _p(_c(topk_idx, np.int64)),
        _p(_c(rank_mask, np.int32)), int(use_fp8), int(round_scale), int(use_ue8m0), _p(out["msgs_by_slot"]),
        _p(out["slot_row"]),
        _p(out["packed_recv_count"]), _p(out["packed_recv_layout_range"])), "ll_dispatch")
    out["status"] = rc
    return out


def ll_combine(y, topk_idx, topk_weights, slot_row, num_max_tokens: int, num_experts: int,
               tokens=None):
    """Low-latency combine: top-k weighted fp32 FMA chain, bf16 out."""
    R, T, K = topk_idx.shape
    H = y.shape[-1]
    out = np.zeros((R, T, H), np.uint16)
    tok = _c(tokens, np.int64)
    _check(_load().oracle_ll_combine(
        R, T, num_max_tokens, H, K, num_experts, _p(_c(y, np.uint16)), _p(_c(topk_idx, np.int64)),
        _p(_c(topk_weights, np.float32)), _p(_c(slot_row, np.int32)), _p(tok),
        0 if tok is None else tok.size, _p(out)), "ll_combine")
    return out
