"""Python binding of the EP C ABI (include/ep.h).

Argument marshalling only: every function checks shapes, dtypes, devices and
contiguity of the torch tensors it is given against the handle's sizes,
allocates missing outputs with torch, and passes raw device pointers and the
current CUDA stream to libep_gb300.so.  All computation happens in the
library's kernels.  The library must be built (``__graft_entry__.build()``);
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

from . import build as _build

EP_OK = 0
STATUS_NAMES = {0: "EP_OK", 1: "EP_ERR_INVALID_ARG", 2: "EP_ERR_CAPACITY", 3: "EP_ERR_TIMEOUT",
                4: "EP_ERR_CUDA", 5: "EP_ERR_UNSUPPORTED", 6: "EP_ERR_INCONSISTENT",
                7: "EP_ERR_BAD_EXPERT", 8: "EP_ERR_STATE"}
EP_BF16, EP_FP8_E4M3, EP_FP32 = 0, 1, 2
EP_DISPATCH_FRESH, EP_DISPATCH_CACHED, EP_DISPATCH_PREPARED = 0, 1, 2
FIELDS = {"rank_prefix_matrix": 0, "channel_prefix_matrix": 1, "recv_channel_prefix_matrix": 2,
          "recv_src_idx": 3, "send_head": 4, "num_recv": 5, "ll_slot_row": 6,
          "rdma_channel_prefix_matrix": 7, "recv_rdma_rank_prefix_sum": 8}


class EPError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class ep_config(ctypes.Structure):
    _fields_ = [("num_ranks", ctypes.c_int32), ("num_max_tokens", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("num_topk", ctypes.c_int32), ("num_channels", ctypes.c_int32),
                ("expert_alignment", ctypes.c_int32), ("max_sms", ctypes.c_int32),
                ("recv_capacity", ctypes.c_int64)]


class ep_sm_model(ctypes.Structure):
    _fields_ = [("hbm_gbs", ctypes.c_double), ("sm_read_gbs", ctypes.c_double), ("sm_write_gbs", ctypes.c_double),
                ("num_device_sms", ctypes.c_int32), ("prefer_overlap_with_compute", ctypes.c_int32)]


_lib = None
EXPORTS = ("ep_handle_create", "ep_handle_destroy", "ep_handle_status", "ep_handle_num_recv",
           "ep_handle_field_bytes", "ep_handle_export", "ep_status_string", "ep_last_error",
           "ep_get_dispatch_layout", "ep_dispatch", "ep_combine", "ep_ll_msg_bytes", "ep_ll_dispatch",
           "ep_ll_combine", "ep_ll_dispatch_noalloc", "ep_notify_dispatch", "ep_update_mask_buffer",
           "ep_query_mask_buffer", "ep_clean_mask_buffer", "ep_selftest_bounded_wait", "ep_ll_combine_strided",
           "ep_expected_topk", "ep_theoretical_num_sms", "ep_layout_notify")


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(path)
        P, I32, I64, S = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int
        L.ep_handle_create.argtypes = [ctypes.POINTER(ep_config), ctypes.POINTER(ctypes.c_void_p)]
        L.ep_handle_destroy.argtypes = [P]
        L.ep_handle_destroy.restype = None
        L.ep_handle_status.argtypes = [P, P, I32]
        L.ep_handle_num_recv.argtypes = [P, P, P]
        L.ep_handle_field_bytes.argtypes = [P, S]
        L.ep_handle_field_bytes.restype = ctypes.c_size_t
        L.ep_handle_export.argtypes = [P, S, P, ctypes.c_size_t, P]
        L.ep_status_string.argtypes = [S]
        L.ep_status_string.restype = ctypes.c_char_p
        L.ep_last_error.argtypes = []
        L.ep_last_error.restype = ctypes.c_char_p
        L.ep_get_dispatch_layout.argtypes = [P, I32, P, P, P, P, P, P]
        L.ep_dispatch.argtypes = [P, I32, P, S, P, I32, P, P, P, P, P, P, P, P, P, P, I32, P]
        L.ep_combine.argtypes = [P, P, P, P, P, P, S, P, P]
        L.ep_ll_msg_bytes.argtypes = [I32, I32]
        L.ep_ll_msg_bytes.restype = I64
        L.ep_ll_dispatch.argtypes = [P, I32, P, P, I32, I32, I32, P, P, P, P, P]
        L.ep_ll_combine.argtypes = [P, P, P, P, P, P]
        L.ep_ll_combine_strided.argtypes = [P, P, I64, P, P, P, P]
        L.ep_expected_topk.argtypes = [I32, I32, I32]
        L.ep_expected_topk.restype = ctypes.c_double
        L.ep_theoretical_num_sms.argtypes = [ctypes.POINTER(ep_sm_model), I32, I32, I32, I32]
        L.ep_theoretical_num_sms.restype = I32
        L.ep_notify_dispatch.argtypes = [P, I32, P, P, P, P, P]
        L.ep_layout_notify.argtypes = [P, I32, P, P, P, P, P, P, P]
        L.ep_update_mask_buffer.argtypes = [P, I32, I32, P]
        L.ep_query_mask_buffer.argtypes = [P, P, P]
        L.ep_clean_mask_buffer.argtypes = [P, P]
        L.ep_selftest_bounded_wait.argtypes = [P, ctypes.c_uint32, I32, P]
        L.ep_ll_dispatch_noalloc.argtypes = [I32, I32, I32, I32, I32, I32, P, P, I32, I32, I32, P, P, P, P, P, P,
                                             P]
        for name in ("ep_handle_create", "ep_handle_status", "ep_handle_num_recv", "ep_handle_export",
                     "ep_get_dispatch_layout", "ep_dispatch", "ep_combine", "ep_ll_dispatch", "ep_ll_combine",
                     "ep_ll_dispatch_noalloc", "ep_notify_dispatch", "ep_update_mask_buffer",
                     "ep_query_mask_buffer", "ep_clean_mask_buffer", "ep_selftest_bounded_wait",
                     "ep_ll_combine_strided", "ep_layout_notify"):
            getattr(L, name).restype = S
        _lib = L
    return _lib


def _raise(rc: int):
    if rc != EP_OK:
        raise EPError(rc, lib().ep_last_error().decode(errors="replace"))


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device):
    """The raw stream handle (an int): `stream`, else the current stream of the handle's device."""
    if stream is None:
        if _raw_stream is not None:  # the current stream's handle without building a Stream object
            return _raw_stream(device.index)
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _ptr(t, name, dtype=None, shape=None, device=None):
    """The device address of a checked tensor (an int; every pointer argument is declared void*)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if shape is not None and t.shape != shape:  # torch.Size compares equal to a tuple
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the handle lives on {device}")
    return t.data_ptr() if t.numel() else _dummy(device).data_ptr()


_dummies = {}


def _dummy(device):
    """A 16-byte aligned device word for zero-sized tensors (their data_ptr may be 0)."""
    if device not in _dummies:
        _dummies[device] = torch.zeros(4, dtype=torch.int32, device=device)
    return _dummies[device]


@dataclasses.dataclass
class Config:
    num_ranks: int
    num_max_tokens: int
    hidden: int
    num_experts: int
    num_topk: int
    num_channels: int = 12
    expert_alignment: int = 1
    recv_capacity: int = 0
    max_sms: int = 0  # 0: fill the GPU; n: at most n SMs' worth of CTAs resident (ep_theoretical_num_sms)

    @property
    def num_nodes(self) -> int:
        """Nodes of 8 ranks in the two-level layout."""
        return (self.num_ranks + 7) // 8

    @property
    def num_local_experts(self) -> int:
        return self.num_experts // self.num_ranks

    def c(self) -> ep_config:
        return ep_config(self.num_ranks, self.num_max_tokens, self.hidden, self.num_experts, self.num_topk,
                         self.num_channels, self.expert_alignment, self.max_sms, self.recv_capacity)


class Handle:
    """Owns an ep_handle* (the Buffer of the pages): sizes, dispatch record, status word."""

    def __init__(self, cfg: Config, device=None):
        self.cfg = cfg
        d = torch.device("cuda") if device is None else torch.device(device)
        if d.type == "cuda" and d.index is None:  # "cuda" means the current device
            d = torch.device("cuda", torch.cuda.current_device())
        self.device = d
        self._ptr = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _raise(lib().ep_handle_create(ctypes.byref(cfg.c()), ctypes.byref(self._ptr)))
        self.normal_tokens = None
        self.ll_tokens = None

    @property
    def ptr(self):
        if not self._ptr:
            raise RuntimeError("handle was destroyed")
        return self._ptr

    def destroy(self):
        if self._ptr:
            lib().ep_handle_destroy(self._ptr)
            self._ptr = ctypes.c_void_p()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.destroy()

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    def status(self, reset: bool = True, stream=None) -> int:
        """Synchronise and return the first device-detected error code (0 = none)."""
        return lib().ep_handle_status(self.ptr, _stream(stream, self.device), int(reset))

    def check(self, stream=None):
        _raise(self.status(True, stream))

    def num_recv(self, stream=None) -> torch.Tensor:
        out = torch.zeros(self.cfg.num_ranks, dtype=torch.int32)
        _raise(lib().ep_handle_num_recv(self.ptr, ctypes.c_void_p(out.data_ptr()),
                                        _stream(stream, self.device)))
        return out

    def export(self, field: str, stream=None) -> torch.Tensor:
        """Device copy of one array of the dispatch record."""
        c = self.cfg
        shapes = {"rank_prefix_matrix": (c.num_ranks, c.num_ranks),
                  "channel_prefix_matrix": (c.num_ranks, c.num_ranks, c.num_channels),
                  "recv_channel_prefix_matrix": (c.num_ranks, c.num_ranks, c.num_channels),
                  "recv_src_idx": (c.num_ranks, c.recv_capacity),
                  "send_head": (c.num_ranks, c.num_max_tokens, c.num_ranks),
                  "num_recv": (c.num_ranks,),
                  "ll_slot_row": (c.num_ranks, c.num_max_tokens, c.num_topk),
                  "rdma_channel_prefix_matrix": (c.num_ranks, c.num_nodes, c.num_channels),
                  "recv_rdma_rank_prefix_sum": (c.num_ranks, c.num_nodes)}
        out = torch.empty(shapes[field], dtype=torch.int32, device=self.device)
        nbytes = lib().ep_handle_field_bytes(self.ptr, FIELDS[field])
        if field.startswith(("rdma_", "recv_rdma_")) and nbytes == 0:
            nbytes = out.numel() * 4  # the call below reports that the record needs whole nodes
        assert nbytes == out.numel() * 4
        if nbytes:
            _raise(lib().ep_handle_export(self.ptr, FIELDS[field], ctypes.c_void_p(out.data_ptr()), nbytes,
                                          _stream(stream, self.device)))
        if field == "send_head":
            # rows are packed for the T of the last fresh dispatch: [R][T][R]
            T = self.normal_tokens or 0
            out = out.view(-1)[:c.num_ranks * T * c.num_ranks].view(c.num_ranks, T, c.num_ranks)
        return out


def ep_update_mask_buffer(h: Handle, rank: int, masked: bool = True, stream=None):
    _raise(lib().ep_update_mask_buffer(h.ptr, rank, int(bool(masked)), _stream(stream, h.device)))


def ep_query_mask_buffer(h: Handle, stream=None) -> torch.Tensor:
    out = torch.zeros(h.cfg.num_ranks, dtype=torch.int32)
    _raise(lib().ep_query_mask_buffer(h.ptr, ctypes.c_void_p(out.data_ptr()), _stream(stream, h.device)))
    return out


def ep_clean_mask_buffer(h: Handle, stream=None):
    _raise(lib().ep_clean_mask_buffer(h.ptr, _stream(stream, h.device)))


def ep_selftest_bounded_wait(h: Handle, max_iterations: int, rank: int, stream=None):
    _raise(lib().ep_selftest_bounded_wait(h.ptr, max_iterations, rank, _stream(stream, h.device)))


def ep_handle_create(cfg: Config, device=None) -> Handle:
    return Handle(cfg, device)


def ep_ll_msg_bytes(hidden: int, use_fp8: bool) -> int:
    return int(lib().ep_ll_msg_bytes(hidden, int(bool(use_fp8))))


def _empty(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


def ep_get_dispatch_layout(h: Handle, topk_idx: torch.Tensor, num_tokens_per_rank=None,
                           num_tokens_per_rdma_rank=None, num_tokens_per_expert=None, is_token_in_rank=None,
                           with_rdma: bool | None = None, stream=None):
    """Layout of a routing: counts per rank / RDMA node / expert and is_token_in_rank."""
    c, d = h.cfg, h.device
    R, E = c.num_ranks, c.num_experts
    if topk_idx.dim() != 3 or topk_idx.shape[0] != R or topk_idx.shape[2] != c.num_topk:
        raise ValueError(f"topk_idx must be [R={R}][T][K={c.num_topk}], got {tuple(topk_idx.shape)}")
    T = topk_idx.shape[1]
    if with_rdma is None:
        with_rdma = R > 8
    nn = (R + 7) // 8
    tpr = num_tokens_per_rank if num_tokens_per_rank is not None else _empty((R, R), torch.int32, d)
    tpe = num_tokens_per_expert if num_tokens_per_expert is not None else _empty((R, E), torch.int32, d)
    itr = is_token_in_rank if is_token_in_rank is not None else _empty((R, T, R), torch.bool, d)
    tprdma = num_tokens_per_rdma_rank
    if tprdma is None and with_rdma:
        tprdma = _empty((R, nn), torch.int32, d)
    _raise(lib().ep_get_dispatch_layout(
        h.ptr, T, _ptr(topk_idx, "topk_idx", torch.int64, (R, T, c.num_topk), d),
        _ptr(tpr, "num_tokens_per_rank", torch.int32, (R, R), d),
        _ptr(tprdma, "num_tokens_per_rdma_rank", torch.int32, (R, nn), d),
        _ptr(tpe, "num_tokens_per_expert", torch.int32, (R, E), d),
        _ptr(itr, "is_token_in_rank", None, (R, T, R), d), _stream(stream, h.device)))
    if itr.dtype not in (torch.bool, torch.uint8):
        raise TypeError("is_token_in_rank must be bool or uint8")
    return dict(num_tokens_per_rank=tpr, num_tokens_per_rdma_rank=tprdma, num_tokens_per_expert=tpe,
                is_token_in_rank=itr)


def ep_notify_dispatch(h: Handle, num_tokens_per_rank, is_token_in_rank, num_tokens_per_expert,
                       num_recv_tokens_per_expert=None, stream=None):
    """Build the dispatch record (notify step); follow with ep_dispatch(..., prepared=True)."""
    c, d = h.cfg, h.device
    R = c.num_ranks
    T = is_token_in_rank.shape[1]
    if is_token_in_rank.dtype not in (torch.bool, torch.uint8):
        raise TypeError("is_token_in_rank must be bool or uint8")
    if num_recv_tokens_per_expert is None:
        num_recv_tokens_per_expert = _empty((R, c.num_local_experts), torch.int32, d)
    _raise(lib().ep_notify_dispatch(
        h.ptr, T, _ptr(num_tokens_per_rank, "num_tokens_per_rank", torch.int32, (R, R), d),
        _ptr(is_token_in_rank, "is_token_in_rank", None, (R, T, R), d),
        _ptr(num_tokens_per_expert, "num_tokens_per_expert", torch.int32, (R, c.num_experts), d),
        _ptr(num_recv_tokens_per_expert, "num_recv_tokens_per_expert", torch.int32, (R, c.num_local_experts), d),
        _stream(stream, h.device)))
    h.normal_tokens = T
    return num_recv_tokens_per_expert


def ep_layout_notify(h: Handle, topk_idx: torch.Tensor, num_tokens_per_rank=None, num_tokens_per_rdma_rank=None,
                     num_tokens_per_expert=None, is_token_in_rank=None, num_recv_tokens_per_expert=None,
                     with_rdma: bool | None = None, stream=None):
    """Layout and the dispatch record in one launch; follow with ep_dispatch(..., prepared=True)."""
    c, d = h.cfg, h.device
    R, E = c.num_ranks, c.num_experts
    if topk_idx.dim() != 3 or topk_idx.shape[0] != R or topk_idx.shape[2] != c.num_topk:
        raise ValueError(f"topk_idx must be [R={R}][T][K={c.num_topk}], got {tuple(topk_idx.shape)}")
    T = topk_idx.shape[1]
    if with_rdma is None:
        with_rdma = R > 8
    nn = (R + 7) // 8
    tpr = num_tokens_per_rank if num_tokens_per_rank is not None else _empty((R, R), torch.int32, d)
    tpe = num_tokens_per_expert if num_tokens_per_expert is not None else _empty((R, E), torch.int32, d)
    itr = is_token_in_rank if is_token_in_rank is not None else _empty((R, T, R), torch.bool, d)
    if itr.dtype not in (torch.bool, torch.uint8):
        raise TypeError("is_token_in_rank must be bool or uint8")
    tprdma = num_tokens_per_rdma_rank
    if tprdma is None and with_rdma:
        tprdma = _empty((R, nn), torch.int32, d)
    nrpe = num_recv_tokens_per_expert
    if nrpe is None:
        nrpe = _empty((R, c.num_local_experts), torch.int32, d)
    _raise(lib().ep_layout_notify(
        h.ptr, T, _ptr(topk_idx, "topk_idx", torch.int64, (R, T, c.num_topk), d),
        _ptr(tpr, "num_tokens_per_rank", torch.int32, (R, R), d),
        _ptr(tprdma, "num_tokens_per_rdma_rank", torch.int32, (R, nn), d),
        _ptr(tpe, "num_tokens_per_expert", torch.int32, (R, E), d),
        _ptr(itr, "is_token_in_rank", None, (R, T, R), d),
        _ptr(nrpe, "num_recv_tokens_per_expert", torch.int32, (R, c.num_local_experts), d),
        _stream(stream, h.device)))
    h.normal_tokens = T
    return dict(num_tokens_per_rank=tpr, num_tokens_per_rdma_rank=tprdma, num_tokens_per_expert=tpe,
                is_token_in_rank=itr, num_recv_tokens_per_expert=nrpe)


def ep_dispatch(h: Handle, x: torch.Tensor, topk_idx=None, topk_weights=None, num_tokens_per_rank=None,
                is_token_in_rank=None, num_tokens_per_expert=None, x_scales=None, cast_to_fp8: bool = False,
                cached: bool = False, recv_x=None, recv_x_scales=None, recv_topk_idx=None, recv_topk_weights=None,
                num_recv_tokens_per_expert=None, with_topk: bool = True, prepared: bool = False, stream=None):
    """Normal-mode dispatch into [R][cap][...] receive buffers (fresh, cached or prepared record)."""
    c, d = h.cfg, h.device
    R, H, K, cap = c.num_ranks, c.hidden, c.num_topk, c.recv_capacity
    T = x.shape[1]
    G = H // 128
    fp8_in = x.dtype == torch.float8_e4m3fn
    if fp8_in:
        _ptr(x, "x", torch.float8_e4m3fn, (R, T, H), d)
    else:
        _ptr(x, "x", torch.bfloat16, (R, T, H), d)
    fp8_out = fp8_in or cast_to_fp8
    if recv_x is None:
        recv_x = _empty((R, cap, H), torch.float8_e4m3fn if fp8_out else torch.bfloat16, d)
    if fp8_out and recv_x_scales is None:
        recv_x_scales = _empty((R, cap, G), torch.float32, d)
    mode = EP_DISPATCH_CACHED if cached else (EP_DISPATCH_PREPARED if prepared else EP_DISPATCH_FRESH)
    if not cached:
        if with_topk and topk_idx is not None:
            if recv_topk_idx is None:
                recv_topk_idx = _empty((R, cap, K), torch.int64, d)
            if topk_weights is not None and recv_topk_weights is None:
                recv_topk_weights = _empty((R, cap, K), torch.float32, d)
        if num_recv_tokens_per_expert is None and not prepared:
            num_recv_tokens_per_expert = _empty((R, c.num_local_experts), torch.int32, d)
    itr_ptr = None
    if is_token_in_rank is not None:
        if is_token_in_rank.dtype not in (torch.bool, torch.uint8):
            raise TypeError("is_token_in_rank must be bool or uint8")
        itr_ptr = _ptr(is_token_in_rank, "is_token_in_rank", None, (R, T, R), d)
    _raise(lib().ep_dispatch(
        h.ptr, T, _ptr(x, "x", None, None, d), EP_FP8_E4M3 if fp8_in else EP_BF16,
        _ptr(x_scales, "x_scales", torch.float32, (R, T, G), d), int(bool(cast_to_fp8)),
        _ptr(topk_idx, "topk_idx", torch.int64, (R, T, K), d),
        _ptr(topk_weights, "topk_weights", torch.float32, (R, T, K), d),
        _ptr(num_tokens_per_rank, "num_tokens_per_rank", torch.int32, (R, R), d), itr_ptr,
        _ptr(num_tokens_per_expert, "num_tokens_per_expert", torch.int32, (R, c.num_experts), d),
        _ptr(recv_x, "recv_x", torch.float8_e4m3fn if fp8_out else torch.bfloat16, (R, cap, H), d),
        _ptr(recv_x_scales, "recv_x_scales", torch.float32, (R, cap, G), d),
        _ptr(recv_topk_idx, "recv_topk_idx", torch.int64, (R, cap, K), d),
        _ptr(recv_topk_weights, "recv_topk_weights", torch.float32, (R, cap, K), d),
        _ptr(num_recv_tokens_per_expert, "num_recv_tokens_per_expert", torch.int32, (R, c.num_local_experts), d),
        mode, _stream(stream, h.device)))
    if mode == EP_DISPATCH_FRESH:
        h.normal_tokens = T
    return dict(recv_x=recv_x, recv_x_scales=recv_x_scales, recv_topk_idx=recv_topk_idx,
                recv_topk_weights=recv_topk_weights, num_recv_tokens_per_expert=num_recv_tokens_per_expert)


def ep_combine(h: Handle, x: torch.Tensor, topk_weights=None, bias_0=None, bias_1=None,
               out_dtype=torch.bfloat16, combined_x=None, combined_topk_weights=None, stream=None):
    """Normal-mode combine: fp32 sum of the received rows (+ biases) back in source order."""
    c, d = h.cfg, h.device
    R, H, K, cap = c.num_ranks, c.hidden, c.num_topk, c.recv_capacity
    if h.normal_tokens is None:
        raise EPError(8, "combine without a prior dispatch on this handle")
    T = h.normal_tokens
    if combined_x is None:
        combined_x = _empty((R, T, H), out_dtype, d)
    if topk_weights is not None and combined_topk_weights is None:
        combined_topk_weights = _empty((R, T, K), torch.float32, d)
    _raise(lib().ep_combine(
        h.ptr, _ptr(x, "x", torch.bfloat16, (R, cap, H), d),
        _ptr(topk_weights, "topk_weights", torch.float32, (R, cap, K), d),
        _ptr(bias_0, "bias_0", torch.bfloat16, (R, T, H), d), _ptr(bias_1, "bias_1", torch.bfloat16, (R, T, H), d),
        _ptr(combined_x, "combined_x", out_dtype, (R, T, H), d),
        EP_FP32 if out_dtype == torch.float32 else EP_BF16,
        _ptr(combined_topk_weights, "combined_topk_weights", torch.float32, (R, T, K), d),
        _stream(stream, h.device)))
    return dict(combined_x=combined_x, combined_topk_weights=combined_topk_weights)


def ep_ll_dispatch(h: Handle, x: torch.Tensor, topk_idx: torch.Tensor, use_fp8: bool = True,
                   round_scale: bool = False, use_ue8m0: bool = False, recv_msgs=None, packed_recv_count=None,
                   packed_recv_layout_range=None, cumulative_local_expert_recv_stats=None, stream=None):
    """Low-latency dispatch into packed per-local-expert message slots."""
    c, d = h.cfg, h.device
    R, H, K, EL, maxT = c.num_ranks, c.hidden, c.num_topk, c.num_local_experts, c.num_max_tokens
    T = x.shape[1]
    msg = ep_ll_msg_bytes(H, use_fp8)
    if recv_msgs is None:
        recv_msgs = _empty((R, EL, R * maxT, msg), torch.uint8, d)
    if packed_recv_count is None:
        packed_recv_count = _empty((R, EL), torch.int32, d)
    if packed_recv_layout_range is None:
        packed_recv_layout_range = _empty((R, EL, R), torch.int64, d)
    _raise(lib().ep_ll_dispatch(
        h.ptr, T, _ptr(x, "x", torch.bfloat16, (R, T, H), d), _ptr(topk_idx, "topk_idx", torch.int64, (R, T, K), d),
        int(bool(use_fp8)), int(bool(round_scale)), int(bool(use_ue8m0)),
        _ptr(recv_msgs, "recv_msgs", torch.uint8, (R, EL, R * maxT, msg), d),
        _ptr(packed_recv_count, "packed_recv_count", torch.int32, (R, EL), d),
        _ptr(packed_recv_layout_range, "packed_recv_layout_range", torch.int64, (R, EL, R), d),
        _ptr(cumulative_local_expert_recv_stats, "cumulative_local_expert_recv_stats", torch.int32, (R, EL), d),
        _stream(stream, h.device)))
    h.ll_tokens = T
    return dict(recv_msgs=recv_msgs, packed_recv_count=packed_recv_count,
                packed_recv_layout_range=packed_recv_layout_range)


def ll_views(recv_msgs: torch.Tensor, hidden: int, use_fp8: bool):
    """Strided views of the message buffer: (packed_recv_x, packed_recv_x_scales, packed_recv_src_info)."""
    R, EL, rows, msg = recv_msgs.shape
    base = recv_msgs.reshape(-1)
    st = (EL * rows * msg, rows * msg, msg)

    def view(dtype, shape, strides_bytes, offset_bytes):
        t = base.view(dtype)
        size = t.element_size()
        return t.as_strided(shape, tuple(s // size for s in strides_bytes),
                            t.storage_offset() + offset_bytes // size)

    src_info = view(torch.int32, (R, EL, rows), st, 0)
    if use_fp8:
        px = view(torch.float8_e4m3fn, (R, EL, rows, hidden), st + (1,), 16)
        scales = view(torch.uint8, (R, EL, rows, 4 * (hidden // 128)), st + (1,), 16 + hidden)
    else:
        px = view(torch.bfloat16, (R, EL, rows, hidden), st + (2,), 16)
        scales = None
    return px, scales, src_info


def _row_stride_bytes(x: torch.Tensor, R: int, EL: int, rows: int, H: int):
    """Row stride in bytes of a [R][EL][rows][H] view whose rows are evenly spaced (contiguous rows
    or the payloads of the message buffer), else None."""
    if tuple(x.shape) != (R, EL, rows, H) or x.stride(3) != 1:
        return None
    r = x.stride(2)
    if x.stride(1) != rows * r or x.stride(0) != EL * rows * r:
        return None
    return r * x.element_size()


def ep_ll_combine(h: Handle, x: torch.Tensor, topk_idx: torch.Tensor, topk_weights: torch.Tensor,
                  combined_x=None, stream=None):
    """Low-latency combine: top-k weighted fp32 sum of the expert outputs, bf16 out.

    x is [R][EL][R*maxT][H] bf16, contiguous or with evenly spaced rows -- e.g. the packed_recv_x
    view of a bf16 message buffer (ll_views), which the experts overwrite in place (zero-copy)."""
    c, d = h.cfg, h.device
    R, H, K, EL, maxT = c.num_ranks, c.hidden, c.num_topk, c.num_local_experts, c.num_max_tokens
    if h.ll_tokens is None:
        raise EPError(8, "low-latency combine without a prior low-latency dispatch")
    T = h.ll_tokens
    if combined_x is None:
        combined_x = _empty((R, T, H), torch.bfloat16, d)
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16 or x.device != d:
        raise TypeError(f"x must be a bf16 tensor on {d}")
    row_bytes = _row_stride_bytes(x, R, EL, R * maxT, H)
    if row_bytes is None:
        raise ValueError(f"x must be [R={R}][EL={EL}][{R * maxT}][H={H}] with evenly spaced rows")
    _raise(lib().ep_ll_combine_strided(
        h.ptr, ctypes.c_void_p(x.data_ptr()), row_bytes,
        _ptr(topk_idx, "topk_idx", torch.int64, (R, T, K), d),
        _ptr(topk_weights, "topk_weights", torch.float32, (R, T, K), d),
        _ptr(combined_x, "combined_x", torch.bfloat16, (R, T, H), d), _stream(stream, h.device)))
    return combined_x


def recv_hook(stream=None):
    """Deferred receive (the return_recv_hook of the low-latency calls, [P3] section 4.3): records an
    event on `stream` (default: the current stream) after the calls already enqueued there and
    returns a function that makes the stream current at call time wait for it.  Launch a dispatch
    on a communication stream, keep computing, call the hook where the received data is needed."""
    s = stream if stream is not None else torch.cuda.current_stream()
    ev = torch.cuda.Event()
    ev.record(s)

    def hook(wait_stream=None):
        (wait_stream if wait_stream is not None else torch.cuda.current_stream()).wait_event(ev)

    return hook


def expected_topk(num_groups: int, num_experts: int, num_topk: int) -> float:
    """Expected groups (ranks) hit by one token's top-k (the library's launch model)."""
    v = lib().ep_expected_topk(num_groups, num_experts, num_topk)
    if v < 0:
        raise ValueError(lib().ep_last_error().decode())
    return v


def theoretical_num_sms(num_ranks: int, num_experts: int, num_topk: int, *, hbm_gbs: float, sm_read_gbs: float,
                        sm_write_gbs: float, num_device_sms: int, prefer_overlap_with_compute: bool = True,
                        for_combine: bool = False) -> int:
    """SMs a dispatch (or combine) needs to keep HBM busy; a value for Config.max_sms."""
    m = ep_sm_model(hbm_gbs, sm_read_gbs, sm_write_gbs, num_device_sms, int(bool(prefer_overlap_with_compute)))
    n = lib().ep_theoretical_num_sms(ctypes.byref(m), num_ranks, num_experts, num_topk, int(bool(for_combine)))
    if n < 0:
        raise ValueError(lib().ep_last_error().decode())
    return n
