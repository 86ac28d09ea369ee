"""Shared plumbing of the GPU parity tests: run the CUDA path through the C ABI
(binding in combine_get_dispatch_03_gb300.ep) and the CPU oracle on the same
seeded inputs, then compare element by element."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from combine_get_dispatch_03_gb300 import ep
from combine_get_dispatch_03_gb300 import workloads as W

DEV = "cuda"
CANARY = 0x5A  # byte written around and into every output before a call


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    if t.dtype == torch.bool:
        return t.numpy().astype(np.uint8)
    return t.numpy()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


class Guarded:
    """A tensor carved out of a larger canary-filled buffer; check() proves nothing was written outside it."""

    PAD = 4096

    def __init__(self, shape, dtype, fill_byte=CANARY):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((n + 2 * self.PAD,), fill_byte, dtype=torch.uint8, device=DEV)
        self.fill = fill_byte
        self.n = n
        self.t = self.buf[self.PAD:self.PAD + n].view(dtype).view(shape)

    def check(self):
        head = self.buf[:self.PAD]
        tail = self.buf[self.PAD + self.n:]
        assert bool((head == self.fill).all()) and bool((tail == self.fill).all()), "write outside the buffer"


def config_of(shape: W.Shape, cap: int, max_sms: int = 0) -> ep.Config:
    return ep.Config(num_ranks=shape.R, num_max_tokens=max(shape.max_tokens or shape.T, shape.T), hidden=shape.H,
                     num_experts=shape.E, num_topk=shape.K, num_channels=shape.C,
                     expert_alignment=shape.A, recv_capacity=cap, max_sms=max_sms)


def needed_capacity(idx: np.ndarray, E: int) -> int:
    lay = O.get_dispatch_layout(idx, E)
    return int(lay["num_tokens_per_rank"].sum(axis=0).max()) if idx.size else 0


def compare_layout(gpu: dict, ora: dict):
    np.testing.assert_array_equal(host(gpu["num_tokens_per_rank"]), ora["num_tokens_per_rank"])
    np.testing.assert_array_equal(host(gpu["num_tokens_per_expert"]), ora["num_tokens_per_expert"])
    np.testing.assert_array_equal(host(gpu["is_token_in_rank"]), ora["is_token_in_rank"])
    if gpu["num_tokens_per_rdma_rank"] is not None:
        np.testing.assert_array_equal(host(gpu["num_tokens_per_rdma_rank"]), ora["num_tokens_per_rdma_rank"])


def compare_record(h: ep.Handle, ora_notify: dict, T: int):
    for key in ("rank_prefix_matrix", "channel_prefix_matrix", "recv_channel_prefix_matrix", "num_recv"):
        np.testing.assert_array_equal(host(h.export(key)), ora_notify[key], err_msg=key)
    np.testing.assert_array_equal(host(h.export("send_head")), ora_notify["send_head"], err_msg="send_head")
    src = host(h.export("recv_src_idx"))
    for r, n in enumerate(ora_notify["num_recv"]):
        n = min(int(n), src.shape[1])
        np.testing.assert_array_equal(src[r, :n], ora_notify["recv_src_idx"][r, :n], err_msg=f"recv_src_idx[{r}]")


def valid_rows(num_recv: np.ndarray, cap: int):
    """Boolean [R][cap] mask of receive rows that the dispatch writes."""
    R = num_recv.shape[0]
    return np.arange(cap)[None, :] < np.minimum(num_recv, cap)[:, None]


def run_normal(shape: W.Shape, *, mode: int = O.MODE_BF16, cap: int | None = None, with_weights=True,
               biases=False, out_fp32=False, y_seed: int | None = None, max_sms: int = 0):
    """Layout -> fresh dispatch -> combine on the GPU and in the oracle; returns both sides' outputs."""
    idx, w = W.routing(shape)
    x = W.tokens_x(shape)  # bf16 on the host
    xb = W.bf16_bits(x)
    need = needed_capacity(idx, shape.E)
    if cap is None:
        cap = max(need, 1)
    cfg = config_of(shape, cap, max_sms)
    h = ep.Handle(cfg)
    idx_d = torch.from_numpy(idx).to(DEV)
    w_d = torch.from_numpy(w).to(DEV)
    x_d = x.to(DEV)
    lay = ep.ep_get_dispatch_layout(h, idx_d)
    ora_lay = O.get_dispatch_layout(idx, shape.E)
    ora_n = O.dispatch_notify(ora_lay["num_tokens_per_rank"], ora_lay["is_token_in_rank"],
                              ora_lay["num_tokens_per_expert"], shape.C, shape.A, cap)
    fp8_out = mode != O.MODE_BF16
    recv_x = Guarded((shape.R, cap, shape.H), torch.float8_e4m3fn if fp8_out else torch.bfloat16)
    recv_s = Guarded((shape.R, cap, shape.H // 128), torch.float32) if fp8_out else None
    recv_i = Guarded((shape.R, cap, shape.K), torch.int64)
    recv_w = Guarded((shape.R, cap, shape.K), torch.float32) if with_weights else None
    x_in, xs_in, xs_host, x_host = x_d, None, None, xb
    if mode == O.MODE_FP8_IN:
        g = np.random.default_rng(shape.seed + 5)
        x_host = g.integers(0, 256, (shape.R, shape.T, shape.H), dtype=np.uint8)
        x_host[(x_host & 0x7F) == 0x7F] = 0  # no NaN codes
        xs_host = g.random((shape.R, shape.T, shape.H // 128), dtype=np.float32)
        x_in = torch.from_numpy(x_host).to(DEV).view(torch.float8_e4m3fn)
        xs_in = torch.from_numpy(xs_host).to(DEV)
    d = ep.ep_dispatch(h, x_in, topk_idx=idx_d, topk_weights=w_d if with_weights else None,
                       num_tokens_per_rank=lay["num_tokens_per_rank"], is_token_in_rank=lay["is_token_in_rank"],
                       num_tokens_per_expert=lay["num_tokens_per_expert"], x_scales=xs_in,
                       cast_to_fp8=mode == O.MODE_CAST_FP8, recv_x=recv_x.t,
                       recv_x_scales=recv_s.t if recv_s else None, recv_topk_idx=recv_i.t,
                       recv_topk_weights=recv_w.t if recv_w else None)
    status = h.status()
    ora_d = O.dispatch(x_host, ora_n["send_head"], cap, shape.E, mode=mode, x_scales=xs_host, topk_idx=idx,
                       topk_weights=w if with_weights else None)
    out = dict(h=h, idx=idx, w=w, x=xb, cap=cap, need=need, lay=lay, ora_lay=ora_lay, ora_n=ora_n, d=d,
               ora_d=ora_d, status=status, guards=[g_ for g_ in (recv_x, recv_s, recv_i, recv_w) if g_])
    if mode == O.MODE_BF16:
        # expert outputs: the received rows themselves, or fresh N(0,1) rows
        if y_seed is None:
            y_host, y_dev = ora_d["recv_x"], d["recv_x"]
        else:
            y_host = W.bf16_bits(W.normal_bf16((shape.R, cap, shape.H), y_seed, "y"))
            y_dev = dev_bf16(y_host)
        b0 = b1 = None
        b0h = b1h = None
        if biases:
            b0, b1 = W.normal_bf16((shape.R, shape.T, shape.H), shape.seed, "b0", std=0.1), \
                W.normal_bf16((shape.R, shape.T, shape.H), shape.seed, "b1", std=0.1)
            b0h, b1h = W.bf16_bits(b0), W.bf16_bits(b1)
            b0, b1 = b0.to(DEV), b1.to(DEV)
        c = ep.ep_combine(h, y_dev, topk_weights=d["recv_topk_weights"] if with_weights else None, bias_0=b0,
                          bias_1=b1, out_dtype=torch.float32 if out_fp32 else torch.bfloat16)
        ora_c = O.combine(y_host, ora_n["send_head"], recv_topk_weights=ora_d.get("recv_topk_weights"),
                          bias0=b0h, bias1=b1h, out_fp32=out_fp32, num_topk=shape.K)
        out.update(c=c, ora_c=ora_c, combine_status=h.status())
    return out


def compare_dispatch(res: dict, shape: W.Shape, mode: int):
    R, K, cap = shape.R, shape.K, res["cap"]
    ora_n, ora_d, d = res["ora_n"], res["ora_d"], res["d"]
    rows = valid_rows(ora_n["num_recv"], cap)
    gx = host(d["recv_x"])
    np.testing.assert_array_equal(gx[rows], ora_d["recv_x"][rows])
    if mode != O.MODE_BF16:
        np.testing.assert_array_equal(host(d["recv_x_scales"])[rows], ora_d["recv_x_scales"][rows])
    np.testing.assert_array_equal(host(d["recv_topk_idx"])[rows], ora_d["recv_topk_idx"][rows])
    if d["recv_topk_weights"] is not None:
        np.testing.assert_array_equal(host(d["recv_topk_weights"])[rows], ora_d["recv_topk_weights"][rows])
    np.testing.assert_array_equal(host(d["num_recv_tokens_per_expert"]), ora_n["num_recv_tokens_per_expert"])
    # rows past num_recv keep the canary
    if (~rows).any():
        raw = host(d["recv_x"].view(torch.uint8))
        assert (raw[~rows] == CANARY).all()
    for g_ in res["guards"]:
        g_.check()


def rel_err(a: np.ndarray, b: np.ndarray) -> float:
    """max |a-b| / max(|b|, 1e-3 * rms(b)) -- the combine tolerance measure."""
    a = a.astype(np.float64)
    b = b.astype(np.float64)
    if b.size == 0:
        return 0.0
    floor = 1e-3 * max(np.sqrt(np.mean(b * b)), 1e-30)
    return float(np.max(np.abs(a - b) / np.maximum(np.abs(b), floor)))


def host_threads() -> int:
    import os
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def oracle_dispatch_all(x, send_head, cap, E, mode=O.MODE_BF16, x_scales=None, topk_idx=None, topk_weights=None):
    """oracle.dispatch over every token, its token loop split into contiguous blocks over the host cores
    (the C calls release the interpreter lock; the blocks write disjoint receive rows)."""
    from concurrent.futures import ThreadPoolExecutor
    R, T, H = x.shape
    K = topk_idx.shape[2] if topk_idx is not None else 1
    pay = np.uint16 if mode == O.MODE_BF16 else np.uint8
    out = dict(recv_x=np.zeros((R, cap, H), pay))
    if mode != O.MODE_BF16:
        out["recv_x_scales"] = np.zeros((R, cap, H // 128), np.float32)
    if topk_idx is not None:
        out["recv_topk_idx"] = np.full((R, cap, K), -2, np.int64)
        if topk_weights is not None:
            out["recv_topk_weights"] = np.full((R, cap, K), np.nan, np.float32)
    n = host_threads()
    blocks = np.array_split(np.arange(R * T, dtype=np.int64), n)
    with ThreadPoolExecutor(n) as ex:
        list(ex.map(lambda b: O.dispatch(x, send_head, cap, E, mode=mode, x_scales=x_scales, topk_idx=topk_idx,
                                         topk_weights=topk_weights, tokens=b, out=out), blocks))
    return out


def oracle_combine_all(y, send_head, recv_topk_weights=None, bias0=None, bias1=None, out_fp32=False, num_topk=1):
    """oracle.combine over every token, split over the host cores like oracle_dispatch_all."""
    from concurrent.futures import ThreadPoolExecutor
    R, T, _ = send_head.shape
    H = y.shape[2]
    K = recv_topk_weights.shape[2] if recv_topk_weights is not None else num_topk
    out = dict(out=np.zeros((R, T, H), np.float32 if out_fp32 else np.uint16),
               combined_topk_weights=np.zeros((R, T, K), np.float32) if recv_topk_weights is not None else None)
    n = host_threads()
    blocks = np.array_split(np.arange(R * T, dtype=np.int64), n)
    with ThreadPoolExecutor(n) as ex:
        list(ex.map(lambda b: O.combine(y, send_head, recv_topk_weights=recv_topk_weights, bias0=bias0, bias1=bias1,
                                        out_fp32=out_fp32, num_topk=num_topk, tokens=b, out=out), blocks))
    return out


def assert_rows_equal(gpu: torch.Tensor, ora: np.ndarray, num_recv, name: str):
    """Receive rows [0, num_recv[r]) of every rank r, whole, one rank at a time (bounded host memory)."""
    for r, n in enumerate(num_recv):
        n = int(min(n, ora.shape[1]))
        np.testing.assert_array_equal(host(gpu[r, :n]), ora[r, :n], err_msg=f"{name}[{r}]")
