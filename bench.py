#!/usr/bin/env python3
"""Benchmark of the EP layout / dispatch / combine path on one GB300.

Headline (one JSON line on stdout): the normal-mode step on the
DeepSeek-V3-shaped workload ``normal_v3`` (R=8 virtual ranks x 4096 tokens,
hidden 7168, 256 experts, top-8, Gumbel routing, expert_alignment 128):
get_dispatch_layout -> dispatch (fresh record, bf16) -> combine (the
received rows as expert outputs, with the top-k weight reduction), all
inputs resident in HBM.  ``value`` is payload GB/s of that step (hidden
bytes read + written by dispatch and combine / step time); tokens/s and the
HBM fraction ride along.  ``ops`` adds per-operation timings of the other
workloads (FP8 dispatch with Zipf routing, low-latency dispatch/combine,
combine with biases on a cached record).

``--impl reference`` times the CPU oracle (the reference arm of this
project) on a bounded sample of the same workload.  Under torchrun every
rank runs an independent replica (the single-GPU path has no exchange step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from combine_get_dispatch_03_gb300 import workloads as W  # noqa: E402

METRIC = "dispatch+combine payload GB/s and tokens/s on 1 GB300; % of HBM peak"
HEADLINE = "normal_v3"


# ----------------------------------------------------------------------------- byte model

def normal_bytes(R, T, H, K, hits, fp8=False, biases=0):
    """Algorithmic bytes of one normal-mode step, split by operation.

    payload: hidden (and FP8 scale) bytes; meta: routing / index / weight bytes.
    hits = number of (token, destination rank) pairs = sum of num_tokens_per_rank.
    """
    n = R * T
    row_in = 2 * H
    row_out = (H + 4 * (H // 128)) if fp8 else 2 * H
    layout = dict(payload=0, meta=n * K * 8 + n * R + R * R * 4 + R * 256 * 4)
    notify = dict(payload=0, meta=n * R + n * R * 4 + hits * 4)
    dispatch = dict(payload=n * row_in + hits * row_out,
                    meta=n * R * 4 + n * K * 12 + hits * K * 12)
    combine = dict(payload=hits * 2 * H + biases * n * 2 * H + n * 2 * H,
                   meta=n * R * 4 + hits * K * 4 + n * K * 4)
    return dict(layout=layout, notify=notify, dispatch=dispatch, combine=combine)


def ll_bytes(R, T, H, K, n_valid, msg):
    n = R * T
    return dict(ll_dispatch=dict(payload=n * 2 * H + n_valid * msg, meta=n * K * 8 + n_valid * 8),
                ll_combine=dict(payload=n_valid * 2 * H + n * 2 * H, meta=n * K * 16))


def total(d):
    return d["payload"] + d["meta"]


# ----------------------------------------------------------------------------- environment

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


KERNEL_SOURCES = ("ep_common.cuh", "ep_dispatch.cu")  # where the dispatch and combine kernels live


def source_digest(names=None):
    """Hash of the kernel sources (all of csrc/ when names is None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "combine_get_dispatch_03_gb300", "csrc")
    for name in sorted(names or os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch from a committed ncu summary, if taken on the kernel's current sources."""
    path = os.path.join(ROOT, "profiles", "traffic_per_launch.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(kernel)
    if not ent or ent.get("source_digest") != source_digest(ent.get("sources")):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            target = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            target = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[device_index]
        self.cmd = ["nvidia-smi", "-i", target, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "100"]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        time.sleep(0.15)
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append(parts)

    def __exit__(self, *exc):
        time.sleep(0.15)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if s[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


# ----------------------------------------------------------------------------- distributed plumbing

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_replicas(elapsed_s: float, units: float, world: int):
    """Whole-job aggregate over independent replicas: max time over ranks, sum of units."""
    if world == 1:
        return elapsed_s, units
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ----------------------------------------------------------------------------- our arm

class Events:
    def __init__(self, n):
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]

    def rec(self, i, stream):
        self.ev[i].record(stream)

    def ms(self, a, b):
        return self.ev[a].elapsed_time(self.ev[b])


STEP_OPS = ("layout_notify", "dispatch", "combine")  # timed parts of the headline step
EV_PER_STEP = len(STEP_OPS) + 1


def headline_config(T, recv_gb, world):
    """The `config` of the headline line (both arms)."""
    return {"workload": f"{HEADLINE}: R=8 T={T} H=7168 E=256 K=8 Gumbel routing A=128 C=12; step = "
                        "get_dispatch_layout + notify_dispatch (one launch) + dispatch (bf16, top-k metadata) + "
                        "combine (received rows, top-k weight reduction)",
            "l2": "no flush; inputs larger than L2 (x 470 MB, receive buffer %.2f GB vs 129 MB L2)" % recv_gb,
            "parallelism": "replicas" if world > 1 else "single GPU, R=8 virtual ranks"}


def receive_capacity(shape):
    """Rows of the largest destination rank for the workload's routing (host arithmetic)."""
    idx, _ = W.routing(shape)
    dest = np.where(idx >= 0, idx // shape.EL, -1)  # [R][T][K] destination rank per slot
    hit = np.zeros((shape.R, shape.T, shape.R), dtype=bool)
    s_, t_, k_ = np.nonzero(dest >= 0)
    hit[s_, t_, dest[s_, t_, k_]] = True
    return int(hit.sum(axis=(0, 1)).max())


def prepare_normal(ep, shape, dev, with_e2e=True):
    idx, w = W.routing(shape)
    idx_d = torch.from_numpy(idx).to(dev)
    w_d = torch.from_numpy(w).to(dev)
    x_d = W.tokens_x(shape, device=dev)
    probe = ep.Handle(ep.Config(shape.R, shape.T, shape.H, shape.E, shape.K, shape.C, shape.A, 0), dev)
    lay = ep.ep_get_dispatch_layout(probe, idx_d)
    probe.check()
    tpr = lay["num_tokens_per_rank"].to("cpu")
    probe.destroy()
    cap = int(tpr.sum(0).max())
    hits = int(tpr.sum())
    h = ep.Handle(ep.Config(shape.R, shape.T, shape.H, shape.E, shape.K, shape.C, shape.A, cap), dev)
    return dict(idx=idx, w=w, idx_d=idx_d, w_d=w_d, x_d=x_d, cap=cap, hits=hits, h=h)


# ----------------------------------------------------------------------------- parity capture
# After each timed region the outputs of its last call are copied to host memory: the layout and
# the dispatch record whole, payload rows and combined tokens on a seeded sample of tokens.  The
# CPU-oracle leg (cpu_parity) later runs the oracle on the same inputs and compares.

PARITY_TOKENS = 1024  # sampled tokens per checked call (plus the first and the last)


def _host(t):
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    if t.dtype == torch.bool:
        return t.numpy().astype(np.uint8)
    return t.numpy()


def _pairs(send_head_host, toks, R):
    """(rank, row) of every destination of the sampled tokens."""
    sh = send_head_host.reshape(-1, R)[toks]
    i, r = np.nonzero(sh >= 0)
    return np.stack([r, sh[i, r]], axis=1).astype(np.int64)


def _rows(t, pairs):
    idx = torch.from_numpy(pairs).to(t.device)
    return _host(t[idx[:, 0], idx[:, 1]])


def capture_normal(name, shape, h, idx, w, x_d, cap, *, mode=0, layout=None, nrpe=None, recv=None,
                   x_scales=None, combine=None):
    """Host copies of one normal-mode call's outputs for the oracle check.

    layout: the four layout outputs (or None); nrpe: num_recv_tokens_per_expert (or None);
    recv: receive buffers of the dispatch (recv_x, and optionally recv_x_scales, recv_topk_idx,
    recv_topk_weights); combine: dict(y, out, and optionally out_w, b0, b1) of a combine (or None)."""
    toks = W.sample_tokens(shape, PARITY_TOKENS, field="bench_parity")
    t_idx = torch.from_numpy(toks).to(x_d.device)
    rec = dict(kind="normal", name=name, shape=shape, idx=idx, w=w, cap=cap, mode=mode, toks=toks,
               x_rows=_host(x_d.reshape(-1, shape.H)[t_idx]))
    if x_scales is not None:
        rec["x_scale_rows"] = _host(x_scales.reshape(-1, shape.H // 128)[t_idx])
    rec["record"] = {k: _host(h.export(k)) for k in
                     ("rank_prefix_matrix", "channel_prefix_matrix", "recv_channel_prefix_matrix", "num_recv",
                      "send_head", "recv_src_idx")}
    if layout is not None:
        rec["layout"] = {k: (_host(v) if v is not None else None) for k, v in layout.items()}
    if nrpe is not None:
        rec["nrpe"] = _host(nrpe)
    pairs = _pairs(rec["record"]["send_head"], toks, shape.R)
    rec["pairs"] = pairs
    if recv is not None:
        rec["recv"] = {k: _rows(v, pairs) for k, v in recv.items() if v is not None}
    if combine is not None:
        c = dict(out_rows=_host(combine["out"].reshape(-1, shape.H)[t_idx]), y_rows=_rows(combine["y"], pairs))
        if combine.get("out_w") is not None:
            c["out_w"] = _host(combine["out_w"])
        for b in ("b0", "b1"):
            if combine.get(b) is not None:
                c[b + "_rows"] = _host(combine[b].reshape(-1, shape.H)[t_idx])
        rec["combine"] = c
    return rec


def capture_ll(name, shape, h, idx, w, x_d, out, use_fp8=True, use_ue8m0=True, rank_mask=None):
    """Host copies of one low-latency dispatch (messages of the sampled tokens' slots, counts, layout
    range, the slot map whole) and combine (the sampled tokens' outputs and the rows they read; the
    expert outputs `y` may be a strided view such as the payloads of the message buffer)."""
    toks = W.sample_tokens(shape, PARITY_TOKENS, field="bench_parity")
    t_idx = torch.from_numpy(toks).to(x_d.device)
    rec = dict(kind="ll", name=name, shape=shape, idx=idx, w=w, toks=toks, use_fp8=use_fp8, use_ue8m0=use_ue8m0,
               rank_mask=rank_mask,
               x_rows=_host(x_d.reshape(-1, shape.H)[t_idx]), slot_row=_host(h.export("ll_slot_row"))[:, :shape.T])
    rec.update({k: _host(v) for k, v in out.items() if k in ("packed_recv_count", "packed_recv_layout_range")})
    sl = rec["slot_row"].reshape(-1, shape.K)[toks]          # [n][K]
    e = idx.reshape(-1, shape.K)[toks]
    ok = (e >= 0) & (sl >= 0)
    flat = torch.from_numpy(np.where(ok, e * (shape.R * shape.max_tokens) + sl, 0).reshape(-1)).to(x_d.device)
    msgs = out["recv_msgs"].reshape(-1, out["recv_msgs"].shape[-1])
    rec["msg_rows"] = _host(msgs[flat]).reshape(len(toks), shape.K, -1)
    rec["ok"] = ok
    if "y" in out:
        ee, ss = np.where(ok, e, 0).reshape(-1), np.where(ok, sl, 0).reshape(-1)
        at = [torch.from_numpy(a.astype(np.int64)).to(x_d.device) for a in (ee // shape.EL, ee % shape.EL, ss)]
        rec["y_rows"] = _host(out["y"][at[0], at[1], at[2]]).reshape(len(toks), shape.K, shape.H)
        rec["out_rows"] = _host(out["combined_x"].reshape(-1, shape.H)[t_idx])
    return rec


def run_ours(args):
    from combine_get_dispatch_03_gb300 import ep
    rank, world, local = dist_setup()
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    shape = W.WORKLOADS[HEADLINE]
    if args.tokens:
        shape = shape.scaled(T=args.tokens)
    R, T, H, E, K = shape.R, shape.T, shape.H, shape.E, shape.K
    st = prepare_normal(ep, shape, dev)
    h, cap, hits = st["h"], st["cap"], st["hits"]
    idx_d, w_d, x_d = st["idx_d"], st["w_d"], st["x_d"]

    lay = dict(num_tokens_per_rank=torch.empty((R, R), dtype=torch.int32, device=dev),
               num_tokens_per_rdma_rank=None,
               num_tokens_per_expert=torch.empty((R, E), dtype=torch.int32, device=dev),
               is_token_in_rank=torch.empty((R, T, R), dtype=torch.bool, device=dev))
    recv_x = torch.empty((R, cap, H), dtype=torch.bfloat16, device=dev)
    recv_i = torch.empty((R, cap, K), dtype=torch.int64, device=dev)
    recv_w = torch.empty((R, cap, K), dtype=torch.float32, device=dev)
    nrpe = torch.empty((R, E // R), dtype=torch.int32, device=dev)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device=dev)
    out_w = torch.empty((R, T, K), dtype=torch.float32, device=dev)

    # The layout and the dispatch record come from one call (one launch); the
    # prepared dispatch then moves the rows, so the data kernel has its own pair of events.
    def layout_notify(idx_in):
        if args.layout_two_launches:
            ep.ep_get_dispatch_layout(h, idx_in, **lay)
            ep.ep_notify_dispatch(h, lay["num_tokens_per_rank"], lay["is_token_in_rank"],
                                  lay["num_tokens_per_expert"], num_recv_tokens_per_expert=nrpe)
        else:
            ep.ep_layout_notify(h, idx_in, num_recv_tokens_per_expert=nrpe, **lay)

    def step(idx_in, w_in, x_in, ev=None, base=0):
        if ev: ev.rec(base, stream)
        layout_notify(idx_in)
        if ev: ev.rec(base + 1, stream)
        ep.ep_dispatch(h, x_in, topk_idx=idx_in, topk_weights=w_in, recv_x=recv_x, recv_topk_idx=recv_i,
                       recv_topk_weights=recv_w, prepared=True)
        if ev: ev.rec(base + 2, stream)
        ep.ep_combine(h, recv_x, topk_weights=recv_w, combined_x=out, combined_topk_weights=out_w)
        if ev: ev.rec(base + 3, stream)

    for _ in range(args.warmup):
        step(idx_d, w_d, x_d)
    torch.cuda.synchronize(dev)
    h.check()

    # The timed region: the K steps with one event pair around them.  An event recorded between two
    # kernels ends their programmatic launch overlap (measured: 904 against 890 us per step), so the
    # per-op times come from a second run of the same K steps with an event between every two
    # kernels, right after; the roofline's kernel duration is from that run.
    span = Events(2)
    barrier(world)
    with ClockSampler(dev.index) as clocks:
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        span.rec(0, stream)
        for i in range(args.steps):
            step(idx_d, w_d, x_d)
        span.rec(1, stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
    barrier(world)
    h.check()
    # the last timed step's outputs, for the oracle check of the CPU leg
    checks = [capture_normal(HEADLINE + ".step", shape, h, st["idx"], st["w"], x_d, cap, layout=lay, nrpe=nrpe,
                             recv=dict(recv_x=recv_x, recv_topk_idx=recv_i, recv_topk_weights=recv_w),
                             combine=dict(y=recv_x, out=out, out_w=out_w))]
    step_ms = span.ms(0, 1) / args.steps

    ev = Events(EV_PER_STEP * args.steps + 1)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        step(idx_d, w_d, x_d, ev, EV_PER_STEP * i)
    ev.rec(EV_PER_STEP * args.steps, stream)
    torch.cuda.synchronize(dev)
    h.check()
    step_ms_instrumented = ev.ms(0, EV_PER_STEP * args.steps) / args.steps
    op_ms = {name: statistics.mean(ev.ms(EV_PER_STEP * i + j, EV_PER_STEP * i + j + 1) for i in range(args.steps))
             for j, name in enumerate(STEP_OPS)}

    # the layout and the record as one launch against the two separate calls (same outputs)
    layout_notify_times = None
    if not args.no_ops:
        ln_one = None if args.layout_two_launches else \
            timed(lambda: ep.ep_layout_notify(h, idx_d, num_recv_tokens_per_expert=nrpe, **lay), 10, stream)

        def two_calls():
            ep.ep_get_dispatch_layout(h, idx_d, **lay)
            ep.ep_notify_dispatch(h, lay["num_tokens_per_rank"], lay["is_token_in_rank"],
                                  lay["num_tokens_per_expert"], num_recv_tokens_per_expert=nrpe)

        ln_two = timed(two_calls, 10, stream)
        h.check()
        layout_notify_times = {"one_launch_us": round(ln_one * 1e3, 2) if ln_one else None,
                         "two_launches_us": round(ln_two * 1e3, 2),
                         "step_uses": "two launches" if args.layout_two_launches else "one launch"}

    bm = normal_bytes(R, T, H, K, hits)
    payload = bm["dispatch"]["payload"] + bm["combine"]["payload"]
    alg = sum(total(v) for v in bm.values())
    elapsed, units = reduce_replicas(step_ms * args.steps / 1e3, payload * args.steps, world)
    value = units / elapsed / 1e9
    peak, peak_kind = load_peaks()

    # dominant operation of the step and its roofline
    dom = max(("dispatch", "combine"), key=lambda k: op_ms[k])
    dom_bytes = total(bm[dom])
    achieved = dom_bytes / (op_ms[dom] / 1e3) / 1e9
    kernel_name = "dispatch_bulk_kernel<0>" if dom == "dispatch" else \
        ("combine_kernel<false, 8>" if R <= 8 else "combine_kernel<false, 4>")  # all rows in one batch at R <= 8
    traffic = recorded_traffic(kernel_name)

    # End to end through the binding: every step copies its inputs from pinned host memory and its
    # result (the combined tokens and weights) back to pinned host memory.  Copies run on their own
    # streams with two buffer sets, so step i's upload, step i-1's compute and step i-2's download
    # overlap, as a serving loop would run them.
    e2e = None
    if not args.no_e2e:
        e2e_steps = min(args.steps, args.e2e_steps)
        n_in = 2
        x_h = [x_d.to("cpu").pin_memory() for _ in range(n_in)]
        idx_h = [st["idx_d"].to("cpu").pin_memory() for _ in range(n_in)]
        w_h = [st["w_d"].to("cpu").pin_memory() for _ in range(n_in)]
        out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(n_in)]
        outw_h = [torch.empty(out_w.shape, dtype=out_w.dtype).pin_memory() for _ in range(n_in)]
        x_in = [torch.empty_like(x_d) for _ in range(n_in)]
        idx_in = [torch.empty_like(idx_d) for _ in range(n_in)]
        w_in = [torch.empty_like(w_d) for _ in range(n_in)]
        outs = [torch.empty_like(out) for _ in range(n_in)]
        outws = [torch.empty_like(out_w) for _ in range(n_in)]
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        uploaded = [torch.cuda.Event() for _ in range(n_in)]
        computed = [torch.cuda.Event() for _ in range(n_in)]
        downloaded = [torch.cuda.Event() for _ in range(n_in)]
        for e_ in downloaded:
            e_.record(down)
        for e_ in computed:
            e_.record(stream)

        def e2e_step(i):
            b = i % n_in
            with torch.cuda.stream(up):
                up.wait_event(computed[b])           # the compute that read this input set is done
                x_in[b].copy_(x_h[b], non_blocking=True)
                idx_in[b].copy_(idx_h[b], non_blocking=True)
                w_in[b].copy_(w_h[b], non_blocking=True)
                uploaded[b].record(up)
            stream.wait_event(uploaded[b])
            stream.wait_event(downloaded[b])         # this output set has been read back
            layout_notify(idx_in[b])
            ep.ep_dispatch(h, x_in[b], topk_idx=idx_in[b], topk_weights=w_in[b], recv_x=recv_x,
                           recv_topk_idx=recv_i, recv_topk_weights=recv_w, prepared=True)
            ep.ep_combine(h, recv_x, topk_weights=recv_w, combined_x=outs[b], combined_topk_weights=outws[b])
            computed[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(computed[b])
                out_h[b].copy_(outs[b], non_blocking=True)
                outw_h[b].copy_(outws[b], non_blocking=True)
                downloaded[b].record(down)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        e0.record(up)
        for i in range(e2e_steps):
            e2e_step(i)
        e1.record(down)
        torch.cuda.synchronize(dev)
        barrier(world)
        e2e_ms = e0.elapsed_time(e1) / e2e_steps
        el, un = reduce_replicas(e2e_ms * e2e_steps / 1e3, payload * e2e_steps, world)
        h2d_b = x_h[0].numel() * 2 + idx_h[0].numel() * 8 + w_h[0].numel() * 4
        d2h_b = out_h[0].numel() * 2 + outw_h[0].numel() * 4

        # the host link alone: the same copies with no compute, each way and both ways at once.  The
        # link is shared with the rest of the host, so each figure is the best of three trials.
        def copies(do_up, do_down, reps=3, trials=3):
            return min(copies_once(do_up, do_down, reps) for _ in range(trials))

        def copies_once(do_up, do_down, reps):
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            a_.record(up)
            down.wait_event(a_)
            for r in range(reps):
                b = r % n_in
                if do_up:
                    with torch.cuda.stream(up):
                        x_in[b].copy_(x_h[b], non_blocking=True)
                        idx_in[b].copy_(idx_h[b], non_blocking=True)
                        w_in[b].copy_(w_h[b], non_blocking=True)
                if do_down:
                    with torch.cuda.stream(down):
                        out_h[b].copy_(outs[b], non_blocking=True)
                        outw_h[b].copy_(outws[b], non_blocking=True)
            up.wait_stream(down)
            b_.record(up)
            torch.cuda.synchronize(dev)
            return a_.elapsed_time(b_) / reps

        up_ms, down_ms, both_ms = copies(True, False), copies(False, True), copies(True, True)
        e2e = {"value": round(un / el / 1e9, 2), "unit": "GB/s", "ms_per_step": round(e2e_ms, 4),
               "steps": e2e_steps, "pipelined": "upload / compute / download on three streams, two buffer sets",
               "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b,
               "host_link": {"h2d_gbs": round(h2d_b / up_ms / 1e6, 1), "d2h_gbs": round(d2h_b / down_ms / 1e6, 1),
                             "both_ways_gbs": round((h2d_b + d2h_b) / both_ms / 1e6, 1),
                             "copies_ms_per_step": round(both_ms, 4),
                             "frac": round(both_ms / e2e_ms, 4),
                             "note": "one step's copies with no compute (best of three trials), both ways at "
                                     "once; frac = that time / the e2e step: the e2e number is bound by the "
                                     "host link"}}
        h.check()
        del x_in, idx_in, w_in, outs, outws

    ops, launch_model = {}, None
    if not args.no_ops and rank == 0:
        del recv_x, recv_i, recv_w, out, out_w
        h.destroy()
        torch.cuda.empty_cache()
        launch_model = measure_launch_model(ep, dev, peak, st)
        del st
        torch.cuda.empty_cache()
        ops = measure_other_ops(ep, dev, peak, checks)

    cpu = cpu_all = None
    parity = {"checked": False, "note": "the oracle check runs in the CPU leg (rank 0, one GPU, without --no-cpu)"}
    if rank == 0 and world == 1 and not args.no_cpu:
        parity = cpu_parity(checks)
        cpu = cpu_baseline(W.WORKLOADS[HEADLINE], args.cpu_seconds)
        cpu_all = cpu_baseline_all_cores(W.WORKLOADS[HEADLINE], args.cpu_seconds)

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded routing and N(0,1) bf16 tokens)",
        "config": headline_config(T, R * cap * H * 2 / 1e9, world),
        "tokens_per_s": round(R * T * world / (elapsed / args.steps), 1),
        "launch_model": launch_model,
        "layout_notify": layout_notify_times,
        "hbm_frac_step": round(alg / (step_ms / 1e3) / 1e9 / peak, 4),
        "op_ms": {k: round(v, 4) for k, v in op_ms.items()},
        "timing": {"ms_per_step": "K steps between one pair of events (the timed region)",
                   "op_ms": "the same K steps again with an event between every two kernels, which ends their "
                            "programmatic launch overlap; the roofline's kernel duration is from this run",
                   "ms_per_step_instrumented": round(step_ms_instrumented, 4)},
        "roofline": {"bound": "hbm", "kernel": kernel_name, "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "algorithmic_bytes": dom_bytes},
        "cpu_baseline": cpu, "cpu_baseline_all_cores": cpu_all, "clocks": clocks.summary(), "e2e": e2e,
        "gpu_launches": (4 if args.layout_two_launches else 3) * args.steps,  # per step: layout + notify
                                                                              # (one or two), dispatch, combine
        "wall_s_timed": round(wall, 3), "ops": ops, "parity": parity,
    }
    if rank == 0:
        print(json.dumps(result), flush=True)
    if parity.get("checked") and not parity.get("ok"):
        sys.exit(1)


def timed(fn, reps, stream, warmup=3, batches=5):
    """Steady-state time of one call: `reps` calls queued back to back between two events
    (host launch overhead hidden behind the GPU work), median over `batches` such runs."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(batches):
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b) / reps)
    return statistics.median(times)


def l2_bytes(dev):
    """The device's L2 size (129 MB on GB300 if the property is missing)."""
    return int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 129 << 20))


def timed_cold(fn, reps, stream, flush, warmup=3, clean=False):
    """Time of one call that starts with a cold L2: `flush` (a buffer twice the L2) is written
    before each call, outside the events -- which leaves the L2 full of dirty lines that the timed
    call writes back -- or, with clean=True, read (the L2 then holds only clean lines of the flush
    buffer); median over `reps` calls."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    flush64 = flush.view(torch.int64)
    for _ in range(reps):
        if clean:
            flush64.sum()
        else:
            flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.median(times)


def measure_launch_model(ep, dev, peak, st, reps=10, probe_sms=(16, 32)):
    """The SM-count model on the headline workload: per-SM rates of the dispatch (writes) and the
    combine (reads) measured with max_sms capping the data kernels, the SM counts the model then
    suggests, and the dispatch / combine timed at those counts against the full GPU."""
    stream = torch.cuda.current_stream(dev)
    shape = W.WORKLOADS[HEADLINE]
    R, T, H, E, K = shape.R, shape.T, shape.H, shape.E, shape.K
    n, hits, cap = R * T, st["hits"], st["cap"]
    disp_read, disp_write = 2 * H * n, 2 * H * hits
    comb_read, comb_write = 2 * H * hits, 2 * H * n
    recv_x = torch.empty((R, cap, H), dtype=torch.bfloat16, device=dev)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device=dev)

    def timed_pair(max_sms):
        h = ep.Handle(ep.Config(R, T, H, E, K, shape.C, shape.A, cap, max_sms=max_sms), dev)
        lay = ep.ep_get_dispatch_layout(h, st["idx_d"])
        ep.ep_dispatch(h, st["x_d"], topk_idx=st["idx_d"], num_tokens_per_rank=lay["num_tokens_per_rank"],
                       is_token_in_rank=lay["is_token_in_rank"], num_tokens_per_expert=lay["num_tokens_per_expert"],
                       recv_x=recv_x)
        d_ms = timed(lambda: ep.ep_dispatch(h, st["x_d"], cached=True, recv_x=recv_x), reps, stream)
        c_ms = timed(lambda: ep.ep_combine(h, recv_x, combined_x=out), reps, stream)
        h.check()
        h.destroy()
        return d_ms, c_ms

    per_sm = {}
    for m in probe_sms:
        d_ms, c_ms = timed_pair(m)
        per_sm[str(m)] = {"dispatch_us": round(d_ms * 1e3, 2), "combine_us": round(c_ms * 1e3, 2),
                          "dispatch_write_gbs_per_sm": round(disp_write / (d_ms / 1e3) / 1e9 / m, 2),
                          "combine_read_gbs_per_sm": round(comb_read / (c_ms / 1e3) / 1e9 / m, 2)}
    # the model's per-SM capabilities: the best rates seen with the GPU not yet saturated
    sm_write = max(v["dispatch_write_gbs_per_sm"] for v in per_sm.values())
    sm_read = max(v["combine_read_gbs_per_sm"] for v in per_sm.values())
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    model = dict(hbm_gbs=peak, sm_read_gbs=sm_read, sm_write_gbs=sm_write, num_device_sms=num_sms,
                 prefer_overlap_with_compute=True)
    n_d = ep.theoretical_num_sms(R, E, K, for_combine=False, **model)
    n_c = ep.theoretical_num_sms(R, E, K, for_combine=True, **model)
    d_ms, _ = timed_pair(n_d)
    _, c_ms = timed_pair(n_c)
    d_full, c_full = timed_pair(0)
    del recv_x, out
    return {"workload": f"{HEADLINE} (cached dispatch, combine of the received rows)",
            "rho_model": round(ep.expected_topk(R, E, K), 4), "rho_measured": round(hits / n, 4),
            "probe": per_sm, "sm_read_gbs": sm_read, "sm_write_gbs": sm_write, "hbm_gbs": peak,
            "suggested_sms": {"dispatch": n_d, "combine": n_c},
            "at_suggested": {"dispatch_us": round(d_ms * 1e3, 2), "combine_us": round(c_ms * 1e3, 2),
                             "full_gpu_dispatch_us": round(d_full * 1e3, 2),
                             "full_gpu_combine_us": round(c_full * 1e3, 2),
                             "dispatch_vs_full_gpu": round(d_full / d_ms, 3),
                             "combine_vs_full_gpu": round(c_full / c_ms, 3)}}


def run_ll_calls(n, small=False, hidden=0):
    """The low-latency path of ll_v3 alone, n dispatches then n combines back to back (a short, fixed
    launch sequence for profilers); prints the CUDA-event time per call.  small: 8 ranks, 16 experts,
    1024 tokens per rank -- the combine still reads 940 MB of rows (more than L2) while the expert
    output buffer holds 1.9 GB instead of ll_v3's 15 GB (for captures that save device memory).
    hidden: ll_v3's routing with this hidden size (the slot-row kernels do not depend on it; at 512
    the buffers hold 1.6 GB)."""
    from combine_get_dispatch_03_gb300 import ep
    dev = torch.device("cuda", 0)
    shape = W.WORKLOADS["ll_v3"]
    if small:
        shape = W.Shape("ll_v3_small", R=8, T=1024, H=shape.H, E=16, K=shape.K, routing=shape.routing,
                        max_tokens=1024, seed=shape.seed)
    if hidden:
        shape = W.Shape(**{**shape.__dict__, "H": hidden})
    idx, w = W.routing(shape)
    idx_d, w_d = torch.from_numpy(idx).to(dev), torch.from_numpy(w).to(dev)
    x_d = W.tokens_x(shape, device=dev)
    h = ep.Handle(ep.Config(shape.R, shape.max_tokens, shape.H, shape.E, shape.K, shape.C, 1, 0), dev)
    rows = shape.R * shape.max_tokens
    msgs = torch.empty((shape.R, shape.EL, rows, ep.ep_ll_msg_bytes(shape.H, True)), dtype=torch.uint8, device=dev)
    y = W.normal_bf16((shape.R, shape.EL, rows, shape.H), shape.seed, "lly", device=dev)
    out = torch.empty((shape.R, shape.T, shape.H), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.current_stream(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    for _ in range(n):
        ep.ep_ll_dispatch(h, x_d, idx_d, use_fp8=True, use_ue8m0=True, recv_msgs=msgs)
    b.record(s)
    b.synchronize()
    d_us = a.elapsed_time(b) * 1e3 / n
    a.record(s)
    for _ in range(n):
        ep.ep_ll_combine(h, y, idx_d, w_d, combined_x=out)
    b.record(s)
    b.synchronize()
    h.check()
    print(json.dumps({"ll_calls": n, "ll_dispatch_us": round(d_us, 2),
                      "ll_combine_us": round(a.elapsed_time(b) * 1e3 / n, 2)}))


def run_scan_calls(n, workload, tokens=0):
    """ep_layout_notify alone (the one-pass layout + record scan; with whole nodes of 8 ranks it also
    builds the node-level record), n calls back to back on a workload's routing, for profilers;
    prints the CUDA-event time per call."""
    from combine_get_dispatch_03_gb300 import ep
    dev = torch.device("cuda", 0)
    shape = W.WORKLOADS[workload]
    if tokens:
        shape = shape.scaled(T=tokens)
    idx, _ = W.routing(shape)
    idx_d = torch.from_numpy(idx).to(dev)
    h = ep.Handle(ep.Config(shape.R, shape.T, shape.H, shape.E, shape.K, shape.C, shape.A, receive_capacity(shape)),
                  dev)
    s = torch.cuda.current_stream(dev)
    lay = ep.ep_layout_notify(h, idx_d)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    for _ in range(n):
        ep.ep_layout_notify(h, idx_d, **lay)
    b.record(s)
    b.synchronize()
    h.check()
    one = a.elapsed_time(b) * 1e3 / n
    if n >= 3:  # the steady state of calls back to back, as bench times them (median of batches)
        one = timed(lambda: ep.ep_layout_notify(h, idx_d, **lay), n, s) * 1e3

    def two_calls():
        ep.ep_get_dispatch_layout(h, idx_d, **{k: lay[k] for k in ("num_tokens_per_rank", "num_tokens_per_rdma_rank",
                                                                   "num_tokens_per_expert", "is_token_in_rank")})
        ep.ep_notify_dispatch(h, lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                              num_recv_tokens_per_expert=lay["num_recv_tokens_per_expert"])

    two = timed(two_calls, max(n, 3), s) * 1e3 if n >= 3 else None
    h.check()
    print(json.dumps({"scan_calls": n, "workload": shape.name, "R": shape.R, "T": shape.T,
                      "layout_notify_us": round(one, 2),
                      "two_separate_calls_us": round(two, 2) if two is not None else None}))


def fp8_inputs(shape, dev):
    """Already-cast tokens for the FP8-input dispatch: e4m3 codes (no NaN codes) and fp32 scales."""
    x8 = torch.randint(0, 126, (shape.R, shape.T, shape.H), dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
    xs = torch.rand((shape.R, shape.T, shape.H // 128), dtype=torch.float32, device=dev)
    return x8, xs


def run_fp8_calls(n, tokens=0, fp8_input=False):
    """The FP8 dispatch of fp8_zipf alone (fresh record, fused cast, top-k metadata), n calls back to
    back for profilers (tokens per rank cut to `tokens` if given); prints the CUDA-event time per call.
    fp8_input: one cast dispatch builds the record, then n cached dispatches move e4m3 codes and
    fp32 scales unchanged."""
    from combine_get_dispatch_03_gb300 import ep
    dev = torch.device("cuda", 0)
    shape = W.WORKLOADS["fp8_zipf"]
    if tokens:
        shape = shape.scaled(T=tokens)
    st = prepare_normal(ep, shape, dev)
    h, cap = st["h"], st["cap"]
    lay = ep.ep_get_dispatch_layout(h, st["idx_d"])
    bufs = dict(recv_x=torch.empty((shape.R, cap, shape.H), dtype=torch.float8_e4m3fn, device=dev),
                recv_x_scales=torch.empty((shape.R, cap, shape.H // 128), dtype=torch.float32, device=dev))
    s = torch.cuda.current_stream(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def cast_call():
        ep.ep_dispatch(h, st["x_d"], topk_idx=st["idx_d"], topk_weights=st["w_d"], cast_to_fp8=True,
                       num_tokens_per_rank=lay["num_tokens_per_rank"], is_token_in_rank=lay["is_token_in_rank"],
                       num_tokens_per_expert=lay["num_tokens_per_expert"], **bufs)

    call = cast_call
    if fp8_input:
        cast_call()
        codes, scales = fp8_inputs(shape, dev)
        call = lambda: ep.ep_dispatch(h, codes, x_scales=scales, cached=True, **bufs)  # noqa: E731
    a.record(s)
    for _ in range(n):
        call()
    b.record(s)
    b.synchronize()
    h.check()
    print(json.dumps({"fp8_calls": n, "tokens_per_rank": shape.T, "fp8_input": fp8_input,
                      "fp8_dispatch_us": round(a.elapsed_time(b) * 1e3 / n, 2)}))


def measure_other_ops(ep, dev, peak, checks, reps=10):
    """Per-op times of the other workloads (median of reps, after warm-up); the outputs of each
    timed op's last call are appended to `checks` for the oracle check."""
    stream = torch.cuda.current_stream(dev)
    res = {}

    def report(name, ms, b, extra=None):
        d = {"us": round(ms * 1e3, 2), "GBps": round(total(b) / (ms / 1e3) / 1e9, 1),
             "payload_GBps": round(b["payload"] / (ms / 1e3) / 1e9, 1),
             "frac": round(total(b) / (ms / 1e3) / 1e9 / peak, 4)}
        d.update(extra or {})
        res[name] = d

    # FP8 dispatch with Zipf routing and masked slots
    shape = W.WORKLOADS["fp8_zipf"]
    st = prepare_normal(ep, shape, dev)
    h = st["h"]
    lay = ep.ep_get_dispatch_layout(h, st["idx_d"])
    bufs = dict(recv_x=torch.empty((shape.R, st["cap"], shape.H), dtype=torch.float8_e4m3fn, device=dev),
                recv_x_scales=torch.empty((shape.R, st["cap"], shape.H // 128), dtype=torch.float32, device=dev),
                recv_topk_idx=torch.empty((shape.R, st["cap"], shape.K), dtype=torch.int64, device=dev),
                recv_topk_weights=torch.empty((shape.R, st["cap"], shape.K), dtype=torch.float32, device=dev),
                num_recv_tokens_per_expert=torch.empty((shape.R, shape.EL), dtype=torch.int32, device=dev))
    fn = lambda: ep.ep_dispatch(h, st["x_d"], topk_idx=st["idx_d"], topk_weights=st["w_d"], cast_to_fp8=True,
                                num_tokens_per_rank=lay["num_tokens_per_rank"],
                                is_token_in_rank=lay["is_token_in_rank"],
                                num_tokens_per_expert=lay["num_tokens_per_expert"], **bufs)
    ms = timed(fn, reps, stream)
    h.check()
    checks.append(capture_normal("fp8_zipf.dispatch_fp8", shape, h, st["idx"], st["w"], st["x_d"], st["cap"], mode=1,
                                 layout=lay, nrpe=bufs["num_recv_tokens_per_expert"],
                                 recv={k: bufs[k] for k in ("recv_x", "recv_x_scales", "recv_topk_idx",
                                                            "recv_topk_weights")}))
    b = normal_bytes(shape.R, shape.T, shape.H, shape.K, st["hits"], fp8=True)
    report("fp8_zipf.dispatch_fp8", ms, {"payload": b["dispatch"]["payload"],
                                         "meta": b["dispatch"]["meta"] + total(b["notify"])},
           {"rho": round(st["hits"] / (shape.R * shape.T), 3)})
    # FP8 input (already cast: e4m3 codes and fp32 scales), cached record: bytes are moved as they are
    n, G = shape.R * shape.T, shape.H // 128
    x8, xs = fp8_inputs(shape, dev)
    fn8 = lambda: ep.ep_dispatch(h, x8, x_scales=xs, cached=True, recv_x=bufs["recv_x"],
                                 recv_x_scales=bufs["recv_x_scales"])
    ms8 = timed(fn8, reps, stream)
    h.check()
    checks.append(capture_normal("fp8_zipf.dispatch_fp8_input_cached", shape, h, st["idx"], st["w"], x8, st["cap"],
                                 mode=2, x_scales=xs, recv={k: bufs[k] for k in ("recv_x", "recv_x_scales")}))
    row8 = shape.H + 4 * G
    report("fp8_zipf.dispatch_fp8_input_cached", ms8,
           {"payload": n * row8 + st["hits"] * row8, "meta": n * shape.R * 4},
           {"note": "e4m3 codes + fp32 scales in, moved unchanged; record of the cast dispatch reused"})
    h.destroy()
    del bufs, st, lay, x8, xs
    torch.cuda.empty_cache()

    # combine-heavy: cached record, fresh expert outputs, two biases, weight reduction
    shape = W.WORKLOADS["combine_heavy"]
    st = prepare_normal(ep, shape, dev)
    h = st["h"]
    lay = ep.ep_get_dispatch_layout(h, st["idx_d"])
    d = ep.ep_dispatch(h, st["x_d"], topk_idx=st["idx_d"], topk_weights=st["w_d"],
                       num_tokens_per_rank=lay["num_tokens_per_rank"], is_token_in_rank=lay["is_token_in_rank"],
                       num_tokens_per_expert=lay["num_tokens_per_expert"])
    ms_disp = timed(lambda: ep.ep_dispatch(h, st["x_d"], cached=True, recv_x=d["recv_x"]), reps, stream)
    b0, b1 = W.biases(shape, device=dev)
    ys = [W.expert_outputs(shape, shape.R * st["cap"], i, device=dev).view(shape.R, st["cap"], shape.H)
          for i in range(2)]
    out = torch.empty((shape.R, shape.T, shape.H), dtype=torch.bfloat16, device=dev)
    cw = torch.empty((shape.R, shape.T, shape.K), dtype=torch.float32, device=dev)
    it = [0]

    def comb():
        it[0] += 1
        ep.ep_combine(h, ys[it[0] % 2], topk_weights=d["recv_topk_weights"], bias_0=b0, bias_1=b1,
                      combined_x=out, combined_topk_weights=cw)

    ms = timed(comb, reps, stream)
    h.check()
    checks.append(capture_normal("combine_heavy.combine", shape, h, st["idx"], st["w"], st["x_d"], st["cap"],
                                 layout=lay, recv=dict(recv_x=d["recv_x"]),
                                 combine=dict(y=ys[it[0] % 2], out=out, out_w=cw, b0=b0, b1=b1)))
    b = normal_bytes(shape.R, shape.T, shape.H, shape.K, st["hits"], biases=2)
    report("combine_heavy.combine", ms, b["combine"], {"rho": round(st["hits"] / (shape.R * shape.T), 3)})
    report("combine_heavy.dispatch_cached", ms_disp, {"payload": b["dispatch"]["payload"],
                                                      "meta": shape.R * shape.T * shape.R * 4})
    # the one-launch layout + record with the node-level record: 16 ranks are 2 nodes of 8
    R16, T16 = shape.R, shape.T
    lay_n = dict(num_tokens_per_rank=torch.empty((R16, R16), dtype=torch.int32, device=dev),
                 num_tokens_per_rdma_rank=torch.empty((R16, (R16 + 7) // 8), dtype=torch.int32, device=dev),
                 num_tokens_per_expert=torch.empty((R16, shape.E), dtype=torch.int32, device=dev),
                 is_token_in_rank=torch.empty((R16, T16, R16), dtype=torch.bool, device=dev),
                 num_recv_tokens_per_expert=torch.empty((R16, shape.EL), dtype=torch.int32, device=dev))
    ms_ln = timed(lambda: ep.ep_layout_notify(h, st["idx_d"], **lay_n), reps, stream)
    h.check()
    checks.append(capture_layout("combine_heavy.layout_notify_nodes", shape, h, st["idx"], lay_n))
    res["combine_heavy.layout_notify_nodes"] = {
        "us": round(ms_ln * 1e3, 2),
        "note": "one launch of the look-back scan with the node-level record (2 nodes of 8 ranks); latency-bound "
                "(about 5 MB moved), so no bandwidth fraction"}
    h.destroy()
    del d, ys, out, cw, b0, b1, st, lay
    torch.cuda.empty_cache()

    # low latency: FP8 + UE8M0 dispatch, weighted combine
    shape = W.WORKLOADS["ll_v3"]
    idx, w = W.routing(shape)
    idx_d, w_d = torch.from_numpy(idx).to(dev), torch.from_numpy(w).to(dev)
    x_d = W.tokens_x(shape, device=dev)
    h = ep.Handle(ep.Config(shape.R, shape.max_tokens, shape.H, shape.E, shape.K, shape.C, 1, 0), dev)
    msg = ep.ep_ll_msg_bytes(shape.H, True)
    msgs = torch.empty((shape.R, shape.EL, shape.R * shape.max_tokens, msg), dtype=torch.uint8, device=dev)
    cnt = torch.empty((shape.R, shape.EL), dtype=torch.int32, device=dev)
    rng_ = torch.empty((shape.R, shape.EL, shape.R), dtype=torch.int64, device=dev)
    fn = lambda: ep.ep_ll_dispatch(h, x_d, idx_d, use_fp8=True, use_ue8m0=True, recv_msgs=msgs,
                                   packed_recv_count=cnt, packed_recv_layout_range=rng_)
    ms_d = timed(fn, reps, stream)
    flush = torch.empty(2 * l2_bytes(dev), dtype=torch.uint8, device=dev)
    cold_d = timed_cold(fn, 2 * reps, stream, flush)
    clean_d = timed_cold(fn, 2 * reps, stream, flush, clean=True)
    y = W.normal_bf16((shape.R, shape.EL, shape.R * shape.max_tokens, shape.H), shape.seed, "lly", device=dev)
    out = torch.empty((shape.R, shape.T, shape.H), dtype=torch.bfloat16, device=dev)
    ms_c = timed(lambda: ep.ep_ll_combine(h, y, idx_d, w_d, combined_x=out), reps, stream)
    cold_c = timed_cold(lambda: ep.ep_ll_combine(h, y, idx_d, w_d, combined_x=out), 2 * reps, stream, flush)
    clean_c = timed_cold(lambda: ep.ep_ll_combine(h, y, idx_d, w_d, combined_x=out), 2 * reps, stream, flush,
                         clean=True)
    h.check()
    checks.append(capture_ll("ll_v3.ll_dispatch_fp8_ue8m0+ll_combine", shape, h, idx, w, x_d,
                             dict(recv_msgs=msgs, packed_recv_count=cnt, packed_recv_layout_range=rng_, y=y,
                                  combined_x=out)))
    n_valid = int((idx >= 0).sum())
    b = ll_bytes(shape.R, shape.T, shape.H, shape.K, n_valid, msg)
    warm = "calls back to back (the 58.7 MB of tokens can stay in the 129 MB L2)"
    cold_note = ("cold_us: L2 written over before each call (the call also writes back the flush's dirty lines); "
                 "cold_clean_us: L2 filled by reading a 2x-L2 buffer before each call (clean lines)")
    for name, ms, bb, cold, clean in (("ll_v3.ll_dispatch_fp8_ue8m0", ms_d, b["ll_dispatch"], cold_d, clean_d),
                                      ("ll_v3.ll_combine", ms_c, b["ll_combine"], cold_c, clean_c)):
        report(name, ms, bb, {"note": warm, "cold_us": round(cold * 1e3, 2), "cold_clean_us": round(clean * 1e3, 2),
                              "cold_clean_frac": round(total(bb) / clean / 1e6 / peak, 4), "cold_note": cold_note})
    del flush, y

    # the same dispatch with rank 5 masked in the mask buffer: its slots are dropped on both sides
    masked = 5
    hm = ep.Handle(ep.Config(shape.R, shape.max_tokens, shape.H, shape.E, shape.K, shape.C, 1, 0), dev)
    ep.ep_update_mask_buffer(hm, masked, True)
    ms_m = timed(lambda: ep.ep_ll_dispatch(hm, x_d, idx_d, use_fp8=True, use_ue8m0=True, recv_msgs=msgs,
                                           packed_recv_count=cnt, packed_recv_layout_range=rng_), reps, stream)
    hm.check()
    mask = np.zeros(shape.R, np.int32)
    mask[masked] = 1
    checks.append(capture_ll("ll_v3.ll_dispatch_fp8_ue8m0_rank_masked", shape, hm, idx, w, x_d,
                             dict(recv_msgs=msgs, packed_recv_count=cnt, packed_recv_layout_range=rng_),
                             rank_mask=mask))
    src = np.arange(shape.R)[:, None, None]
    n_valid_m = int(((idx >= 0) & (src != masked) & (idx // shape.EL != masked)).sum())
    report("ll_v3.ll_dispatch_fp8_ue8m0_rank_masked", ms_m,
           ll_bytes(shape.R, shape.T, shape.H, shape.K, n_valid_m, msg)["ll_dispatch"],
           {"note": f"rank {masked} masked: its {n_valid - n_valid_m} slots are dropped on both sides; every token "
                    "row is still read"})
    hm.destroy()
    del msgs

    # bf16 messages, and the combine reading the expert outputs in place in the message buffer (the
    # payloads as dispatched stand for the experts' outputs: identity experts)
    msg16 = ep.ep_ll_msg_bytes(shape.H, False)
    msgs16 = torch.empty((shape.R, shape.EL, shape.R * shape.max_tokens, msg16), dtype=torch.uint8, device=dev)
    ep.ep_ll_dispatch(h, x_d, idx_d, use_fp8=False, recv_msgs=msgs16, packed_recv_count=cnt,
                      packed_recv_layout_range=rng_)
    px, _, _ = ep.ll_views(msgs16, shape.H, False)
    ms_z = timed(lambda: ep.ep_ll_combine(h, px, idx_d, w_d, combined_x=out), reps, stream)
    h.check()
    checks.append(capture_ll("ll_v3.ll_dispatch_bf16+ll_combine_zero_copy", shape, h, idx, w, x_d,
                             dict(recv_msgs=msgs16, packed_recv_count=cnt, packed_recv_layout_range=rng_, y=px,
                                  combined_x=out), use_fp8=False, use_ue8m0=False))
    report("ll_v3.ll_combine_zero_copy", ms_z, b["ll_combine"],
           {"note": "the expert outputs read in place from the payloads of the bf16 message buffer (row stride "
                    f"{msg16} B)"})
    h.destroy()
    del msgs16, px, out
    torch.cuda.empty_cache()

    # the small case (L2-resident, launch-bound): eager calls and one CUDA graph of the step
    shape = W.WORKLOADS["normal_small"]
    st = prepare_normal(ep, shape, dev)
    h = st["h"]
    R, T, H, E, K, cap = shape.R, shape.T, shape.H, shape.E, shape.K, st["cap"]
    lay = dict(num_tokens_per_rank=torch.empty((R, R), dtype=torch.int32, device=dev), num_tokens_per_rdma_rank=None,
               num_tokens_per_expert=torch.empty((R, E), dtype=torch.int32, device=dev),
               is_token_in_rank=torch.empty((R, T, R), dtype=torch.bool, device=dev))
    bufs = dict(recv_x=torch.empty((R, cap, H), dtype=torch.bfloat16, device=dev),
                recv_topk_idx=torch.empty((R, cap, K), dtype=torch.int64, device=dev),
                recv_topk_weights=torch.empty((R, cap, K), dtype=torch.float32, device=dev),
                num_recv_tokens_per_expert=torch.empty((R, shape.EL), dtype=torch.int32, device=dev))
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device=dev)
    cw = torch.empty((R, T, K), dtype=torch.float32, device=dev)

    def small_step():
        ep.ep_get_dispatch_layout(h, st["idx_d"], **lay)
        ep.ep_dispatch(h, st["x_d"], topk_idx=st["idx_d"], topk_weights=st["w_d"],
                       num_tokens_per_rank=lay["num_tokens_per_rank"], is_token_in_rank=lay["is_token_in_rank"],
                       num_tokens_per_expert=lay["num_tokens_per_expert"], **bufs)
        ep.ep_combine(h, bufs["recv_x"], topk_weights=bufs["recv_topk_weights"], combined_x=out,
                      combined_topk_weights=cw)

    ms = timed(small_step, reps, stream)
    h.check()
    b = normal_bytes(R, T, H, K, st["hits"])
    step_b = {"payload": b["dispatch"]["payload"] + b["combine"]["payload"],
              "meta": sum(v["meta"] for v in b.values())}
    flush = torch.empty(2 * l2_bytes(dev), dtype=torch.uint8, device=dev)
    cold = timed_cold(small_step, 2 * reps, stream, flush)
    del flush
    report("normal_small.step", ms, step_b, {"note": "L2-resident; eager calls, launch-bound",
                                             "cold_us": round(cold * 1e3, 2),
                                             "cold_note": "L2 written over before each step"})
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        small_step()
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        small_step()
    ms = timed(graph.replay, reps, stream)
    h.check()
    checks.append(capture_normal("normal_small.step_graph", shape, h, st["idx"], st["w"], st["x_d"], cap, layout=lay,
                                 nrpe=bufs["num_recv_tokens_per_expert"],
                                 recv={k: bufs[k] for k in ("recv_x", "recv_topk_idx", "recv_topk_weights")},
                                 combine=dict(y=bufs["recv_x"], out=out, out_w=cw)))
    report("normal_small.step_graph", ms, step_b, {"note": "the same step captured once in a CUDA graph"})
    h.destroy()
    return res


# ----------------------------------------------------------------------------- CPU oracle

def capture_layout(name, shape, h, idx, lay):
    """Host copies of one ep_layout_notify call: layout outputs, the record and, with whole nodes of 8
    ranks, the node-level record -- all whole."""
    rec = dict(kind="layout", name=name, shape=shape, idx=idx, cap=h.cfg.recv_capacity,
               layout={k: (_host(v) if v is not None else None) for k, v in lay.items()},
               record={k: _host(h.export(k)) for k in
                       ("rank_prefix_matrix", "channel_prefix_matrix", "recv_channel_prefix_matrix", "num_recv",
                        "send_head", "recv_src_idx")})
    if shape.R > 8 and shape.R % 8 == 0:
        rec["nodes"] = {k: _host(h.export(k)) for k in ("rdma_channel_prefix_matrix", "recv_rdma_rank_prefix_sum")}
    return rec


def _check_layout(O, rec):
    """The oracle on one captured layout + record call, every output whole."""
    shape, cap = rec["shape"], rec["cap"]
    bad = []
    lay = O.get_dispatch_layout(rec["idx"], shape.E, with_rdma=True)
    n = O.dispatch_notify(lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                          shape.C, shape.A, cap)
    for k, v in rec["layout"].items():
        if k == "num_recv_tokens_per_expert":
            if v is not None and not np.array_equal(v, n["num_recv_tokens_per_expert"]):
                bad.append(k)
        elif v is not None and not np.array_equal(v, lay[k]):
            bad.append(k)
    for k, v in rec["record"].items():
        want = n[k]
        if k == "recv_src_idx":
            m = np.arange(cap)[None, :] < np.minimum(n["num_recv"], cap)[:, None]
            v, want = v[m], want[m]
        if not np.array_equal(v, want):
            bad.append(k)
    if "nodes" in rec:
        nodes = O.rdma_prefix(lay["is_token_in_rank"], shape.C)
        for k, v in rec["nodes"].items():
            if not np.array_equal(v, nodes[k]):
                bad.append(k)
    return bad, shape.R * shape.T


def _check_normal(O, rec):
    """The oracle on one captured normal-mode call: layout and record whole, rows and tokens sampled."""
    shape, cap, toks, pairs = rec["shape"], rec["cap"], rec["toks"], rec["pairs"]
    R, T, H, E, K = shape.R, shape.T, shape.H, shape.E, shape.K
    bad = []
    lay = O.get_dispatch_layout(rec["idx"], E, with_rdma=True)
    n = O.dispatch_notify(lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                          shape.C, shape.A, cap)
    for k, v in rec.get("layout", {}).items():
        if v is not None and not np.array_equal(v, lay[k]):
            bad.append(k)
    for k, v in rec["record"].items():
        want = n[k]
        if k == "recv_src_idx":
            m = np.arange(cap)[None, :] < np.minimum(n["num_recv"], cap)[:, None]
            v, want = v[m], want[m]
        if not np.array_equal(v, want):
            bad.append(k)
    if "nrpe" in rec and not np.array_equal(rec["nrpe"], n["num_recv_tokens_per_expert"]):
        bad.append("num_recv_tokens_per_expert")
    mode = rec["mode"]
    x = np.zeros((R * T, H), np.uint8 if mode == 2 else np.uint16)  # only the sampled rows are touched
    x[toks] = rec["x_rows"]
    xs = None
    if "x_scale_rows" in rec:
        xs = np.zeros((R * T, H // 128), np.float32)
        xs[toks] = rec["x_scale_rows"]
        xs = xs.reshape(R, T, H // 128)
    c = rec.get("combine")
    with_topk = "recv_topk_idx" in rec.get("recv", {}) or (c is not None and "out_w" in c)
    d = O.dispatch(x.reshape(R, T, H), n["send_head"], cap, E, mode=mode, x_scales=xs,
                   topk_idx=rec["idx"] if with_topk else None, topk_weights=rec["w"] if with_topk else None,
                   tokens=toks)
    for k, v in rec.get("recv", {}).items():
        if not np.array_equal(v, d[k][pairs[:, 0], pairs[:, 1]]):
            bad.append(k)
    if c is not None:
        y = np.zeros((R, cap, H), np.uint16)
        y[pairs[:, 0], pairs[:, 1]] = c["y_rows"]
        rw = d["recv_topk_weights"] if "out_w" in c else None  # the oracle's own dispatched weights
        bias = {}
        for b in ("b0", "b1"):
            if b + "_rows" in c:
                a = np.zeros((R * T, H), np.uint16)
                a[toks] = c[b + "_rows"]
                bias[b] = a.reshape(R, T, H)
        oc = O.combine(y, n["send_head"], recv_topk_weights=rw, bias0=bias.get("b0"), bias1=bias.get("b1"),
                       num_topk=K, tokens=toks)
        if not np.array_equal(c["out_rows"], oc["out"].reshape(-1, H)[toks]):
            bad.append("combined_x")
        if "out_w" in c:
            # every token: one nonzero term per valid slot, so the reduction returns the routing's weights
            want = np.where(rec["idx"] >= 0, rec["w"], 0).astype(np.float32)
            if not np.array_equal(c["out_w"], want) or \
                    not np.array_equal(c["out_w"].reshape(-1, K)[toks], oc["combined_topk_weights"].reshape(-1, K)[toks]):
                bad.append("combined_topk_weights")
    return bad, len(toks)


def _check_ll(O, rec):
    """The oracle on one captured low-latency dispatch + combine: counts, layout range and the slot map
    whole, the sampled tokens' messages and combined outputs."""
    shape, toks = rec["shape"], rec["toks"]
    R, T, H, E, K, maxT = shape.R, shape.T, shape.H, shape.E, shape.K, shape.max_tokens
    bad = []
    x = np.zeros((R * T, H), np.uint16)
    x[toks] = rec["x_rows"]
    o = O.ll_dispatch(x.reshape(R, T, H), rec["idx"], maxT, E, use_fp8=rec.get("use_fp8", True),
                      use_ue8m0=rec.get("use_ue8m0", True), rank_mask=rec.get("rank_mask"))
    for k in ("packed_recv_count", "packed_recv_layout_range", "slot_row"):
        if not np.array_equal(rec[k], o[k]):
            bad.append(k)
    want = o["msgs_by_slot"].reshape(R * T, K, -1)[toks]
    ok = rec["ok"]
    if not np.array_equal(rec["msg_rows"][ok], want[ok]):
        bad.append("messages")
    if "y_rows" in rec:
        y = np.zeros((R, E // R, R * maxT, H), np.uint16)
        e = rec["idx"].reshape(-1, K)[toks]
        sl = o["slot_row"].reshape(-1, K)[toks]
        for i in range(len(toks)):
            for k in range(K):
                if ok[i, k]:
                    y[e[i, k] // (E // R), e[i, k] % (E // R), sl[i, k]] = rec["y_rows"][i, k]
        got = O.ll_combine(y, rec["idx"], rec["w"], o["slot_row"], maxT, E, tokens=toks)
        if not np.array_equal(rec["out_rows"], got.reshape(-1, H)[toks]):
            bad.append("ll combined_x")
    return bad, len(toks)


def cpu_parity(checks):
    """The CPU-oracle leg's check of the timed calls: each captured call against the oracle."""
    import oracle as O
    t0 = time.perf_counter()
    res, ok = {}, True
    for rec in checks:
        bad, n = {"ll": _check_ll, "layout": _check_layout}.get(rec["kind"], _check_normal)(O, rec)
        res[rec["name"]] = {"status": "ok" if not bad else "MISMATCH: " + ", ".join(bad), "tokens_sampled": n}
        ok = ok and not bad
    return {"checked": True, "ok": ok, "calls": res,
            "whole": "layout outputs, the dispatch record, num_recv_tokens_per_expert, the combined top-k weights, "
                     "LL counts / layout range / slot map",
            "sampled": "receive rows and scales of the sampled tokens' destinations, their combined tokens, "
                       "their LL messages",
            "what": "the outputs of the last timed call of each line, against the CPU oracle on the same inputs",
            "seconds": round(time.perf_counter() - t0, 2)}


def cpu_sample(shape, tokens: int):
    """Inputs of the oracle sample: the first `tokens` tokens of every rank of the workload."""
    sub = W.Shape(**{**shape.__dict__, "T": tokens})
    idx, w = W.routing(shape)
    idx, w = np.ascontiguousarray(idx[:, :tokens]), np.ascontiguousarray(w[:, :tokens])
    x = W.bf16_bits(W.tokens_x(shape, device="cuda" if torch.cuda.is_available() else "cpu")[:, :tokens])
    return sub, idx, w, x


def cpu_step(sub, idx, w, x):
    """One oracle pass (layout + notify + dispatch + combine); returns (seconds, hits)."""
    import oracle as O
    t0 = time.perf_counter()
    lay = O.get_dispatch_layout(idx, sub.E, with_rdma=sub.R > 8)
    cap = int(lay["num_tokens_per_rank"].sum(axis=0).max())
    n = O.dispatch_notify(lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                          sub.C, sub.A, cap)
    d = O.dispatch(x, n["send_head"], cap, sub.E, topk_idx=idx, topk_weights=w)
    O.combine(d["recv_x"], n["send_head"], recv_topk_weights=d["recv_topk_weights"])
    return time.perf_counter() - t0, int(lay["num_tokens_per_rank"].sum())


def cpu_step_threads(sub, idx, w, x, threads: int):
    """The same oracle pass with the dispatch and combine token loops split over `threads` host
    threads, contiguous token blocks each (the oracle's C calls release the interpreter lock; the
    blocks write disjoint rows of the shared outputs).  Layout and notify stay single-threaded."""
    import oracle as O
    from concurrent.futures import ThreadPoolExecutor
    t0 = time.perf_counter()
    lay = O.get_dispatch_layout(idx, sub.E, with_rdma=sub.R > 8)
    cap = int(lay["num_tokens_per_rank"].sum(axis=0).max())
    n = O.dispatch_notify(lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                          sub.C, sub.A, cap)
    blocks = np.array_split(np.arange(sub.R * sub.T, dtype=np.int64), threads)
    d = dict(recv_x=np.zeros((sub.R, cap, sub.H), np.uint16),
             recv_topk_idx=np.full((sub.R, cap, sub.K), -2, np.int64),
             recv_topk_weights=np.full((sub.R, cap, sub.K), np.nan, np.float32))
    c = dict(out=np.zeros((sub.R, sub.T, sub.H), np.uint16),
             combined_topk_weights=np.zeros((sub.R, sub.T, sub.K), np.float32))
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda b: O.dispatch(x, n["send_head"], cap, sub.E, topk_idx=idx, topk_weights=w, tokens=b,
                                         out=d), blocks))
        list(ex.map(lambda b: O.combine(d["recv_x"], n["send_head"], recv_topk_weights=d["recv_topk_weights"],
                                        tokens=b, out=c), blocks))
    return time.perf_counter() - t0, int(lay["num_tokens_per_rank"].sum())


def cpu_describe(shape, tokens, threads: int = 1):
    how = "single-threaded C oracle" if threads == 1 else \
        f"C oracle with its dispatch and combine token loops over {threads} threads"
    return (f"{HEADLINE} restricted to the first {tokens} of {shape.T} tokens of each of the {shape.R} ranks: "
            f"layout + notify + dispatch + combine, {how}")


def cpu_tokens(shape, budget_s: float, passes: int) -> int:
    """Tokens per rank of the oracle sample so that `passes` passes take about budget_s seconds: one
    pass over 64 tokens per rank gives the oracle's cost per token (its work is linear in tokens)."""
    sub, idx, w, x = cpu_sample(shape, 64)
    dt, _ = cpu_step(sub, idx, w, x)
    t = int(budget_s / passes / (dt / 64)) // 64 * 64
    return max(64, min(shape.T, t))


def cpu_baseline(shape, budget_s: float, passes: int = 3):
    """The CPU oracle, as it stands, timed over `passes` passes of a sample of the workload sized to
    about budget_s seconds of CPU work in all."""
    tokens = cpu_tokens(shape, budget_s, passes)
    sub, idx, w, x = cpu_sample(shape, tokens)
    total, hits = 0.0, 0
    for _ in range(passes):
        dt, hits = cpu_step(sub, idx, w, x)
        total += dt
    b = normal_bytes(sub.R, tokens, sub.H, sub.K, hits)
    payload = b["dispatch"]["payload"] + b["combine"]["payload"]
    return {"value": round(payload * passes / total / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{cpu_describe(shape, tokens)}; {passes} passes", "seconds": round(total, 3),
            "tokens_per_s": round(sub.R * tokens * passes / total, 1)}


def cpu_baseline_all_cores(shape, budget_s: float, passes: int = 3):
    """The same oracle with its dispatch and combine token loops split over every host core the
    process may run on; the sample is sized like cpu_baseline's, scaled by the core count."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    tokens = cpu_tokens(shape, budget_s * cores, passes)
    sub, idx, w, x = cpu_sample(shape, tokens)
    total, hits = 0.0, 0
    for _ in range(passes):
        dt, hits = cpu_step_threads(sub, idx, w, x, cores)
        total += dt
    b = normal_bytes(sub.R, tokens, sub.H, sub.K, hits)
    payload = b["dispatch"]["payload"] + b["combine"]["payload"]
    return {"value": round(payload * passes / total / 1e9, 3), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{cpu_describe(shape, tokens, cores)}; {passes} passes", "seconds": round(total, 3),
            "tokens_per_s": round(sub.R * tokens * passes / total, 1)}


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores, W warm-up and K timed sample steps."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    shape = W.WORKLOADS[HEADLINE]
    tokens = cpu_tokens(shape, args.reference_seconds, args.warmup + args.steps)
    sub, idx, w, x = cpu_sample(shape, tokens)
    for _ in range(args.warmup):
        cpu_step(sub, idx, w, x)
    secs, hits = [], 0
    for _ in range(args.steps):
        dt, hits = cpu_step(sub, idx, w, x)
        secs.append(dt)
    b = normal_bytes(sub.R, tokens, sub.H, sub.K, hits)
    payload = b["dispatch"]["payload"] + b["combine"]["payload"]
    value = round(payload * len(secs) / sum(secs) / 1e9, 4)
    desc = cpu_describe(shape, tokens)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * sum(secs) / len(secs), 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": headline_config(shape.T, shape.R * receive_capacity(shape) * shape.H * 2 / 1e9, 1),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=24.0,
                    help="CPU work of the oracle baseline (three passes of a sample sized to it)")
    ap.add_argument("--reference-seconds", type=float, default=120.0,
                    help="--impl reference: the warm-up and timed steps together take about this long")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-ops", action="store_true")
    ap.add_argument("--ll-calls", type=int, default=0,
                    help="only run the ll_v3 low-latency dispatch and combine this many times each (profiling)")
    ap.add_argument("--ll-small", action="store_true",
                    help="with --ll-calls: 8 ranks, 16 experts, 1024 tokens per rank instead of ll_v3")
    ap.add_argument("--ll-hidden", type=int, default=0,
                    help="with --ll-calls: this hidden size instead of 7168 (a multiple of 512)")
    ap.add_argument("--fp8-calls", type=int, default=0,
                    help="only run the fp8_zipf FP8 dispatch (fresh record, cast) this many times (profiling)")
    ap.add_argument("--fp8-input", action="store_true",
                    help="with --fp8-calls: time cached dispatches of already-cast e4m3 tokens and scales")
    ap.add_argument("--scan-calls", type=int, default=0,
                    help="only run ep_layout_notify this many times on --scan-workload (profiling)")
    ap.add_argument("--scan-workload", default="combine_heavy",
                    help="with --scan-calls: the workload whose routing is scanned (combine_heavy: 2 nodes of 8)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--layout-two-launches", action="store_true",
                    help="run the step's layout and notify as the two separate calls (ep_get_dispatch_layout, "
                         "ep_notify_dispatch) instead of ep_layout_notify")
    ap.add_argument("--tokens", type=int, default=0,
                    help="tokens per rank of the headline workload (0 = its full 4096; smaller only for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.scan_calls:
        run_scan_calls(args.scan_calls, args.scan_workload, args.tokens)
    elif args.ll_calls:
        run_ll_calls(args.ll_calls, args.ll_small, args.ll_hidden)
    elif args.fp8_calls:
        run_fp8_calls(args.fp8_calls, args.tokens, args.fp8_input)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
