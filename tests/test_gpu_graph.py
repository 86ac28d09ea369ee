"""The path captured in CUDA graphs: layout -> dispatch -> combine and LL dispatch -> LL combine,
recorded once through the C ABI and replayed on new inputs copied into the captured buffers.
Every replay is compared with the CPU oracle, bit for bit."""
import numpy as np
import pytest
import torch

import oracle as O
from combine_get_dispatch_03_gb300 import ep
from combine_get_dispatch_03_gb300 import workloads as W

import _parity as P

pytestmark = pytest.mark.gpu


def test_normal_step_graph_replays_match_oracle():
    base = W.Shape("graph", R=8, T=200, H=1024, E=64, K=6, routing="gumbel", mask_p=0.05, A=4, seed=7001)
    routes = [W.routing(W.Shape(**{**base.__dict__, "seed": base.seed + i})) for i in range(3)]
    xs = [W.tokens_x(W.Shape(**{**base.__dict__, "seed": base.seed + i})) for i in range(3)]
    cap = max(P.needed_capacity(r[0], base.E) for r in routes)
    h = ep.Handle(P.config_of(base, cap))
    idx_d = torch.empty((base.R, base.T, base.K), dtype=torch.int64, device=P.DEV)
    w_d = torch.empty((base.R, base.T, base.K), dtype=torch.float32, device=P.DEV)
    x_d = torch.empty((base.R, base.T, base.H), dtype=torch.bfloat16, device=P.DEV)
    idx_d.copy_(torch.from_numpy(routes[0][0]))
    w_d.copy_(torch.from_numpy(routes[0][1]))
    x_d.copy_(xs[0])
    lay = dict(num_tokens_per_rank=torch.empty((base.R, base.R), dtype=torch.int32, device=P.DEV),
               num_tokens_per_rdma_rank=None,
               num_tokens_per_expert=torch.empty((base.R, base.E), dtype=torch.int32, device=P.DEV),
               is_token_in_rank=torch.empty((base.R, base.T, base.R), dtype=torch.bool, device=P.DEV))
    recv_x = torch.empty((base.R, cap, base.H), dtype=torch.bfloat16, device=P.DEV)
    recv_w = torch.empty((base.R, cap, base.K), dtype=torch.float32, device=P.DEV)
    recv_i = torch.empty((base.R, cap, base.K), dtype=torch.int64, device=P.DEV)
    nrpe = torch.empty((base.R, base.EL), dtype=torch.int32, device=P.DEV)
    out = torch.empty((base.R, base.T, base.H), dtype=torch.float32, device=P.DEV)
    out_w = torch.empty((base.R, base.T, base.K), dtype=torch.float32, device=P.DEV)

    def step():
        ep.ep_get_dispatch_layout(h, idx_d, **lay)
        ep.ep_dispatch(h, x_d, topk_idx=idx_d, topk_weights=w_d, num_tokens_per_rank=lay["num_tokens_per_rank"],
                       is_token_in_rank=lay["is_token_in_rank"], num_tokens_per_expert=lay["num_tokens_per_expert"],
                       recv_x=recv_x, recv_topk_idx=recv_i, recv_topk_weights=recv_w,
                       num_recv_tokens_per_expert=nrpe)
        ep.ep_combine(h, recv_x, topk_weights=recv_w, combined_x=out, combined_topk_weights=out_w,
                      out_dtype=torch.float32)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    assert h.status() == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for i in range(3):
        idx, w = routes[i]
        idx_d.copy_(torch.from_numpy(idx))
        w_d.copy_(torch.from_numpy(w))
        x_d.copy_(xs[i])
        graph.replay()
        torch.cuda.synchronize()
        assert h.status() == 0
        xb = W.bf16_bits(xs[i])
        lay_o = O.get_dispatch_layout(idx, base.E)
        n = O.dispatch_notify(lay_o["num_tokens_per_rank"], lay_o["is_token_in_rank"],
                              lay_o["num_tokens_per_expert"], base.C, base.A, cap)
        d = O.dispatch(xb, n["send_head"], cap, base.E, topk_idx=idx, topk_weights=w)
        c = O.combine(d["recv_x"], n["send_head"], recv_topk_weights=d["recv_topk_weights"], out_fp32=True)
        np.testing.assert_array_equal(P.host(lay["is_token_in_rank"]), lay_o["is_token_in_rank"])
        np.testing.assert_array_equal(P.host(nrpe), n["num_recv_tokens_per_expert"])
        rows = P.valid_rows(n["num_recv"], cap)
        np.testing.assert_array_equal(P.host(recv_x)[rows], d["recv_x"][rows])
        np.testing.assert_array_equal(P.host(out), c["out"])
        np.testing.assert_array_equal(P.host(out_w), c["combined_topk_weights"])


def test_low_latency_graph_replays_match_oracle():
    base = W.Shape("llgraph", R=8, T=24, H=1024, E=32, K=4, routing="uniform", max_tokens=32, seed=7101)
    maxT = base.max_tokens
    h = ep.Handle(P.config_of(base, 0))
    idx_d = torch.empty((base.R, base.T, base.K), dtype=torch.int64, device=P.DEV)
    w_d = torch.empty((base.R, base.T, base.K), dtype=torch.float32, device=P.DEV)
    x_d = torch.empty((base.R, base.T, base.H), dtype=torch.bfloat16, device=P.DEV)
    msg = ep.ep_ll_msg_bytes(base.H, True)
    msgs = torch.zeros((base.R, base.EL, base.R * maxT, msg), dtype=torch.uint8, device=P.DEV)
    cnt = torch.empty((base.R, base.EL), dtype=torch.int32, device=P.DEV)
    rng = torch.empty((base.R, base.EL, base.R), dtype=torch.int64, device=P.DEV)
    y = torch.empty((base.R, base.EL, base.R * maxT, base.H), dtype=torch.bfloat16, device=P.DEV)
    out = torch.empty((base.R, base.T, base.H), dtype=torch.bfloat16, device=P.DEV)
    cases = []
    for i in range(3):
        sh = W.Shape(**{**base.__dict__, "seed": base.seed + i})
        idx, w = W.routing(sh)
        cases.append((idx, w, W.tokens_x(sh), W.normal_bf16(tuple(y.shape), sh.seed, "gy")))
    idx_d.copy_(torch.from_numpy(cases[0][0]))
    w_d.copy_(torch.from_numpy(cases[0][1]))
    x_d.copy_(cases[0][2])
    y.copy_(cases[0][3])

    def step():
        ep.ep_ll_dispatch(h, x_d, idx_d, use_fp8=True, use_ue8m0=True, recv_msgs=msgs, packed_recv_count=cnt,
                          packed_recv_layout_range=rng)
        ep.ep_ll_combine(h, y, idx_d, w_d, combined_x=out)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    assert h.status() == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for idx, w, x, yv in cases:
        idx_d.copy_(torch.from_numpy(idx))
        w_d.copy_(torch.from_numpy(w))
        x_d.copy_(x)
        y.copy_(yv)
        graph.replay()
        torch.cuda.synchronize()
        assert h.status() == 0
        ora = O.ll_dispatch(W.bf16_bits(x), idx, maxT, base.E, use_fp8=True, use_ue8m0=True)
        np.testing.assert_array_equal(P.host(cnt), ora["packed_recv_count"])
        np.testing.assert_array_equal(P.host(rng), ora["packed_recv_layout_range"])
        s_, t_, k_ = np.nonzero(idx >= 0)
        e = idx[s_, t_, k_]
        rows = ora["slot_row"][s_, t_, k_]
        np.testing.assert_array_equal(P.host(msgs)[e // base.EL, e % base.EL, rows], ora["msgs_by_slot"][s_, t_, k_])
        want = O.ll_combine(W.bf16_bits(yv), idx, w, ora["slot_row"], maxT, base.E)
        np.testing.assert_array_equal(P.host(out), want)


def test_layout_notify_graph_replays():
    """The one-launch layout + record (its grid barrier counts generations) captured in a graph with
    the prepared dispatch and the combine, replayed on three routings."""
    base = W.Shape("graph_ln", R=16, T=300, H=512, E=128, K=8, routing="zipf", mask_p=0.05, seed=7201)
    routes = [W.routing(W.Shape(**{**base.__dict__, "seed": base.seed + i})) for i in range(3)]
    x_h = W.tokens_x(base)
    cap = max(P.needed_capacity(r[0], base.E) for r in routes)
    h = ep.Handle(P.config_of(base, cap))
    idx_d = torch.empty((base.R, base.T, base.K), dtype=torch.int64, device=P.DEV)
    x_d = x_h.to(P.DEV)
    idx_d.copy_(torch.from_numpy(routes[0][0]))
    R, E, EL = base.R, base.E, base.EL
    lay = dict(num_tokens_per_rank=torch.empty((R, R), dtype=torch.int32, device=P.DEV),
               num_tokens_per_rdma_rank=torch.empty((R, 2), dtype=torch.int32, device=P.DEV),
               num_tokens_per_expert=torch.empty((R, E), dtype=torch.int32, device=P.DEV),
               is_token_in_rank=torch.empty((R, base.T, R), dtype=torch.bool, device=P.DEV),
               num_recv_tokens_per_expert=torch.empty((R, EL), dtype=torch.int32, device=P.DEV))
    recv_x = torch.empty((R, cap, base.H), dtype=torch.bfloat16, device=P.DEV)
    out = torch.empty((R, base.T, base.H), dtype=torch.bfloat16, device=P.DEV)

    def step():
        ep.ep_layout_notify(h, idx_d, **lay)
        ep.ep_dispatch(h, x_d, topk_idx=idx_d, prepared=True, recv_x=recv_x, with_topk=False)
        ep.ep_combine(h, recv_x, combined_x=out)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    assert h.status() == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    xb = W.bf16_bits(x_h)
    for idx, _ in routes:
        idx_d.copy_(torch.from_numpy(idx))
        graph.replay()
        torch.cuda.synchronize()
        assert h.status() == 0
        ora_lay = O.get_dispatch_layout(idx, E)
        n = O.dispatch_notify(ora_lay["num_tokens_per_rank"], ora_lay["is_token_in_rank"],
                              ora_lay["num_tokens_per_expert"], base.C, base.A, cap)
        d = O.dispatch(xb, n["send_head"], cap, E)
        c = O.combine(d["recv_x"], n["send_head"])
        np.testing.assert_array_equal(P.host(lay["num_tokens_per_rdma_rank"]), ora_lay["num_tokens_per_rdma_rank"])
        np.testing.assert_array_equal(P.host(lay["num_recv_tokens_per_expert"]), n["num_recv_tokens_per_expert"])
        np.testing.assert_array_equal(P.host(out), c["out"])

