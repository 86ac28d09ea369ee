"""The five named workloads at their full sizes, in the launch configuration bench.py times.

The benchmark's own step and ops (test_*_timed_*) are compared whole with the
oracle: every layout output, the whole dispatch record, every receive row and
every combined token, with the oracle's token loops split over the host cores.
The other tests compare integer outputs whole and payload rows and combine
outputs on a seeded sample of tokens, plus properties over every token.
"""
import numpy as np
import pytest
import torch

import oracle as O
from combine_get_dispatch_03_gb300 import ep
from combine_get_dispatch_03_gb300 import workloads as W

import _parity as P

pytestmark = pytest.mark.gpu

N_SAMPLE = 384


def setup_normal(shape, dev="cuda"):
    idx, w = W.routing(shape)
    idx_d, w_d = torch.from_numpy(idx).to(dev), torch.from_numpy(w).to(dev)
    x_d = W.tokens_x(shape, device=dev)
    ora_lay = O.get_dispatch_layout(idx, shape.E, with_rdma=shape.R > 8)
    cap = int(ora_lay["num_tokens_per_rank"].sum(axis=0).max())
    h = ep.Handle(P.config_of(shape, cap))
    lay = ep.ep_get_dispatch_layout(h, idx_d)
    ora_n = O.dispatch_notify(ora_lay["num_tokens_per_rank"], ora_lay["is_token_in_rank"],
                              ora_lay["num_tokens_per_expert"], shape.C, shape.A, cap)
    return dict(idx=idx, w=w, idx_d=idx_d, w_d=w_d, x_d=x_d, cap=cap, h=h, lay=lay, ora_lay=ora_lay, ora_n=ora_n)


def rows_of(send_head, tokens, R):
    """(r, row) pairs of every destination of the sampled tokens."""
    sh = send_head.reshape(-1, R)[tokens]
    rr, kk = np.nonzero(sh >= 0)
    return np.stack([kk, sh[rr, kk]], axis=1)


def gather_rows(t, pairs):
    r = torch.from_numpy(pairs[:, 0]).to(t.device)
    row = torch.from_numpy(pairs[:, 1]).to(t.device)
    return t[r, row]


def lazy_host_rows(shape3, dtype, pairs, values):
    """A (lazily zero-filled) host array holding `values` at the given (r, row) pairs."""
    a = np.zeros(shape3, dtype)
    a[pairs[:, 0], pairs[:, 1]] = values
    return a


@pytest.mark.parametrize("name", ["normal_small", "normal_v3", "fp8_zipf", "combine_heavy"])
def test_layout_and_record_full(name):
    shape = W.WORKLOADS[name]
    st = setup_normal(shape)
    P.compare_layout(st["lay"], st["ora_lay"])
    d = ep.ep_dispatch(st["h"], st["x_d"], topk_idx=st["idx_d"], topk_weights=st["w_d"],
                       num_tokens_per_rank=st["lay"]["num_tokens_per_rank"],
                       is_token_in_rank=st["lay"]["is_token_in_rank"],
                       num_tokens_per_expert=st["lay"]["num_tokens_per_expert"],
                       cast_to_fp8=name == "fp8_zipf")
    assert st["h"].status() == 0
    P.compare_record(st["h"], st["ora_n"], shape.T)
    np.testing.assert_array_equal(P.host(d["num_recv_tokens_per_expert"]), st["ora_n"]["num_recv_tokens_per_expert"])


def test_normal_small_end_to_end():
    """The small workload whole: every output against the oracle, and combine / ranks_hit == x."""
    shape = W.WORKLOADS["normal_small"]
    res = P.run_normal(shape, with_weights=True)
    assert res["status"] == 0 and res["combine_status"] == 0
    P.compare_dispatch(res, shape, O.MODE_BF16)
    np.testing.assert_array_equal(P.host(res["c"]["combined_x"]), res["ora_c"]["out"])
    res32 = P.run_normal(shape, with_weights=True, out_fp32=True)
    n = res32["ora_lay"]["is_token_in_rank"].sum(axis=2).astype(np.float32)
    x = (res32["x"].astype(np.uint32) << 16).view(np.float32)
    got = P.host(res32["c"]["combined_x"])
    hit = n > 0
    np.testing.assert_array_equal((got / np.where(hit, n, 1)[..., None])[hit], x[hit])


@pytest.mark.parametrize("name,mode", [("normal_v3", O.MODE_BF16), ("fp8_zipf", O.MODE_CAST_FP8)])
def test_dispatch_combine_full_sampled(name, mode):
    shape = W.WORKLOADS[name]
    st = setup_normal(shape)
    h = st["h"]
    d = ep.ep_dispatch(h, st["x_d"], topk_idx=st["idx_d"], topk_weights=st["w_d"],
                       num_tokens_per_rank=st["lay"]["num_tokens_per_rank"],
                       is_token_in_rank=st["lay"]["is_token_in_rank"],
                       num_tokens_per_expert=st["lay"]["num_tokens_per_expert"], cast_to_fp8=mode == O.MODE_CAST_FP8)
    assert h.status() == 0
    toks = W.sample_tokens(shape, N_SAMPLE)
    x_rows = P.host(st["x_d"].view(-1, shape.H)[torch.from_numpy(toks).to(st["x_d"].device)])
    x_host = np.zeros((shape.R * shape.T, shape.H), np.uint16)
    x_host[toks] = x_rows
    x_host = x_host.reshape(shape.R, shape.T, shape.H)
    cap = st["cap"]
    pairs = rows_of(st["ora_n"]["send_head"], toks, shape.R)
    ora = O.dispatch(x_host, st["ora_n"]["send_head"], cap, shape.E, mode=mode, topk_idx=st["idx"],
                     topk_weights=st["w"], tokens=toks)
    np.testing.assert_array_equal(P.host(gather_rows(d["recv_x"], pairs)), ora["recv_x"][pairs[:, 0], pairs[:, 1]])
    np.testing.assert_array_equal(P.host(gather_rows(d["recv_topk_idx"], pairs)),
                                  ora["recv_topk_idx"][pairs[:, 0], pairs[:, 1]])
    np.testing.assert_array_equal(P.host(gather_rows(d["recv_topk_weights"], pairs)),
                                  ora["recv_topk_weights"][pairs[:, 0], pairs[:, 1]])
    if mode == O.MODE_CAST_FP8:
        np.testing.assert_array_equal(P.host(gather_rows(d["recv_x_scales"], pairs)),
                                      ora["recv_x_scales"][pairs[:, 0], pairs[:, 1]])
        return
    # every token: src index of every received row
    src = P.host(h.export("recv_src_idx"))
    for r, n in enumerate(st["ora_n"]["num_recv"]):
        np.testing.assert_array_equal(src[r, :n], st["ora_n"]["recv_src_idx"][r, :n])
    # combine of the received rows, sampled, bf16 and the weight reduction over all tokens
    c = ep.ep_combine(h, d["recv_x"], topk_weights=d["recv_topk_weights"])
    assert h.status() == 0
    y_host = lazy_host_rows((shape.R, cap, shape.H), np.uint16, pairs, P.host(gather_rows(d["recv_x"], pairs)))
    oc = O.combine(y_host, st["ora_n"]["send_head"], out_fp32=False, num_topk=shape.K, tokens=toks)
    np.testing.assert_array_equal(P.host(c["combined_x"]).reshape(-1, shape.H)[toks],
                                  oc["out"].reshape(-1, shape.H)[toks])
    valid = st["idx"] >= 0
    np.testing.assert_array_equal(P.host(c["combined_topk_weights"]), np.where(valid, st["w"], 0).astype(np.float32))


def test_combine_heavy_ten_combines_sampled():
    """Cached record, ten combines of fresh expert outputs with two biases, fp32 reduction of the weights."""
    shape = W.WORKLOADS["combine_heavy"]
    st = setup_normal(shape)
    h = st["h"]
    d = ep.ep_dispatch(h, st["x_d"], topk_idx=st["idx_d"], topk_weights=st["w_d"],
                       num_tokens_per_rank=st["lay"]["num_tokens_per_rank"],
                       is_token_in_rank=st["lay"]["is_token_in_rank"],
                       num_tokens_per_expert=st["lay"]["num_tokens_per_expert"])
    b0, b1 = W.biases(shape, device="cuda")
    cap = st["cap"]
    toks = W.sample_tokens(shape, 256)
    pairs = rows_of(st["ora_n"]["send_head"], toks, shape.R)
    t_idx = torch.from_numpy(toks).to("cuda")
    b0h = np.zeros((shape.R * shape.T, shape.H), np.uint16)
    b1h = np.zeros_like(b0h)
    b0h[toks] = P.host(b0.view(-1, shape.H)[t_idx])
    b1h[toks] = P.host(b1.view(-1, shape.H)[t_idx])
    b0h, b1h = b0h.reshape(shape.R, shape.T, shape.H), b1h.reshape(shape.R, shape.T, shape.H)
    out = torch.empty((shape.R, shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
    for i in range(shape.n_combines):
        y = W.expert_outputs(shape, shape.R * cap, i, device="cuda").view(shape.R, cap, shape.H)
        c = ep.ep_combine(h, y, topk_weights=d["recv_topk_weights"], bias_0=b0, bias_1=b1, combined_x=out)
        assert h.status() == 0
        y_host = lazy_host_rows((shape.R, cap, shape.H), np.uint16, pairs, P.host(gather_rows(y, pairs)))
        oc = O.combine(y_host, st["ora_n"]["send_head"], bias0=b0h, bias1=b1h, num_topk=shape.K, tokens=toks)
        np.testing.assert_array_equal(P.host(out).reshape(-1, shape.H)[toks], oc["out"].reshape(-1, shape.H)[toks])
        del y
    valid = st["idx"] >= 0
    np.testing.assert_array_equal(P.host(c["combined_topk_weights"]), np.where(valid, st["w"], 0).astype(np.float32))


def test_ll_v3_full():
    """Low-latency workload whole: every message, count, range and slot, then the weighted combine."""
    shape = W.WORKLOADS["ll_v3"]
    idx, w = W.routing(shape)
    idx_d, w_d = torch.from_numpy(idx).to("cuda"), torch.from_numpy(w).to("cuda")
    x = W.tokens_x(shape, device="cuda")
    maxT = shape.max_tokens
    h = ep.Handle(P.config_of(shape, 0))
    out = ep.ep_ll_dispatch(h, x, idx_d, use_fp8=True, use_ue8m0=True)
    assert h.status() == 0
    ora = O.ll_dispatch(P.host(x), idx, maxT, shape.E, use_fp8=True, use_ue8m0=True)
    np.testing.assert_array_equal(P.host(out["packed_recv_count"]), ora["packed_recv_count"])
    np.testing.assert_array_equal(P.host(out["packed_recv_layout_range"]), ora["packed_recv_layout_range"])
    np.testing.assert_array_equal(P.host(h.export("ll_slot_row"))[:, :shape.T], ora["slot_row"])
    s_, t_, k_ = np.nonzero(idx >= 0)
    e = idx[s_, t_, k_]
    flat = torch.from_numpy(e.astype(np.int64) * shape.R * maxT + ora["slot_row"][s_, t_, k_]).to("cuda")
    msgs = out["recv_msgs"].view(-1, out["recv_msgs"].shape[-1])
    np.testing.assert_array_equal(P.host(msgs[flat]), ora["msgs_by_slot"][s_, t_, k_])
    del msgs, out
    # expert outputs on the valid rows, weighted combine
    y = torch.zeros((shape.R, shape.EL, shape.R * maxT, shape.H), dtype=torch.bfloat16, device="cuda")
    vals = W.normal_bf16((flat.numel(), shape.H), shape.seed, "lly", device="cuda")
    y.view(-1, shape.H)[flat] = vals
    got = ep.ep_ll_combine(h, y, idx_d, w_d)
    assert h.status() == 0
    y_host = np.zeros((shape.R, shape.EL, shape.R * maxT, shape.H), np.uint16)
    y_host.reshape(-1, shape.H)[flat.cpu().numpy()] = P.host(vals)
    want = O.ll_combine(y_host, idx, w, ora["slot_row"], maxT, shape.E)
    np.testing.assert_array_equal(P.host(got), want)


def test_headline_step_timed_whole():
    """normal_v3 exactly as the benchmark's timed step runs it: layout + record in one launch
    (ep_layout_notify), the prepared bf16 dispatch with top-k metadata, then the combine of the
    received rows with the top-k weight reduction.  Every output against the oracle, whole."""
    shape = W.WORKLOADS["normal_v3"]
    R, T, H, E, K = shape.R, shape.T, shape.H, shape.E, shape.K
    idx, w = W.routing(shape)
    ora_lay = O.get_dispatch_layout(idx, E, with_rdma=False)
    cap = int(ora_lay["num_tokens_per_rank"].sum(axis=0).max())
    ora_n = O.dispatch_notify(ora_lay["num_tokens_per_rank"], ora_lay["is_token_in_rank"],
                              ora_lay["num_tokens_per_expert"], shape.C, shape.A, cap)
    dev = torch.device("cuda")
    idx_d, w_d = torch.from_numpy(idx).to(dev), torch.from_numpy(w).to(dev)
    x_d = W.tokens_x(shape, device=dev)
    h = ep.Handle(P.config_of(shape, cap), dev)
    lay = dict(num_tokens_per_rank=torch.empty((R, R), dtype=torch.int32, device=dev), num_tokens_per_rdma_rank=None,
               num_tokens_per_expert=torch.empty((R, E), dtype=torch.int32, device=dev),
               is_token_in_rank=torch.empty((R, T, R), dtype=torch.bool, device=dev))
    nrpe = torch.empty((R, E // R), dtype=torch.int32, device=dev)
    recv_x = torch.empty((R, cap, H), dtype=torch.bfloat16, device=dev)
    recv_i = torch.empty((R, cap, K), dtype=torch.int64, device=dev)
    recv_w = torch.empty((R, cap, K), dtype=torch.float32, device=dev)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device=dev)
    out_w = torch.empty((R, T, K), dtype=torch.float32, device=dev)
    for _ in range(2):  # the second step runs on a handle and buffers the first one used, as in the benchmark
        ep.ep_layout_notify(h, idx_d, num_recv_tokens_per_expert=nrpe, **lay)
        ep.ep_dispatch(h, x_d, topk_idx=idx_d, topk_weights=w_d, recv_x=recv_x, recv_topk_idx=recv_i,
                       recv_topk_weights=recv_w, prepared=True)
        ep.ep_combine(h, recv_x, topk_weights=recv_w, combined_x=out, combined_topk_weights=out_w)
    assert h.status() == 0
    P.compare_layout(lay, ora_lay)
    P.compare_record(h, ora_n, T)
    np.testing.assert_array_equal(P.host(nrpe), ora_n["num_recv_tokens_per_expert"])
    ora_d = P.oracle_dispatch_all(P.host(x_d), ora_n["send_head"], cap, E, topk_idx=idx, topk_weights=w)
    P.assert_rows_equal(recv_x, ora_d["recv_x"], ora_n["num_recv"], "recv_x")
    P.assert_rows_equal(recv_i, ora_d["recv_topk_idx"], ora_n["num_recv"], "recv_topk_idx")
    P.assert_rows_equal(recv_w, ora_d["recv_topk_weights"], ora_n["num_recv"], "recv_topk_weights")
    ora_c = P.oracle_combine_all(ora_d["recv_x"], ora_n["send_head"], recv_topk_weights=ora_d["recv_topk_weights"])
    np.testing.assert_array_equal(P.host(out), ora_c["out"])
    np.testing.assert_array_equal(P.host(out_w), ora_c["combined_topk_weights"])
    h.destroy()


def test_fp8_zipf_timed_dispatch_whole():
    """fp8_zipf as the benchmark times it: a fresh dispatch with the fused FP8 cast and top-k
    metadata after ep_get_dispatch_layout, then the FP8-input dispatch (codes and scales moved
    unchanged) on the cached record.  Every receive row, scale and top-k entry, whole."""
    shape = W.WORKLOADS["fp8_zipf"]
    R, T, H, E, K = shape.R, shape.T, shape.H, shape.E, shape.K
    st = setup_normal(shape)
    h, cap, ora_n = st["h"], st["cap"], st["ora_n"]
    bufs = dict(recv_x=torch.empty((R, cap, H), dtype=torch.float8_e4m3fn, device="cuda"),
                recv_x_scales=torch.empty((R, cap, H // 128), dtype=torch.float32, device="cuda"),
                recv_topk_idx=torch.empty((R, cap, K), dtype=torch.int64, device="cuda"),
                recv_topk_weights=torch.empty((R, cap, K), dtype=torch.float32, device="cuda"),
                num_recv_tokens_per_expert=torch.empty((R, shape.EL), dtype=torch.int32, device="cuda"))
    P.compare_layout(st["lay"], st["ora_lay"])
    ep.ep_dispatch(h, st["x_d"], topk_idx=st["idx_d"], topk_weights=st["w_d"], cast_to_fp8=True,
                   num_tokens_per_rank=st["lay"]["num_tokens_per_rank"], is_token_in_rank=st["lay"]["is_token_in_rank"],
                   num_tokens_per_expert=st["lay"]["num_tokens_per_expert"], **bufs)
    assert h.status() == 0
    P.compare_record(h, ora_n, T)
    np.testing.assert_array_equal(P.host(bufs["num_recv_tokens_per_expert"]), ora_n["num_recv_tokens_per_expert"])
    ora = P.oracle_dispatch_all(P.host(st["x_d"]), ora_n["send_head"], cap, E, mode=O.MODE_CAST_FP8,
                                topk_idx=st["idx"], topk_weights=st["w"])
    for key in ("recv_x", "recv_x_scales", "recv_topk_idx", "recv_topk_weights"):
        P.assert_rows_equal(bufs[key], ora[key], ora_n["num_recv"], key)
    del ora
    # FP8 input on the cached record: already-cast codes (no NaN codes) and scales
    g = torch.Generator(device="cuda")
    g.manual_seed(shape.seed + 11)
    x8 = torch.randint(0, 126, (R, T, H), dtype=torch.uint8, device="cuda", generator=g).view(torch.float8_e4m3fn)
    xs = torch.rand((R, T, H // 128), dtype=torch.float32, device="cuda", generator=g)
    ep.ep_dispatch(h, x8, x_scales=xs, cached=True, recv_x=bufs["recv_x"], recv_x_scales=bufs["recv_x_scales"])
    assert h.status() == 0
    ora = P.oracle_dispatch_all(P.host(x8), ora_n["send_head"], cap, E, mode=O.MODE_FP8_IN, x_scales=P.host(xs))
    for key in ("recv_x", "recv_x_scales"):
        P.assert_rows_equal(bufs[key], ora[key], ora_n["num_recv"], key)
    h.destroy()


def test_combine_heavy_timed_combine_whole():
    """combine_heavy as the benchmark times it: one fresh dispatch, then combines of fresh expert
    outputs with two biases and the top-k weight reduction on the cached record.  The second
    combine (it runs on the claim counters the first one left) against the oracle, whole."""
    shape = W.WORKLOADS["combine_heavy"]
    R, T, H, K = shape.R, shape.T, shape.H, shape.K
    st = setup_normal(shape)
    h, cap, ora_n = st["h"], st["cap"], st["ora_n"]
    d = ep.ep_dispatch(h, st["x_d"], topk_idx=st["idx_d"], topk_weights=st["w_d"],
                       num_tokens_per_rank=st["lay"]["num_tokens_per_rank"],
                       is_token_in_rank=st["lay"]["is_token_in_rank"],
                       num_tokens_per_expert=st["lay"]["num_tokens_per_expert"])
    b0, b1 = W.biases(shape, device="cuda")
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
    cw = torch.empty((R, T, K), dtype=torch.float32, device="cuda")
    for i in range(2):
        y = W.expert_outputs(shape, R * cap, i, device="cuda").view(R, cap, H)
        ep.ep_combine(h, y, topk_weights=d["recv_topk_weights"], bias_0=b0, bias_1=b1, combined_x=out,
                      combined_topk_weights=cw)
    assert h.status() == 0
    ora_w = P.oracle_dispatch_all(np.zeros((R, T, 8), np.uint16), ora_n["send_head"], cap, shape.E,
                                  topk_idx=st["idx"], topk_weights=st["w"])["recv_topk_weights"]
    ora_c = P.oracle_combine_all(P.host(y), ora_n["send_head"], recv_topk_weights=ora_w, bias0=P.host(b0),
                                 bias1=P.host(b1))
    np.testing.assert_array_equal(P.host(out), ora_c["out"])
    np.testing.assert_array_equal(P.host(cw), ora_c["combined_topk_weights"])
    h.destroy()
