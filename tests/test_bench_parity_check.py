"""The bench's oracle check of its timed calls must flag a wrong output.

CPU only: a captured call is built from the oracle's own outputs on a small shape (what a correct
GPU run would have copied back), the check must pass it, and then each output in turn is altered
in one element and the check must name that output.  This guards the `parity` key of the bench
line against a checker that passes everything.
"""
import numpy as np
import pytest

import bench
import oracle as O
from combine_get_dispatch_03_gb300 import workloads as W

NORMAL = W.Shape("check_normal", R=4, T=48, H=256, E=16, K=4, routing="zipf", mask_p=0.05, C=5, A=4, seed=7101)
LL = W.Shape("check_ll", R=4, T=24, H=512, E=16, K=4, routing="uniform", max_tokens=32, seed=7102)
SAMPLED = 16


def normal_record():
    s = NORMAL
    R, T, H, E, K = s.R, s.T, s.H, s.E, s.K
    idx, w = W.routing(s)
    x = W.bf16_bits(W.tokens_x(s))
    lay = O.get_dispatch_layout(idx, E, with_rdma=True)
    cap = int(lay["num_tokens_per_rank"].sum(axis=0).max())
    n = O.dispatch_notify(lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                          s.C, s.A, cap)
    d = O.dispatch(x, n["send_head"], cap, E, topk_idx=idx, topk_weights=w)
    y = W.bf16_bits(W.normal_bf16((R, cap, H), s.seed, "check_y"))
    oc = O.combine(y, n["send_head"], recv_topk_weights=d["recv_topk_weights"], num_topk=K)
    toks = W.sample_tokens(s, SAMPLED, field="bench_parity")
    pairs = bench._pairs(n["send_head"], toks, R)
    at = (pairs[:, 0], pairs[:, 1])
    return dict(kind="normal", name="normal", shape=s, idx=idx, w=w, cap=cap, mode=0, toks=toks,
                x_rows=x.reshape(-1, H)[toks], pairs=pairs,
                layout={k: lay[k] for k in ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank")},
                record={k: n[k].copy() for k in ("rank_prefix_matrix", "channel_prefix_matrix",
                                                 "recv_channel_prefix_matrix", "num_recv", "send_head",
                                                 "recv_src_idx")},
                nrpe=n["num_recv_tokens_per_expert"].copy(),
                recv={k: d[k][at].copy() for k in ("recv_x", "recv_topk_idx", "recv_topk_weights")},
                combine=dict(out_rows=oc["out"].reshape(-1, H)[toks].copy(), y_rows=y[at].copy(),
                             out_w=oc["combined_topk_weights"].copy()))


def ll_record():
    s = LL
    R, T, H, E, K, maxT = s.R, s.T, s.H, s.E, s.K, s.max_tokens
    idx, w = W.routing(s)
    x = W.bf16_bits(W.tokens_x(s))
    o = O.ll_dispatch(x, idx, maxT, E, use_fp8=True, use_ue8m0=True)
    y = W.bf16_bits(W.normal_bf16((R, E // R, R * maxT, H), s.seed, "check_lly"))
    out = O.ll_combine(y, idx, w, o["slot_row"], maxT, E)
    toks = W.sample_tokens(s, SAMPLED, field="bench_parity")
    e = idx.reshape(-1, K)[toks]
    sl = o["slot_row"].reshape(-1, K)[toks]
    ok = (e >= 0) & (sl >= 0)
    ee, ss = np.where(ok, e, 0), np.where(ok, sl, 0)
    y_rows = y[ee // (E // R), ee % (E // R), ss]
    return dict(kind="ll", name="ll", shape=s, idx=idx, w=w, toks=toks, x_rows=x.reshape(-1, H)[toks],
                slot_row=o["slot_row"].copy(), packed_recv_count=o["packed_recv_count"].copy(),
                packed_recv_layout_range=o["packed_recv_layout_range"].copy(),
                msg_rows=o["msgs_by_slot"].reshape(R * T, K, -1)[toks].copy(), ok=ok,
                y_rows=y_rows.copy(), out_rows=out.reshape(-1, H)[toks].copy())


def bump(a, flat_index=0):
    """a with one element changed (the integer or bit pattern +1)."""
    a = a.copy()
    v = a.reshape(-1)
    if v.dtype == np.float32:
        v.view(np.int32)[flat_index] += 1
    elif v.dtype == np.bool_:
        v[flat_index] = not v[flat_index]
    else:
        v[flat_index] += 1
    return a


def test_correct_normal_call_passes():
    rec = normal_record()
    bad, n = bench._check_normal(O, rec)
    assert bad == [] and n == len(rec["toks"]) >= SAMPLED


def test_correct_ll_call_passes():
    rec = ll_record()
    bad, n = bench._check_ll(O, rec)
    assert bad == [] and n == len(rec["toks"]) >= SAMPLED


NORMAL_FIELDS = [
    ("layout", "num_tokens_per_rank", "num_tokens_per_rank"),
    ("layout", "num_tokens_per_expert", "num_tokens_per_expert"),
    ("layout", "is_token_in_rank", "is_token_in_rank"),
    ("record", "rank_prefix_matrix", "rank_prefix_matrix"),
    ("record", "channel_prefix_matrix", "channel_prefix_matrix"),
    ("record", "recv_channel_prefix_matrix", "recv_channel_prefix_matrix"),
    ("record", "send_head", "send_head"),
    ("record", "recv_src_idx", "recv_src_idx"),
    ("recv", "recv_x", "recv_x"),
    ("recv", "recv_topk_idx", "recv_topk_idx"),
    ("recv", "recv_topk_weights", "recv_topk_weights"),
    ("combine", "out_rows", "combined_x"),
    ("combine", "out_w", "combined_topk_weights"),
]


@pytest.mark.parametrize("group,key,flagged", NORMAL_FIELDS, ids=[f[1] for f in NORMAL_FIELDS])
def test_wrong_normal_output_is_flagged(group, key, flagged):
    rec = normal_record()
    if group == "record" and key == "recv_src_idx":
        rec[group][key] = bump(rec[group][key], 0)  # row 0 of rank 0 is always a received row here
    else:
        rec[group][key] = bump(rec[group][key])
    bad, _ = bench._check_normal(O, rec)
    assert flagged in bad


def test_wrong_aligned_expert_count_is_flagged():
    rec = normal_record()
    rec["nrpe"] = bump(rec["nrpe"])
    assert "num_recv_tokens_per_expert" in bench._check_normal(O, rec)[0]


@pytest.mark.parametrize("key,flagged", [("packed_recv_count", "packed_recv_count"),
                                         ("packed_recv_layout_range", "packed_recv_layout_range"),
                                         ("slot_row", "slot_row"), ("out_rows", "ll combined_x")])
def test_wrong_ll_output_is_flagged(key, flagged):
    rec = ll_record()
    rec[key] = bump(rec[key])
    assert flagged in bench._check_ll(O, rec)[0]


def test_wrong_ll_message_is_flagged():
    rec = ll_record()
    i, k = np.argwhere(rec["ok"])[0]
    rec["msg_rows"] = rec["msg_rows"].copy()
    rec["msg_rows"][i, k, 20] ^= 1  # a payload byte
    assert "messages" in bench._check_ll(O, rec)[0]


def test_cpu_parity_reports_a_mismatch():
    good, wrong = normal_record(), normal_record()
    wrong["name"] = "wrong"
    wrong["recv"]["recv_x"] = bump(wrong["recv"]["recv_x"])
    res = bench.cpu_parity([good, wrong])
    assert res["ok"] is False
    assert res["calls"]["normal"]["status"] == "ok"
    assert res["calls"]["wrong"]["status"].startswith("MISMATCH") and "recv_x" in res["calls"]["wrong"]["status"]


NODES = W.Shape("check_nodes", R=16, T=40, H=256, E=32, K=4, routing="zipf", mask_p=0.05, C=5, A=4, seed=7103)


def layout_record():
    s = NODES
    idx, _ = W.routing(s)
    lay = O.get_dispatch_layout(idx, s.E, with_rdma=True)
    cap = int(lay["num_tokens_per_rank"].sum(axis=0).max())
    n = O.dispatch_notify(lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                          s.C, s.A, cap)
    nodes = O.rdma_prefix(lay["is_token_in_rank"], s.C)
    layout = {k: lay[k].copy() for k in ("num_tokens_per_rank", "num_tokens_per_rdma_rank", "num_tokens_per_expert",
                                         "is_token_in_rank")}
    layout["num_recv_tokens_per_expert"] = n["num_recv_tokens_per_expert"].copy()
    return dict(kind="layout", name="layout", shape=s, idx=idx, cap=cap, layout=layout,
                record={k: n[k].copy() for k in ("rank_prefix_matrix", "channel_prefix_matrix",
                                                 "recv_channel_prefix_matrix", "num_recv", "send_head",
                                                 "recv_src_idx")},
                nodes={k: v.copy() for k, v in nodes.items()})


def test_correct_layout_call_passes():
    bad, n = bench._check_layout(O, layout_record())
    assert bad == [] and n == NODES.R * NODES.T


@pytest.mark.parametrize("group,key", [("layout", "num_tokens_per_rdma_rank"), ("layout", "num_recv_tokens_per_expert"),
                                       ("record", "send_head"), ("nodes", "rdma_channel_prefix_matrix"),
                                       ("nodes", "recv_rdma_rank_prefix_sum")])
def test_wrong_layout_output_is_flagged(group, key):
    rec = layout_record()
    rec[group][key] = bump(rec[group][key])
    assert key in bench._check_layout(O, rec)[0]


def ll_record_with(mask=None, use_fp8=True):
    rec = ll_record()
    s = LL
    x = W.bf16_bits(W.tokens_x(s))
    o = O.ll_dispatch(x, rec["idx"], s.max_tokens, s.E, use_fp8=use_fp8, use_ue8m0=use_fp8, rank_mask=mask)
    toks = rec["toks"]
    sl = o["slot_row"].reshape(-1, s.K)[toks]
    e = rec["idx"].reshape(-1, s.K)[toks]
    rec.update(slot_row=o["slot_row"].copy(), packed_recv_count=o["packed_recv_count"].copy(),
               packed_recv_layout_range=o["packed_recv_layout_range"].copy(),
               msg_rows=o["msgs_by_slot"].reshape(s.R * s.T, s.K, -1)[toks].copy(), ok=(e >= 0) & (sl >= 0),
               use_fp8=use_fp8, use_ue8m0=use_fp8, rank_mask=mask)
    for k in ("y_rows", "out_rows"):
        rec.pop(k)
    return rec


def test_masked_ll_call_passes_only_with_its_mask():
    mask = np.zeros(LL.R, np.int32)
    mask[1] = 1
    rec = ll_record_with(mask)
    assert bench._check_ll(O, rec)[0] == []
    rec["rank_mask"] = None  # the unmasked oracle disagrees with a masked dispatch
    assert "slot_row" in bench._check_ll(O, rec)[0]


def test_bf16_ll_call_passes_and_its_message_is_checked():
    rec = ll_record_with(use_fp8=False)
    assert bench._check_ll(O, rec)[0] == []
    i, k = np.argwhere(rec["ok"])[0]
    rec["msg_rows"][i, k, 100] ^= 1
    assert "messages" in bench._check_ll(O, rec)[0]
