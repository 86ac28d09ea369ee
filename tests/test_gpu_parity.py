"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element by element.

Sizes span several CTA tiles / scan rounds and ragged tails; integer, index,
bf16 and FP8 outputs must be bit-exact; combine outputs are compared exactly
as well (same fp32 order) and additionally against the 5e-6 relative bound.
"""
import numpy as np
import pytest
import torch

import oracle as O
from combine_get_dispatch_03_gb300 import ep
from combine_get_dispatch_03_gb300 import workloads as W

import _parity as P

pytestmark = pytest.mark.gpu

REL_TOL = 5e-6  # combine tolerance (fp32 accumulation)


def S(name, R, T, H, E, K, routing="uniform", mask_p=0.0, C=12, A=1, seed=0, **kw):
    return W.Shape(name, R=R, T=T, H=H, E=E, K=K, routing=routing, mask_p=mask_p, C=C, A=A,
                   seed=90000 + seed, **kw)


NORMAL_CASES = [
    S("r1", 1, 37, 256, 4, 2, seed=1),
    S("r2_ragged", 2, 1500, 512, 8, 3, mask_p=0.1, C=5, A=4, seed=2),
    S("r3_odd", 3, 1025, 128, 12, 4, routing="zipf", mask_p=0.05, C=7, seed=3),
    S("r8_small", 8, 256, 1024, 32, 4, seed=4),
    S("r8_v3_like", 8, 700, 7168, 256, 8, routing="gumbel", A=128, seed=5),
    S("r16_zipf", 16, 333, 2048, 256, 8, routing="zipf", mask_p=0.05, seed=6),
    S("r32", 32, 65, 1024, 256, 8, seed=7),
    S("r5_multiround", 5, 4100, 256, 20, 2, mask_p=0.3, C=12, seed=8),
    S("r8_allmasked", 8, 40, 256, 32, 4, mask_p=1.0, seed=9),
    S("r4_T1", 4, 1, 256, 16, 4, seed=10),
    S("r17_nodes", 17, 50, 256, 34, 5, routing="zipf", mask_p=0.1, seed=11),
]


@pytest.mark.parametrize("shape", NORMAL_CASES, ids=lambda s: s.name)
def test_layout_and_record(shape):
    res = P.run_normal(shape, with_weights=True)
    assert res["status"] == 0
    P.compare_layout(res["lay"], res["ora_lay"])
    P.compare_record(res["h"], res["ora_n"], shape.T)


@pytest.mark.parametrize("shape", NORMAL_CASES, ids=lambda s: s.name)
def test_dispatch_bf16_and_combine(shape):
    res = P.run_normal(shape, with_weights=True)
    assert res["status"] == 0 and res["combine_status"] == 0
    P.compare_dispatch(res, shape, O.MODE_BF16)
    np.testing.assert_array_equal(P.host(res["c"]["combined_x"]), res["ora_c"]["out"])
    np.testing.assert_array_equal(P.host(res["c"]["combined_topk_weights"]), res["ora_c"]["combined_topk_weights"])


@pytest.mark.parametrize("shape", NORMAL_CASES[:7], ids=lambda s: s.name)
def test_combine_fp32_biases_fresh_outputs(shape):
    res = P.run_normal(shape, with_weights=True, biases=True, out_fp32=True, y_seed=shape.seed + 77)
    assert res["combine_status"] == 0
    got = P.host(res["c"]["combined_x"])
    want = res["ora_c"]["out"]
    assert P.rel_err(got, want) <= REL_TOL
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("shape", NORMAL_CASES[:7], ids=lambda s: s.name)
def test_combine_bf16_biases(shape):
    res = P.run_normal(shape, with_weights=False, biases=True, out_fp32=False, y_seed=shape.seed + 78)
    assert res["combine_status"] == 0
    np.testing.assert_array_equal(P.host(res["c"]["combined_x"]), res["ora_c"]["out"])


FP8_CASES = [c for c in NORMAL_CASES if c.H % 128 == 0]


@pytest.mark.parametrize("shape", FP8_CASES, ids=lambda s: s.name)
def test_dispatch_cast_fp8(shape):
    shape = W.Shape(**{**shape.__dict__, "outlier_frac": 0.01, "outlier_scale": 50.0})
    res = P.run_normal(shape, mode=O.MODE_CAST_FP8)
    assert res["status"] == 0
    P.compare_dispatch(res, shape, O.MODE_CAST_FP8)


@pytest.mark.parametrize("shape", FP8_CASES[:5], ids=lambda s: s.name)
def test_dispatch_fp8_input(shape):
    res = P.run_normal(shape, mode=O.MODE_FP8_IN)
    assert res["status"] == 0
    P.compare_dispatch(res, shape, O.MODE_FP8_IN)


def test_cached_dispatch_reuses_record():
    shape = S("cached", 8, 900, 1024, 64, 6, routing="gumbel", mask_p=0.05, seed=20)
    res = P.run_normal(shape)
    h = res["h"]
    x2 = W.normal_bf16((shape.R, shape.T, shape.H), 4321, "x2")
    out = P.Guarded((shape.R, res["cap"], shape.H), torch.bfloat16)
    ep.ep_dispatch(h, x2.to(P.DEV), cached=True, recv_x=out.t)
    assert h.status() == 0
    ora = O.dispatch(W.bf16_bits(x2), res["ora_n"]["send_head"], res["cap"], shape.E)
    rows = P.valid_rows(res["ora_n"]["num_recv"], res["cap"])
    np.testing.assert_array_equal(P.host(out.t)[rows], ora["recv_x"][rows])
    out.check()
    # cached FP8 cast as well
    q = P.Guarded((shape.R, res["cap"], shape.H), torch.float8_e4m3fn)
    s = P.Guarded((shape.R, res["cap"], shape.H // 128), torch.float32)
    ep.ep_dispatch(h, x2.to(P.DEV), cached=True, cast_to_fp8=True, recv_x=q.t, recv_x_scales=s.t)
    assert h.status() == 0
    ora = O.dispatch(W.bf16_bits(x2), res["ora_n"]["send_head"], res["cap"], shape.E, mode=O.MODE_CAST_FP8)
    np.testing.assert_array_equal(P.host(q.t)[rows], ora["recv_x"][rows])
    np.testing.assert_array_equal(P.host(s.t)[rows], ora["recv_x_scales"][rows])
    q.check()
    s.check()


def test_notify_then_prepared_dispatch_equals_fresh():
    """ep_notify_dispatch + the prepared mode give the fresh dispatch's record and rows."""
    shape = S("prepared", 8, 700, 1024, 64, 6, routing="zipf", mask_p=0.05, A=4, seed=26)
    res = P.run_normal(shape)
    h2 = ep.Handle(P.config_of(shape, res["cap"]))
    idx_d = torch.from_numpy(res["idx"]).to(P.DEV)
    w_d = torch.from_numpy(res["w"]).to(P.DEV)
    lay = ep.ep_get_dispatch_layout(h2, idx_d)
    nrpe = ep.ep_notify_dispatch(h2, lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"])
    assert (h2.num_recv().numpy() == res["ora_n"]["num_recv"]).all()  # counts readable before any row moves
    d = ep.ep_dispatch(h2, P.dev_bf16(res["x"]), topk_idx=idx_d, topk_weights=w_d, prepared=True)
    assert h2.status() == 0
    np.testing.assert_array_equal(P.host(nrpe), res["ora_n"]["num_recv_tokens_per_expert"])
    P.compare_record(h2, res["ora_n"], shape.T)
    rows = P.valid_rows(res["ora_n"]["num_recv"], res["cap"])
    np.testing.assert_array_equal(P.host(d["recv_x"])[rows], res["ora_d"]["recv_x"][rows])
    np.testing.assert_array_equal(P.host(d["recv_topk_idx"])[rows], res["ora_d"]["recv_topk_idx"][rows])
    np.testing.assert_array_equal(P.host(d["recv_topk_weights"])[rows], res["ora_d"]["recv_topk_weights"][rows])
    # the record is consumed: a second prepared dispatch needs a new notify
    with pytest.raises(ep.EPError):
        ep.ep_dispatch(h2, P.dev_bf16(res["x"]), topk_idx=idx_d, prepared=True)


@pytest.mark.parametrize("shape", NORMAL_CASES, ids=lambda s: s.name)
def test_layout_notify_in_one_launch(shape):
    """ep_layout_notify (layout and record in one launch) then a prepared dispatch and a combine:
    every output equals the oracle, as with the separate calls."""
    _layout_notify_round(shape)


# The one-pass scan's look-back reads 32 tiles of 512 tokens per round of loads: T = 16384 is one
# window per source, T = 16385 and 32768 need more (a source's same-source sum then stops at the
# nearest inclusive tile of that source), the R = 16 shape adds the node-level record to many tiles
# per source; the last shape has a single tile with a 1-token tail.
SCAN_EDGE_CASES = [S("scan_32_tiles", 2, 16384, 16, 8, 2, routing="gumbel", mask_p=0.05, C=7, seed=80),
                   S("scan_33_tiles", 3, 16385, 16, 12, 3, routing="zipf", C=5, A=4, seed=81),
                   S("scan_64_tiles", 2, 32768, 16, 8, 2, routing="uniform", mask_p=0.1, C=12, seed=83),
                   S("scan_nodes_40_tiles", 16, 20000, 16, 64, 4, routing="zipf", mask_p=0.05, C=9, seed=84),
                   S("scan_tail", 5, 513, 16, 20, 4, mask_p=0.2, C=3, seed=82)]


@pytest.mark.parametrize("shape", SCAN_EDGE_CASES, ids=lambda s: s.name)
def test_layout_notify_scan_edges(shape):
    """The one-pass layout + record at the edges of its tiling (one look-back window per source,
    more than one, with the node-level record, a 1-token last tile) equals the oracle."""
    _layout_notify_round(shape)


# (shape, masked ranks): one or two ranks masked in the handle's mask buffer
MASK_CASES = [(NORMAL_CASES[0], [NORMAL_CASES[0].R - 1]), (NORMAL_CASES[1], [0]),
              (S("mask_r16_nodes", 16, 700, 256, 64, 6, routing="gumbel", mask_p=0.05, C=12, seed=85), [3, 12]),
              (S("mask_r5_multitile", 5, 1500, 128, 20, 4, routing="zipf", C=7, A=4, seed=86), [2])]


@pytest.mark.parametrize("case", MASK_CASES, ids=[c[0].name for c in MASK_CASES])
def test_normal_rank_mask(case):
    """Masked ranks in the mask buffer: the layout leaves out every slot that starts or ends on one,
    through both layout paths (ep_get_dispatch_layout + fresh dispatch, ep_layout_notify + prepared
    dispatch); record, rows and combine equal the oracle's masked layout; a masked rank receives no
    row; cleaning the mask restores the unmasked layout."""
    shape, masked = case
    mask = np.zeros(shape.R, np.int32)
    mask[masked] = 1
    idx, _ = W.routing(shape)
    cap = max(P.needed_capacity(idx, shape.E), 1)
    h = ep.Handle(P.config_of(shape, cap))
    for r in masked:
        ep.ep_update_mask_buffer(h, r, True)
    _layout_notify_round(shape, h=h, rank_mask=mask)
    lay = ep.ep_get_dispatch_layout(h, torch.from_numpy(idx).to(P.DEV))
    ora_lay = O.get_dispatch_layout(idx, shape.E, rank_mask=mask)
    P.compare_layout(lay, ora_lay)
    assert (ora_lay["num_tokens_per_rank"][:, masked] == 0).all()
    x = W.tokens_x(shape).to(P.DEV)
    ep.ep_dispatch(h, x, topk_idx=torch.from_numpy(idx).to(P.DEV), num_tokens_per_rank=lay["num_tokens_per_rank"],
                   is_token_in_rank=lay["is_token_in_rank"], num_tokens_per_expert=lay["num_tokens_per_expert"])
    assert h.status() == 0
    ora_n = O.dispatch_notify(ora_lay["num_tokens_per_rank"], ora_lay["is_token_in_rank"],
                              ora_lay["num_tokens_per_expert"], shape.C, shape.A, cap)
    P.compare_record(h, ora_n, shape.T)
    assert (P.host(h.export("num_recv"))[masked] == 0).all()
    ep.ep_clean_mask_buffer(h)
    P.compare_layout(ep.ep_get_dispatch_layout(h, torch.from_numpy(idx).to(P.DEV)), O.get_dispatch_layout(idx, shape.E))
    h.destroy()


def _layout_notify_round(shape, h=None, rank_mask=None):
    idx, w = W.routing(shape)
    cap = max(P.needed_capacity(idx, shape.E), 1)
    if h is None:
        h = ep.Handle(P.config_of(shape, cap))
    idx_d, w_d = torch.from_numpy(idx).to(P.DEV), torch.from_numpy(w).to(P.DEV)
    x = W.tokens_x(shape)
    lay = ep.ep_layout_notify(h, idx_d)
    assert h.status() == 0
    ora_lay = O.get_dispatch_layout(idx, shape.E, rank_mask=rank_mask)
    P.compare_layout(lay, ora_lay)
    ora_n = O.dispatch_notify(ora_lay["num_tokens_per_rank"], ora_lay["is_token_in_rank"],
                              ora_lay["num_tokens_per_expert"], shape.C, shape.A, cap)
    P.compare_record(h, ora_n, shape.T)
    np.testing.assert_array_equal(P.host(lay["num_recv_tokens_per_expert"]), ora_n["num_recv_tokens_per_expert"])
    if shape.R > 8 and shape.R % 8 == 0:
        want = O.rdma_prefix(ora_lay["is_token_in_rank"], shape.C)
        for key in want:
            np.testing.assert_array_equal(P.host(h.export(key)), want[key], err_msg=key)
    d = ep.ep_dispatch(h, x.to(P.DEV), topk_idx=idx_d, topk_weights=w_d, prepared=True)
    assert h.status() == 0
    ora_d = O.dispatch(W.bf16_bits(x), ora_n["send_head"], cap, shape.E, topk_idx=idx, topk_weights=w)
    rows = P.valid_rows(ora_n["num_recv"], cap)
    np.testing.assert_array_equal(P.host(d["recv_x"])[rows], ora_d["recv_x"][rows])
    np.testing.assert_array_equal(P.host(d["recv_topk_idx"])[rows], ora_d["recv_topk_idx"][rows])
    c = ep.ep_combine(h, d["recv_x"], topk_weights=d["recv_topk_weights"])
    ora_c = O.combine(ora_d["recv_x"], ora_n["send_head"], recv_topk_weights=ora_d["recv_topk_weights"],
                      num_topk=shape.K)
    np.testing.assert_array_equal(P.host(c["combined_x"]), ora_c["out"])


def test_combine_of_dispatch_restores_x():
    """combine(dispatch(x)) / (number of receiving ranks) == x exactly (fp32 out)."""
    shape = S("roundtrip", 8, 300, 1024, 32, 4, mask_p=0.1, seed=21)
    res = P.run_normal(shape, out_fp32=True)
    got = P.host(res["c"]["combined_x"])
    n = res["ora_lay"]["is_token_in_rank"].sum(axis=2).astype(np.float32)
    x = (res["x"].astype(np.uint32) << 16).view(np.float32)
    hit = n > 0
    np.testing.assert_array_equal((got / np.where(hit, n, 1)[..., None])[hit], x[hit])
    assert (got[~hit] == 0).all()


def test_capacity_overflow_is_reported_and_bounded():
    shape = S("cap", 4, 200, 256, 16, 4, seed=22)
    idx, _ = W.routing(shape)
    need = P.needed_capacity(idx, shape.E)
    res = P.run_normal(shape, cap=need - 5)
    assert res["status"] == 2  # EP_ERR_CAPACITY
    P.compare_dispatch(res, shape, O.MODE_BF16)  # rows that fit are exact; guards intact


def test_bad_expert_is_reported():
    shape = S("bad", 2, 64, 128, 8, 2, seed=23)
    h = ep.Handle(P.config_of(shape, 256))
    idx, _ = W.routing(shape)
    idx[1, 5, 1] = 8  # == E
    ep.ep_get_dispatch_layout(h, torch.from_numpy(idx).to(P.DEV))
    assert h.status() == 7


def test_inconsistent_counts_are_reported():
    shape = S("inc", 4, 64, 128, 16, 2, seed=24)
    idx, w = W.routing(shape)
    h = ep.Handle(P.config_of(shape, 512))
    lay = ep.ep_get_dispatch_layout(h, torch.from_numpy(idx).to(P.DEV))
    tpr = lay["num_tokens_per_rank"].clone()
    tpr[1, 2] += 1
    ep.ep_dispatch(h, W.tokens_x(shape).to(P.DEV), topk_idx=torch.from_numpy(idx).to(P.DEV),
                   num_tokens_per_rank=tpr, is_token_in_rank=lay["is_token_in_rank"],
                   num_tokens_per_expert=lay["num_tokens_per_expert"])
    assert h.status() == 6


def test_zero_tokens():
    shape = S("empty", 4, 0, 256, 16, 4, seed=25)
    h = ep.Handle(ep.Config(4, 8, 256, 16, 4, 12, 4, 8))
    idx = torch.zeros((4, 0, 4), dtype=torch.int64, device=P.DEV)
    lay = ep.ep_get_dispatch_layout(h, idx)
    x = torch.zeros((4, 0, 256), dtype=torch.bfloat16, device=P.DEV)
    d = ep.ep_dispatch(h, x, topk_idx=idx, topk_weights=torch.zeros((4, 0, 4), device=P.DEV),
                       num_tokens_per_rank=lay["num_tokens_per_rank"], is_token_in_rank=lay["is_token_in_rank"],
                       num_tokens_per_expert=lay["num_tokens_per_expert"])
    c = ep.ep_combine(h, d["recv_x"])
    assert h.status() == 0
    assert (P.host(lay["num_tokens_per_rank"]) == 0).all()
    assert (P.host(h.export("rank_prefix_matrix")) == 0).all()
    assert (P.host(d["num_recv_tokens_per_expert"]) == 0).all()
    assert c["combined_x"].shape == (4, 0, 256)


def test_host_side_validation():
    h = ep.Handle(ep.Config(4, 8, 256, 16, 4, 12, 1, 8))
    x = torch.zeros((4, 9, 256), dtype=torch.bfloat16, device=P.DEV)  # T > num_max_tokens
    idx = torch.zeros((4, 9, 4), dtype=torch.int64, device=P.DEV)
    with pytest.raises(ep.EPError):
        ep.ep_get_dispatch_layout(h, idx)
    with pytest.raises(ep.EPError):
        ep.ep_combine(h, torch.zeros((4, 8, 256), dtype=torch.bfloat16, device=P.DEV))  # no dispatch yet
    with pytest.raises(ep.EPError):
        ep.ep_dispatch(h, x[:, :8].contiguous(), cached=True)  # no fresh dispatch yet


# ----------------------------------------------------------------------------- low latency

LL_CASES = [
    S("ll_r2", 2, 5, 512, 8, 3, mask_p=0.1, seed=30, max_tokens=7),
    S("ll_r4", 4, 33, 1024, 16, 4, seed=31, max_tokens=40),
    S("ll_r8_zipf", 8, 64, 2048, 64, 8, routing="zipf", mask_p=0.05, seed=32, max_tokens=64),
    S("ll_r32", 32, 12, 7168, 256, 8, seed=33, max_tokens=16),
    S("ll_r3_full", 3, 100, 512, 6, 2, seed=34, max_tokens=100),
    # an odd number of slots per source
    S("ll_r5_odd", 5, 37, 512, 20, 3, routing="zipf", mask_p=0.1, seed=36, max_tokens=41),
    # many slots per source: 32768, in 32 chunks of the slot-row pass's 1024-thread block
    S("ll_r4_long", 4, 4096, 512, 32, 8, mask_p=0.05, seed=35, max_tokens=4096),
    # 20 sources, 2 local experts each, zipf routing with masked slots
    S("ll_r20", 20, 50, 512, 40, 6, routing="zipf", mask_p=0.05, seed=37, max_tokens=50),
    # 32 sources with 800, 2048 and 2056 slots each: one ragged chunk, two whole chunks, and two
    # whole chunks plus an 8-slot tail in the count kernel
    S("ll_r32_t100", 32, 100, 512, 64, 8, routing="zipf", mask_p=0.05, seed=38, max_tokens=128),
    S("ll_r32_t256", 32, 256, 512, 64, 8, seed=39, max_tokens=256),
    S("ll_r32_t257", 32, 257, 512, 64, 8, seed=40, max_tokens=257),
]
LL_FORMATS = ["bf16", "fp8", "fp8_round", "fp8_ue8m0"]


def run_ll(shape, fmt, mask=None, h=None):
    use_fp8 = fmt != "bf16"
    idx, w = W.routing(shape)
    x = W.tokens_x(shape)
    maxT = shape.max_tokens
    cfg = P.config_of(shape, 0)
    if h is None:
        h = ep.Handle(cfg)
    msg = ep.ep_ll_msg_bytes(shape.H, use_fp8)
    msgs = P.Guarded((shape.R, shape.EL, shape.R * maxT, msg), torch.uint8)
    stats = torch.full((shape.R, shape.EL), 3, dtype=torch.int32, device=P.DEV)
    out = ep.ep_ll_dispatch(h, x.to(P.DEV), torch.from_numpy(idx).to(P.DEV), use_fp8=use_fp8,
                            round_scale=fmt == "fp8_round", use_ue8m0=fmt == "fp8_ue8m0", recv_msgs=msgs.t,
                            cumulative_local_expert_recv_stats=stats)
    status = h.status()
    ora = O.ll_dispatch(W.bf16_bits(x), idx, maxT, shape.E, use_fp8=use_fp8, round_scale=fmt == "fp8_round",
                        use_ue8m0=fmt == "fp8_ue8m0", rank_mask=mask)
    return dict(h=h, idx=idx, w=w, x=x, out=out, ora=ora, msgs=msgs, stats=stats, status=status, msg=msg)


def compare_ll(r, shape):
    ora, out, idx = r["ora"], r["out"], r["idx"]
    np.testing.assert_array_equal(P.host(out["packed_recv_count"]), ora["packed_recv_count"])
    np.testing.assert_array_equal(P.host(out["packed_recv_layout_range"]), ora["packed_recv_layout_range"])
    slot = P.host(r["h"].export("ll_slot_row"))[:, :shape.T]
    np.testing.assert_array_equal(slot, ora["slot_row"])
    msgs = P.host(out["recv_msgs"])
    s_, t_, k_ = np.nonzero(ora["slot_row"] >= 0)
    e = idx[s_, t_, k_]
    rows = ora["slot_row"][s_, t_, k_]
    np.testing.assert_array_equal(msgs[e // shape.EL, e % shape.EL, rows], ora["msgs_by_slot"][s_, t_, k_])
    r["msgs"].check()


@pytest.mark.parametrize("fmt", LL_FORMATS)
@pytest.mark.parametrize("shape", LL_CASES, ids=lambda s: s.name)
def test_ll_dispatch(shape, fmt):
    r = run_ll(shape, fmt)
    assert r["status"] == 0
    ora, out, idx = r["ora"], r["out"], r["idx"]
    np.testing.assert_array_equal(P.host(out["packed_recv_count"]), ora["packed_recv_count"])
    np.testing.assert_array_equal(P.host(out["packed_recv_layout_range"]), ora["packed_recv_layout_range"])
    np.testing.assert_array_equal(P.host(r["stats"]), ora["packed_recv_count"] + 3)
    slot = P.host(r["h"].export("ll_slot_row"))[:, :shape.T]
    np.testing.assert_array_equal(slot, ora["slot_row"])
    msgs = P.host(out["recv_msgs"])
    EL = shape.EL
    s_, t_, k_ = np.nonzero(idx >= 0)
    e = idx[s_, t_, k_]
    rows = ora["slot_row"][s_, t_, k_]
    np.testing.assert_array_equal(msgs[e // EL, e % EL, rows], ora["msgs_by_slot"][s_, t_, k_])
    # rows past packed_recv_count are untouched
    cnt = ora["packed_recv_count"]
    untouched = np.arange(shape.R * shape.max_tokens)[None, None, :] >= cnt[:, :, None]
    assert (msgs[untouched] == P.CANARY).all()
    r["msgs"].check()


@pytest.mark.parametrize("shape", LL_CASES, ids=lambda s: s.name)
def test_ll_combine(shape):
    r = run_ll(shape, "fp8_ue8m0")
    idx, w = r["idx"], r["w"]
    maxT = shape.max_tokens
    y_host = np.zeros((shape.R, shape.EL, shape.R * maxT, shape.H), np.uint16)
    cnt = r["ora"]["packed_recv_count"]
    fresh = W.bf16_bits(W.normal_bf16((int(cnt.sum()), shape.H), shape.seed, "lly"))
    mask = np.arange(shape.R * maxT)[None, None, :] < cnt[:, :, None]
    y_host[mask] = fresh
    y_dev = P.dev_bf16(y_host)
    got = ep.ep_ll_combine(r["h"], y_dev, torch.from_numpy(idx).to(P.DEV), torch.from_numpy(w).to(P.DEV))
    assert r["h"].status() == 0
    want = O.ll_combine(y_host, idx, w, r["ora"]["slot_row"], maxT, shape.E)
    np.testing.assert_array_equal(P.host(got), want)


def test_ll_back_to_back_calls_with_changing_routing():
    """Four dispatch + combine pairs queued on one handle with no host sync between them, each with
    its own routing and token count.  Every kernel of a call may be scheduled, and run the part of
    its body that precedes its grid-dependency wait, while the previous call's kernels still run;
    every call's messages, counts, ranges and combine must still equal the oracle's."""
    maxT = 64
    shapes = [S(f"b2b{i}", 8, T, 512, 64, 8, routing="zipf", mask_p=0.05, seed=50 + i, max_tokens=maxT)
              for i, T in enumerate([64, 33, 64, 1])]
    h = ep.Handle(P.config_of(shapes[0], 0))
    runs = []
    for sh in shapes:
        idx, w = W.routing(sh)
        x = W.tokens_x(sh)
        idx_d, w_d = torch.from_numpy(idx).to(P.DEV), torch.from_numpy(w).to(P.DEV)
        out = ep.ep_ll_dispatch(h, x.to(P.DEV), idx_d, use_fp8=True, use_ue8m0=True)
        y = W.normal_bf16((sh.R, sh.EL, sh.R * maxT, sh.H), sh.seed, "b2by", device=P.DEV)
        got = ep.ep_ll_combine(h, y, idx_d, w_d)
        runs.append((sh, idx, w, x, out, y, got))
    assert h.status() == 0
    for sh, idx, w, x, out, y, got in runs:
        ora = O.ll_dispatch(W.bf16_bits(x), idx, maxT, sh.E, use_fp8=True, use_ue8m0=True)
        np.testing.assert_array_equal(P.host(out["packed_recv_count"]), ora["packed_recv_count"], err_msg=sh.name)
        np.testing.assert_array_equal(P.host(out["packed_recv_layout_range"]), ora["packed_recv_layout_range"],
                                      err_msg=sh.name)
        s_, t_, k_ = np.nonzero(ora["slot_row"] >= 0)
        e = idx[s_, t_, k_]
        msgs = P.host(out["recv_msgs"])
        np.testing.assert_array_equal(msgs[e // sh.EL, e % sh.EL, ora["slot_row"][s_, t_, k_]],
                                      ora["msgs_by_slot"][s_, t_, k_], err_msg=sh.name)
        want = O.ll_combine(P.host(y), idx, w, ora["slot_row"], maxT, sh.E)
        np.testing.assert_array_equal(P.host(got), want, err_msg=sh.name)
    # the handle keeps the last call's slot rows
    np.testing.assert_array_equal(P.host(h.export("ll_slot_row"))[:, :shapes[-1].T], ora["slot_row"])
    h.destroy()


def test_ll_dispatch_with_8_byte_aligned_topk_idx():
    """topk_idx needs only its natural 8-byte alignment: an offset view gives the same messages."""
    shape = LL_CASES[2]
    idx, _ = W.routing(shape)
    x = W.tokens_x(shape)
    flat = torch.full((idx.size + 1,), -1, dtype=torch.int64, device=P.DEV)
    idx_d = flat[1:].view(idx.shape)
    idx_d.copy_(torch.from_numpy(idx))
    assert idx_d.data_ptr() % 16 == 8
    h = ep.Handle(P.config_of(shape, 0))
    out = ep.ep_ll_dispatch(h, x.to(P.DEV), idx_d, use_fp8=True, use_ue8m0=True)
    assert h.status() == 0
    ora = O.ll_dispatch(W.bf16_bits(x), idx, shape.max_tokens, shape.E, use_fp8=True, use_ue8m0=True)
    np.testing.assert_array_equal(P.host(out["packed_recv_count"]), ora["packed_recv_count"])
    np.testing.assert_array_equal(P.host(out["packed_recv_layout_range"]), ora["packed_recv_layout_range"])
    np.testing.assert_array_equal(P.host(h.export("ll_slot_row"))[:, :shape.T], ora["slot_row"])
    h.destroy()


def test_ll_views():
    shape = LL_CASES[1]
    r = run_ll(shape, "fp8")
    px, sc, src = ep.ll_views(r["out"]["recv_msgs"], shape.H, True)
    idx = r["idx"]
    s_, t_, k_ = np.nonzero(idx >= 0)
    e = idx[s_, t_, k_]
    rows = r["ora"]["slot_row"][s_, t_, k_]
    np.testing.assert_array_equal(P.host(src)[e // shape.EL, e % shape.EL, rows], t_)
    q = P.host(px.contiguous())[e // shape.EL, e % shape.EL, rows]
    np.testing.assert_array_equal(q, r["ora"]["msgs_by_slot"][s_, t_, k_, 16:16 + shape.H])


@pytest.mark.parametrize("shape", LL_CASES[:4], ids=lambda s: s.name)
def test_ll_zero_copy_combine_in_message_buffer(shape):
    """bf16 messages: the experts overwrite the payloads in place and the combine reads them there
    (strided rows, no copy); same result as the oracle on the same outputs.  Headers stay intact."""
    r = run_ll(shape, "bf16")
    assert r["status"] == 0
    maxT = shape.max_tokens
    px, _, src = ep.ll_views(r["out"]["recv_msgs"], shape.H, False)
    src_before = P.host(src).copy()
    y = W.normal_bf16((shape.R, shape.EL, shape.R * maxT, shape.H), shape.seed, "zcy", device=P.DEV)
    px.copy_(y)  # the expert writes its outputs over the payloads
    idx_d, w_d = torch.from_numpy(r["idx"]).to(P.DEV), torch.from_numpy(r["w"]).to(P.DEV)
    got = ep.ep_ll_combine(r["h"], px, idx_d, w_d)
    assert r["h"].status() == 0
    want = O.ll_combine(P.host(y), r["idx"], r["w"], r["ora"]["slot_row"], maxT, shape.E)
    np.testing.assert_array_equal(P.host(got), want)
    np.testing.assert_array_equal(P.host(src), src_before)
    r["msgs"].check()
    # the contiguous call on a copy of the same outputs agrees bit for bit
    np.testing.assert_array_equal(P.host(ep.ep_ll_combine(r["h"], px.contiguous(), idx_d, w_d)), want)
    with pytest.raises(ValueError):
        ep.ep_ll_combine(r["h"], px[:, :, ::2], idx_d, w_d)


def test_ll_recv_hook_defers_the_wait():
    """Dispatch on a communication stream, take the hook, run other work on the compute stream,
    call the hook, then combine: the received messages are complete and correct."""
    shape = LL_CASES[2]
    h = ep.Handle(P.config_of(shape, 0))
    idx, w = W.routing(shape)
    x = W.tokens_x(shape).to(P.DEV)
    idx_d, w_d = torch.from_numpy(idx).to(P.DEV), torch.from_numpy(w).to(P.DEV)
    comm = torch.cuda.Stream()
    comm.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(comm):
        out = ep.ep_ll_dispatch(h, x, idx_d, use_fp8=True, use_ue8m0=True, stream=comm)
        hook = ep.recv_hook(comm)
    busy = torch.randn(2048, 2048, device=P.DEV) @ torch.randn(2048, 2048, device=P.DEV)  # overlapped work
    hook()
    msgs = P.host(out["recv_msgs"])
    ora = O.ll_dispatch(W.bf16_bits(W.tokens_x(shape)), idx, shape.max_tokens, shape.E, use_fp8=True,
                        use_ue8m0=True)
    s_, t_, k_ = np.nonzero(ora["slot_row"] >= 0)
    e = idx[s_, t_, k_]
    rows = ora["slot_row"][s_, t_, k_]
    np.testing.assert_array_equal(msgs[e // shape.EL, e % shape.EL, rows], ora["msgs_by_slot"][s_, t_, k_])
    assert torch.isfinite(busy).all()
    assert h.status() == 0


@pytest.mark.parametrize("shape", LL_CASES[:4], ids=lambda s: s.name)
def test_ll_rank_mask(shape):
    """A masked rank neither sends nor receives; cleaning the mask restores the full dispatch."""
    h = ep.Handle(P.config_of(shape, 0))
    masked_rank = shape.R - 1
    ep.ep_update_mask_buffer(h, masked_rank, True)
    mask = np.zeros(shape.R, np.int32)
    mask[masked_rank] = 1
    np.testing.assert_array_equal(ep.ep_query_mask_buffer(h).numpy(), mask)
    r = run_ll(shape, "fp8_ue8m0", mask=mask, h=h)
    assert r["status"] == 0
    compare_ll(r, shape)
    assert (P.host(r["out"]["packed_recv_count"])[masked_rank] == 0).all()
    # weighted combine skips every masked slot
    maxT = shape.max_tokens
    y = W.normal_bf16((shape.R, shape.EL, shape.R * maxT, shape.H), shape.seed, "masky", device=P.DEV)
    got = ep.ep_ll_combine(h, y, torch.from_numpy(r["idx"]).to(P.DEV), torch.from_numpy(r["w"]).to(P.DEV))
    want = O.ll_combine(P.host(y), r["idx"], r["w"], r["ora"]["slot_row"], maxT, shape.E)
    np.testing.assert_array_equal(P.host(got), want)
    ep.ep_clean_mask_buffer(h)
    assert (ep.ep_query_mask_buffer(h).numpy() == 0).all()
    r2 = run_ll(shape, "fp8_ue8m0", h=h)
    compare_ll(r2, shape)


def test_maximum_sizes():
    """The largest configuration the library takes: 32 ranks, 2048 experts, top-32, with masked
    slots; normal dispatch (bf16 and FP8 cast) and combine at H = 7168, and the LL path, against the
    oracle."""
    shape = S("max", 32, 24, 7168, 2048, 32, routing="zipf", mask_p=0.05, C=12, A=128, seed=90)
    for mode in (O.MODE_BF16, O.MODE_CAST_FP8):
        res = P.run_normal(shape, mode=mode, biases=mode == O.MODE_BF16)
        assert res["status"] == 0
        P.compare_layout(res["lay"], res["ora_lay"])
        P.compare_record(res["h"], res["ora_n"], shape.T)
        P.compare_dispatch(res, shape, mode)
        if mode == O.MODE_BF16:
            np.testing.assert_array_equal(P.host(res["c"]["combined_x"]), res["ora_c"]["out"])
            np.testing.assert_array_equal(P.host(res["c"]["combined_topk_weights"]),
                                          res["ora_c"]["combined_topk_weights"])
    # LL at H = 512: its buffers hold E * R * maxT rows (64 local experts x 768 rows per rank here)
    ll = S("max_ll", 32, 24, 512, 2048, 32, routing="zipf", mask_p=0.05, seed=91, max_tokens=24)
    r = run_ll(ll, "fp8_ue8m0")
    assert r["status"] == 0
    compare_ll(r, ll)
    y = W.normal_bf16((ll.R, ll.EL, ll.R * ll.max_tokens, ll.H), ll.seed, "maxy", device=P.DEV)
    got = ep.ep_ll_combine(r["h"], y, torch.from_numpy(r["idx"]).to(P.DEV), torch.from_numpy(r["w"]).to(P.DEV))
    want = O.ll_combine(P.host(y), r["idx"], r["w"], r["ora"]["slot_row"], ll.max_tokens, ll.E)
    np.testing.assert_array_equal(P.host(got), want)


@pytest.mark.parametrize("max_sms", [1, 7, 16])
def test_max_sms_keeps_every_result(max_sms):
    """With the data kernels capped to a few SMs' worth of CTAs (one resident wave takes every
    token), dispatch (bf16 and FP8 cast), combine and the LL path stay bit-exact."""
    shape = NORMAL_CASES[3]
    for mode in (O.MODE_BF16, O.MODE_CAST_FP8):
        res = P.run_normal(shape, mode=mode, biases=mode == O.MODE_BF16, max_sms=max_sms)
        assert res["status"] == 0
        P.compare_dispatch(res, shape, mode)
        if mode == O.MODE_BF16:
            np.testing.assert_array_equal(P.host(res["c"]["combined_x"]), res["ora_c"]["out"])
    ll = LL_CASES[2]
    r = run_ll(ll, "fp8_ue8m0", h=ep.Handle(P.config_of(ll, 0, max_sms)))
    assert r["status"] == 0
    compare_ll(r, ll)
    y = W.normal_bf16((ll.R, ll.EL, ll.R * ll.max_tokens, ll.H), ll.seed, "msy", device=P.DEV)
    got = ep.ep_ll_combine(r["h"], y, torch.from_numpy(r["idx"]).to(P.DEV), torch.from_numpy(r["w"]).to(P.DEV))
    want = O.ll_combine(P.host(y), r["idx"], r["w"], r["ora"]["slot_row"], ll.max_tokens, ll.E)
    np.testing.assert_array_equal(P.host(got), want)


@pytest.mark.parametrize("R", [8, 16])
def test_claimed_token_combines_back_to_back(R):
    """With several tokens per warp the combine's warps claim tokens from a counter in the handle,
    which each launch must leave at zero: three combines on one handle (fresh outputs each, fp32
    and bf16, with and without weights and biases) all equal the oracle."""
    shape = S(f"claims{R}", R, 2048 if R == 8 else 1024, 128, 4 * R, 6, routing="gumbel", mask_p=0.05, seed=70 + R)
    n_tokens = shape.R * shape.T
    warps = torch.cuda.get_device_properties(0).multi_processor_count * 24  # at most 24 resident warps/SM
    assert n_tokens >= 2 * warps, "the shape must put several tokens on every warp"
    idx, w = W.routing(shape)
    x = W.tokens_x(shape)
    cap = P.needed_capacity(idx, shape.E)
    h = ep.Handle(P.config_of(shape, cap))
    idx_d, w_d = torch.from_numpy(idx).to(P.DEV), torch.from_numpy(w).to(P.DEV)
    ep.ep_layout_notify(h, idx_d)
    d = ep.ep_dispatch(h, x.to(P.DEV), topk_idx=idx_d, topk_weights=w_d, prepared=True)
    assert h.status() == 0
    lay = O.get_dispatch_layout(idx, shape.E)
    n = O.dispatch_notify(lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                          shape.C, shape.A, cap)
    ora_d = O.dispatch(W.bf16_bits(x), n["send_head"], cap, shape.E, topk_idx=idx, topk_weights=w)
    for i, (out_f32, weights, biases) in enumerate([(True, True, False), (False, False, True), (False, True, True)]):
        y = W.normal_bf16((shape.R, cap, shape.H), shape.seed, f"cy{i}")
        b0 = W.normal_bf16((shape.R, shape.T, shape.H), shape.seed, f"cb0{i}", std=0.1) if biases else None
        b1 = W.normal_bf16((shape.R, shape.T, shape.H), shape.seed, f"cb1{i}", std=0.1) if biases else None
        c = ep.ep_combine(h, y.to(P.DEV), topk_weights=d["recv_topk_weights"] if weights else None,
                          bias_0=None if b0 is None else b0.to(P.DEV), bias_1=None if b1 is None else b1.to(P.DEV),
                          out_dtype=torch.float32 if out_f32 else torch.bfloat16)
        assert h.status() == 0
        ora = O.combine(W.bf16_bits(y), n["send_head"],
                        recv_topk_weights=ora_d["recv_topk_weights"] if weights else None,
                        bias0=None if b0 is None else W.bf16_bits(b0), bias1=None if b1 is None else W.bf16_bits(b1),
                        out_fp32=out_f32, num_topk=shape.K)
        np.testing.assert_array_equal(P.host(c["combined_x"]), ora["out"], err_msg=f"combine {i}")
        if weights:
            np.testing.assert_array_equal(P.host(c["combined_topk_weights"]), ora["combined_topk_weights"])


def test_bounded_wait_times_out_and_masks():
    """A wait on an mbarrier that nothing completes gives up, reports EP_ERR_TIMEOUT and masks the
    rank; the context stays usable and the next dispatch leaves that rank out."""
    shape = LL_CASES[1]
    h = ep.Handle(P.config_of(shape, 0))
    ep.ep_selftest_bounded_wait(h, 2000, 2)
    assert h.status() == 3  # EP_ERR_TIMEOUT
    mask = ep.ep_query_mask_buffer(h).numpy()
    np.testing.assert_array_equal(mask, [0, 0, 1, 0])
    r = run_ll(shape, "fp8", mask=mask, h=h)
    assert r["status"] == 0
    compare_ll(r, shape)
