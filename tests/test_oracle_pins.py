"""Pins of the CPU oracle to facts that do not come from the oracle itself.

* hand-enumerated worked cases (tests/golden/*.json, each with its source);
* library routines for the number formats (torch's bf16 and float8_e4m3fn
  conversions) and a brute-force nearest-code search over the e4m3 table
  decoded here from the format definition;
* invariants that must hold for any routing: histograms, exactly-once
  delivery, permutation closure, combine(dispatch(x)) / n == x exactly,
  top-k weight round trip, low-latency slot order and packing;
* floating-point sums checked against an exact (math.fsum) value within the
  rounding bound of the stated fp32 order.
All CPU-only; they run under ``-m "not gpu"``.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from combine_get_dispatch_03_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")
U = 2.0 ** -24  # unit roundoff of binary32


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def bits_of(values):
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f32_of_bits(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------- P1

def load_p1():
    g = gold("p1_hand_case.json")
    g["idx"] = np.array(g["topk_idx"], np.int64)
    return g


@pytest.fixture(scope="module")
def p1():
    return load_p1()


def test_p1_layout(p1):
    lay = O.get_dispatch_layout(p1["idx"], p1["E"])
    np.testing.assert_array_equal(lay["is_token_in_rank"], p1["is_token_in_rank"])
    np.testing.assert_array_equal(lay["num_tokens_per_rank"], p1["num_tokens_per_rank"])
    np.testing.assert_array_equal(lay["num_tokens_per_rdma_rank"], p1["num_tokens_per_rdma_rank"])
    np.testing.assert_array_equal(lay["num_tokens_per_expert"], p1["num_tokens_per_expert"])


@pytest.mark.parametrize("align", [1, 4])
def test_p1_notify(p1, align):
    lay = O.get_dispatch_layout(p1["idx"], p1["E"])
    n = O.dispatch_notify(lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                          p1["C"], align, capacity=3)
    assert n["status"] == O.OK
    for key in ("rank_prefix_matrix", "num_recv", "channel_prefix_matrix", "recv_channel_prefix_matrix",
                "recv_src_idx", "send_head"):
        np.testing.assert_array_equal(n[key], p1[key], err_msg=key)
    np.testing.assert_array_equal(n["num_recv_tokens_per_expert"], p1[f"num_recv_tokens_per_expert_align{align}"])


def test_p1_dispatch_combine(p1):
    R, T, H = p1["R"], p1["T"], 128
    lay = O.get_dispatch_layout(p1["idx"], p1["E"])
    n = O.dispatch_notify(lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                          p1["C"], 1, capacity=3)
    # token (s,t) carries the value s*T+t+1 in every channel
    x = np.stack([np.stack([bits_of([float(s * T + t + 1)] * H) for t in range(T)]) for s in range(R)])
    w = np.arange(R * T * p1["K"], dtype=np.float32).reshape(R, T, p1["K"]) + 0.5
    d = O.dispatch(x, n["send_head"], 3, p1["E"], topk_idx=p1["idx"], topk_weights=w)
    np.testing.assert_array_equal(d["recv_topk_idx"], p1["recv_topk_idx"])
    for r in range(R):
        for row, t in enumerate(p1["recv_src_idx"][r]):
            s = 0 if row < p1["rank_prefix_matrix"][0][r] else 1
            assert f32_of_bits(d["recv_x"][r, row, :1])[0] == s * T + t + 1
    c = O.combine(d["recv_x"], n["send_head"], recv_topk_weights=d["recv_topk_weights"], out_fp32=True)
    mult = np.array(p1["combine_multiplicity"], np.float32)
    expect = mult[:, :, None] * f32_of_bits(x)
    np.testing.assert_array_equal(c["out"], expect)
    valid = p1["idx"] >= 0
    np.testing.assert_array_equal(c["combined_topk_weights"], np.where(valid, w, 0.0).astype(np.float32))


def test_p1_low_latency(p1):
    R, T, H = p1["R"], p1["T"], 128
    x = np.stack([np.stack([bits_of([float(s * T + t + 1)] * H) for t in range(T)]) for s in range(R)])
    ll = O.ll_dispatch(x, p1["idx"], p1["max_tokens"], p1["E"], use_fp8=False)
    assert ll["status"] == O.OK
    np.testing.assert_array_equal(ll["slot_row"], p1["ll_slot_row"])
    np.testing.assert_array_equal(ll["packed_recv_count"], p1["ll_packed_recv_count"])
    lr = ll["packed_recv_layout_range"]
    got = np.stack([lr >> 32, lr & 0xFFFFFFFF], axis=-1)
    np.testing.assert_array_equal(got, p1["ll_layout_range_count_begin"])
    # headers of local expert 1 on rank 1 (expert 3), in row order
    hdr = ll["msgs_by_slot"][..., :16].copy().view(np.int32)
    rows = {}
    for s in range(R):
        for t in range(T):
            for k in range(p1["K"]):
                if p1["idx"][s, t, k] == 3:
                    rows[ll["slot_row"][s, t, k]] = hdr[s, t, k]
    assert [int(rows[i][0]) for i in range(3)] == p1["ll_src_info_rank1_expert1"]
    assert all((rows[i][1:] == 0).all() for i in range(3))


# --------------------------------------------------------------------- number formats

def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(5)
    v = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** g.integers(-30, 30, 20000),
        # exact ties: low half-word 0x8000 with even and odd upper halves
        ((g.integers(0, 0x7F00, 4000).astype(np.uint32) << 16) | 0x8000).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.389e38, -3.39e38, 1e-40, -1e-45], np.float32),
    ]).astype(np.float32)
    ours = np.array([O.f32_to_bf16(float(f)) for f in v], np.uint16)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def _e4m3_table():
    """Positive finite e4m3 magnitudes for codes 0x00..0x7e, from the format definition."""
    vals = []
    for c in range(0x7F):
        ef, m = c >> 3, c & 7
        vals.append(m * 2.0 ** -9 if ef == 0 else (1 + m / 8) * 2.0 ** (ef - 7))
    return np.array(vals)


def _brute_e4m3(v):
    """Nearest finite e4m3 code by exhaustive search, ties to the even code, sign kept."""
    tab = _e4m3_table()
    # beyond 448 the nearest finite code is 448 for every magnitude; the clamp only keeps the
    # float64 distances from absorbing for huge inputs
    a = np.minimum(np.abs(v.astype(np.float64)), 1024.0)
    dist = np.abs(a[:, None] - tab[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # among equal distances take the even code (only two candidates can tie)
    even = cand & (np.arange(0x7F)[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1)).astype(np.uint8)
    return pick | np.where(np.signbit(v), 0x80, 0).astype(np.uint8)


def test_e4m3_exhaustive_against_brute_force():
    every_bf16 = np.arange(0x10000, dtype=np.uint32)
    finite = (every_bf16 & 0x7F80) != 0x7F80
    v_bf = f32_of_bits(every_bf16[finite].astype(np.uint16))
    g = np.random.default_rng(7)
    v_rand = (g.uniform(-1, 1, 60000) * 2.0 ** g.uniform(-14, 10, 60000)).astype(np.float32)
    tab = _e4m3_table()
    mids = ((tab[1:] + tab[:-1]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    v = np.concatenate([v_bf, v_rand, near, -near]).astype(np.float32)
    ours = O.f32_to_e4m3_array(v)
    np.testing.assert_array_equal(ours, _brute_e4m3(v))


def test_e4m3_matches_torch_in_range():
    g = np.random.default_rng(11)
    v = (g.uniform(-1, 1, 50000) * 2.0 ** g.uniform(-12, 8.8, 50000)).astype(np.float32)
    v = v[np.abs(v) <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.f32_to_e4m3_array(v), ref)


def test_e4m3_hand_codes():
    for case in gold("fp8_hand_values.json")["e4m3_codes"]:
        assert O.f32_to_e4m3(case["x"]) == int(case["code"], 16), case


def test_e4m3_decode_table():
    tab = _e4m3_table()
    for c in range(0x7F):
        assert O.e4m3_to_f32(c) == np.float32(tab[c])
        assert O.e4m3_to_f32(c | 0x80) == -np.float32(tab[c])
    assert math.isnan(O.e4m3_to_f32(0x7F)) and math.isnan(O.e4m3_to_f32(0xFF))


def test_fp8_group_hand_values():
    for case in gold("fp8_hand_values.json")["groups"]:
        vals = case["values"]
        if vals == "all 1.0":
            vals = [1.0] * 128
        elif vals == "all 0.0":
            vals = [0.0] * 128
        vals = list(vals) + [0.0] * (128 - len(vals))
        q, scale, e = O.fp8_quantize_group(bits_of(vals), round_scale=case["round_scale"])
        codes = [int(c, 16) for c in case["codes"]]
        assert list(q[:len(codes)]) == codes, case
        if "scale" in case:
            assert scale == case["scale"], case
        if case.get("scale_is_fp32_of") == "1/448":
            assert scale == float(np.float32(1.0) / np.float32(448.0))
        if case.get("scale_is_fp32_of") == "1e-4/448":
            assert scale == float(np.float32(1e-4) / np.float32(448.0))
        if "exponent" in case:
            assert e == case["exponent"] and e + 127 == case["ue8m0_byte"]


@pytest.mark.parametrize("round_scale", [False, True])
def test_fp8_group_properties(round_scale):
    """Scale rule, code = library e4m3 cast of the fp32 product, dequantisation error bound."""
    g = np.random.default_rng(13)
    for trial in range(300):
        mag = 2.0 ** g.uniform(-20, 20)
        x = bits_of((g.standard_normal(128) * mag).tolist())
        if trial % 7 == 0:
            x[g.integers(0, 128, 3)] = bits_of([0.0])[0]
        xf = f32_of_bits(x)
        q, scale, e = O.fp8_quantize_group(x, round_scale=round_scale)
        amax = max(np.float32(np.abs(xf).max()), np.float32(1e-4))
        s = np.float32(amax) / np.float32(448.0)
        if round_scale:
            assert scale == 2.0 ** e
            assert 2.0 ** (e - 1) < float(s) <= 2.0 ** e
            prod = xf * np.float32(2.0 ** -e)
        else:
            assert scale == float(s)
            prod = xf * (np.float32(448.0) / np.float32(amax))
        ref = torch.from_numpy(prod.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        np.testing.assert_array_equal(q, ref)
        deq = np.array([O.e4m3_to_f32(int(c)) for c in q], np.float64) * scale
        err = np.abs(deq - xf.astype(np.float64))
        bound = np.maximum(2.0 ** -4 * np.abs(xf), 2.0 ** -10 * scale) * (1 + 1e-6)
        assert (err <= bound).all()


# --------------------------------------------------------------------- invariants on random routings

CASES = [
    # (R, T, E, K, routing, mask_p, C, A)
    (1, 5, 4, 2, "uniform", 0.0, 3, 1),
    (2, 7, 8, 3, "uniform", 0.2, 2, 4),
    (3, 33, 12, 4, "zipf", 0.1, 5, 3),
    (4, 1, 16, 4, "gumbel", 0.0, 12, 1),
    (5, 17, 20, 2, "uniform", 0.5, 4, 2),
    (8, 40, 32, 4, "gumbel", 0.05, 12, 128),
    (2, 0, 4, 2, "uniform", 0.0, 2, 1),
    (4, 9, 8, 3, "uniform", 1.0, 3, 1),   # every slot masked
    (16, 6, 64, 8, "zipf", 0.05, 12, 1),  # two RDMA nodes
]


def _case(R, T, E, K, routing, mask_p, C, A, H=256, seed=0):
    shape = W.Shape("pin", R=R, T=T, H=H, E=E, K=K, routing=routing, C=C, A=A, mask_p=mask_p,
                    seed=4242 + seed + 97 * R + T)
    idx, w = W.routing(shape)
    x = W.bf16_bits(W.tokens_x(shape))
    return shape, idx, w, x


@pytest.mark.parametrize("case", CASES)
def test_layout_invariants(case):
    shape, idx, w, x = _case(*case)
    R, T, E, K = shape.R, shape.T, shape.E, shape.K
    lay = O.get_dispatch_layout(idx, E)
    for s in range(R):
        flat = idx[s].ravel()
        np.testing.assert_array_equal(lay["num_tokens_per_expert"][s], np.bincount(flat[flat >= 0], minlength=E))
    hit = np.zeros((R, T, R), bool)
    for s, t, k in zip(*np.nonzero(idx >= 0)):
        hit[s, t, idx[s, t, k] // shape.EL] = True
    np.testing.assert_array_equal(lay["is_token_in_rank"], hit.astype(np.uint8))
    np.testing.assert_array_equal(lay["num_tokens_per_rank"], hit.sum(axis=1))
    nodes = (R + 7) // 8
    node_hit = np.stack([hit[:, :, 8 * n:8 * n + 8].any(axis=2) for n in range(nodes)], axis=2)
    np.testing.assert_array_equal(lay["num_tokens_per_rdma_rank"], node_hit.sum(axis=1))
    assert lay["num_tokens_per_expert"].sum() == (idx >= 0).sum()


@pytest.mark.parametrize("case", CASES)
def test_dispatch_invariants(case):
    shape, idx, w, x = _case(*case)
    R, T, E, K, C, A = shape.R, shape.T, shape.E, shape.K, shape.C, shape.A
    lay = O.get_dispatch_layout(idx, E)
    tpr, itr = lay["num_tokens_per_rank"], lay["is_token_in_rank"]
    cap = max(int(tpr.sum(axis=0).max()), 1)
    n = O.dispatch_notify(tpr, itr, lay["num_tokens_per_expert"], C, A, cap)
    assert n["status"] == O.OK
    rp = n["rank_prefix_matrix"]
    # I3: prefix matrices
    np.testing.assert_array_equal(rp[-1], tpr.sum(axis=0))
    np.testing.assert_array_equal(n["num_recv"], tpr.sum(axis=0))
    assert (np.diff(rp, axis=0) >= 0).all()
    cp = n["channel_prefix_matrix"]
    np.testing.assert_array_equal(cp[:, :, -1], tpr)
    assert (np.diff(cp, axis=2) >= 0).all()
    excl = np.vstack([np.zeros((1, R), np.int32), rp[:-1]])
    np.testing.assert_array_equal(n["recv_channel_prefix_matrix"][:, :, 0], excl.T)
    # channel c's slice of the receive rows holds exactly the hits of its token range
    chunk = -(-T // C) if T else 0
    for s in range(R):
        for r in range(R):
            for c in range(C):
                lo, hi = min(T, c * chunk), min(T, (c + 1) * chunk)
                start = n["recv_channel_prefix_matrix"][r, s, c]
                rows = n["send_head"][s, lo:hi, r]
                rows = rows[rows >= 0]
                np.testing.assert_array_equal(rows, start + np.arange(rows.size))
    # aligned per-expert receive counts
    raw = lay["num_tokens_per_expert"].sum(axis=0).reshape(R, shape.EL)
    got = n["num_recv_tokens_per_expert"]
    assert ((got % A) == 0).all() and (got >= raw).all() and (got - raw < A).all()
    # I2 / I8: exactly-once delivery in (source, token) order, payload intact
    d = O.dispatch(x, n["send_head"], cap, E, topk_idx=idx, topk_weights=w)
    for r in range(R):
        expect = [(s, t) for s in range(R) for t in range(T) if itr[s, t, r]]
        assert len(expect) == n["num_recv"][r]
        for row, (s, t) in enumerate(expect):
            assert n["send_head"][s, t, r] == row
            assert n["recv_src_idx"][r, row] == t
            np.testing.assert_array_equal(d["recv_x"][r, row], x[s, t])
            mine = (idx[s, t] >= 0) & (idx[s, t] // shape.EL == r)
            np.testing.assert_array_equal(d["recv_topk_idx"][r, row], np.where(mine, idx[s, t] % shape.EL, -1))
            np.testing.assert_array_equal(d["recv_topk_weights"][r, row], np.where(mine, w[s, t], 0))
    assert ((n["send_head"] >= 0) == (itr == 1)).all()
    # I4 / I5: combine of the received rows, divided by the number of receiving ranks
    c = O.combine(d["recv_x"], n["send_head"], recv_topk_weights=d["recv_topk_weights"], out_fp32=True)
    nrecv = itr.sum(axis=2).astype(np.float32)
    xf = f32_of_bits(x)
    hitany = nrecv > 0
    np.testing.assert_array_equal((c["out"] / np.where(hitany, nrecv, 1)[..., None])[hitany], xf[hitany])
    assert (c["out"][~hitany] == 0).all()
    np.testing.assert_array_equal(c["combined_topk_weights"], np.where(idx >= 0, w, 0).astype(np.float32))
    cb = O.combine(d["recv_x"], n["send_head"], out_fp32=False, num_topk=K)
    ref = torch.from_numpy(c["out"]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(cb["out"], ref)


@pytest.mark.parametrize("case", CASES[:6])
def test_combine_sum_bound_with_biases(case):
    """fp32 sum (biases, then ranks ascending) within the rounding bound of the exact sum."""
    shape, idx, w, x = _case(*case)
    R, T, H = shape.R, shape.T, shape.H
    lay = O.get_dispatch_layout(idx, shape.E)
    cap = max(int(lay["num_tokens_per_rank"].sum(axis=0).max()), 1)
    n = O.dispatch_notify(lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                          shape.C, 1, cap)
    g = np.random.default_rng(3)
    y = bits_of((g.standard_normal(R * cap * H) * 3).tolist()).reshape(R, cap, H)
    b0 = bits_of((g.standard_normal(R * T * H) * 0.1).tolist()).reshape(R, T, H)
    b1 = bits_of((g.standard_normal(R * T * H) * 0.1).tolist()).reshape(R, T, H)
    c = O.combine(y, n["send_head"], bias0=b0, bias1=b1, out_fp32=True, num_topk=shape.K)
    yf, b0f, b1f = f32_of_bits(y), f32_of_bits(b0), f32_of_bits(b1)
    for s in range(R):
        for t in range(T):
            rows = [(r, n["send_head"][s, t, r]) for r in range(R) if n["send_head"][s, t, r] >= 0]
            terms = [b0f[s, t].astype(np.float64), b1f[s, t].astype(np.float64)] + \
                    [yf[r, row].astype(np.float64) for r, row in rows]
            for h in range(0, H, 37):
                col = [float(v[h]) for v in terms]
                exact = math.fsum(col)
                bound = (len(col) - 1) * U * sum(abs(v) for v in col) * (1 + 1e-6)
                assert abs(float(c["out"][s, t, h]) - exact) <= bound


@pytest.mark.parametrize("case", CASES)
def test_notify_capacity_and_consistency(case):
    shape, idx, w, x = _case(*case)
    lay = O.get_dispatch_layout(idx, shape.E)
    need = int(lay["num_tokens_per_rank"].sum(axis=0).max())
    if need > 0:
        n = O.dispatch_notify(lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                              shape.C, 1, need - 1)
        assert n["status"] == O.CAPACITY
        bad = lay["num_tokens_per_rank"].copy()
        bad[0, 0] += 1
        n = O.dispatch_notify(bad, lay["is_token_in_rank"], lay["num_tokens_per_expert"], shape.C, 1, need + 1)
        assert n["status"] == O.INCONSISTENT


# --------------------------------------------------------------------- low latency

@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("fmt", ["bf16", "fp8", "fp8_round", "fp8_ue8m0"])
def test_low_latency_invariants(case, fmt):
    # 512 channels: the FP8 message 16 + H + H/32 bytes is then a whole number of 16-byte units
    shape, idx, w, x = _case(*case, H=512)
    R, T, E, K, EL, H = shape.R, shape.T, shape.E, shape.K, shape.EL, shape.H
    use_fp8 = fmt != "bf16"
    maxT = T + 2
    ll = O.ll_dispatch(x, idx, maxT, E, use_fp8=use_fp8, round_scale=fmt == "fp8_round",
                       use_ue8m0=fmt == "fp8_ue8m0")
    assert ll["status"] == O.OK
    msg = O.ll_msg_bytes(H, use_fp8)
    assert msg % 16 == 0 and msg == (16 + H + 4 * (H // 128) if use_fp8 else 16 + 2 * H)
    # I6: counts and packing
    for d in range(R):
        assert ll["packed_recv_count"][d].sum() == ((idx >= 0) & (idx // EL == d)).sum()
    lr = ll["packed_recv_layout_range"]
    cnt, beg = lr >> 32, lr & 0xFFFFFFFF
    np.testing.assert_array_equal(cnt.sum(axis=2), ll["packed_recv_count"])
    np.testing.assert_array_equal(beg[:, :, 1:], np.cumsum(cnt, axis=2)[:, :, :-1])
    assert (beg[:, :, 0] == 0).all()
    for e in range(E):
        slots = [(s, t, k) for s in range(R) for t in range(T) for k in range(K) if idx[s, t, k] == e]
        assert [ll["slot_row"][s, t, k] for s, t, k in slots] == list(range(len(slots)))
    assert ((ll["slot_row"] < 0) == (idx < 0)).all()
    xf = f32_of_bits(x)
    for s, t, k in zip(*np.nonzero(idx >= 0)):
        m = ll["msgs_by_slot"][s, t, k]
        hdr = m[:16].view(np.int32)
        assert hdr[0] == t and (hdr[1:] == 0).all()
        if not use_fp8:
            np.testing.assert_array_equal(m[16:].view(np.uint16), x[s, t])
            continue
        q = m[16:16 + H]
        tail = m[16 + H:]
        for grp in range(H // 128):
            qq, sc, ex = O.fp8_quantize_group(x[s, t, grp * 128:(grp + 1) * 128],
                                              round_scale=fmt != "fp8")
            np.testing.assert_array_equal(q[grp * 128:(grp + 1) * 128], qq)
            if fmt == "fp8_ue8m0":
                assert tail[grp] == ex + 127
            else:
                assert tail[grp * 4:grp * 4 + 4].view(np.float32)[0] == np.float32(sc)
        if fmt == "fp8_ue8m0":
            assert (tail[H // 128:] == 0).all()
    # masked slots carry no message
    assert (ll["msgs_by_slot"][idx < 0] == 0).all()


@pytest.mark.parametrize("case", CASES[:6])
def test_low_latency_combine(case):
    """bf16 messages as expert outputs: combine == sum_k w_k x within bf16 rounding; random y within the
    fma-chain bound of the exact weighted sum."""
    shape, idx, w, x = _case(*case, H=128)
    R, T, E, K, EL, H = shape.R, shape.T, shape.E, shape.K, shape.EL, shape.H
    maxT = T + 1
    ll = O.ll_dispatch(x, idx, maxT, E, use_fp8=False)
    y = np.zeros((R, EL, R * maxT, H), np.uint16)
    for s, t, k in zip(*np.nonzero(idx >= 0)):
        e = idx[s, t, k]
        y[e // EL, e % EL, ll["slot_row"][s, t, k]] = x[s, t]
    out = O.ll_combine(y, idx, w, ll["slot_row"], maxT, E)
    xf = f32_of_bits(x).astype(np.float64)
    wsum = np.where(idx >= 0, w, 0).astype(np.float64).sum(axis=2)
    exact = wsum[..., None] * xf
    got = f32_of_bits(out).astype(np.float64)
    bound = 2.0 ** -8 * np.abs(exact) + (K + 1) * U * np.abs(xf) * 2 + 1e-30
    assert (np.abs(got - exact) <= bound).all()
    g = np.random.default_rng(9)
    yr = bits_of(g.standard_normal(y.size).tolist()).reshape(y.shape)
    out2 = O.ll_combine(yr, idx, w, ll["slot_row"], maxT, E)
    yrf = f32_of_bits(yr).astype(np.float64)
    for s in range(R):
        for t in range(T):
            terms = []
            for k in range(K):
                e = idx[s, t, k]
                if e >= 0:
                    terms.append(float(w[s, t, k]) * yrf[e // EL, e % EL, ll["slot_row"][s, t, k]])
            exact = np.array([math.fsum(v[h] for v in terms) for h in range(H)]) if terms else np.zeros(H)
            mag = np.sum(np.abs(terms), axis=0) if terms else np.zeros(H)
            got = f32_of_bits(out2[s, t]).astype(np.float64)
            assert (np.abs(got - exact) <= 2.0 ** -8 * np.abs(exact) + (K + 1) * U * mag * 1.01 + 1e-30).all()


def test_dispatch_fp8_modes():
    """Cast-in-dispatch writes the group cast of each token; FP8 input is copied with its scales."""
    shape, idx, w, x = _case(3, 11, 12, 4, "zipf", 0.1, 4, 1, H=384)
    R, E = shape.R, shape.E
    lay = O.get_dispatch_layout(idx, E)
    cap = max(int(lay["num_tokens_per_rank"].sum(axis=0).max()), 1)
    n = O.dispatch_notify(lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                          shape.C, 1, cap)
    d = O.dispatch(x, n["send_head"], cap, E, mode=O.MODE_CAST_FP8)
    for s in range(R):
        for t in range(shape.T):
            for r in range(R):
                row = n["send_head"][s, t, r]
                if row < 0:
                    continue
                for grp in range(3):
                    q, sc, _ = O.fp8_quantize_group(x[s, t, grp * 128:(grp + 1) * 128])
                    np.testing.assert_array_equal(d["recv_x"][r, row, grp * 128:(grp + 1) * 128], q)
                    assert d["recv_x_scales"][r, row, grp] == np.float32(sc)
    xq = np.random.default_rng(1).integers(0, 256, x.shape, dtype=np.uint8)
    xs = np.random.default_rng(2).random((R, shape.T, 3), dtype=np.float32)
    d2 = O.dispatch(xq, n["send_head"], cap, E, mode=O.MODE_FP8_IN, x_scales=xs)
    for s in range(R):
        for t in range(shape.T):
            for r in range(R):
                row = n["send_head"][s, t, r]
                if row >= 0:
                    np.testing.assert_array_equal(d2["recv_x"][r, row], xq[s, t])
                    np.testing.assert_array_equal(d2["recv_x_scales"][r, row], xs[s, t])


def test_sampled_tokens_match_full():
    """Token-subset evaluation (used at full sizes) equals the full evaluation on those tokens."""
    shape, idx, w, x = _case(4, 25, 16, 4, "uniform", 0.1, 3, 1)
    lay = O.get_dispatch_layout(idx, shape.E)
    cap = int(lay["num_tokens_per_rank"].sum(axis=0).max())
    n = O.dispatch_notify(lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                          shape.C, 1, cap)
    full = O.dispatch(x, n["send_head"], cap, shape.E, topk_idx=idx, topk_weights=w)
    toks = np.array([0, 7, 30, 99], np.int64)
    part = O.dispatch(x, n["send_head"], cap, shape.E, topk_idx=idx, topk_weights=w, tokens=toks)
    for g_ in toks:
        s, t = divmod(int(g_), shape.T)
        for r in range(shape.R):
            row = n["send_head"][s, t, r]
            if row >= 0:
                np.testing.assert_array_equal(part["recv_x"][r, row], full["recv_x"][r, row])
    cf = O.combine(full["recv_x"], n["send_head"], out_fp32=True, num_topk=shape.K)
    cp = O.combine(full["recv_x"], n["send_head"], out_fp32=True, num_topk=shape.K, tokens=toks)
    np.testing.assert_array_equal(cp["out"].reshape(-1, shape.H)[toks], cf["out"].reshape(-1, shape.H)[toks])


def test_token_blocks_into_shared_outputs_match_full():
    """Dispatch and combine over disjoint token blocks into one set of preallocated outputs (the
    all-cores CPU baseline) give the full evaluation's outputs."""
    shape, idx, w, x = _case(4, 25, 16, 4, "uniform", 0.1, 3, 1)
    lay = O.get_dispatch_layout(idx, shape.E)
    cap = int(lay["num_tokens_per_rank"].sum(axis=0).max())
    n = O.dispatch_notify(lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                          shape.C, 1, cap)
    full = O.dispatch(x, n["send_head"], cap, shape.E, topk_idx=idx, topk_weights=w)
    d = dict(recv_x=np.zeros_like(full["recv_x"]), recv_topk_idx=np.full_like(full["recv_topk_idx"], -2),
             recv_topk_weights=np.full_like(full["recv_topk_weights"], np.nan))
    blocks = np.array_split(np.arange(shape.R * shape.T, dtype=np.int64), 3)
    for b in blocks:
        O.dispatch(x, n["send_head"], cap, shape.E, topk_idx=idx, topk_weights=w, tokens=b, out=d)
    for key in d:
        np.testing.assert_array_equal(d[key], full[key], err_msg=key)
    cf = O.combine(full["recv_x"], n["send_head"], recv_topk_weights=full["recv_topk_weights"])
    c = dict(out=np.zeros_like(cf["out"]), combined_topk_weights=np.zeros_like(cf["combined_topk_weights"]))
    for b in blocks:
        O.combine(full["recv_x"], n["send_head"], recv_topk_weights=full["recv_topk_weights"], tokens=b, out=c)
    np.testing.assert_array_equal(c["out"], cf["out"])
    np.testing.assert_array_equal(c["combined_topk_weights"], cf["combined_topk_weights"])
    with pytest.raises(ValueError):
        O.combine(full["recv_x"], n["send_head"], out=dict(out=np.zeros((1, 1, 1), np.uint16)))


@pytest.mark.parametrize("case", CASES[1:6])
def test_low_latency_rank_mask(case):
    """Masking a rank equals removing every slot that starts or ends on it (both sides agree)."""
    shape, idx, w, x = _case(*case, H=512)
    R, T, E, EL = shape.R, shape.T, shape.E, shape.EL
    mask = np.zeros(R, np.int32)
    mask[R // 2] = 1
    masked = O.ll_dispatch(x, idx, T + 1, E, use_fp8=True, use_ue8m0=True, rank_mask=mask)
    idx2 = idx.copy()
    for s in range(R):
        for t in range(T):
            for k in range(shape.K):
                e = idx2[s, t, k]
                if e >= 0 and (mask[s] or mask[e // EL]):
                    idx2[s, t, k] = -1
    plain = O.ll_dispatch(x, idx2, T + 1, E, use_fp8=True, use_ue8m0=True)
    for key in ("slot_row", "packed_recv_count", "packed_recv_layout_range", "msgs_by_slot"):
        np.testing.assert_array_equal(masked[key], plain[key], err_msg=key)
    assert (masked["packed_recv_count"][R // 2] == 0).all()
    assert (masked["slot_row"][R // 2] == -1).all()


def _mask_slots(idx, mask, EL):
    """topk_idx with every slot that starts or ends on a masked rank set to -1 (numpy, no oracle)."""
    R = idx.shape[0]
    src = np.asarray(mask, bool)[:, None, None].repeat(idx.shape[1], 1).repeat(idx.shape[2], 2)
    dst = np.where(idx >= 0, np.asarray(mask, bool)[np.clip(idx, 0, None) // EL], False)
    out = idx.copy()
    out[(idx >= 0) & (src | dst)] = -1
    assert out.shape[0] == R
    return out


def test_p1_rank_mask():
    """The hand case with rank 1 masked: layout, record, rows, combine multiplicity, weights."""
    g = gold("p1_rank_mask_case.json")
    idx = np.array(g["topk_idx"], np.int64)
    R, T, K, E = g["R"], g["T"], g["K"], g["E"]
    lay = O.get_dispatch_layout(idx, E, rank_mask=np.array(g["rank_mask"], np.int32))
    for key in ("is_token_in_rank", "num_tokens_per_rank", "num_tokens_per_rdma_rank", "num_tokens_per_expert"):
        np.testing.assert_array_equal(lay[key], g[key], err_msg=key)
    n = O.dispatch_notify(lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"],
                          g["C"], 1, capacity=3)
    assert n["status"] == O.OK
    for key in ("rank_prefix_matrix", "num_recv", "channel_prefix_matrix", "recv_channel_prefix_matrix",
                "send_head"):
        np.testing.assert_array_equal(n[key], g[key], err_msg=key)
    np.testing.assert_array_equal(n["recv_src_idx"][0, :2], g["recv_src_idx_rank0"])
    np.testing.assert_array_equal(n["num_recv_tokens_per_expert"], g["num_recv_tokens_per_expert_align1"])
    H = 128
    x = np.stack([np.stack([bits_of([float(s * T + t + 1)] * H) for t in range(T)]) for s in range(R)])
    w = np.arange(R * T * K, dtype=np.float32).reshape(R, T, K) + 0.5
    d = O.dispatch(x, n["send_head"], 3, E, topk_idx=idx, topk_weights=w)
    np.testing.assert_array_equal(d["recv_topk_idx"][0, :2], g["recv_topk_idx_rank0"])
    c = O.combine(d["recv_x"], n["send_head"], recv_topk_weights=d["recv_topk_weights"], out_fp32=True)
    mult = np.array(g["combine_multiplicity"], np.float32)
    np.testing.assert_array_equal(c["out"], mult[:, :, None] * f32_of_bits(x))
    np.testing.assert_array_equal(c["combined_topk_weights"],
                                  np.where(np.array(g["combined_topk_weights_valid"], bool), w, 0).astype(np.float32))


@pytest.mark.parametrize("case", CASES)
def test_normal_rank_mask(case):
    """Masking ranks in the layout equals removing every slot that starts or ends on them; the masked
    ranks then receive no row and their tokens go nowhere."""
    shape, idx, w, x = _case(*case)
    R, T, E, EL = shape.R, shape.T, shape.E, shape.EL
    for masked in ({R // 2}, {0, R - 1}):
        mask = np.zeros(R, np.int32)
        mask[list(masked)] = 1
        got = O.get_dispatch_layout(idx, E, rank_mask=mask)
        want = O.get_dispatch_layout(_mask_slots(idx, mask, EL), E)
        for key in ("is_token_in_rank", "num_tokens_per_rank", "num_tokens_per_rdma_rank", "num_tokens_per_expert"):
            np.testing.assert_array_equal(got[key], want[key], err_msg=key)
        for r in masked:
            assert not got["is_token_in_rank"][r].any() and not got["is_token_in_rank"][:, :, r].any()
            assert not got["num_tokens_per_expert"][r].any()
            assert not got["num_tokens_per_expert"][:, r * EL:(r + 1) * EL].any()
        n = O.dispatch_notify(got["num_tokens_per_rank"], got["is_token_in_rank"], got["num_tokens_per_expert"],
                              shape.C, shape.A, max(1, int(got["num_tokens_per_rank"].sum(axis=0).max())))
        assert n["status"] == O.OK
        for r in masked:
            assert n["num_recv"][r] == 0 and (n["send_head"][:, :, r] == -1).all() and (n["send_head"][r] == -1).all()
    no_mask = O.get_dispatch_layout(idx, E, rank_mask=np.zeros(R, np.int32))
    plain = O.get_dispatch_layout(idx, E)
    for key in plain:
        np.testing.assert_array_equal(no_mask[key], plain[key], err_msg=key)


# --------------------------------------------------------------------- two-level (node) record

def _two_level_hand():
    g = gold("two_level_hand_case.json")
    R, T = g["R"], g["T"]
    itr = np.zeros((R, T, R), np.uint8)
    for s, toks in g["hits"].items():
        for t, ranks in enumerate(toks):
            for r in ranks:
                itr[int(s), t, r] = 1
    return g, itr


def test_two_level_hand_case():
    g, itr = _two_level_hand()
    R, C = g["R"], g["C"]
    out = O.rdma_prefix(itr, C)
    rcp = np.zeros((R, R // 8, C), np.int32)
    for s, v in g["rdma_channel_prefix_matrix"].items():
        rcp[int(s)] = v
    rrp = np.zeros((R, R // 8), np.int32)
    for r, v in g["recv_rdma_rank_prefix_sum"].items():
        rrp[int(r)] = v
    np.testing.assert_array_equal(out["rdma_channel_prefix_matrix"], rcp)
    np.testing.assert_array_equal(out["recv_rdma_rank_prefix_sum"], rrp)


def test_two_level_needs_whole_nodes():
    for R in (8, 9, 17):
        with pytest.raises(ValueError):
            O.rdma_prefix(np.zeros((R, 2, R), np.uint8), 2)


TWO_LEVEL_CASES = [c for c in CASES if c[0] > 8 and c[0] % 8 == 0] + [
    (24, 40, 48, 3, "zipf", 0.1, 5, 1), (32, 20, 64, 4, "uniform", 0.0, 12, 1), (16, 0, 32, 2, "uniform", 0.0, 3, 1),
    (16, 30, 32, 4, "uniform", 1.0, 4, 1)]


@pytest.mark.parametrize("case", TWO_LEVEL_CASES)
def test_two_level_invariants(case):
    shape, idx, w, x = _case(*case)
    R, T, C = shape.R, shape.T, shape.C
    lay = O.get_dispatch_layout(idx, shape.E)
    out = O.rdma_prefix(lay["is_token_in_rank"], C)
    rcp, rrp = out["rdma_channel_prefix_matrix"], out["recv_rdma_rank_prefix_sum"]
    NN = R // 8
    # last channel = the layout's per-node token counts; prefixes never decrease
    np.testing.assert_array_equal(rcp[:, :, -1], lay["num_tokens_per_rdma_rank"])
    assert (np.diff(rcp, axis=2) >= 0).all() and (np.diff(rrp, axis=1) >= 0).all()
    # channel bins by an independent formulation: node hit per token, cumulative count at each channel end
    node_hit = lay["is_token_in_rank"].reshape(R, T, NN, 8).any(axis=3)
    chunk = -(-T // C) if T else 0
    ends = [min(T, (c + 1) * chunk) for c in range(C)]
    csum = np.concatenate([np.zeros((R, 1, NN), np.int64), np.cumsum(node_hit, axis=1)], axis=1)
    np.testing.assert_array_equal(rcp, np.stack([csum[:, e, :] for e in ends], axis=2))
    # rank (n, l) receives from the sources (m, l): per node, its 8 receivers together get every token
    # that reaches the node exactly once, and each receiver's total is a column of the layout counts
    tprdma = lay["num_tokens_per_rdma_rank"]
    for n in range(NN):
        np.testing.assert_array_equal(rrp[8 * n:8 * n + 8, -1].sum(), tprdma[:, n].sum())
        for l in range(8):
            np.testing.assert_array_equal(rrp[8 * n + l], np.cumsum(tprdma[l::8, n]))
