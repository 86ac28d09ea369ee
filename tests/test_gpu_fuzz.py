"""Seeded random shapes across the ABI's limits, every output against the oracle.

Each case draws R, experts per rank, top-k, tokens (0 included), hidden (down to 8 channels),
channels, alignment, routing, masked slots, an SM cap for the data kernels and a masked rank (in
the handle's mask buffer, for the normal and the LL path).  It runs the one-call layout + record (with the node-level record when the ranks
form whole nodes of 8), the prepared bf16 dispatch, the combine with biases and fp32 output, the
cached FP8 cast and FP8-input dispatches when H allows, and the LL dispatch (bf16 and, when H
allows, FP8 + UE8M0) and combine."""
import numpy as np
import pytest
import torch

import oracle as O
from combine_get_dispatch_03_gb300 import ep
from combine_get_dispatch_03_gb300 import workloads as W

import _parity as P

pytestmark = pytest.mark.gpu

N_CASES = 40


def draw(i):
    g = np.random.default_rng(20261202 + i)
    R = int(g.choice([1, 2, 3, 5, 8, 9, 12, 16, 24, 32]))
    EL = int(g.integers(1, 9))
    E = R * EL
    K = int(g.integers(1, min(E, 9) + 1))
    H = int(g.choice([8, 16, 128, 256, 512, 1024]))
    # the LL expert outputs [R][EL][R * max tokens][H] bf16 stay under 64 MB
    T = int(g.choice([t for t in (0, 1, 7, 33, 100, 257) if R * EL * R * (t + 3) * H * 2 <= 1 << 26]))
    C = int(g.integers(1, 17))
    A = int(g.choice([1, 4, 128]))
    routing = str(g.choice(["uniform", "zipf", "gumbel"]))
    mask_p = float(g.choice([0.0, 0.1, 0.5]))
    shape = W.Shape(f"fuzz{i}", R=R, T=T, H=H, E=E, K=K, routing=routing, C=C, A=A, mask_p=mask_p,
                    max_tokens=max(T, 1) + int(g.integers(0, 4)), seed=30000 + i)
    max_sms = int(g.choice([0, 0, 0, 1, 3, 16]))     # data kernels capped to this many SMs' worth
    masked = int(g.integers(-1, R)) if R > 1 else -1  # a rank masked in the mask buffer, or none
    return shape, max_sms, masked


@pytest.mark.parametrize("i", range(N_CASES))
def test_fuzz_normal_and_ll(i):
    shape, max_sms, masked = draw(i)
    idx, w = W.routing(shape)
    x = W.tokens_x(shape)
    xb = W.bf16_bits(x)
    mask = None
    if masked >= 0:
        mask = np.zeros(shape.R, np.int32)
        mask[masked] = 1
    cap = max(P.needed_capacity(idx, shape.E), 1)
    h = ep.Handle(P.config_of(shape, cap, max_sms))
    if mask is not None:
        ep.ep_update_mask_buffer(h, masked, True)
    idx_d, w_d, x_d = torch.from_numpy(idx).to(P.DEV), torch.from_numpy(w).to(P.DEV), x.to(P.DEV)

    # layout and record in one call, then the prepared dispatch and the combine
    lay = ep.ep_layout_notify(h, idx_d)
    ora_lay = O.get_dispatch_layout(idx, shape.E, rank_mask=mask)
    ora_n = O.dispatch_notify(ora_lay["num_tokens_per_rank"], ora_lay["is_token_in_rank"],
                              ora_lay["num_tokens_per_expert"], shape.C, shape.A, cap)
    assert h.status() == 0, shape
    P.compare_layout(lay, ora_lay)
    P.compare_record(h, ora_n, shape.T)
    np.testing.assert_array_equal(P.host(lay["num_recv_tokens_per_expert"]), ora_n["num_recv_tokens_per_expert"])
    if shape.R > 8 and shape.R % 8 == 0:  # whole nodes of 8: the node-level record
        ora_rdma = O.rdma_prefix(ora_lay["is_token_in_rank"], shape.C)
        for key in ("rdma_channel_prefix_matrix", "recv_rdma_rank_prefix_sum"):
            np.testing.assert_array_equal(P.host(h.export(key)), ora_rdma[key], err_msg=f"{key} {shape}")
    d = ep.ep_dispatch(h, x_d, topk_idx=idx_d, topk_weights=w_d, prepared=True)
    assert h.status() == 0, shape
    ora_d = O.dispatch(xb, ora_n["send_head"], cap, shape.E, topk_idx=idx, topk_weights=w)
    rows = P.valid_rows(ora_n["num_recv"], cap)
    for key in ("recv_x", "recv_topk_idx", "recv_topk_weights"):
        np.testing.assert_array_equal(P.host(d[key])[rows], ora_d[key][rows], err_msg=f"{key} {shape}")
    b0 = W.normal_bf16((shape.R, shape.T, shape.H), shape.seed, "fb0", std=0.1)
    b1 = W.normal_bf16((shape.R, shape.T, shape.H), shape.seed, "fb1", std=0.1)
    c = ep.ep_combine(h, d["recv_x"], topk_weights=d["recv_topk_weights"], bias_0=b0.to(P.DEV),
                      bias_1=b1.to(P.DEV), out_dtype=torch.float32)
    assert h.status() == 0, shape
    ora_c = O.combine(ora_d["recv_x"], ora_n["send_head"], recv_topk_weights=ora_d["recv_topk_weights"],
                      bias0=W.bf16_bits(b0), bias1=W.bf16_bits(b1), out_fp32=True, num_topk=shape.K)
    np.testing.assert_array_equal(P.host(c["combined_x"]), ora_c["out"], err_msg=str(shape))
    np.testing.assert_array_equal(P.host(c["combined_topk_weights"]), ora_c["combined_topk_weights"])

    if shape.H % 128 == 0:  # the fused FP8 cast, cached record
        d8 = ep.ep_dispatch(h, x_d, cached=True, cast_to_fp8=True)
        assert h.status() == 0, shape
        ora8 = O.dispatch(xb, ora_n["send_head"], cap, shape.E, mode=O.MODE_CAST_FP8)
        np.testing.assert_array_equal(P.host(d8["recv_x"])[rows], ora8["recv_x"][rows], err_msg=str(shape))
        np.testing.assert_array_equal(P.host(d8["recv_x_scales"])[rows], ora8["recv_x_scales"][rows])
        # FP8 input: e4m3 codes (no NaN codes) and fp32 scales moved unchanged
        g = np.random.default_rng(shape.seed + 11)
        codes = g.integers(0, 256, (shape.R, shape.T, shape.H), dtype=np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0
        xs = g.random((shape.R, shape.T, shape.H // 128), dtype=np.float32)
        dq = ep.ep_dispatch(h, torch.from_numpy(codes).to(P.DEV).view(torch.float8_e4m3fn), cached=True,
                            x_scales=torch.from_numpy(xs).to(P.DEV))
        assert h.status() == 0, shape
        oraq = O.dispatch(codes, ora_n["send_head"], cap, shape.E, mode=O.MODE_FP8_IN, x_scales=xs)
        np.testing.assert_array_equal(P.host(dq["recv_x"])[rows], oraq["recv_x"][rows], err_msg=str(shape))
        np.testing.assert_array_equal(P.host(dq["recv_x_scales"])[rows], oraq["recv_x_scales"][rows])
    h.destroy()

    # low-latency dispatch and combine
    maxT = shape.max_tokens
    for use_fp8 in ([False, True] if shape.H % 512 == 0 else [False]):
        hl = ep.Handle(P.config_of(shape, 0, max_sms))
        if mask is not None:
            ep.ep_update_mask_buffer(hl, masked, True)
        out = ep.ep_ll_dispatch(hl, x_d, idx_d, use_fp8=use_fp8, use_ue8m0=use_fp8)
        assert hl.status() == 0, shape
        ora = O.ll_dispatch(xb, idx, maxT, shape.E, use_fp8=use_fp8, use_ue8m0=use_fp8, rank_mask=mask)
        np.testing.assert_array_equal(P.host(out["packed_recv_count"]), ora["packed_recv_count"])
        np.testing.assert_array_equal(P.host(out["packed_recv_layout_range"]), ora["packed_recv_layout_range"])
        np.testing.assert_array_equal(P.host(hl.export("ll_slot_row"))[:, :shape.T], ora["slot_row"])
        s_, t_, k_ = np.nonzero(ora["slot_row"] >= 0)
        e = idx[s_, t_, k_]
        msgs = P.host(out["recv_msgs"])
        np.testing.assert_array_equal(msgs[e // shape.EL, e % shape.EL, ora["slot_row"][s_, t_, k_]],
                                      ora["msgs_by_slot"][s_, t_, k_], err_msg=str(shape))
        y = W.normal_bf16((shape.R, shape.EL, shape.R * maxT, shape.H), shape.seed, "fy", device=P.DEV)
        got = ep.ep_ll_combine(hl, y, idx_d, w_d)
        want = O.ll_combine(P.host(y), idx, w, ora["slot_row"], maxT, shape.E)
        np.testing.assert_array_equal(P.host(got), want, err_msg=str(shape))
        hl.destroy()
