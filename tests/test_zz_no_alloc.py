"""ep_ll_dispatch_noalloc: the low-latency dispatch for callers that cannot allocate device memory.

Such callers (an engine plugin whose enqueue path may not allocate, a server
that reserves all device memory once at start-up, a latency-critical loop that
cannot take cudaMalloc's synchronisation) get the same results as the
handle-based ep_ll_dispatch, with the kernels' count array in a fixed
file-scope device array.  This test calls the new entry point through the C
ABI twice in a row and checks every output against ep_ll_dispatch on the same
inputs.  It runs last (file name) and needs no state from other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from combine_get_dispatch_03_gb300 import ep
from combine_get_dispatch_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def p(t):
    return ctypes.c_void_p(t.data_ptr())


def host(t):
    return t.detach().cpu().numpy()


# (R, maxT, H, E, K, calls): 16 ranks x 128 experts run the count kernel's 1024-thread block; 8 ranks
# x 2048 experts (R * E at the scratch's limit) its 512-thread block, whose shared-memory size the
# first call's set-up plans for the most experts; 4 ranks x 4096 tokens x top-8 count 32768 slots per
# source in 32 chunks, then a shorter second call on the same fixed array
CASES = [
    (16, 48, 2048, 128, 8, [dict(T=48, fmt=(1, 1, 1), seed=501, mask=0.05), dict(T=37, fmt=(1, 0, 0), seed=502, mask=0.0)]),
    (8, 8, 512, 2048, 8, [dict(T=8, fmt=(1, 1, 1), seed=503, mask=0.05), dict(T=5, fmt=(0, 0, 0), seed=504, mask=0.1)]),
    (4, 4096, 512, 32, 8, [dict(T=4096, fmt=(1, 1, 1), seed=505, mask=0.05), dict(T=2000, fmt=(1, 0, 0), seed=506, mask=0.0)]),
]


@pytest.mark.parametrize("R,maxT,H,E,K,calls", CASES, ids=["r16_e128", "r8_e2048", "r4_t4096"])
def test_noalloc_matches_handle_dispatch_on_two_calls(R, maxT, H, E, K, calls):
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    EL = E // R
    L = ep.lib()
    h = ep.Handle(ep.Config(R, maxT, H, E, K, 12, 1, 0), dev)
    slot = torch.full((R, maxT, K), -7, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for c in calls:
        shape = W.Shape("noalloc", R=R, T=c["T"], H=H, E=E, K=K, routing="zipf", mask_p=c["mask"],
                        max_tokens=maxT, seed=c["seed"])
        idx, _ = W.routing(shape)
        x = W.tokens_x(shape, device=dev)
        idx_d = torch.from_numpy(idx).to(dev)
        use_fp8, round_scale, ue8m0 = c["fmt"]
        msg = ep.ep_ll_msg_bytes(H, use_fp8)

        ref = ep.ep_ll_dispatch(h, x, idx_d, use_fp8=bool(use_fp8), round_scale=bool(round_scale),
                                use_ue8m0=bool(ue8m0),
                                cumulative_local_expert_recv_stats=torch.zeros((R, EL), dtype=torch.int32,
                                                                               device=dev))
        assert h.status() == 0
        ref_slot = host(h.export("ll_slot_row"))[:, :c["T"]]

        msgs = torch.zeros((R, EL, R * maxT, msg), dtype=torch.uint8, device=dev)
        cnt = torch.zeros((R, EL), dtype=torch.int32, device=dev)
        rng = torch.zeros((R, EL, R), dtype=torch.int64, device=dev)
        stats = torch.zeros((R, EL), dtype=torch.int32, device=dev)
        rc = L.ep_ll_dispatch_noalloc(R, c["T"], maxT, H, E, K, p(x), p(idx_d), use_fp8, round_scale, ue8m0,
                                      p(msgs), p(cnt), p(rng), p(stats), p(slot), p(status), stream)
        assert rc == 0, L.ep_last_error()
        torch.cuda.synchronize()
        assert int(status.item()) == 0

        np.testing.assert_array_equal(host(cnt), host(ref["packed_recv_count"]))
        np.testing.assert_array_equal(host(rng), host(ref["packed_recv_layout_range"]))
        np.testing.assert_array_equal(host(stats), host(ref["packed_recv_count"]))
        np.testing.assert_array_equal(host(slot)[:, :c["T"]], ref_slot)
        valid = np.arange(R * maxT)[None, None, :] < host(cnt)[:, :, None]
        np.testing.assert_array_equal(host(msgs)[valid], host(ref["recv_msgs"])[valid])
        assert valid.sum() == (idx >= 0).sum()
    h.destroy()


def test_noalloc_rejects_sizes_past_its_scratch():
    dev = torch.device("cuda", torch.cuda.current_device())
    L = ep.lib()
    buf = torch.zeros(64, dtype=torch.int64, device=dev)
    # 32 ranks x 1024 experts needs 32768 count entries; the fixed scratch holds 16384
    rc = L.ep_ll_dispatch_noalloc(32, 1, 4, 512, 1024, 8, p(buf), p(buf), 1, 0, 0, p(buf), p(buf), p(buf), None,
                                  p(buf), p(buf), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 5  # EP_ERR_UNSUPPORTED, nothing enqueued
    assert b"scratch" in L.ep_last_error()
