"""The node-level record of the two-level layout (two or more whole nodes of 8
ranks): rdma_channel_prefix_matrix [R][NN][C] and recv_rdma_rank_prefix_sum
[R][NN] from the notify step, against the oracle, bit for bit; with the
rank-level record of the same call, and the rows of a dispatch that follows it."""
import numpy as np
import pytest
import torch

import oracle as O
from combine_get_dispatch_03_gb300 import ep
from combine_get_dispatch_03_gb300 import workloads as W

import _parity as P

pytestmark = pytest.mark.gpu

CASES = [
    # (R, T, E, K, routing, mask_p, C): 2, 3 and 4 nodes; T < C; T = 0; no token reaching any node
    (16, 1000, 128, 8, "gumbel", 0.05, 12),
    (24, 257, 72, 6, "zipf", 0.1, 7),
    (32, 2100, 256, 8, "gumbel", 0.02, 24),
    (32, 5, 64, 8, "zipf", 0.0, 12),
    (16, 0, 32, 2, "uniform", 0.0, 3),
    (24, 64, 48, 3, "uniform", 1.0, 5),
]


def _shape(R, T, E, K, routing, mask_p, C):
    return W.Shape("two_level", R=R, T=T, H=256, E=E, K=K, routing=routing, C=C, A=1, mask_p=mask_p,
                   seed=9100 + 31 * R + T)


def _record(h, key):
    return P.host(h.export(key))


@pytest.mark.parametrize("case", CASES, ids=[f"R{c[0]}-T{c[1]}-C{c[6]}" for c in CASES])
def test_node_record_matches_oracle(case):
    shape = _shape(*case)
    idx, _ = W.routing(shape)
    cap = max(P.needed_capacity(idx, shape.E), 1)
    h = ep.Handle(P.config_of(shape, cap))
    lay = ep.ep_get_dispatch_layout(h, torch.from_numpy(idx).to(P.DEV))
    ep.ep_notify_dispatch(h, lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"])
    assert h.status() == 0
    ora_lay = O.get_dispatch_layout(idx, shape.E)
    P.compare_layout(lay, ora_lay)
    ora_n = O.dispatch_notify(ora_lay["num_tokens_per_rank"], ora_lay["is_token_in_rank"],
                              ora_lay["num_tokens_per_expert"], shape.C, shape.A, cap)
    P.compare_record(h, ora_n, shape.T)
    want = O.rdma_prefix(ora_lay["is_token_in_rank"], shape.C)
    for key in ("rdma_channel_prefix_matrix", "recv_rdma_rank_prefix_sum"):
        np.testing.assert_array_equal(_record(h, key), want[key], err_msg=key)
    h.destroy()


def test_fresh_dispatch_builds_node_record_and_cached_keeps_it():
    shape = _shape(16, 700, 64, 6, "zipf", 0.05, 12)
    shape = W.Shape(**{**shape.__dict__, "H": 512})
    res = P.run_normal(shape)
    assert res["status"] == 0
    P.compare_dispatch(res, shape, O.MODE_BF16)
    h = res["h"]
    want = O.rdma_prefix(res["ora_lay"]["is_token_in_rank"], shape.C)
    for key in want:
        np.testing.assert_array_equal(_record(h, key), want[key], err_msg=key)
    # a cached dispatch moves rows again and leaves the record as it was
    x_d = W.tokens_x(shape).to(P.DEV)
    ep.ep_dispatch(h, x_d, cached=True)
    assert h.status() == 0
    for key in want:
        np.testing.assert_array_equal(_record(h, key), want[key], err_msg=f"{key} after cached dispatch")


@pytest.mark.parametrize("R", [8, 9, 17])
def test_node_record_needs_whole_nodes(R):
    shape = _shape(R, 40, 4 * R, 4, "zipf", 0.0, 4)
    idx, _ = W.routing(shape)
    h = ep.Handle(P.config_of(shape, max(P.needed_capacity(idx, shape.E), 1)))
    lay = ep.ep_get_dispatch_layout(h, torch.from_numpy(idx).to(P.DEV))
    ep.ep_notify_dispatch(h, lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["num_tokens_per_expert"])
    assert h.status() == 0
    ora_lay = O.get_dispatch_layout(idx, shape.E)
    P.compare_layout(lay, ora_lay)  # the per-node counts of a partial last node still hold
    for key in ("rdma_channel_prefix_matrix", "recv_rdma_rank_prefix_sum"):
        with pytest.raises(ep.EPError) as err:
            h.export(key)
        assert err.value.status == 5  # EP_ERR_UNSUPPORTED
    h.destroy()


@pytest.mark.parametrize("case", CASES, ids=[f"R{c[0]}-T{c[1]}-C{c[6]}" for c in CASES])
def test_layout_notify_builds_node_record(case):
    """ep_layout_notify (the one-pass scan for T >= 1, the two separate kernels for T = 0) builds the
    same node-level record as the separate calls: every array against the oracle."""
    shape = _shape(*case)
    idx, _ = W.routing(shape)
    cap = max(P.needed_capacity(idx, shape.E), 1)
    h = ep.Handle(P.config_of(shape, cap))
    for _ in range(2):  # the second call runs on the scratch the first one left
        lay = ep.ep_layout_notify(h, torch.from_numpy(idx).to(P.DEV))
    assert h.status() == 0
    ora_lay = O.get_dispatch_layout(idx, shape.E)
    P.compare_layout(lay, ora_lay)
    ora_n = O.dispatch_notify(ora_lay["num_tokens_per_rank"], ora_lay["is_token_in_rank"],
                              ora_lay["num_tokens_per_expert"], shape.C, shape.A, cap)
    P.compare_record(h, ora_n, shape.T)
    np.testing.assert_array_equal(P.host(lay["num_recv_tokens_per_expert"]), ora_n["num_recv_tokens_per_expert"])
    want = O.rdma_prefix(ora_lay["is_token_in_rank"], shape.C)
    for key in ("rdma_channel_prefix_matrix", "recv_rdma_rank_prefix_sum"):
        np.testing.assert_array_equal(_record(h, key), want[key], err_msg=key)
    h.destroy()
