"""The SM-count launch model: the oracle pinned (brute force, limits, a hand-worked case, planted
mistakes), then the library's host entry points against the oracle.  CPU only."""
import itertools
import json
import math
import os
import types
from fractions import Fraction

import pytest

from oracle import launch_model as LM

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "launch_model_hand_case.json")
SMALL = [(G, E, K) for E in (2, 4, 6, 8, 12, 16) for G in range(1, E + 1) if E % G == 0 for K in range(1, min(E, 5) + 1)]


def brute_expected(G, E, K):
    """Mean number of distinct groups over every K-subset of the experts."""
    per = E // G
    subsets = list(itertools.combinations(range(E), K))
    return Fraction(sum(len({e // per for e in c}) for c in subsets), len(subsets))


def check_expected_topk(m=LM):
    for G, E, K in SMALL:
        assert m.expected_topk(G, E, K) == brute_expected(G, E, K), (G, E, K)
    for E, G in ((256, 8), (2048, 32), (64, 16)):
        assert m.expected_topk(G, E, 1) == 1  # one expert, one group
        assert m.expected_topk(1, E, 5) == 1  # one group holds everything
        assert m.expected_topk(G, E, E - E // G + 1) == G  # more picks than experts outside a group
        prev = Fraction(0)
        for K in range(1, 12):
            cur = m.expected_topk(G, E, K)
            assert prev < cur <= min(G, K)
            prev = cur


def check_hand_case(m=LM):
    g = json.load(open(GOLDEN))
    e = g["expected_topk"]
    assert m.expected_topk(e["G"], e["E"], e["K"]) == Fraction(e["num"], e["den"])
    mo = g["model"]
    for c in g["cases"]:
        got = m.theoretical_num_sms(mo["hbm_gbs"], mo["sm_read_gbs"], mo["sm_write_gbs"], c["device"],
                                    c["prefer_overlap"], mo["R"], mo["E"], mo["K"], c["for_combine"])
        assert got == c["sms"], c


def check_sm_invariants(m=LM):
    for R, E, K in ((8, 256, 8), (16, 256, 8), (32, 256, 8), (4, 64, 6), (2, 8, 2)):
        for dev in (8, 64, 152):
            for ov in (True, False):
                prev = 0
                for hbm in (500.0, 2000.0, 6770.5, 20000.0):
                    n = m.theoretical_num_sms(hbm, 200.0, 50.0, dev, ov, R, E, K, False)
                    assert n <= dev and (n == dev or (n % 2 == 0 and n >= 4))
                    assert ov or n >= min(64, dev)
                    assert n >= prev  # more bandwidth to fill never needs fewer SMs
                    prev = n
                # faster SMs never need more of them
                assert m.theoretical_num_sms(6770.5, 400.0, 100.0, dev, ov, R, E, K, True) <= \
                    m.theoretical_num_sms(6770.5, 200.0, 50.0, dev, ov, R, E, K, True)


def test_expected_topk_is_the_brute_force_mean():
    check_expected_topk()


def test_hand_worked_case():
    check_hand_case()


def test_sm_count_invariants():
    check_sm_invariants()


def test_oracle_rejects_invalid_groups():
    for args in ((3, 8, 2), (0, 8, 2), (2, 8, 0), (2, 8, 9)):
        with pytest.raises(ValueError):
            LM.expected_topk(*args)


MUTATIONS = [
    ("group size taken as the group count", "num_experts - num_experts // num_groups", "num_experts - num_groups"),
    ("miss probability returned", "return num_groups * (1 - miss)", "return num_groups * miss"),
    ("combine with the dispatch demand", "sm_read, sm_write = Fraction(1), 1 / rho",
     "sm_read, sm_write = 1 / rho, Fraction(1)"),
    ("HBM traffic without the source reads", "hbm_traffic = 1 + 1 / rho", "hbm_traffic = 1"),
    ("no margin", "math.ceil(need * Fraction(5, 4))", "math.ceil(need)"),
    ("odd counts kept", "n = n + (n % 2)", "n = n"),
    ("overlap floor inverted", "if not prefer_overlap_with_compute:", "if prefer_overlap_with_compute:"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new):
    src = open(LM.__file__).read()
    assert src.count(old) == 1, f"mutation anchor not found: {old!r}"
    mutant = types.ModuleType("mutant_launch_model")
    exec(compile(src.replace(old, new), "mutant_launch_model.py", "exec"), mutant.__dict__)
    caught = False
    for check in (check_expected_topk, check_hand_case, check_sm_invariants):
        try:
            check(mutant)
        except AssertionError:
            caught = True
            break
    assert caught, f"no pin caught the planted mistake '{name}'"


# --------------------------------------------------------------- library (host entry points)

def test_library_expected_topk_matches_oracle():
    from combine_get_dispatch_03_gb300 import ep
    for G, E, K in SMALL + [(8, 256, 8), (16, 256, 8), (32, 256, 8), (32, 2048, 9), (8, 2048, 32), (4, 64, 64)]:
        want = float(LM.expected_topk(G, E, K))
        assert ep.expected_topk(G, E, K) == pytest.approx(want, rel=1e-12, abs=1e-12), (G, E, K)
    with pytest.raises(ValueError, match="num_groups"):
        ep.expected_topk(3, 8, 2)


def test_library_num_sms_matches_oracle():
    from combine_get_dispatch_03_gb300 import ep
    g = json.load(open(GOLDEN))
    mo = g["model"]
    for c in g["cases"]:
        assert ep.theoretical_num_sms(mo["R"], mo["E"], mo["K"], hbm_gbs=mo["hbm_gbs"], sm_read_gbs=mo["sm_read_gbs"],
                                      sm_write_gbs=mo["sm_write_gbs"], num_device_sms=c["device"],
                                      prefer_overlap_with_compute=c["prefer_overlap"],
                                      for_combine=c["for_combine"]) == c["sms"]
    for R, E, K in ((8, 256, 8), (16, 256, 8), (32, 256, 8), (4, 64, 6), (2, 8, 2), (32, 2048, 9)):
        for hbm, rd, wr in ((6770.5, 200.0, 50.0), (6770.5, 90.0, 60.0), (3000.0, 45.0, 44.0)):
            for dev in (24, 152):
                for ov in (True, False):
                    for fc in (False, True):
                        want = LM.theoretical_num_sms(hbm, rd, wr, dev, ov, R, E, K, fc)
                        got = ep.theoretical_num_sms(R, E, K, hbm_gbs=hbm, sm_read_gbs=rd, sm_write_gbs=wr,
                                                     num_device_sms=dev, prefer_overlap_with_compute=ov,
                                                     for_combine=fc)
                        assert got == want, (R, E, K, hbm, rd, wr, dev, ov, fc)
    with pytest.raises(ValueError, match="positive"):
        ep.theoretical_num_sms(8, 256, 8, hbm_gbs=0.0, sm_read_gbs=1.0, sm_write_gbs=1.0, num_device_sms=152)
