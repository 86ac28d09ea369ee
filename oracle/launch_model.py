"""Oracle of the SM-count launch model (test infrastructure: only tests/, smoke() and bench.py's
CPU leg use it).

"DeepEP Normal vs Low-Latency 双模式深度分析", get_theoretical_num_sms (elastic.py): the expected
number of groups one token's top-k touches, then the SMs needed to keep the bottleneck link busy
from per-token traffic and per-SM read / write rates.  On one GPU the bottleneck link is HBM; per
received row a dispatch reads 1/rho source rows and writes one row, a combine reads one row and
writes 1/rho rows, and HBM carries 1 + 1/rho rows (rho = expected destination ranks per token).

Written with exact rationals: the binomial ratio comes from math.comb as the pages state it."""
from __future__ import annotations

import math
from fractions import Fraction


def expected_topk(num_groups: int, num_experts: int, num_topk: int) -> Fraction:
    """num_groups * (1 - C(E - E/G, k) / C(E, k)), exactly (the pages' get_expected_topk)."""
    if not (1 <= num_groups <= num_experts and num_experts % num_groups == 0):
        raise ValueError("need 1 <= num_groups <= num_experts, num_experts % num_groups == 0")
    if not 1 <= num_topk <= num_experts:
        raise ValueError("need 1 <= num_topk <= num_experts")
    miss = Fraction(math.comb(num_experts - num_experts // num_groups, num_topk), math.comb(num_experts, num_topk))
    return num_groups * (1 - miss)


def theoretical_num_sms(hbm_gbs: float, sm_read_gbs: float, sm_write_gbs: float, num_device_sms: int,
                        prefer_overlap_with_compute: bool, num_ranks: int, num_experts: int, num_topk: int,
                        for_combine: bool) -> int:
    """The steps of get_theoretical_num_sms with HBM as the bounded link."""
    rho = expected_topk(num_ranks, num_experts, num_topk)
    if rho == 0:
        return num_device_sms
    # 1. per received row: reads and writes of the SMs, bytes through HBM
    if for_combine:
        sm_read, sm_write = Fraction(1), 1 / rho
    else:
        sm_read, sm_write = 1 / rho, Fraction(1)
    hbm_traffic = 1 + 1 / rho
    # 2. SMs to keep HBM busy: bounded bandwidth / traffic * per-SM demand / per-SM capability
    need = max(Fraction(hbm_gbs) / hbm_traffic * sm_read / Fraction(sm_read_gbs),
               Fraction(hbm_gbs) / hbm_traffic * sm_write / Fraction(sm_write_gbs))
    # 3. margin, floor of 4, even count, the non-overlap floor, the device
    n = max(4, math.ceil(need * Fraction(5, 4)))
    n = n + (n % 2)
    if not prefer_overlap_with_compute:
        n = max(n, 64)
    return min(n, num_device_sms)
