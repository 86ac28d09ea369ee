"""Planted mistakes: each is written into a copy of the oracle's C source, built on the CPU, and
must make at least one pin of tests/test_oracle_pins.py fail.  Shows that the pins constrain every
part of the oracle (a dropped term, a wrong sign or index, a transposed operand, a rounding slip)."""
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle as O
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(O.__file__), "ep_oracle.c")

MUTATIONS = [
    ("combine sign", "acc = acc + oracle_bf16_to_f32(y[", "acc = acc - oracle_bf16_to_f32(y["),
    ("combine drops bias_1", "float acc = b0 + b1;", "float acc = b0;"),
    ("combine weights keep only the last rank", "w = w + recv_topk_weights[", "w = recv_topk_weights["),
    ("rank of an expert by modulo", "hit[e / EL] = 1;", "hit[e % R] = 1;"),
    ("expert histogram index", "num_tokens_per_expert[(size_t)s * E + e] += 1;",
     "num_tokens_per_expert[(size_t)s * E + (e + 1) % E] += 1;"),
    ("rdma node of 4 ranks", "for (int r = 8 * n; r < 8 * n + 8 && r < R; ++r) any |= hit[r];",
     "for (int r = 4 * n; r < 4 * n + 4 && r < R; ++r) any |= hit[r];"),
    ("rank prefix exclusive",
     "acc += num_tokens_per_rank[(size_t)s * R + r];\n            rank_prefix_matrix[(size_t)s * R + r] = acc;",
     "rank_prefix_matrix[(size_t)s * R + r] = acc;\n            acc += num_tokens_per_rank[(size_t)s * R + r];"),
    ("channel start inclusive", "if (t < start) n_start += h;", "if (t <= start) n_start += h;"),
    ("recv_src_idx off by one", "recv_src_idx[(size_t)r * cap + row] = t;", "recv_src_idx[(size_t)r * cap + row] = t + 1;"),
    ("alignment rounds down", "((sum + A - 1) / A) * A", "(sum / A) * A"),
    ("recv_topk_idx keeps the global id", "recv_topk_idx[dst * K + k] = mine ? e % EL : -1;",
     "recv_topk_idx[dst * K + k] = mine ? e : -1;"),
    ("fp8 inverse transposed", "float inv = 448.0f / amax;", "float inv = amax / 448.0f;"),
    ("fp8 amax clamp", "if (amax < 1e-4f) amax = 1e-4f;", "if (amax < 1e-2f) amax = 1e-2f;"),
    ("e4m3 truncates", "double n = nearbyint(a / quantum);", "double n = floor(a / quantum);"),
    ("e4m3 saturates to NaN", "if (a >= 448.0) return sign | 0x7e;", "if (a > 464.0) return 0x7f;"),
    ("ue8m0 rounds the scale down", "return (m == 0.5f) ? e2 - 1 : e2;", "return e2 - 1;"),
    ("bf16 rounds ties up", "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;",
     "if (lower >= 0x8000u) upper += 1u;"),
    ("ll slots in reverse order", "int64_t row = begin[(size_t)e * R + s] + running[e];",
     "int64_t row = begin[(size_t)e * R + s] + (cnt[(size_t)s * E + e] - 1 - running[e]);"),
    ("ll header carries the source rank", "int32_t header[4] = {t, 0, 0, 0};", "int32_t header[4] = {t, s, 0, 0};"),
    ("ll combine ignores the weight", "acc = fmaf(topk_weights[(size_t)g * K + k], v, acc);", "acc = acc + v;"),
    ("node record with 4 ranks per node", "for (int r = 8 * n; r < 8 * n + 8; ++r)\n                        goes |=",
     "for (int r = 4 * n; r < 4 * n + 4; ++r)\n                        goes |="),
    ("node receive prefix from every source of the node",
     "acc += rdma_channel_prefix[((size_t)(8 * m + l) * NN + n) * C + (C - 1)];",
     "for (int q = 0; q < 8; ++q) acc += rdma_channel_prefix[((size_t)(8 * m + q) * NN + n) * C + (C - 1)];"),
    ("node receive prefix from the first channel",
     "acc += rdma_channel_prefix[((size_t)(8 * m + l) * NN + n) * C + (C - 1)];",
     "acc += rdma_channel_prefix[((size_t)(8 * m + l) * NN + n) * C + 0];"),
    ("node receive prefix with node and GPU index swapped", "const int n = r / 8, l = r % 8;",
     "const int l = r / 8, n = r % 8 % NN;"),
    ("ll mask ignores the source", "if (rank_mask && (rank_mask[s] != 0 || rank_mask[e / EL] != 0)) return -1;",
     "if (rank_mask && rank_mask[e / EL] != 0) return -1;"),
    ("layout mask ignores the source", "if (rank_mask && (rank_mask[s] != 0 || rank_mask[e / EL] != 0)) continue;",
     "if (rank_mask && rank_mask[e / EL] != 0) continue;"),
    ("layout mask ignores the destination",
     "if (rank_mask && (rank_mask[s] != 0 || rank_mask[e / EL] != 0)) continue;",
     "if (rank_mask && rank_mask[s] != 0) continue;"),
]


def _pin_checks():
    """The pins, as (name, callable) pairs."""
    p1 = pins.load_p1()
    checks = [
        ("p1 layout", lambda: pins.test_p1_layout(p1)),
        ("p1 notify", lambda: pins.test_p1_notify(p1, 4)),
        ("p1 dispatch/combine", lambda: pins.test_p1_dispatch_combine(p1)),
        ("p1 low latency", lambda: pins.test_p1_low_latency(p1)),
        ("p1 rank mask", pins.test_p1_rank_mask),
        ("bf16 vs torch", pins.test_bf16_rounding_matches_torch),
        ("e4m3 hand codes", pins.test_e4m3_hand_codes),
        ("e4m3 brute force", pins.test_e4m3_exhaustive_against_brute_force),
        ("fp8 group hand values", pins.test_fp8_group_hand_values),
        ("fp8 group properties", lambda: pins.test_fp8_group_properties(False)),
        ("ue8m0 group properties", lambda: pins.test_fp8_group_properties(True)),
    ]
    for case in pins.CASES[:8]:
        checks.append((f"layout {case}", lambda c=case: pins.test_layout_invariants(c)))
        checks.append((f"dispatch {case}", lambda c=case: pins.test_dispatch_invariants(c)))
    for case in pins.CASES[1:6]:
        checks.append((f"combine bound {case}", lambda c=case: pins.test_combine_sum_bound_with_biases(c)))
        checks.append((f"ll invariants {case}", lambda c=case: pins.test_low_latency_invariants(c, "fp8_ue8m0")))
        checks.append((f"ll combine {case}", lambda c=case: pins.test_low_latency_combine(c)))
        checks.append((f"ll rank mask {case}", lambda c=case: pins.test_low_latency_rank_mask(c)))
        checks.append((f"normal rank mask {case}", lambda c=case: pins.test_normal_rank_mask(c)))
    checks.append(("dispatch fp8 modes", pins.test_dispatch_fp8_modes))
    checks.append(("two-level hand case", pins.test_two_level_hand_case))
    for case in pins.TWO_LEVEL_CASES:
        checks.append((f"two-level {case}", lambda c=case: pins.test_two_level_invariants(c)))
    return checks


def _first_failing_pin(lib_path):
    with O.use_library(lib_path):
        for name, check in _pin_checks():
            try:
                check()
            except (AssertionError, ValueError) as exc:  # noqa: F841  (a pin caught the mistake)
                return name
    return None


def test_unmutated_copy_passes_every_pin(tmp_path):
    lib = tmp_path / "oracle_copy.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(lib), SRC,
                           "-lm"])
    assert _first_failing_pin(str(lib)) is None


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation anchor not found: {old!r}"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new, 1))
    lib = tmp_path / "mutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(lib),
                           str(src), "-lm"])
    caught = _first_failing_pin(str(lib))
    assert caught is not None, f"no pin caught the planted mistake '{name}'"
