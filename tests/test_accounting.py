"""The benchmark's FLOP / byte accounting against the values printed by the
handbook page "MLA inference: two computation paths and FlashMLA" (section
"Which is faster: count new tokens and cached tokens"), stored in
tests/golden/p1_flop_accounting.txt."""
import os

import pytest

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "p1_flop_accounting.txt")
H, NOPE, ROPE, DV, DC = 128, 128, 64, 128, 512


def golden():
    scalars, shapes = {}, []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        parts = line.split()
        if parts[0] == "shape":
            shapes.append((parts[1], int(parts[2]), int(parts[3]), float(parts[4]), float(parts[5])))
        else:
            scalars[parts[0]] = (float(parts[1]), int(parts[3]))
    return scalars, shapes


def close(value, printed, digits):
    return abs(value - printed) <= 0.5 * 10 ** (-digits) + 1e-12


def expand_cost_per_cached_token():   # path one's fixed cost: W_UK and W_UV applied to one cached latent
    return 2 * DC * H * (NOPE + DV)


def absorb_cost_per_new_token():      # path two's fixed cost: W_UK folded into q, W_UV applied to the output
    return 2 * H * NOPE * DC + 2 * H * DC * DV


def pair_expand():
    return 2 * H * (NOPE + ROPE) + 2 * H * DV


def test_pair_flops_match_printed():
    s, _ = golden()
    v, d = s["pair_absorb_kflops"]
    assert bench.pair_flops(H) == 278528 and close(bench.pair_flops(H) / 1e3, v, d)
    v, d = s["pair_expand_kflops"]
    assert close(pair_expand() / 1e3, v, d)
    v, d = s["pair_ratio"]
    assert close(bench.pair_flops(H) / pair_expand(), v, d)


def test_fixed_costs_match_printed():
    s, _ = golden()
    assert close(expand_cost_per_cached_token() / 1e6, *s["expand_per_cached_mflops"])
    assert close(absorb_cost_per_new_token() / 1e6, *s["absorb_per_new_mflops"])


@pytest.mark.parametrize("row", golden()[1], ids=lambda r: r[0])
def test_shape_totals_match_printed(row):
    name, q, k, p1, p2 = row
    pairs = bench.causal_pairs(q, k)
    path1 = k * expand_cost_per_cached_token() + pairs * pair_expand()
    path2 = q * absorb_cost_per_new_token() + pairs * bench.pair_flops(H)
    assert close(path1 / 1e9, p1, 1), (name, path1 / 1e9, p1)
    assert close(path2 / 1e9, p2, 1), (name, path2 / 1e9, p2)


def test_crossover_and_intensities_match_printed():
    s, _ = golden()
    cross = expand_cost_per_cached_token() / (bench.pair_flops(H) - pair_expand())
    assert close(cross, *s["crossover_new_tokens"])
    bf16_row = (DC + ROPE) * 2
    assert close(bench.pair_flops(H) / bf16_row, *s["decode_intensity_mla"])
    assert close(2 * 64 * 128 * 2 / (8 * 128 * 2 * 2), *s["decode_intensity_gqa"])
    assert close(989e12 / 3.35e12, *s["h800_ridge"])


def test_toy_cache_sizes_match_printed():
    s, _ = golden()
    h, nope, rope, dv, dc = 4, 8, 4, 8, 16
    assert h * (nope + rope) + h * dv == s["toy_mha_numbers_per_token"][0]
    assert dc + rope == s["toy_mla_numbers_per_token"][0]


def test_algorithmic_totals_of_the_workloads():
    import numpy as np
    # single decode token, 8192 cached tokens, one sequence: the printed "decode 8K" pair count
    assert bench.algorithmic_flops([8192], 1, H) == 8192 * 278528
    # two new tokens, causal: q*k - q(q-1)/2 pairs
    assert bench.algorithmic_flops([100], 2, H) == (2 * 100 - 1) * 278528
    # bytes: each visible cache row once (1152 B bf16 / 656 B fp8), plus q, out, lse, block table, lengths
    b = bench.algorithmic_bytes([4096] * 32, 1, 128, 1152, 2)
    assert b == 32 * 4096 * 1152 + 32 * 128 * 576 * 2 + 32 * 128 * 512 * 2 + 32 * 128 * 4 + 32 * 64 * 4 + 32 * 4


@pytest.mark.parametrize("row", golden()[1], ids=lambda r: r[0])
def test_extend_flops_match_printed_path_one(row):
    """bench.extend_flops (the extend leg's FLOP count) reproduces the printed path-one totals."""
    name, q, k, p1, _ = row
    assert close(bench.extend_flops(q, k, H) / 1e9, p1, 1), (name, bench.extend_flops(q, k, H) / 1e9, p1)


def test_fp8_qk_tensor_peak_weights_each_contraction_by_its_rate():
    """The FP8-QK decode's tensor roofline: per pair and head, 2*d_c FLOPs of QK on E4M3 codes at
    twice the bf16 rate and 2*d_r (RoPE QK) + 2*d_c (PV) at the bf16 rate, so the time of a pair is
    the sum of the two parts' times; the effective peak is FLOPs over that time."""
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0}
    fp8, bf16 = 2 * DC, 2 * ROPE + 2 * DC
    t_pair = fp8 / (2 * 100.0) + bf16 / 100.0
    assert abs(bench.qk8_tensor_peak(peaks) - (fp8 + bf16) / t_pair) < 1e-9
    assert 100.0 < bench.qk8_tensor_peak(peaks) < 200.0
    # a compute-bound case picks that peak; a byte-bound one is unchanged
    t_q8, bound = bench.roofline_time_s(10 ** 15, 10 ** 6, peaks, qk8=True)
    assert bound == "tensor" and abs(t_q8 - 10 ** 15 / (bench.qk8_tensor_peak(peaks) * 1e12)) < 1e-12
    assert bench.roofline_time_s(10 ** 6, 10 ** 12, peaks, qk8=True) == bench.roofline_time_s(10 ** 6, 10 ** 12, peaks)
