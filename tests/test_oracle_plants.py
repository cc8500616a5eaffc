"""Plant plausible mistakes in the CPU oracle (compiled variants, CPU only) and check the pins fail.

Each variant of ``oracle.cpp`` is built with ``-DORACLE_PLANT=k`` into a temporary directory and
swapped in for the real oracle while the pin tests run. A variant that every pin accepts would mean
the pins cannot tell that mistake from the real method; the test fails in that case.
"""
import ctypes
import os
import subprocess
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

from oracle import oracle as O
from tests import test_oracle_pins as P

PLANTS = {
    1: "sfb block row taken as n/64 instead of n/128",
    2: "last K block dropped",
    3: "e4m3 exponent bias off by one for normal codes",
    4: "BF16 rounding done through FP32 (double rounding)",
    5: "sign error on odd K blocks",
    6: "wgrad sfb taken per 128-row block instead of per row",
    7: "masked layout writes row masked_m",
    8: "contiguous layout ignores the group of the row",
    9: "sfa taken per 128-row block instead of per row",
    10: "BF16 rounding truncates toward zero",
    11: "k-grouped expert windows start one K block late",
    12: "B read as [K, N] instead of [N, K]",
    13: "contiguous padding rows (group -1) computed as group 0",
    14: "every K block scaled by the first block's scales",
}

PINS = [
    P.test_e4m3_decode_all_codes_match_torch,
    lambda: P.test_bf16_rounding_from_double_is_single_rounding(),
    lambda: P.test_normal_gemm_matches_exact_rational_bruteforce(2, 136, 256),
    lambda: P.test_normal_gemm_matches_exact_rational_bruteforce(3, 5, 128),
    lambda: P.test_normal_gemm_integer_exact(256),
    P.test_worked_example_closed_form,
    P.test_pow2_scaling_of_sfb_block_row_scales_its_128_columns_exactly,
    P.test_contiguous_bruteforce_small,
    P.test_contiguous_equals_per_group_normal_and_skips_padding,
    P.test_masked_equals_per_group_normal_and_leaves_rows_untouched,
    P.test_kgrouped_bruteforce_with_accumulation,
    P.test_kgrouped_g1_equals_dense_definition,
]


def _build(tmp, k):
    out = os.path.join(tmp, f"liboracle_plant{k}.so")
    subprocess.run(["g++", "-O1", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                    f"-DORACLE_PLANT={k}", O._SRC, "-o", out], check=True)
    return out


@pytest.fixture(scope="module")
def plant_libs():
    O.lib()  # the real oracle, with its ctypes signatures
    with tempfile.TemporaryDirectory() as tmp:
        with ThreadPoolExecutor(max_workers=4) as ex:
            paths = dict(zip(PLANTS, ex.map(lambda k: _build(tmp, k), PLANTS)))
        yield paths


def _with_lib(path):
    real = O._lib
    L = ctypes.CDLL(path)
    for name in dir(real):
        if name.startswith("oracle_"):
            f, g = getattr(real, name), getattr(L, name)
            g.restype, g.argtypes = f.restype, f.argtypes
    return real, L


@pytest.mark.parametrize("k", sorted(PLANTS))
def test_pins_catch_planted_mistake(plant_libs, k):
    real, L = _with_lib(plant_libs[k])
    caught = []
    try:
        O._lib = L
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                caught.append(getattr(pin, "__name__", "pin"))
    finally:
        O._lib = real
    assert caught, f"no pin detects plant {k}: {PLANTS[k]}"
