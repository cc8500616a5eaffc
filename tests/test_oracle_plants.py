"""Plant plausible mistakes in the CPU oracle (compiled variants, CPU only) and check the pins fail.

Each variant is a copy of ``oracle.cpp`` with one textual patch (every patched snippet must occur
exactly once in the oracle source, so a patch cannot silently stop applying), compiled into a temporary
directory and swapped in for the real oracle while the pin tests run. A variant that every pin accepts
would mean the pins cannot tell that mistake from the method; the test fails in that case. The oracle
source itself holds only the plain definition.
"""
import ctypes
import os
import subprocess
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

from oracle import oracle as O
from tests import test_oracle_pins as P

SFB_ROW = "const float* sfb_row = sfb + (per_col_sfb ? n : n / 128) * kbs;"
KB_LOOP = "for (int64_t kb = kb0; kb < kb1; ++kb) {"
B_READ = "p += a_dec[k] * tab[b_row[k]];"
SCALE = "const double s = static_cast<double>(sfa_row[kb]) * static_cast<double>(sfb_row[kb]);"
ACC = "acc += s * p;"
MAG = "std::ldexp(static_cast<double>(8 + f), e - 10)"
ROUND = "double r = std::nearbyint(std::ldexp(a, -q));"
BF16_ENTRY = "    return bf16_bits(x);\n}"
SFA_ROW = "row_sums(A + m * K, sfa + m * kbs, B, sfb, N, K, kbs, 0, kbs, false, a_dec, acc.data());"
GROUP = "const int64_t g = m_indices[r];"
MASK = "if (r >= lim) return;"
WINDOW = "const int64_t kb0 = koff / 128, kb1 = (koff + ks[g]) / 128;"

# plant number -> (the mistake, [(snippet of the oracle, its planted replacement), ...])
PLANTS = {
    1: ("sfb block row taken as n/64 instead of n/128",
        [(SFB_ROW, "const float* sfb_row = sfb + (per_col_sfb ? n : n / 64 % ((N + 127) / 128)) * kbs;")]),
    2: ("last K block dropped", [(KB_LOOP, "for (int64_t kb = kb0; kb < kb1 - 1; ++kb) {")]),
    3: ("e4m3 exponent bias off by one for normal codes", [(MAG, "std::ldexp(static_cast<double>(8 + f), e - 11)")]),
    4: ("BF16 rounding done through FP32 (double rounding)",
        [(BF16_ENTRY, "    return bf16_bits(static_cast<float>(x));\n}")]),
    5: ("sign error on odd K blocks", [(ACC, "acc += (kb % 2) ? -s * p : s * p;")]),
    6: ("wgrad sfb taken per 128-row block instead of per row",
        [(SFB_ROW, "const float* sfb_row = sfb + (n / 128) * kbs;")]),
    7: ("masked layout writes row masked_m", [(MASK, "if (r >= lim + 1) return;")]),
    8: ("contiguous layout ignores the group of the row", [(GROUP, "const int64_t g = 0;")]),
    9: ("sfa taken per 128-row block instead of per row",
        [(SFA_ROW, "row_sums(A + m * K, sfa + (m / 128) * 128 * kbs, B, sfb, N, K, kbs, 0, kbs, false, a_dec, acc.data());")]),
    10: ("BF16 rounding truncates toward zero", [(ROUND, "double r = std::trunc(std::ldexp(a, -q));")]),
    11: ("k-grouped expert windows start one K block late",
         [(WINDOW, "const int64_t late = (ks[g] > 0 && (koff + ks[g]) / 128 < kbs) ? 1 : 0;\n"
                   "            const int64_t kb0 = koff / 128 + late, kb1 = (koff + ks[g]) / 128 + late;")]),
    12: ("B read as [K, N] instead of [N, K]", [(B_READ, "p += a_dec[k] * tab[B[k * N + n]];")]),
    13: ("contiguous padding rows (group -1) computed as group 0",
         [(GROUP, "const int64_t g = m_indices[r] < 0 ? 0 : m_indices[r];")]),
    14: ("every K block scaled by the first block's scales",
         [(SCALE, "const double s = static_cast<double>(sfa_row[kb0]) * static_cast<double>(sfb_row[kb0]);")]),
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


def planted_source(k):
    """The oracle source with plant k applied."""
    with open(O._SRC) as f:
        src = f.read()
    for old, new in PLANTS[k][1]:
        assert src.count(old) == 1, f"plant {k}: snippet {old!r} occurs {src.count(old)} times in the oracle"
        src = src.replace(old, new)
    return src


def _build(tmp, k):
    src = os.path.join(tmp, f"oracle_plant{k}.cpp")
    with open(src, "w") as f:
        f.write(planted_source(k))
    out = os.path.join(tmp, f"liboracle_plant{k}.so")
    subprocess.run(["g++", "-O1", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                    src, "-o", out], check=True)
    return out


def test_every_plant_applies_and_changes_the_source():
    with open(O._SRC) as f:
        clean = f.read()
    for k in PLANTS:
        assert planted_source(k) != clean


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
    assert caught, f"no pin detects plant {k}: {PLANTS[k][0]}"
