"""Every plausible mistake planted in a copy of the oracle trips a pin.

Each mutant is the oracle's C source with one textual change, compiled into a
temporary directory on the CPU.  The pins in ``pins.py`` must reject every
one of them; a mutant that passes them all would mean the pins cannot tell a
broken oracle from a correct one.
"""

import os
import shutil
import subprocess

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kmassign_oracle.c")

MUTANTS = {
    "sign_of_dot_term": ("cnorm - 2.0 * dot(x, c, D)", "cnorm + 2.0 * dot(x, c, D)"),
    "dropped_norm_term": ("cnorm - 2.0 * dot(x, c, D)", "0.0 - 2.0 * dot(x, c, D)"),
    "dropped_factor_two": ("cnorm - 2.0 * dot(x, c, D)", "cnorm - 1.0 * dot(x, c, D)"),
    "dot_uses_one_operand": ("bf16_to_double(a[d]) * bf16_to_double(b[d])",
                             "bf16_to_double(a[d]) * bf16_to_double(a[d])"),
    "ties_go_to_highest_index": ("return a < b;", "return a <= b;"),
    "nan_ordered_lowest": ("if (isnan(a))\n        return 0;\n    if (isnan(b))\n        return 1;",
                           "if (isnan(a))\n        return 1;\n    if (isnan(b))\n        return 0;"),
    "scan_skips_last_centroid": ("for (int64_t j = 1; j < K; ++j)", "for (int64_t j = 1; j + 1 < K; ++j)"),
    "norm_of_abs_not_square": ("acc += v * v;", "acc += fabs(v);"),
    "row_stride_off": ("const uint16_t *x = X + i * D;", "const uint16_t *x = X + i * (D > 1 ? D - 1 : D);"),
    "fp32_dot_accumulator": ("    double acc = 0.0;\n    for (int64_t d = 0; d < D; ++d)\n        acc += bf16",
                             "    float acc = 0.0f;\n    for (int64_t d = 0; d < D; ++d)\n        acc += (float)bf16"),
    "centroid_index_off_by_one": ("score(x, C + j * D, cnorm[j], D)", "score(x, C + j * D, cnorm[j > 0 ? j - 1 : 0], D)"),
    "update_counts_twice": ("        counts[j] += 1;", "        counts[j] += 2;"),
    "update_wrong_dimension": ("sums[(int64_t)j * D + d] += bf16_to_double(X[i * D + d]);",
                               "sums[(int64_t)j * D + d] += bf16_to_double(X[i * D + (d + 1) % D]);"),
    "update_keeps_invalid_ids": ("        if (j < 0 || j >= K)\n            continue;",
                                 "        if (j < 0 || j >= K)\n            j = 0;"),
    "topk_ties_to_higher_index": ("    return ja < jb;   /* equal scores, or both NaN */",
                                  "    return ja > jb;   /* equal scores, or both NaN */"),
    "topk_drops_last_slot": ("            if (pos >= k)\n                continue;",
                             "            if (pos >= k - 1 && k > 1)\n                continue;"),
    "topk_centroid_index_off_by_one": ("score(xi, C + j * D, cnorm[j], D)",
                                       "score(xi, C + j * D, cnorm[j > 0 ? j - 1 : 0], D)"),
    "sqdist_adds_instead_of_subtracting": (
        "double diff = bf16_to_double(x[d]) - bf16_to_double(c[d]);",
        "double diff = bf16_to_double(x[d]) + bf16_to_double(c[d]);"),
    "sqdist_skips_last_dimension": ("        for (int64_t d = 0; d < D; ++d) {\n            double diff",
                                    "        for (int64_t d = 0; d + 1 < D; ++d) {\n            double diff"),
    "update_skips_first_point": ("    for (int64_t i = 0; i < N; ++i) {\n        int32_t j",
                                 "    for (int64_t i = 1; i < N; ++i) {\n        int32_t j"),
}


@pytest.fixture(scope="module")
def workdir(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    return tmp_path_factory.mktemp("mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(workdir, name):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) == 1, f"mutation site for {name} not unique/present"
    src = workdir / f"{name}.c"
    src.write_text(text.replace(old, new))
    lib_path = str(workdir / f"lib{name}.so")
    oracle.build(force=True, src=str(src), out=lib_path)
    orc = oracle.Oracle(oracle.load_library(lib_path))
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
