"""Planted mistakes in the CPU oracle fail its pins.

Each case edits a copy of oracle/oracle.c in a temporary directory (never the
committed file), builds it with the same flags, and expects at least one pin in
tests/oracle_pins.py to fail on it.  This shows that the pins would catch a
dropped term, a wrong summation order or start value, a wrong index, a
transposed operand or a wrong rounding rule in the oracle itself.
"""
import os
import subprocess
import sys

import pytest

import oracle.build as obuild

MUTATIONS = {
    "fold_drops_last_rank": ("for (int r = 1; r < R; ++r)\n        acc = acc +",
                             "for (int r = 1; r < R - 1; ++r)\n        acc = acc +"),
    "fold_starts_from_plus_zero": ("float acc = load_f32(bufs[0], dtype, idx[0]);\n    for (int r = 1; r < R; ++r)\n"
                                   "        acc = acc +",
                                   "float acc = 0.0f;\n    for (int r = 0; r < R; ++r)\n        acc = acc +"),
    "fold_reverse_order": ("float acc = load_f32(bufs[0], dtype, idx[0]);\n    for (int r = 1; r < R; ++r)\n"
                           "        acc = acc + load_f32(bufs[r], dtype, idx[r]);",
                           "float acc = load_f32(bufs[R - 1], dtype, idx[R - 1]);\n    for (int r = R - 2; r >= 0; --r)\n"
                           "        acc = acc + load_f32(bufs[r], dtype, idx[r]);"),
    "rounding_ties_toward_zero": ("if (dt < da)\n        pick = t;", "if (dt <= da)\n        pick = t;"),
    "rounding_truncates": ("uint32_t pick;\n", "uint32_t pick = t; if (1) return (uint16_t)(pick >> 16);\n"),
    "allgather_wrong_source": ("copy_elem(out[r], base + i, in[j], i, dtype);",
                               "copy_elem(out[r], base + i, in[r], i, dtype);"),
    "reducescatter_ignores_offset": ("idx[r] = o + i;\n            store_f32(out[k]",
                                     "idx[r] = i;\n            store_f32(out[k]"),
    "alltoall_transposed_lengths": ("src_base += nm[(uint64_t)r * R + jj];",
                                    "src_base += nm[(uint64_t)jj * R + r];"),
    "alltoall_dest_order_by_dest": ("uint64_t len = nm[(uint64_t)r * R + j];",
                                    "uint64_t len = nm[(uint64_t)j * R + r];"),
    "ulysses_head_index_swapped": ("in[r], (s * H + (uint64_t)j * hs + h) * D + d",
                                   "in[r], (s * H + h * (uint64_t)R + j) * D + d"),
    "layout_region_ignores_stride": ("return p->offset + (j / p->len) * p->row_stride + (j % p->len);",
                                     "return p->offset + j;"),
    "max_keeps_later_ties": ("        if (v > acc)\n            acc = v;", "        if (v >= acc)\n            acc = v;"),
    "max_is_min": ("        if (v > acc)\n            acc = v;", "        if (v < acc)\n            acc = v;"),
    "f16_ties_away_from_zero": ("        n = fmod(t, 2.0) == 0.0 ? t : t + 1.0;", "        n = t + 1.0;"),
    "f16_wrong_subnormal_spacing": ("        ulp = ldexp(1.0, -24);\n    } else {", "        ulp = ldexp(1.0, -25);\n    } else {"),
    "f16_no_overflow_to_inf": ("    if (v >= 65536.0)\n        return (uint16_t)(sign | 0x7C00u);", "    if (v > 1e300)\n        return (uint16_t)(sign | 0x7C00u);"),
    "layout_sum_accepts_any_rank_order": ("if (src_rank[r] != r || region_count(src[r]) != cnt)",
                                          "if (region_count(src[r]) != cnt)"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, f"mutation {name}: anchor not found exactly once"
    path = os.path.join(tmp_path, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(tmp_path, f"lib{name}.so")
    subprocess.run(["gcc", *[c for c in obuild.CFLAGS if c != "-Werror"], path, "-o", lib, "-lm"],
                   check=True)
    return lib


_CHILD = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
m = oracle.Oracle({lib!r})
failed = []
for check in oracle_pins.ALL_CHECKS:
    try:
        check(m)
    except (AssertionError, ValueError, TypeError):
        failed.append(check.__name__)
print("FAILED_PINS", ",".join(failed))
"""


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    lib = _build_mutant(str(tmp_path), name, old, new)
    tests = os.path.dirname(os.path.abspath(__file__))
    code = _CHILD.format(root=os.path.dirname(tests), tests=tests, lib=lib)
    # A mutant may also read out of bounds and crash: that is a failure the pins expose too.
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if p.returncode != 0:
        return
    line = [ln for ln in p.stdout.splitlines() if ln.startswith("FAILED_PINS")][-1]
    failed = [x for x in line.split(" ", 1)[1].split(",") if x]
    assert failed, f"no pin caught the planted mistake {name!r}"
