"""Planted mistakes: each plausible error in the oracle must fail some pin.

Every case copies the oracle source to a temporary directory, plants one
mistake by text replacement, builds it with the oracle's own flags and runs the
pins of ``test_oracle_pins`` against that build.  The real oracle is never
modified.  A mutant that survives every pin would mean the pins cannot tell
that mistake from the definition.
"""

from __future__ import annotations

import os
import subprocess

import pytest

import oracle
from tests.test_oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "rpa_oracle.cpp")

# name -> (text in the oracle, planted replacement, replace every occurrence)
MUTANTS = {
    "window_off_by_one": ("if (w > 0 && pos - (w - 1) > 0) first = pos - (w - 1);",
                          "if (w > 0 && pos - w > 0) first = pos - w;", False),
    "gqa_head_mapping": ("const int32_t g = h / group;",
                         "const int32_t g = h % pr.hkv;", False),
    "dropped_scale": ("T xj = scale * dot;", "T xj = dot;", False),
    "softmax_sign": ("std::exp(x[j - lo] - m)", "std::exp(m - x[j - lo])", False),
    "query_position": ("static_cast<int64_t>(pr.kv_lens[s]) - ql + i;",
                       "static_cast<int64_t>(pr.kv_lens[s]) - ql + i - 1;", False),
    "kv_layout_transposed": ("((page * pr.p + slot) * pr.hkv + g) * pr.d + dd",
                             "((page * pr.hkv + g) * pr.p + slot) * pr.d + dd", False),
    "page_table_ignored": ("const int64_t page = pt[j / pr.p];",
                           "const int64_t page = j / pr.p;", True),
    "missing_normalisation": ("out_row[dd] = static_cast<double>(acc / l);",
                              "out_row[dd] = static_cast<double>(acc);", False),
    "values_read_from_keys": ("load(pr, pr.v_pages, kv_index(pr, page, slot, g, dd))",
                              "load(pr, pr.k_pages, kv_index(pr, page, slot, g, dd))",
                              False),
    "fp32_accumulates_in_half_order": ("dot = dot + qv * kv;",
                                       "dot = dot + qv * kv * (dd % 2 == 0 ? 1 : 0);",
                                       False),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new, every = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, "mutation anchor not found: " + old
    text = text.replace(old, new) if every else text.replace(old, new, 1)
    src = tmp_path / "mutant.cpp"
    src.write_text(text)
    lib = str(tmp_path / ("liboracle_%s.so" % name))
    subprocess.run(["g++"] + oracle.CXXFLAGS + ["-o", lib, str(src)], check=True)
    caught = []
    for pin in PINS:
        try:
            ok, detail = pin(lib)
        except (ValueError, FloatingPointError, AssertionError) as e:
            ok, detail = False, repr(e)
        if not ok:
            caught.append(pin.__name__)
            break
    assert caught, "planted mistake %r passed every pin" % name
