"""Plant plausible mistakes in copies of the oracle and require the pins to catch each.

Every mutant is built on the CPU from a modified copy of oracle/msa_oracle.c
in a temporary directory; the real oracle is never touched.
"""

import os

import pytest

import oracle
import oracle_pins as pins

MUTANTS = [
    ("drop the last dimension", "d < DIM; ++d", "d < DIM - 1; ++d"),
    ("read the whole last page", "if (valid > PAGE)\n                    valid = PAGE;", "valid = PAGE;"),
    ("skip the last valid token", "t < valid; ++t", "t < valid - 1; ++t"),
    ("head 0's query for every head", "q + ((int64_t)b * HEADS + h) * DIM", "q + ((int64_t)b * HEADS) * DIM"),
    ("min instead of max", "if (dot > best)", "if (best == -INFINITY || dot < best)"),
    ("transposed key tile",
     "bf16_to_double(krow[d])",
     "bf16_to_double(pool[((int64_t)page * DIM + d) * PAGE + t])"),
    ("scaled scores", "if (dot > best)", "dot *= 0.08838834764831845;\n                    if (dot > best)"),
    ("tie-break toward the higher id",
     "if (a->id < b->id)\n        return -1;\n    if (a->id > b->id)\n        return 1;",
     "if (a->id < b->id)\n        return 1;\n    if (a->id > b->id)\n        return -1;"),
    ("lower score first",
     "if (a->score > b->score)\n        return -1;\n    if (a->score < b->score)\n        return 1;",
     "if (a->score > b->score)\n        return 1;\n    if (a->score < b->score)\n        return -1;"),
    ("window pin off by one", "|| j >= nb - n_window;", "|| j > nb - n_window;"),
    ("sink pin off by one", "return j < n_sink ||", "return j <= n_sink ||"),
    ("pad ids with 0", "out_ids[filled] = -1;", "out_ids[filled] = 0;"),
    ("bf16 read as the low half", "((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    ("e4m3 exponent bias 6", "ldexp(1.0 + mantissa / 8.0, exponent - 7)", "ldexp(1.0 + mantissa / 8.0, exponent - 6)"),
    ("e4m3 subnormals read as normals", "magnitude = ldexp(mantissa / 8.0, -6);", "magnitude = ldexp(1.0 + mantissa / 8.0, -7);"),
    ("fp8 scale ignored", "double scale = (double)kscale[(int64_t)page * PAGE + t];", "double scale = 1.0;"),
    ("expansion keeps the selection order", "qsort(sel, (size_t)n_sel, sizeof(int), cmp_int);", ""),
    ("expansion includes the pages past the end", "if (p < small_pages)\n                        out[n++]", "if (p <= small_pages)\n                        out[n++]"),
]


def _cases():
    """Each mutant at every place its anchor occurs (the bf16 and fp8 scoring
    loops share some text): one test per (mutant, occurrence)."""
    src = open(oracle.SOURCE).read()
    out = []
    for name, old, new in MUTANTS:
        n = src.count(old)
        assert n >= 1, f"mutation anchor for {name!r} not found"
        for i in range(n):
            out.append(pytest.param(name, old, new, i, id=f"{name} #{i}" if n > 1 else name))
    return out


def _replace_nth(text, old, new, n):
    at = -1
    for _ in range(n + 1):
        at = text.index(old, at + 1)
    return text[:at] + new + text[at + len(old):]


@pytest.mark.parametrize("name,old,new,which", _cases())
def test_pins_catch_mutant(tmp_path, name, old, new, which):
    src = open(oracle.SOURCE).read()
    mutated = tmp_path / "msa_oracle_mutant.c"
    mutated.write_text(_replace_nth(src, old, new, which))
    lib = oracle.build(src=str(mutated), out=str(tmp_path / "libmutant.so"))
    mutant = oracle.load(lib)
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            check(mutant)
        except (AssertionError, ValueError):
            caught.append(check.__name__)
    assert caught, f"no pin caught the mutant {name!r}"
