"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of the oracle's C source, on the CPU
(a shifted field, a wrong mask, OR for XOR, a swapped direction, a wrong
index, a wrong bank modulus, broken broadcast, ...), compiles the copy and
runs the pin battery of test_oracle.py against it.  At least one pin must
fail for every mistake; the unmodified copy must pass them all.
"""
import pytest

import oracle
import test_oracle as pins

MUTATIONS = [
    ("y field one bit too high", "int ypos = ylo + i;", "int ypos = ylo + 1 + i;"),
    ("y field one bit too low", "int ypos = ylo + i;", "int ypos = ylo - 1 + i;"),
    ("z field one bit too high", "int zpos = zlo + i;", "int zpos = zlo + 1 + i;"),
    ("negative shift read below MBase (the formula taken literally)",
     "int zlo = shift >= 0 ? base : base - shift;   /* the field that is written */\n    int ylo = shift >= 0 ? base + shift : base;",
     "int zlo = base;   /* the field that is written */\n    int ylo = base + shift;"),
    ("negative shift taken as its magnitude",
     "int zlo = shift >= 0 ? base : base - shift;   /* the field that is written */\n    int ylo = shift >= 0 ? base + shift : base;",
     "int zlo = base;   /* the field that is written */\n    int ylo = shift >= 0 ? base + shift : base - shift;"),
    ("field one bit short", "for (i = 0; i < bits; ++i) {", "for (i = 0; i < bits - 1; ++i) {"),
    ("OR instead of XOR", "v = orc_bit(offset, zpos) ^ orc_bit(offset, ypos);",
     "v = orc_bit(offset, zpos) | orc_bit(offset, ypos);"),
    ("z bit never cleared", "out &= ~((uint64_t)1 << zpos);", "out = out;"),
    ("set bit written one place up", "out |= (uint64_t)1 << zpos;", "out |= (uint64_t)1 << (zpos + 1);"),
    ("relayout forward as a gather",
     "memcpy(d + (size_t)(tile0 + (int64_t)j) * esize,\n                       s + (size_t)(tile0 + i) * esize, (size_t)esize);",
     "memcpy(d + (size_t)(tile0 + i) * esize,\n                       s + (size_t)(tile0 + (int64_t)j) * esize, (size_t)esize);"),
    ("relayout on global offsets", "uint64_t j = orc_swizzle((uint64_t)i, base, bits, shift);",
     "uint64_t j = orc_swizzle((uint64_t)(tile0 + i), base, bits, shift) - (uint64_t)tile0;"),
    ("transpose writes with the wrong stride", "memcpy(d + (size_t)(c * rows + r) * esize,",
     "memcpy(d + (size_t)(c * cols + r) * esize,"),
    ("bank modulus 16", "if ((int)(words[k] % 32) == bank)", "if ((int)(words[k] % 16) == bank)"),
    ("last word one too far", "last = (a + (uint64_t)width - 1) / 4;", "last = (a + (uint64_t)width) / 4;"),
    ("16-byte accesses in two passes", "passes = (width <= 4) ? 1 : width / 4;",
     "passes = (width <= 4) ? 1 : 2;"),
    ("8-byte accesses in one pass", "passes = (width <= 4) ? 1 : width / 4;",
     "passes = (width <= 8) ? 1 : width / 4;"),
    ("passes interleave the lanes",
     "for (lane = pass * lanes_per_pass; lane < (pass + 1) * lanes_per_pass; ++lane) {",
     "for (lane = pass; lane < 32; lane += passes) {"),
    ("no broadcast: repeated words counted",
     "for (k = 0; k < n_words; ++k)\n                        if (words[k] == wd)\n                            seen = 1;",
     "(void)seen;"),
    ("wavefronts = worst pass", "total += cost;", "total = worst;"),
    ("fused: relayout before the transpose",
     "rc = orc_transpose(tmp, src, rows, cols, esize);\n    if (rc != ORC_OK)\n        return rc;\n    return orc_relayout(dst, tmp, (rows * cols) / tile_elems, tile_elems, esize, base, bits, shift, 0);",
     "rc = orc_relayout(tmp, src, (rows * cols) / tile_elems, tile_elems, esize, base, bits, shift, 0);\n    if (rc != ORC_OK)\n        return rc;\n    return orc_transpose(dst, tmp, rows, cols, esize);"),
    ("fused: inverse relayout",
     "return orc_relayout(dst, tmp, (rows * cols) / tile_elems, tile_elems, esize, base, bits, shift, 0);",
     "return orc_relayout(dst, tmp, (rows * cols) / tile_elems, tile_elems, esize, base, bits, shift, 1);"),
    ("collision keeps A & sw(A)", "return A & ~orc_swizzle(A, base, bits, shift);",
     "return A & orc_swizzle(A, base, bits, shift);"),
]


def battery(orc):
    """Run the pins on `orc`; return the names of the ones that fail."""
    checks = [
        ("worked_example", lambda: pins.test_worked_example_673(orc)),
        ("mapping_32x32", lambda: pins.test_two_d_mappings(orc, 32, 32, pins._mapping_32x32, (5, 0, 5))),
        ("mapping_64x32", lambda: pins.test_two_d_mappings(orc, 64, 32, pins._mapping_64x32, (5, 0, 5))),
        ("mapping_32x64", lambda: pins.test_two_d_mappings(orc, 32, 64, pins._mapping_32x64, (5, 0, 6))),
        ("mapping_half", lambda: pins.test_two_d_mappings(orc, 32, 64, pins._mapping_half_pairs, (5, 1, 5))),
        ("bit_diagrams", lambda: pins.test_bit_diagrams(orc)),
        ("invariants_333", lambda: pins.test_swizzle_invariants(orc, 3, 3, 3)),
        ("invariants_525", lambda: pins.test_swizzle_invariants(orc, 5, 2, 5)),
        ("degenerate", lambda: pins.test_swizzle_degenerate(orc)),
        ("negative_mirror", lambda: pins.test_negative_shift_mirrors_positive(orc, 3, 4, 10, 4)),
        ("negative_mirror_overlap", lambda: pins.test_negative_shift_mirrors_positive(orc, 3, 0, 1, 2)),
        ("negative_invariants", lambda: pins.test_negative_shift_invariants(orc, 3, 2, -4)),
        ("relayout_roundtrip", lambda: pins.test_relayout_roundtrip_and_closed(orc)),
        ("relayout_tile_local", lambda: pins.test_relayout_tile_local(orc, 48)),
        ("relayout_usage_loop", lambda: pins.test_relayout_usage_loop(orc)),
        ("transpose_small", lambda: pins.test_transpose_small(orc)),
        ("transpose_relayout", lambda: pins.test_transpose_relayout_composes(orc)),
        ("bank_column", lambda: pins.test_bank_column_fp32(orc)),
        ("bank_padding_xor", lambda: pins.test_bank_padding_and_xor(orc)),
        ("bank_fp16", lambda: pins.test_bank_fp16_64_columns(orc)),
        ("bank_usage", lambda: pins.test_bank_usage_examples(orc)),
        ("bank_broadcast", lambda: pins.test_bank_broadcast(orc)),
        ("bank_passes", lambda: pins.test_bank_minimum_passes(orc)),
        ("bank_ldmatrix", lambda: pins.test_bank_ldmatrix_x4_passes(orc)),
        ("bank_8byte", lambda: pins.test_bank_8byte_passes(orc)),
        ("bank_unaligned", lambda: pins.test_bank_inactive_and_unaligned(orc)),
        ("collision_table", lambda: pins.test_collision_truth_table(orc)),
        ("collision_layout", lambda: pins.test_collision_predicts_layout(orc, 2, 0, 2)),
        ("dump", lambda: pins.test_dump_layout(orc)),
    ]
    failed = []
    for name, fn in checks:
        try:
            fn()
        except (AssertionError, ValueError, OverflowError):
            failed.append(name)
    return failed


def test_unmodified_copy_passes(tmp_path):
    orc = oracle.Oracle(oracle.compile_copy(oracle.c_source(), str(tmp_path)))
    assert battery(orc) == []


_CHILD = """
import json, sys
sys.path[:0] = [{tests!r}, {root!r}]
import oracle, test_oracle_mutations as tm
print(json.dumps(tm.battery(oracle.Oracle({lib!r}))))
"""


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    """The battery runs on the mutated copy in a child process: a mistake
    that writes out of bounds may crash it, and a crash counts as caught."""
    import json
    import os
    import subprocess
    import sys
    src = oracle.c_source()
    assert src.count(old) == 1, name
    lib = oracle.compile_copy(src.replace(old, new), str(tmp_path))
    tests = os.path.dirname(os.path.abspath(__file__))
    code = _CHILD.format(tests=tests, root=os.path.dirname(tests), lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if r.returncode != 0:
        return  # the planted mistake crashed the pins: caught
    failed = json.loads(r.stdout.strip().splitlines()[-1])
    assert failed, f"no pin caught: {name}"
