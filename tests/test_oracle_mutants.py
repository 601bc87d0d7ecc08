"""Plant plausible mistakes in copies of the C oracle and check that the
pins catch every one of them (CPU only).

Each mutant is a textual edit of ``oracle/dc_oracle.c`` written to a
temporary folder, compiled with the oracle's flags and loaded on its own;
the real oracle is never modified.
"""
from __future__ import annotations

import os

import pytest

import oracle
import oracle_pins
from oracle import build as oracle_build

SRC = os.path.join(os.path.dirname(oracle_build.__file__), "dc_oracle.c")

MUTANTS = {
    # fold order: ranks 1..P-1 added in reverse
    "reverse_rank_order": ("float x = orc_bf16_to_f32(in[q][i]);",
                           "float x = orc_bf16_to_f32(in[P - q][i]);"),
    # accumulator starts at +0 instead of rank 0's value
    "zero_initial_accumulator": ("float acc = orc_bf16_to_f32(in[0][i]);\n    for (int q = 1;",
                                 "float acc = 0.0f;\n    for (int q = 0;"),
    # the last rank is dropped
    "drop_last_rank": ("for (int q = 1; q < P; ++q) {", "for (int q = 1; q < P - 1; ++q) {"),
    # typed linear fold: the last rank dropped
    "typed_drop_last_rank": ("for (int q = 1; q < P; ++q)\n        acc = acc + x[q];",
                             "for (int q = 1; q < P - 1; ++q)\n        acc = acc + x[q];"),
    # BF16 rounding after every add instead of binary32 accumulation
    "bf16_accumulation": ("acc = acc + x;",
                          "acc = orc_bf16_to_f32(orc_f32_to_bf16_rne(acc + x));"),
    # truncation instead of round to nearest even
    "truncate": ("u += 0x7FFFu + lsb;", "u += 0u * lsb;"),
    # ties away from zero instead of ties to even
    "round_half_up": ("u += 0x7FFFu + lsb;", "u += 0x8000u + 0u * lsb;"),
    # NaN is rounded like a number (a carry can turn it into infinity)
    "nan_not_special": ("if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)",
                        "if (0)"),
    # gather writes the ranks in reverse order
    "gather_reverse_ranks": ("= peers[r][j];", "= peers[P - 1 - r][j];"),
    # gather reads each payload shifted by one byte
    "gather_shifted_source": ("out[(size_t)r * B + j] = peers[r][j];",
                              "out[(size_t)r * B + j] = peers[r][(j + 1) % B];"),
    # gather_many reuses the wrong peers for later tensors
    "gather_many_wrong_peers": ("peers + (size_t)t * (size_t)P", "peers + (size_t)t"),
    # reduce_scatter takes interleaved instead of contiguous shards
    "reduce_scatter_interleaved": ("fold_ranks(in, P, (size_t)r * C + j)",
                                   "fold_ranks(in, P, j * (size_t)P + (size_t)r)"),
    # all_reduce only fills rank 0's output
    "all_reduce_one_output": ("out[r][i] = y;", "out[0][i] = y;"),
    # binary16: truncation instead of round to nearest even
    "f16_truncate": ("uint32_t r = a + 0x0FFFu + ((a >> 13) & 1u);", "uint32_t r = a;"),
    # binary16: only infinity saturates; large finite values overflow the exponent
    "f16_no_overflow_check": ("if (a >= 0x477FF000u)", "if (a >= 0x7F800000u)"),
    # binary16 subnormals: off-by-one scale
    "f16_subnormal_scale": ("int sh = -(e + 1);", "int sh = -e;"),
    # binary16 widening: wrong exponent bias
    "f16_widen_bias": ("u = sign | ((e - 15u + 127u) << 23) | (f << 13);",
                       "u = sign | ((e - 15u + 128u) << 23) | (f << 13);"),
    # tree order: halves instead of the largest power of two below the count
    "tree_half_split": ("int m = 1;\n    while (m * 2 < n)\n        m *= 2;", "int m = n / 2;"),
    # tree order ignored
    "tree_is_linear": ("if (order == ORC_ORDER_TREE)", "if (0)"),
    # binary16 payloads widened as BF16
    "f16_read_as_bf16": ("return dtype == ORC_F16 ? orc_f16_to_f32(h) : orc_bf16_to_f32(h);",
                         "return orc_bf16_to_f32(h);"),
}


def _caught(orc) -> str | None:
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(orc)
        except (AssertionError, ValueError) as e:  # the pin rejected the oracle
            return f"{check.__name__}: {type(e).__name__}"
    return None


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib = oracle_build.compile_source(str(src), str(tmp_path / f"lib_{name}.so"))
    caught_by = _caught(oracle.load(lib))
    assert caught_by is not None, f"no pin catches the mutant {name}"
