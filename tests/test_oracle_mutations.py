"""Plant plausible mistakes in a copy of the oracle and check that a pin catches each.

The mutants are built from the oracle's source text on the CPU; the real
oracle module is never modified.
"""
import importlib.util
import os
import types

import pytest

import oracle_pins as P

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "qlin_oracle.py")

MUTANTS = {
    "zero_point_off_by_one": ("return 1 << (BITS[fmt] - 1)", "return (1 << (BITS[fmt] - 1)) - 1"),
    "nibble_order_swapped": ("codes[:, 0::2] = cb & 0xF\n        codes[:, 1::2] = cb >> 4",
                             "codes[:, 0::2] = cb >> 4\n        codes[:, 1::2] = cb & 0xF"),
    "six_bit_fields_reversed": ("codes[:, i::4] = (word >> (6 * i)) & 0x3F", "codes[:, i::4] = (word >> (6 * (3 - i))) & 0x3F"),
    "round_half_away": ("np.clip(np.rint(v[m])", "np.clip(np.trunc(v[m] + 0.5 * np.sign(v[m]))"),
    "scale_over_128_fp64": ("s[m] = amax / 127.0", "s[m] = amax / 128.0"),
    "scale_over_128_fp32": ("np.float32(amax / np.float32(127.0))", "np.float32(amax / np.float32(128.0))"),
    "rmsnorm_drops_eps": ("np.sqrt(mean_sq + float(eps))", "np.sqrt(mean_sq)"),
    "rmsnorm_one_plus_gamma": ("xv * g[None, :]", "xv * (1.0 + g[None, :])"),
    "swiglu_operands_swapped": ("gv / (1.0 + np.exp(-gv)) * uv", "uv / (1.0 + np.exp(-uv)) * gv"),
    "rmsnorm_mean_over_k_minus_1": ("(xv * xv).sum(axis=1) / K", "(xv * xv).sum(axis=1) / (K - 1)"),
    "group_scale_shifted": ("sw.astype(np.float64)[None, :, :]", "np.roll(sw, 1, axis=1).astype(np.float64)[None, :, :]"),
    "scale_matrix_transposed": ("sw.reshape(N_all, K // G)[rows]", "sw.reshape(K // G, N_all).T[rows]"),
    "row_scale_dropped": ("y64 = s[:, None] * (", "y64 = 1.0 * ("),
    "acc_sign_flipped": ("L = np.asarray(codes, dtype=np.int64) - code_offset(fmt)", "L = code_offset(fmt) - np.asarray(codes, dtype=np.int64)"),
    "stream_hi_bits_moved": ("2 * (reg // 2) + 4 * (reg % 2))", "4 * (reg // 2) + 2 * (reg % 2))"),
    "stream_rows_g_g8_swapped": ("row = g + 8 * (reg % 2)", "row = g + 8 * (reg // 2)"),
    "stream_scale_pairs_transposed": ("f.transpose(1, 3, 2, 0)", "f.transpose(1, 2, 3, 0)"),
    "bias_dropped": ("y64 = y64 + (b if cols is None", "y64 = y64 + 0 * (b if cols is None"),
    "moe_expert_rows_offset": ("cols = e * N + sel", "cols = e * N + sel + (N if e == 0 else 0)"),
    "codebook_index_flipped": ("astype(np.float64)[np.asarray(codes)]", "astype(np.float64)[np.asarray(codes) ^ 8]"),
    "codebook_layout_elements_swapped": ("nib_shift = (8 * reg + 4 * elem)", "nib_shift = (8 * reg + 4 * (1 - elem))"),
    "codebook_layout_registers_as_plain": ("nib_shift = (8 * reg + 4 * elem)", "nib_shift = (16 * elem + 4 * reg)"),
    "rows_top_bits_table_permuted": ("TOP2_POS = (4, 8, 0, 12, 20, 24, 16, 28)", "TOP2_POS = (0, 8, 4, 12, 16, 24, 20, 28)"),
    "rows_second_word_offset_dropped": ("2 * (j[:, None] % 2)", "0 * (j[:, None] % 2)"),
    "rows_scale_block_row_major": ("reshape(ng, R)", "reshape(R, ng).T.reshape(ng, R)"),
    "rows_chunk_and_row_swapped": ('reshape(C, R, 4)\n', 'reshape(R, C, 4).transpose(1, 0, 2)\n'),
    "bias_scaled_by_row_scale": ("y64 = y64 + (b if cols is None else b[np.asarray(cols)])[None, :]",
                                 "y64 = y64 + s[:, None] * (b if cols is None else b[np.asarray(cols)])[None, :]"),
}

PINS = ["hand_example", "file_layout", "forward_bruteforce", "quantize", "prologues",
        "closed_forms", "invariants", "stream_positions", "stream_bijection", "stream_positions_codebook", "stream_positions_rows", "bias",
        "moe", "codebook", "float_sanity"]


def build_mutant(old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("qlin_oracle_mutant")
    exec(compile(src.replace(old, new), SRC + ":mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    mod = build_mutant(*MUTANTS[name])
    caught = []
    for pin in PINS:
        try:
            getattr(P, "check_" + pin)(mod)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin)
    assert caught, f"mutant {name} survived every pin"
