"""Planted mistakes: each test patches one plausible bug into a copy of the oracle's C
source, builds it in a temporary directory and checks that the pins in test_oracle.py
catch it.  This shows the pins are sharp enough to notice a dropped term, a wrong sign
or index, or a transposed operand anywhere in the oracle (CPU only)."""
import os

import pytest

import oracle
import test_append_oracle as apins
import test_oracle as pins
from oracle.build import SRC, build

MUTANTS = {
    "gqa_group_by_modulo": ("int g = h / G;", "int g = h % c->num_kv_heads;"),
    "k_wrong_slot": ("int slot = j % bs;\n    if (page < 0",
                     "int slot = (j + 1) % bs;\n    if (page < 0"),
    "v_wrong_slot": ("size_t voff = (((size_t)page * bs + slot)",
                     "size_t voff = (((size_t)page * bs + (bs - 1 - slot))"),
    "causal_off_by_one": ("return p->c->causal ? n - ql + i + 1 : n;",
                          "return p->c->causal ? n - ql + i : n;"),
    "padding_rows_attend": ("if (i >= ql) return 0;", "if (i >= ql + 1) return 0;"),
    "sm_scale_dropped": ("s[j - j0] = (real)c->sm_scale * dot;", "s[j - j0] = dot;"),
    "max_not_subtracted": ("real e = R_EXP(s[j - j0] - m);", "real e = R_EXP(s[j - j0]);"),
    "lse_without_max": ("*lse = m + R_LOG(den);", "*lse = R_LOG(den);"),
    "not_normalised": ("for (int d = 0; d < D; ++d) o[d] /= den;", ""),
    "q_heads_and_rows_transposed": (
        "(((size_t)b * c->max_q_len + i) * c->num_q_heads + h)",
        "(((size_t)b * c->num_q_heads + h) * c->max_q_len + i)"),
    "merge_weight_sign": ("R_EXP(lse_s[s] - mx)", "R_EXP(mx - lse_s[s])"),
    "split_drops_tail": ("int chunk = (L + nsplit - 1) / nsplit;", "int chunk = L / nsplit;"),
    "e4m3_bias": ("v = ldexp((double)(8 + m), e - 10);", "v = ldexp((double)(8 + m), e - 11);"),
    "e4m3_subnormal_scale": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    "fp16_exponent": ("ldexp((double)(1024 + m), e - 25)", "ldexp((double)(1024 + m), e - 24)"),
    "bf16_shift": ("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
    "token_scale_ignores_head": (
        "return (real)s[((size_t)page * c->block_size + slot) * c->num_kv_heads + g];",
        "return (real)s[((size_t)page * c->block_size + slot) * c->num_kv_heads];"),
    "v_scaled_by_k_scale": ("real vs = row_scale(p, 1, page, slot, g);",
                            "real vs = row_scale(p, 0, page, slot, g);"),
    # quantise-on-write append
    "append_wrong_slot": ("      int slot = pos % bs;\n", "      int slot = (pos + 1) % bs;\n"),
    "append_position_ignores_q_len": (
        "int pos = n - ql + i;\n      int page = block_tables[(size_t)b * c->max_blocks_per_seq + pos / bs];\n      int slot",
        "int pos = n - 1 - i;\n      int page = block_tables[(size_t)b * c->max_blocks_per_seq + pos / bs];\n      int slot"),
    "append_scale_divisor": ("s = amax > 0.0f ? amax / 448.0f : 1.0f;",
                             "s = amax > 0.0f ? amax / 447.0f : 1.0f;"),
    "append_zero_row_scale": ("s = amax > 0.0f ? amax / 448.0f : 1.0f;",
                              "s = amax > 0.0f ? amax / 448.0f : 0.0f;"),
    "append_v_uses_k_scale": ("float *scales = t ? v_scale : k_scale;",
                              "float *scales = t ? k_scale : k_scale;"),
    "append_tensor_scale_ignored": ("s = scales[0];", "s = 1.0f;"),
    "encode_ties_away_from_zero": ("(fr == 0.5 && fmod(fl, 2.0) == 1.0)", "(fr == 0.5)"),
    "encode_no_clamp": ("if (a > 448.0) a = 448.0;", ""),
    "encode_subnormal_step": ("  int e = -6;\n", "  int e = -7;\n"),
}


def _pins():
    """The pins, as calls: (name, thunk)."""
    out = []
    for i in range(4):
        out.append((f"golden{i}", lambda i=i: pins.test_golden_hand_cases(i, "f64")))
    out.append(("golden_e4m3", pins.test_golden_e4m3_table))
    out.append(("e4m3_all", pins.test_e4m3_all_codes_match_torch))
    out.append(("bf16_all", lambda: pins.test_16bit_decoders_all_codes("bf16")))
    out.append(("fp16_all", lambda: pins.test_16bit_decoders_all_codes("fp16")))
    for ci in range(len(pins.BRUTE_CASES)):
        out.append((f"brute{ci}",
                    lambda ci=ci: pins.test_oracle_matches_contiguous_brute_force(ci, "f64")))
    out.append(("split3", lambda: pins.test_split_invariance(3, "f64")))
    for i in range(5):
        out.append((f"append_golden{i}", lambda i=i: apins.test_golden_append_cases(i, "f64")))
    out.append(("append_encode_grid",
                apins.test_e4m3_encode_matches_torch_on_grid_midpoints_and_neighbours))
    for mode in ("token", "tensor", "none"):
        out.append((f"append_fp8_{mode}",
                    lambda mode=mode: apins.test_fp8_append_codes_and_scales(mode, "bf16")))
    out.append(("append_16bit", lambda: apins.test_16bit_append_places_rows_bitwise("bf16", "bf16")))
    out.append(("zero_scale", lambda: pins.test_zero_scale_gives_mean_over_visible_keys("f64")))
    return out


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "pa_oracle.c"
    mutated.write_text(src.replace(old, new))
    build(str(mutated), str(tmp_path))
    caught = []
    with oracle.libs_from(str(tmp_path)):
        for pin, thunk in _pins():
            try:
                thunk()
            except (AssertionError, ValueError):
                caught.append(pin)
    assert caught, f"no pin caught the planted mistake {name}"


def test_unpatched_source_passes_the_same_pins(tmp_path):
    build(SRC, str(tmp_path))
    with oracle.libs_from(str(tmp_path)):
        for pin, thunk in _pins():
            thunk()
