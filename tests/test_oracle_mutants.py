"""Planted mistakes: each mutated build of the oracle must fail at least one pin.

A mutation is a one-line textual edit of the C source (a dropped term, a wrong sign, index or
operand), compiled into a temporary library. If every pin still passed, the pins would not be
able to tell that oracle from the real one.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "mask_one_short": ("return p->context_lens[b] - p->q_len + i;",
                       "return p->context_lens[b] - p->q_len + i - 1;"),
    "dropped_softmax_scale": ("return dot / sqrt((double)p->D);", "return dot;"),
    "gqa_head_map_transposed": ("int h = hq / (p->Hq / p->Hkv);", "int h = hq % p->Hkv;"),
    "page_slot_off_by_one": ("int slot = j % p->P;", "int slot = (j + 1) % p->P;"),
    "dropped_v_scale": ("return e4m3[p->v_pool[kv_offset(p, b, j, h) + d]] * p->v_scale;",
                        "return e4m3[p->v_pool[kv_offset(p, b, j, h) + d]];"),
    "merge_weight_dropped": ("L += w * l[r * S + s];", "L += l[r * S + s];"),
    "q_layout_transposed": ("p->q + (((int64_t)b * p->q_len + i) * p->Hq + hq) * p->D;",
                            "p->q + (((int64_t)b * p->Hq + hq) * p->q_len + i) * p->D;"),
    "subnormal_exponent": ("mag = ldexp((double)mant, -9);", "mag = ldexp((double)mant, -10);"),
    "lse_without_max": ("double l = mx + log(sum);", "double l = log(sum);"),
    "partials_max_sign": ("double w = exp(score(&p, e4m3, b, i, hq, j) - mx);",
                          "double w = exp(mx - score(&p, e4m3, b, i, hq, j));"),
    "encode_ties_to_odd": ("(err == best_err && (c & 1) == 0)", "(err == best_err && (c & 1) == 1)"),
    "encode_truncates": ("if (err < best_err || (err == best_err && (c & 1) == 0)) {",
                         "if (oracle_e4m3_value((uint8_t)c) <= a) {"),
    "encode_sign_dropped": ("return (uint8_t)(best | (neg << 7));", "return (uint8_t)best;"),
    "kv_write_position_shift": ("const int pos = n - q_len + i;", "const int pos = n - q_len + i + 1;"),
    "kv_write_slot_off_by_one": ("const int64_t dst = (((int64_t)page * P + pos % P) * Hkv + h) * D;",
                                 "const int64_t dst = (((int64_t)page * P + (pos + 1) % P) * Hkv + h) * D;"),
    "kv_write_wrong_scale": ("const float vq = v_new[src + d] / v_scale;",
                             "const float vq = v_new[src + d] / k_scale;"),
    "kv_write_double_quotient": ("k_pool[dst + d] = oracle_e4m3_encode((double)kq);",
                                 "k_pool[dst + d] = oracle_e4m3_encode((double)k_new[src + d] / k_scale);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.compile_oracle(str(mutated), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in oracle_pins.PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin detects the planted mistake {name}"
