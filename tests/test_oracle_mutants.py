"""Plant plausible mistakes in copies of the oracle and check that the pins catch each.

Each mutant is the oracle's C source with one textual change (a dropped term, a wrong
sign or index, a swapped operand), compiled into a temporary directory.  The unmodified
oracle passes every pin (tests/test_oracle_pins.py); every mutant must fail at least one.
"""

import os

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "paged_attn_oracle.c")

MUTANTS = {
    "causal_off_by_one": ("if (causal && j > pos)", "if (causal && j >= pos)"),
    "window_off_by_one": ("j < pos - window_left", "j <= pos - window_left"),
    "lse_log2": ("lse[r] = m + log(l);", "lse[r] = m + log2(l);"),
    "dropped_sm_scale": ("s[j] = sm_scale * dot;", "s[j] = dot;"),
    "unnormalised_output": ("o[d] /= l;", "o[d] /= 1.0;"),
    "nibble_order_swapped": ("(elem % 2 == 0) ? (byte & 15) : (byte >> 4)",
                             "(elem % 2 == 0) ? (byte >> 4) : (byte & 15)"),
    "e4m3_subnormal_exponent": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "e4m3_bias": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "gqa_head_mapping": ("row_head[r] / group;", "row_head[r] % Hkv;"),
    "page_table_offset_ignored": ("kv->kv_indices[kv->kv_indptr[b] + t / ps]",
                                  "kv->kv_indices[t / ps]"),
    "v_reads_k_block": ("int64_t block_base = is_v ? (int64_t)kv->Hkv * ps * kv->d_qk : 0;",
                        "int64_t block_base = 0;"),
    "last_page_len_ignored": ("return (npages - 1) * (int64_t)kv->page_size + kv->kv_last_page_len[b];",
                              "return npages * (int64_t)kv->page_size;"),
    "merge_weight_wrong_base": ("double w = exp(lse_parts[s] - *lse);",
                                "double w = exp(lse_parts[s] - M);"),
    "bottom_right_alignment_dropped": ("int64_t pos = kv_len - qo_len + i;", "int64_t pos = i;"),
    "fp8_scale_k_for_v": ("double scale = is_v ? kv->v_scale : kv->k_scale;",
                          "double scale = kv->k_scale;"),
    "sf_block_of_32": ("int64_t sf_index = elem / 16;", "int64_t sf_index = elem / 32;"),
    "mask_bit_order": ("if (!((mask[bit >> 3] >> (bit & 7)) & 1)) allowed = 0;",
                       "if (!((mask[bit >> 3] >> (7 - (bit & 7))) & 1)) allowed = 0;"),
    "mask_row_stride": ("int64_t bit = mask_indptr[b] * 8 + i * kv_len + j;",
                        "int64_t bit = mask_indptr[b] * 8 + i * qo_len + j;"),
    "mask_sequence_offset_ignored": ("int64_t bit = mask_indptr[b] * 8 + i * kv_len + j;",
                                     "int64_t bit = i * kv_len + j;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique / missing"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.load(oracle.compile_oracle(str(path), str(tmp_path / "libmutant.so")))
    failed = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
