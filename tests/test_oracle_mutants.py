"""The pins must catch plausible slips in the oracle.

Each case copies oracle.c, plants one mistake on the CPU (a dropped term, a wrong index,
a swapped operand, a wrong offset), builds the copy with gcc and runs the pins against
it: at least one pin must fail. The committed oracle itself is never modified.
"""
import os
import shutil
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins
from tests import test_oracle_fp16_cpu as f16
from tests import test_sampler_oracle_cpu as gs
from tests import test_staged_write_cpu as sw

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement, pins expected to notice)
MUTANTS = [
    ("gqa_modulo", "Hk, h / group, D, block_size, num_blocks, scale, scores, is_fp16);\n      if (lse) lse[dst]",
     "Hk, h % Hk, D, block_size, num_blocks, scale, scores, is_fp16);\n      if (lse) lse[dst]",
     [pins.test_decode_gqa_head_mapping_with_constant_values]),
    ("no_scale", "scores[t] = scale * dot;", "scores[t] = dot;",
     [pins.test_decode_two_keys_closed_form_scale]),
    ("context_minus_one", "max_blocks, context_lens[b],", "max_blocks, context_lens[b] - 1,",
     [pins.test_decode_single_key_returns_its_value]),
    ("causal_offset", "causal ? (c_s + i + 1) : k_s", "causal ? (c_s + i) : k_s",
     [pins.test_prefill_first_row_without_cache_is_its_own_value,
      pins.test_prefill_brute_force_tiny]),
    ("no_max_subtraction", "scores[t] = exp(scores[t] - m);", "scores[t] = exp(scores[t]);",
     [pins.test_decode_dominant_key_and_no_overflow]),
    ("block_offset", "return phys * block_size + t % block_size;",
     "return phys * block_size + (t + 1) % block_size;",
     [pins.test_decode_contiguous_matches_scipy_softmax, pins.test_page_layout_example_slots_and_rows]),
    ("values_from_keys", "const uint16_t* vt = v_cache +", "const uint16_t* vt = k_cache +",
     [pins.test_decode_single_key_returns_its_value, pins.test_decode_zero_query_is_mean_of_values]),
    ("store_ignores_minus_one", "if (slot == -1) continue;", "if (slot == -1) slot = 0;",
     [pins.test_store_slot_minus_one_leaves_cache_byte_identical]),
    ("staged_start_shift", "memcpy(base + (w_row[w] * cols + w_start[w]) * elem_bytes",
     "memcpy(base + (w_row[w] * cols + w_start[w] + 1) * elem_bytes",
     [sw.test_oracle_reproduces_the_pages_usage_example]),
    ("staged_row_pitch", "memcpy(base + (w_row[w] * cols + w_start[w]) * elem_bytes",
     "memcpy(base + (w_row[w] * rows + w_start[w]) * elem_bytes",
     [sw.test_oracle_reproduces_the_pages_usage_example]),
    ("staged_values_not_advanced", "taken += w_len[w];", "taken += 0;",
     [sw.test_oracle_later_write_wins_on_overlap]),
    ("gumbel_is_exponential", "return logit / temperature - log(-log(u));",
     "return logit / temperature - log(u);",
     [gs.test_samples_follow_softmax_over_seeds]),
    ("gumbel_times_temperature", "return logit / temperature - log(-log(u));",
     "return logit * temperature - log(-log(u));",
     [gs.test_samples_follow_softmax_over_seeds]),
    ("philox_no_key_bump", "      k0 += W0;\n", "      k0 += 0;\n",
     [gs.test_philox_known_answer_vectors]),
    ("philox_swapped_product_word", "const uint32_t n1 = (uint32_t)p1;",
     "const uint32_t n1 = (uint32_t)(p1 >> 32);",
     [gs.test_philox_known_answer_vectors]),
    ("uniform_wrong_shift", "(2u * (bits >> 9) + 1u)", "(2u * (bits >> 8) + 1u)",
     [gs.test_uniform_mapping_closed_form]),
    ("f16_exponent_bias", "else v = ldexp((double)(1024 + m), e - 25);",
     "else v = ldexp((double)(1024 + m), e - 24);",
     [f16.test_f16_widening_matches_numpy_on_every_bit_pattern]),
    ("f16_as_bf16", "return is_fp16 ? f16_bits_to_double(bits) : bf16_bits_to_double(bits);",
     "return bf16_bits_to_double(bits);",
     [f16.test_fp16_and_bf16_agree_on_values_exact_in_both]),
    ("ties_to_highest_index", "      if (x > m1) {", "      if (x >= m1) {",
     [gs.test_greedy_is_numpy_argmax_with_lowest_index_on_ties]),
]


def _call(fn):
    import inspect
    params = inspect.signature(fn).parameters
    if "H" in params:
        return fn(4, 2)
    if "causal" in params:
        return fn(True)
    if "bs" in params:
        return fn(4)
    if "D" in params and "bs" in params:
        return fn(64, 16)
    if "D" in params:
        return fn(64)
    if "T" in params:
        return fn(0.7)
    if "dtype" in params:
        import numpy as np
        return fn(np.int32)
    return fn()


@pytest.mark.parametrize("name,old,new,checks", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, checks):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / "oracle_mut.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"liboracle_{name}.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", str(lib), str(path), "-lm"],
                   check=True)
    prev = oracle.use_library(str(lib))
    try:
        caught = 0
        for fn in checks:
            try:
                _call(fn)
            except (AssertionError, ValueError):
                caught += 1
        assert caught > 0, f"no pin noticed mutant {name}"
    finally:
        oracle.restore_library(prev)
