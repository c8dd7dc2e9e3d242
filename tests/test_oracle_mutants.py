"""Plant one plausible mistake at a time in a copy of the oracle's C source
and require that at least one pin catches it.  This shows the pins are
strong enough to notice a dropped term, a wrong index or a swapped operand
anywhere in the oracle (no GPU)."""
import os
import shutil

import pytest

import oracle
import oracle_pins

# (name, exact text in pseq_oracle.c, replacement)
MUTANTS = [
    ("o1_no_row_start", "int row_start = (s == 0);", "int row_start = 0;"),
    ("o1_wrong_neighbour", "read_int(doc_ids, elem_bytes, t - 1);", "read_int(doc_ids, elem_bytes, t > 1 ? t - 2 : 0);"),
    ("o1_no_final_end", "if (total > 0) cu_out[n++] = (int32_t)total;", "if (0) cu_out[n++] = (int32_t)total;"),
    ("o1_max_off_by_one", "int64_t len = (int64_t)cu_out[k + 1] - (int64_t)cu_out[k];",
     "int64_t len = (int64_t)cu_out[k + 1] - (int64_t)cu_out[k] - 1;"),
    ("o1_max_skips_last", "for (int64_t k = 0; k < num_segments; ++k) {", "for (int64_t k = 0; k + 1 < num_segments; ++k) {"),
    ("o2_offset_from_real", "offset_in_row += padded;", "offset_in_row += real;"),
    ("o2_cu_from_padded", "run_real += seq_real[i];", "run_real += seq_padded[i];"),
    ("o2_no_absorption", "if (pad_only_at_end) cu[n] = (int32_t)T;", "if (0) cu[n] = (int32_t)T;"),
    ("o2_gate_includes_last", "for (int64_t i = 0; i + 1 < n; ++i)\n      if (seq_real[i] != seq_padded[i])",
     "for (int64_t i = 0; i < n; ++i)\n      if (seq_real[i] != seq_padded[i])"),
    ("o2_gate_ignored", "if (seq_real[i] != seq_padded[i]) pad_only_at_end = 0;", "if (0) pad_only_at_end = 0;"),
    ("o2_pad_between_inverted", "if (cu[i] != cu_padded[i]) differ = 1;", "if (cu[i] == cu_padded[i]) differ = 1;"),
    ("o2_max_from_padded", "int64_t w = (int64_t)cu[i + 1] - (int64_t)cu[i];",
     "int64_t w = (int64_t)cu_padded[i + 1] - (int64_t)cu_padded[i];"),
    ("o2_no_row_check", "if (offset_in_row > S) return ORC_VALUE;", "if (0) return ORC_VALUE;"),
    ("o2_no_filler_check", "if (real_is_filler != padded_is_filler) return ORC_VALUE;", ""),
    ("o3_row_dropped", "int64_t src_token = (p * B + seq_row[i]) * S + seq_off[i] + j;",
     "int64_t src_token = (p * B) * S + seq_off[i] + j;"),
    ("o3_plane_stride_B", "int64_t dst_token = p * T + (int64_t)cu_padded[i] + j;",
     "int64_t dst_token = p * B + (int64_t)cu_padded[i] + j;"),
    ("o4_clear_padded", "for (int64_t j = 0; j < real; ++j) mask[start + j] = 0;",
     "for (int64_t j = 0; j < padded; ++j) mask[start + j] = 0;"),
    ("o4_start_by_real", "start += padded;\n  }\n  return ORC_OK;", "start += real;\n  }\n  return ORC_OK;"),
    ("o5_floor_not_ceil", "int64_t padded = ((real + multiple - 1) / multiple) * multiple;",
     "int64_t padded = (real / multiple) * multiple;"),
    ("o5_stretch_wrong_entry", "if (stretch) bcup[count] = (int32_t)capacity;", "if (stretch) bcup[count - 1] = (int32_t)capacity;"),
    ("o5_slot_from_real", "int64_t t = run_padded + j;", "int64_t t = run_real + j;"),
    ("o5_cu_from_padded", "run_real += real;\n      run_padded += padded;", "run_real += padded;\n      run_padded += padded;"),
    ("o5_source_row_is_bin", "in[(i * W + j) * elem_bytes + e]", "in[(b * W + j) * elem_bytes + e]"),
    ("o5_no_capacity_check", "if (run_padded + padded > capacity) return ORC_CAPACITY;", ""),
    ("o6_inverted_compare", "mask[t] = (read_int(ids, elem_bytes, t) == pad_id) ? 1 : 0;",
     "mask[t] = (read_int(ids, elem_bytes, t) != pad_id) ? 1 : 0;"),
    ("o6_no_validation", "else if (seen_pad) return ORC_VALUE; /* content after a pad token */", ""),
    ("o7_ascending", "if (sizes[a] > sizes[b] || (sizes[a] == sizes[b] && a < b)) best = j;",
     "if (sizes[a] < sizes[b] || (sizes[a] == sizes[b] && a < b)) best = j;"),
    ("o7_exact_fit_rejected", "while (b < bins && room[b] < sizes[item]) ++b;",
     "while (b < bins && room[b] <= sizes[item]) ++b;"),
    ("o7_ties_by_larger_index", "if (sizes[a] > sizes[b] || (sizes[a] == sizes[b] && a < b)) best = j;",
     "if (sizes[a] > sizes[b] || (sizes[a] == sizes[b] && a > b)) best = j;"),
    ("o8_pad_not_absorbed", "        seq_lens_padded[b * num_packs + slot] += 1;\n      }\n    }",
     "      }\n    }"),
    ("o8_positions_not_reset", "          position_ids[t] = 0;\n        } else {", "          position_ids[t] = s;\n        } else {"),
    ("o8_positions_start_at_one", "          position_ids[t] = 0;\n        } else {", "          position_ids[t] = 1;\n        } else {"),
    ("o8_real_counts_pad", "        seq_lens_padded[b * num_packs + slot] += 1;\n      }\n    }",
     "        seq_lens_padded[b * num_packs + slot] += 1;\n        seq_lens[b * num_packs + slot] += 1;\n      }\n    }"),
    ("o5_real_slots_masked", "        mask[b * width + t] = 0;", "        mask[b * width + t] = 1;"),
    ("o2_offset_ignored", "      seq_off[n] = offset_in_row;", "      seq_off[n] = 0;"),
    ("o8_leading_pad_dropped", "          slot = 0;\n          if (slot >= num_packs) return ORC_CAPACITY;\n          seq_lens[b * num_packs] = 0;\n          seq_lens_padded[b * num_packs] = 0;\n        }\n        seq_lens_padded[b * num_packs + slot] += 1;",
     "          continue;\n        }\n        seq_lens_padded[b * num_packs + slot] += 1;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    with open(oracle.SOURCE) as f:
        text = f.read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / "pseq_oracle.c"
    src.write_text(text.replace(old, new))
    path = oracle.compile_library(str(src), str(tmp_path / "build"), strict=False)
    lib = oracle.load_library(path)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {name}"
