"""Plant plausible mistakes in copies of the CPU oracle and check that the
pins catch every one of them (no GPU).

Each mutant is a one-line textual change of oracle/pagedkv_oracle.c,
compiled into a temporary library and run against every pin in a child
process (a mutant that crashes counts as caught).  The real oracle must pass
every pin (test_oracle_pins.py); each mutant must fail at least one.
"""
import subprocess
import sys
import textwrap
from pathlib import Path

import pytest

import oracle

ROOT = Path(__file__).resolve().parent.parent

# (name, original text, mutated text)
MUTANTS = [
    ("drop_softmax_scale", "p[t] = a->scale * s;", "p[t] = s;"),
    ("gqa_head_modulo", "const int kvh = h / group;",
     "const int kvh = h % a->num_kv_heads;"),
    ("no_max_subtraction", "p[t] = exp(p[t] - mx);", "p[t] = exp(p[t]);"),
    ("no_normalisation", "double w = p[t] / denom;", "double w = p[t];"),
    ("one_token_too_many", "bb, hh, seq_lens[bb],",
     "bb, hh, seq_lens[bb] > 0 ? seq_lens[bb] + 1 : 0,"),
    ("value_read_from_key_cache",
     "V[(size_t)t * d + i] = decode_elem(a->value_cache,",
     "V[(size_t)t * d + i] = decode_elem(a->key_cache,"),
    ("block_offset_ignored",
     "(((size_t)blk * bs + (size_t)(t - j * bs)) * a->num_kv_heads +",
     "(((size_t)blk * bs + (size_t)0) * a->num_kv_heads +"),
    ("logical_block_as_physical",
     "int32_t blk = a->block_tables[(size_t)b * a->max_blocks + j];",
     "int32_t blk = j;"),
    ("query_from_wrong_head",
     "errors += attend_row(&a, q + ((size_t)bb * num_heads + hh) * head_dim,",
     "errors += attend_row(&a, q + ((size_t)bb * num_heads + hh / (num_heads / num_kv_heads)) * head_dim,"),
    ("prefill_not_causal", "bb, hh, c + i + 1, orow", "bb, hh, seq_lens[bb], orow"),
    ("prefill_causal_off_by_one", "bb, hh, c + i + 1, orow", "bb, hh, c + i, orow"),
    ("prefill_history_ignored", "c = seq_lens[bb] - nq; /* tokens before this chunk */",
     "c = 0;"),
    ("prefill_query_row_of_sequence",
     "errors += attend_row(&a, q + ((size_t)t * num_heads + hh) * head_dim,",
     "errors += attend_row(&a, q + ((size_t)query_start_loc[bb] * num_heads + hh) * head_dim,"),
    ("fp8_scale_not_applied",
     "return oracle_e4m3_to_double(cache[idx]) * scale;",
     "return oracle_e4m3_to_double(cache[idx]);"),
    ("e4m3_bias_8", "mag = ldexp(1.0 + (double)m / 8.0, e - 7);",
     "mag = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("e4m3_subnormal_exponent", "mag = ldexp((double)m / 8.0, -6);",
     "mag = ldexp((double)m / 8.0, -7);"),
    ("e4m3_ties_up", "code = (lo % 2 == 0) ? lo : lo + 1;", "code = lo + 1;"),
    ("e4m3_truncate", "else if (a > half)", "else if (a > vhi)"),
    ("e4m3_overflow_to_nan", "return (uint8_t)(sign | 0x7E);",
     "return (uint8_t)(sign | 0x7F);"),
    ("quantise_multiplies", "q = xf / scale;", "q = xf * scale;"),
    ("bf16_wrong_shift", "uint32_t w = ((uint32_t)bits) << 16;",
     "uint32_t w = ((uint32_t)bits) << 15;"),
    ("write_skips_value",
     "memcpy(value_cache + (base + e) * eb, &vb, 2);", "(void)vb;"),
    ("write_swaps_block_offset", "off = s % block_size;",
     "off = (s + 1) % block_size;"),
    ("zero_skips_value_cache",
     "memset(value_cache + (size_t)id * block_bytes, 0, block_bytes);",
     "(void)value_cache;"),
    ("zero_accepts_negative", "if (id < 0 || id >= num_blocks) {",
     "if (id >= num_blocks) {"),
    ("empty_sequence_not_zero", "out_row[i] = 0.0;", "out_row[i] = 1.0;"),
    ("copy_value_from_key",
     "                value_cache + (size_t)src[i] * block_bytes, block_bytes);",
     "                key_cache + (size_t)src[i] * block_bytes, block_bytes);"),
    ("swap_out_wrong_slot", "memcpy(out_k + (size_t)i * block_bytes,",
     "memcpy(out_k + (size_t)(n - 1 - i) * block_bytes,"),
    ("swap_in_skips_value",
     "        memcpy(value_cache + (size_t)ids[i] * block_bytes,\n               in_v + (size_t)i * block_bytes, block_bytes);",
     "        (void)in_v;"),
    ("prepare_positions_from_zero", "                int pos = c + i;",
     "                int pos = i;"),
    ("prepare_table_of_batch_index",
     "                    (int64_t)state_block_table[(size_t)r * max_blocks + pos / 16] *",
     "                    (int64_t)state_block_table[(size_t)b * max_blocks + pos / 16] *"),
    ("prepare_seq_len_without_new", "            seq_lens[b] = c + n;",
     "            seq_lens[b] = c;"),
    ("prepare_start_loc_inclusive", "        query_start_loc[b] = (int32_t)t0;",
     "        query_start_loc[b] = (int32_t)(t0 + n);"),
    ("prepare_negative_count_kept",
     "            ++errors;\n            n = 0;\n",
     "            ++errors;\n"),
    ("prepare_negative_count_not_reported",
     "            ++errors;\n            n = 0;\n",
     "            n = 0;\n"),
    ("prepare_overflow_offset_not_advanced",
     "            ++errors;\n            t0 += n;\n            continue;",
     "            ++errors;\n            continue;"),
    ("prepare_overflow_not_reported",
     "            ++errors;\n            t0 += n;\n            continue;",
     "            t0 += n;\n            continue;"),
]

_RUNNER = textwrap.dedent("""
    import sys
    sys.path[:0] = [{root!r}, {tests!r}]
    import oracle, oracle_pins
    o = oracle.Oracle({lib!r})
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except Exception as e:
            failed.append(pin.__name__)
    print("FAILED", len(failed), ",".join(failed))
""")


def test_mutants_are_distinct_edits():
    src = oracle.SOURCE.read_text()
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, f"{name}: anchor not unique/present"
        assert old != new


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = oracle.SOURCE.read_text()
    assert src.count(old) == 1
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.compile_library(mutated, tmp_path / "libmutant.so")
    code = _RUNNER.format(root=str(ROOT), tests=str(ROOT / "tests"),
                          lib=str(lib))
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True,
                          text=True, timeout=300)
    if proc.returncode != 0:
        return  # the mutant crashed the pins: caught
    line = [l for l in proc.stdout.splitlines() if l.startswith("FAILED")][-1]
    n_failed = int(line.split()[1])
    assert n_failed > 0, f"mutant {name} passed every pin"
