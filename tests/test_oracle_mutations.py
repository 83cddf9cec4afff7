"""The oracle pins must fail when a plausible mistake is planted in the oracle.

Each case rebuilds a copy of the oracle's C source with one edit (a dropped
term, a wrong index, a swapped operand, a wrong sign ...) into a temporary
directory, points the oracle module at that copy, and runs the pin suite in
a subprocess: it must report a failure.  Everything runs on the CPU.
"""
import os
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
SRC = (ROOT / "oracle" / "pkv_oracle.c").read_text()

MUTATIONS = {
    "gqa_modulo": ("const int32_t kv = h / group;", "const int32_t kv = h % P->num_kv_heads;"),
    "block_offset_swapped": ("const int32_t logical_block = t / P->block_size;",
                             "const int32_t logical_block = t % P->block_size;"),
    "scale_dropped": ("scores[t] = P->scale * dot;", "scores[t] = dot;"),
    "softmax_sign": ("scores[t] = exp(scores[t] - m);", "scores[t] = exp(m - scores[t]);"),
    "last_token_dropped": ("for (int32_t t = 0; t < L; ++t) {\n        const int32_t logical_block",
                           "for (int32_t t = 0; t < L - 1; ++t) {\n        const int32_t logical_block"),
    "value_is_key": ("vrows[t] = P->v_cache + row;", "vrows[t] = P->k_cache + row;"),
    "normalisation_dropped": ("const double p = scores[t] / denom;", "const double p = scores[t];"),
    "append_head_stride": (
        "const int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * (int64_t)head_dim;",
        "const int64_t dst = ((block * block_size + offset) * num_kv_heads + h) * (int64_t)head_dim;"),
    "append_value_from_k": ("v_cache[dst + d] = v[src + d];", "v_cache[dst + d] = k[src + d];"),
    "rope_sign": ("const float r1 = a - b;", "const float r1 = a + b;"),
    "rope_cos_sin_swapped": ("const float c = cs[i], s = cs[half + i];", "const float c = cs[half + i], s = cs[i];"),
    "bf16_truncates": ("u += 0x7fffu + lsb;", "u += 0u;"),
    "prefill_causal_off_by_one": ("prefix + i + 1, out_row);", "prefix + i, out_row);"),
    "table_row_stride": ("P->block_tables[(int64_t)b * P->max_blocks_per_seq + logical_block]",
                         "P->block_tables[(int64_t)b * P->block_size + logical_block]"),
    "copy_k_only": ("            v_cache[dst * per_block + e] = v_cache[src * per_block + e];\n", ""),
    "copy_block_stride_without_heads": ("const int64_t per_block = (int64_t)num_kv_heads * block_size * head_dim;",
                                        "const int64_t per_block = (int64_t)block_size * head_dim;"),
    "copy_pairs_reversed": ("const int64_t src = src_dst[2 * i], dst = src_dst[2 * i + 1];",
                            "const int64_t src = src_dst[2 * (num_pairs - 1 - i)], "
                            "dst = src_dst[2 * (num_pairs - 1 - i) + 1];"),
    "copy_src_dst_swapped": ("const int64_t src = src_dst[2 * i], dst = src_dst[2 * i + 1];",
                             "const int64_t dst = src_dst[2 * i], src = src_dst[2 * i + 1];"),
}


def _run_pins_against(source: str, tmp_path) -> subprocess.CompletedProcess:
    src = tmp_path / "pkv_oracle.c"
    src.write_text(source)
    lib = tmp_path / "libpkv_oracle.so"
    subprocess.run(["gcc", "-std=c11", "-O1", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", str(src),
                    "-o", str(lib), "-lm"], check=True)
    # Run the pin suite against the mutated library in a fresh interpreter.
    runner = (
        "import sys, ctypes, oracle, pytest\n"
        f"oracle._LIB_PATH = oracle.Path({str(lib)!r})\n"
        "oracle.build = lambda force=False: oracle._LIB_PATH\n"
        f"sys.exit(pytest.main(['-q', '-x', '-p', 'no:cacheprovider', {str(ROOT / 'tests' / 'test_oracle_pins.py')!r}]))\n"
    )
    env = dict(os.environ, PYTHONPATH=str(ROOT))
    return subprocess.run([sys.executable, "-c", runner], cwd=str(ROOT), env=env, capture_output=True, text=True,
                          timeout=600)


def test_unmutated_copy_passes(tmp_path):
    """Control: the same harness on an unedited copy passes, so a failure below is the edit's."""
    r = _run_pins_against(SRC, tmp_path)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    assert SRC.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    r = _run_pins_against(SRC.replace(old, new), tmp_path)
    assert r.returncode != 0, f"pins did not catch mutation {name}:\n{r.stdout[-2000:]}"
