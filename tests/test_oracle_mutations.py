"""The oracle pins catch planted mistakes (CPU only).

Each case copies ``oracle/lora_oracle.c``, plants one plausible mistake (a
dropped term, a transposed operand, a wrong index or offset, a missing scale, a
wrong tie rule, an unstable sort, an overwrite that still adds or drops the scale, non-zero padding, swapped MoE slices, a wrong
adapter stride, a per-token input row for the down projection, a dropped routing
weight, a non-local expert treated as local, a disabled adapter applied, a reversed rank gather, a dropped rank
partial), compiles the copy into a temporary library and runs the pin
suite against it in a subprocess.  The pins must fail for every mutant.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "lora_oracle.c")

MUTANTS = {
    "dropped_k_term": (
        "                        for (int k = 0; k < k_in; ++k)\n"
        "                            acc += oracle_bf16_to_f32(xrow[k]) * oracle_bf16_to_f32(arow[k]);\n"
        "                        hf[q] = acc;",
        "                        for (int k = 0; k < k_in - 1; ++k)\n"
        "                            acc += oracle_bf16_to_f32(xrow[k]) * oracle_bf16_to_f32(arow[k]);\n"
        "                        hf[q] = acc;"),
    "transposed_b": (
        "                            d += hf[q] * oracle_bf16_to_f32(brow[q]);",
        "                            d += hf[q] * oracle_bf16_to_f32(B[(size_t)q * widths[j] + c]);"),
    "wrong_slice_offset": (
        "                    }\n                }\n            }\n            off += widths[j];",
        "                    }\n                }\n            }\n            off += widths[0];"),
    "missing_scale": ("                        float v = scale * d;", "                        float v = d;"),
    "expand_overwrite_adds": (
        "                    uint16_t *o = out + (size_t)i * ld_out + off + c;\n"
        "                    *o = oracle_f32_to_bf16(add_inputs ? oracle_bf16_to_f32(*o) + v : v);",
        "                    uint16_t *o = out + (size_t)i * ld_out + off + c;\n"
        "                    *o = oracle_f32_to_bf16(oracle_bf16_to_f32(*o) + v);"),
    "expand_overwrite_unscaled": (
        "                    uint16_t *o = out + (size_t)i * ld_out + off + c;\n"
        "                    *o = oracle_f32_to_bf16(add_inputs ? oracle_bf16_to_f32(*o) + v : v);",
        "                    uint16_t *o = out + (size_t)i * ld_out + off + c;\n"
        "                    *o = oracle_f32_to_bf16(add_inputs ? oracle_bf16_to_f32(*o) + v : d);"),
    "ties_away_from_zero": ("(lower == 0x8000u && (upper & 1u))", "(lower == 0x8000u)"),
    "unstable_segments": (
        "        for (int i = 0; i < n; ++i)\n            if (seq_slot[i] == s)",
        "        for (int i = n - 1; i >= 0; --i)\n            if (seq_slot[i] == s)"),
    "nonzero_padding": (
        "a_slot[(size_t)q * k_in + k] = (q < r) ? a_r[(size_t)q * k_in + k] : 0;",
        "a_slot[(size_t)q * k_in + k] = (q < r) ? a_r[(size_t)q * k_in + k] : 0x3f80;"),
    "moe_gate_up_swapped": (
        "            const uint16_t *A = w_ptr_a[(size_t)j * E + e] + (size_t)l * stride_a;",
        "            const uint16_t *A = w_ptr_a[(size_t)(n_slices - 1 - j) * E + e] + (size_t)l * stride_a;"),
    "moe_wrong_adapter_stride": (
        "            const uint16_t *B = w_ptr_b[(size_t)j * E + e] + (size_t)l * stride_b;",
        "            const uint16_t *B = w_ptr_b[(size_t)j * E + e] + (size_t)l * (stride_b / 2);"),
    "moe_w2_x_per_token": (
        "        moe_pair_fold(y + (size_t)p * H, x + (size_t)p * I, I,",
        "        moe_pair_fold(y + (size_t)p * H, x + (size_t)(p / top_k) * I, I,"),
    "moe_w2_weight_dropped": (
        "            if (has_w)\n                v = w * v;",
        "            if (has_w)\n                v = 1.0f * v;"),
    "moe_nonlocal_expert_as_zero": (
        "        else if (expert_map[e] < 0)\n            return 0;",
        "        else if (expert_map[e] < 0)\n            e = 0;"),
    "gather_rank_blocks_reversed": (
        "                    h[((size_t)j * n + i) * R + (size_t)p * Rs + q] =",
        "                    h[((size_t)j * n + i) * R + (size_t)(tp - 1 - p) * Rs + q] ="),
    "rank_sum_drops_last_rank": (
        "        for (int p = 1; p < tp; ++p)\n            s = s + parts[(size_t)p * len + e];",
        "        for (int p = 1; p < tp - 1; ++p)\n            s = s + parts[(size_t)p * len + e];"),
    "moe_disabled_adapter_applied": (
        "adapter_enabled && adapter_enabled[l] == 0)",
        "adapter_enabled && adapter_enabled[l] == 2)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_fail_on_mutant(name, tmp_path):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC",
                    "-shared", "-o", str(so), str(mutant), "-lm"], check=True)
    env = dict(os.environ, LORA_ORACLE_LIBRARY=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
