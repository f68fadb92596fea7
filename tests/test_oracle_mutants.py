"""Mutation tests: the pins must catch a plausible mistake anywhere in the oracle.

Each mutant is a copy of ``oracle/pa_oracle.c`` with ONE planted mistake (a dropped term, a
wrong index or sign, a swapped operand, an off-by-one). The copy is compiled into a temporary
directory and the whole pin suite runs against it in a child process; the test passes only if
some pin fails (or the mutant crashes). The committed oracle is never modified. Every
original snippet must occur exactly once in the source, so an edit to the oracle that moves a
snippet shows up here instead of silently weakening the check.
"""
import subprocess
import sys
from pathlib import Path

import pytest

import oracle

ROOT = Path(__file__).resolve().parents[1]

MUTANTS = {
    # the 16-bit formats
    "f16_exponent_bias": ("mag = ldexp((double)(0x400 | f), e - 15 - 10);",
                          "mag = ldexp((double)(0x400 | f), e - 15 - 9);"),
    "f16_subnormal_scale": ("mag = ldexp((double)f, -24);", "mag = ldexp((double)f, -25);"),
    "bf16_exponent_bias": ("mag = ldexp((double)(0x80 | f), e - 127 - 7);",
                           "mag = ldexp((double)(0x80 | f), e - 127 - 8);"),
    "bf16_hidden_bit": ("mag = ldexp((double)(0x80 | f), e - 127 - 7);",
                        "mag = ldexp((double)(f), e - 127 - 7);"),
    # store
    "store_v_from_k": ("memcpy(v_cache + (size_t)s * row, v + (size_t)t * row",
                       "memcpy(v_cache + (size_t)s * row, k + (size_t)t * row"),
    "store_duplicates_accepted": ("if (s >= num_slots || seen[s]) {", "if (s >= num_slots) {"),
    # addressing
    "block_index_mod": ("long long block = src->table[j / src->block_size];",
                        "long long block = src->table[j % src->block_size];"),
    "offset_div": ("long long slot = block * src->block_size + j % src->block_size;",
                   "long long slot = block * src->block_size + j / src->block_size;"),
    "head_stride_dropped": ("return base_pool + ((size_t)slot * src->Hkv + src->g) * src->D;",
                            "return base_pool + ((size_t)slot + src->g) * src->D;"),
    "packed_row_fixed": ("return base_packed + ((size_t)(src->first + j) * src->Hkv + src->g) * src->D;",
                         "return base_packed + ((size_t)(src->first) * src->Hkv + src->g) * src->D;"),
    # GQA map
    "decode_gqa_modulo": ("NULL, NULL, 0, block_size, Hkv, D, h / G};",
                          "NULL, NULL, 0, block_size, Hkv, D, h % Hkv};"),
    "prefill_gqa_modulo": ("k, v, cu_seqlens_k[s], block_size, Hkv, D, h / G};",
                           "k, v, cu_seqlens_k[s], block_size, Hkv, D, h % Hkv};"),
    # softmax / contraction
    "scale_dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "v_from_k_pool": ("const uint16_t *vr = key_row(src, j, src->v_cache, src->v);",
                      "const uint16_t *vr = key_row(src, j, src->k_cache, src->k);"),
    "not_normalised": ("out[d] /= z;", "out[d] /= (double)n;"),
    "score_sign": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "q_as_key": ("dot += to_double(q[d], dtype) * to_double(kr[d], dtype);",
                 "dot += to_double(q[d], dtype) * to_double(q[d], dtype);"),
    # lengths and masks
    "decode_ctx_short": ("context_lens[i], scale, dtype, s);", "context_lens[i] - 1, scale, dtype, s);"),
    "causal_off_by_one": ("int n = causal ? P + r + 1 : kl;", "int n = causal ? P + r : kl;"),
    "causal_top_left": ("int n = causal ? P + r + 1 : kl;", "int n = causal ? r + 1 : kl;"),
    "noncausal_q_len": ("int n = causal ? P + r + 1 : kl;", "int n = causal ? P + r + 1 : ql;"),
    "prefill_row_base": ("long long row = (long long)cu_seqlens_q[s] + r;", "long long row = r;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    src = oracle.SOURCE.read_text()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"snippet for {name} not found exactly once"
    mutant_src = tmp_path / "pa_oracle_mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = oracle.build(mutant_src, tmp_path / "libmutant.so")
    r = subprocess.run([sys.executable, str(ROOT / "tests" / "pins.py"), str(lib)],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout}{r.stderr}"
