"""Plant plausible mistakes in copies of the oracle source (a wrong index, a
dropped term, a flipped sign, a transposed layout, a wrong format constant)
and check that at least one pin fails for every copy. This is what makes the
pins evidence: they are sensitive to each kind of mistake they guard against.
Each copy is compiled and exercised in a subprocess."""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))

# (name, text in pkv_oracle.c, replacement, which occurrence)
MUTATIONS = [
    ("logical block index reversed",
     "block_tables[(size_t)s * max_blocks_per_seq + t / block_size];\n        if (p < 0 || p >= num_blocks) {\n          rc = -7;",
     "block_tables[(size_t)s * max_blocks_per_seq + ((L - 1) / block_size - t / block_size)];\n        if (p < 0 || p >= num_blocks) {\n          rc = -7;", 0),
    ("row within block reversed",
     "row[t] = (((size_t)p * num_kv_heads + g) * block_size + (size_t)(t % block_size)) * head_dim;",
     "row[t] = (((size_t)p * num_kv_heads + g) * block_size + (size_t)(block_size - 1 - t % block_size)) * head_dim;", 0),
    ("block layout transposed (rows before heads)",
     "row[t] = (((size_t)p * num_kv_heads + g) * block_size + (size_t)(t % block_size)) * head_dim;",
     "row[t] = (((size_t)p * block_size + (size_t)(t % block_size)) * num_kv_heads + g) * head_dim;", 0),
    ("kv head = h % group", "const int g = h / group;", "const int g = h % group;", 0),
    ("dense kv head = h % group", "const int g = h / group;", "const int g = h % group;", 1),
    ("softmax scale dropped",
     "x[t] = scale * dot_rows(q, q_off, k_cache, row[t], head_dim, dtype);",
     "x[t] = dot_rows(q, q_off, k_cache, row[t], head_dim, dtype);", 0),
    ("softmax exponent sign", "x[t] = exp(x[t] - m);", "x[t] = exp(m - x[t]);", 0),
    ("normalisation dropped", "out[d] = acc / z;", "out[d] = acc;", 0),
    ("last token dropped", "softmax_combine(o, x, L, V, head_dim);",
     "softmax_combine(o, x, L > 1 ? L - 1 : L, V, head_dim);", 0),
    ("f16 exponent bias", "ldexp((double)(f + 1024), e - 25)", "ldexp((double)(f + 1024), e - 24)", 0),
    ("f16 subnormal scale", "ldexp((double)f, -24)", "ldexp((double)f, -25)", 0),
    ("bf16 hidden bit", "ldexp((double)(f + 128), e - 134)", "ldexp((double)(f + 127), e - 134)", 0),
    ("f32 exponent bias", "ldexp((double)(f + 0x800000u), e - 150)", "ldexp((double)(f + 0x800000u), e - 149)", 0),
    ("cache write ignores row offset",
     "(((size_t)blk * num_kv_heads + h) * block_size + (size_t)off) * row_bytes",
     "(((size_t)blk * num_kv_heads + h) * block_size + (size_t)0) * row_bytes", 0),
    ("cache write swaps K and V", "memcpy((unsigned char*)k_cache + dst, (const unsigned char*)k + src, row_bytes);",
     "memcpy((unsigned char*)k_cache + dst, (const unsigned char*)v + src, row_bytes);", 0),
    ("block copy direction",
     "memmove((unsigned char*)k_cache + (size_t)dst * block_bytes,\n            (const unsigned char*)k_cache + (size_t)src * block_bytes, block_bytes);",
     "memmove((unsigned char*)k_cache + (size_t)src * block_bytes,\n            (const unsigned char*)k_cache + (size_t)dst * block_bytes, block_bytes);", 0),
    ("merge weight sign", "acc += cl[c] * exp(cm[c] - M) * co", "acc += cl[c] * exp(M - cm[c]) * co", 0),
    ("merge drops chunk exp-sum", "acc += cl[c] * exp(cm[c] - M) * co", "acc += exp(cm[c] - M) * co", 0),
    ("e4m3 exponent bias", "ldexp((double)(m + 8), e - 10)", "ldexp((double)(m + 8), e - 9)", 0),
    ("e4m3 ties away from zero", "(int)rint(ldexp(a, 3 - E))", "(int)floor(ldexp(a, 3 - E) + 0.5)", 0),
    ("e4m3 no saturation", "if (a > 448.0) return sign | 0x7e;", "if (a > 480.0) return sign | 0x7f;", 0),
    ("fp8 cache write skips the scale", "(float)elem(k, src, src_dtype) / k_scale", "(float)elem(k, src, src_dtype)", 0),
    ("fp8 attention drops v_scale", "x[t] * (v_scale * orc_decode_e4m3(", "x[t] * (orc_decode_e4m3(", 0),
    ("prefill causal off by one", "const int pos = L - n + i;", "const int pos = L - n + i - 1;", 0),
    ("prefill positions from the start", "const int pos = L - n + i;", "const int pos = i;", 0),
    ("f16 encoder ties away from zero", "(int)rint(ldexp(a, 10 - E))", "(int)floor(ldexp(a, 10 - E) + 0.5)", 0),
    ("f16 encoder subnormal step", "code = (int)rint(ldexp(a, 24));", "code = (int)rint(ldexp(a, 23));", 0),
    ("q4_0 offset 7", "return (double)(q - 8) * orc_decode_f16(sb);", "return (double)(q - 7) * orc_decode_f16(sb);", 0),
    ("q4_0 nibbles swapped", "qs[j] = (uint8_t)(q[j] | (q[j + 16] << 4));",
     "qs[j] = (uint8_t)(q[j + 16] | (q[j] << 4));", 0),
    ("q4_0 scale sign", "const float d = m / -8.0f;", "const float d = m / 8.0f;", 0),
    ("q4_0 rounds down", "const float y = prod + 8.5f;", "const float y = prod + 8.0f;", 0),
    ("q4_0 last maximum on ties", "if (a > amax) {", "if (a >= amax) {", 0),
    ("q4_0 no clamp", "q[j] = y >= 15.0f ? 15 : (y >= 0.0f ? (int)y : 0);",
     "q[j] = y >= 16.0f ? 16 : (y >= 0.0f ? (int)y : 0) & 15;", 0),
    ("q4_0 scales after the codes", "const uint8_t byte = row[head_dim / 16 + 16 * b + (j % 16)];",
     "const uint8_t byte = row[16 * b + (j % 16)];", 0),
    ("q4_0 cache write swaps K and V",
     "orc_q4_0_quantize_row((const unsigned char*)k + src, src_dtype, head_dim, k_cache + dst);",
     "orc_q4_0_quantize_row((const unsigned char*)v + src, src_dtype, head_dim, k_cache + dst);", 0),
    ("q4_0 attention reads K for V", "acc += x[t] * orc_q4_0_value(v_cache + row[t], head_dim, d);",
     "acc += x[t] * orc_q4_0_value(k_cache + row[t], head_dim, d);", 0),
]


def _mutate(src: str, old: str, new: str, which: int) -> str:
    pos = -1
    for _ in range(which + 1):
        pos = src.find(old, pos + 1)
        assert pos >= 0, f"mutation target not found (occurrence {which}): {old[:60]!r}"
    return src[:pos] + new + src[pos + len(old):]


@pytest.mark.parametrize("name,old,new,which", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new, which):
    src = open(oracle.SOURCE).read()
    mutated = tmp_path / "mutant.c"
    mutated.write_text(_mutate(src, old, new, which))
    so = oracle.build(force=True, src=str(mutated), out=str(tmp_path / "libmutant.so"))
    r = subprocess.run([sys.executable, os.path.join(HERE, "_mutant_runner.py"), so],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 1 and "FAILED pin_" in r.stdout, \
        f"no pin caught '{name}' (rc={r.returncode})\n{r.stdout}\n{r.stderr[-2000:]}"
