"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each.

Every mutant is compiled from a patched copy of ``oracle/pa_oracle.c`` into a
temporary directory and the whole pin suite (test_oracle_pins.py) is run against
it in a child process; the suite must fail.  The oracle itself is never changed.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pa_oracle.c")

MUTANTS = {
    "k-layout-group-and-lane-swapped": ("* (D / x) + d / x) * bs + t) * x + d % x",
                                        "* (D / x) + d % x) * bs + t) * x + d / x"),
    "v-layout-transposed": ("(((int64_t)b * Hkv + h) * D + d) * bs + t",
                            "(((int64_t)b * Hkv + h) * bs + t) * D + d"),
    "fp16-exponent-bias": ("e - 25", "e - 24"),
    "fp16-subnormal-scale": ("ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    "bf16-shift": ("(uint32_t)b << 16", "(uint32_t)b << 15"),
    "scale-dropped": ("z[t] = scale * acc;", "z[t] = acc;"),
    "softmax-sign": ("z[t] = exp(z[t] - m);", "z[t] = exp(m - z[t]);"),
    "softmax-not-normalised": ("z[t] /= Z;", "z[t] /= 1.0;"),
    "gqa-mapping-modulo": ("const int kvh = h / G;", "const int kvh = h % num_kv_heads;"),
    "table-index-offset": ("table_row[t / bs]", "table_row[t % bs]"),
    "in-block-offset-shifted": ("const int off = t % bs;", "const int off = (t + 1) % bs;"),
    "length-off-by-one": ("const int L = seq_lens[s];", "const int L = seq_lens[s] - (seq_lens[s] > 1);"),
    "value-uses-keys": ("acc += z[t] * V[(int64_t)t * D + d];", "acc += z[t] * K[(int64_t)t * D + d];"),
    "query-not-indexed": ("load(q, qo + d, q_dtype)", "load(q, qo, q_dtype)"),
    "slot-block-from-modulo": ("const int64_t blk = slot / block_size;",
                               "const int64_t blk = slot % block_size;"),
    "slot-offset-from-division": ("const int off = (int)(slot % block_size);",
                                  "const int off = (int)(slot / block_size % block_size);"),
    "copy-direction-swapped": ("memmove((char*)k_cache + (size_t)dst * blk_bytes, (const char*)k_cache + (size_t)src * blk_bytes",
                               "memmove((char*)k_cache + (size_t)src * blk_bytes, (const char*)k_cache + (size_t)dst * blk_bytes"),
    # a padding token written instead of skipped (into slot 0, so that the mutant stays in bounds)
    "padding-slot-written": ("if (slot < 0) continue;\n    const int64_t blk = slot / block_size;\n    const int off = (int)(slot % block_size);",
                             "const int64_t blk = slot < 0 ? 0 : slot / block_size;\n    const int off = slot < 0 ? 0 : (int)(slot % block_size);"),
    "e4m3-exponent-bias": ("ldexp((double)(f | 8), e - 10)", "ldexp((double)(f | 8), e - 9)"),
    "e4m3-subnormal-scale": ("v = ldexp((double)f, -9);", "v = ldexp((double)f, -10);"),
    "e4m3-ties-to-odd": ("(d == best_d && (c & 1) == 0)", "(d == best_d && (c & 1) == 1)"),
    "e4m3-no-clamp": ("for (int c = 0; c <= 126; ++c)", "for (int c = 0; c <= 125; ++c)"),
    "k-scale-dropped": ("k_scale * load(k_cache", "load(k_cache"),
    "v-scale-dropped": ("v_scale * load(v_cache", "load(v_cache"),
    "quantise-multiplies": ("(float)load(value, src, key_dtype) / vs", "(float)load(value, src, key_dtype) * vs"),
    "prefill-position-off-by-one": ("const int p = L - n + i;", "const int p = L - n + i - 1 + (i == 0);"),
    "prefill-ignores-history": ("const int p = L - n + i;", "const int p = i;"),
    "prefill-wrong-query-row": ("(int64_t)(query_start_loc[s] + i) * num_heads", "(int64_t)(s + i) * num_heads"),
    "prefill-not-normalised": ("out[qo + d] = acc / Z;", "out[qo + d] = acc;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation anchor missing for {name}"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(text.replace(old, new))
    lib = tmp_path / "libmutant.so"
    r = subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", str(mutant_c), "-o", str(lib), "-lm"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, PA_ORACLE_LIB=str(lib), OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)
    # a pin must fail: exit code 1 (a collection error, exit 2, or a crash would catch nothing)
    caught = r.returncode == 1
    assert caught, f"mutant {name} survived the pins (exit {r.returncode}):\n{r.stdout[-2000:]}"
