"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of oracle/pagedkv_oracle.c (a wrong index, a
dropped term, a transposed operand, a flipped sign), builds the copy separately, and
runs the pin suites (decode and prefill) against it in a child process: they must fail.  The oracle
itself is never modified.
"""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "pagedkv_oracle.c")

MUTATIONS = {
    "gqa_head_modulo": ("const int32_t g = h / G;", "const int32_t g = h % p->num_kv_heads;"),
    "scale_dropped": ("scores[j - t0] = scale * dot;", "scores[j - t0] = dot;"),
    "head_row_transposed": ("return (((size_t)b * p->num_kv_heads + g) * p->block_size + r) * p->head_dim;",
                            "return (((size_t)b * p->block_size + r) * p->num_kv_heads + g) * p->head_dim;"),
    "row_reversed": ("size_t row = orc_row(p, b, g, j % p->block_size);",
                     "size_t row = orc_row(p, b, g, p->block_size - 1 - j % p->block_size);"),
    "exp_sign": ("double w = exp(scores[j - t0] - m);", "double w = exp(m - scores[j - t0]);"),
    "normalisation_dropped": ("for (int32_t d = 0; d < head_dim; ++d) o[d] /= l;", "(void)l;"),
    "last_token_dropped": ("num_q_heads, s, h, 0, context_lens[s], scale,",
                           "num_q_heads, s, h, 0, context_lens[s] - (context_lens[s] > 1), scale,"),
    "causal_diagonal_dropped": ("max_blocks_per_seq, num_q_heads, s, h, 0, pos + 1, scale,",
                                "max_blocks_per_seq, num_q_heads, s, h, 0, pos + (pos == 0), scale,"),
    "prefill_position_from_start": ("const int32_t pos = context_lens[s] - n + (t - query_start[s]);",
                                    "const int32_t pos = t - query_start[s];"),
    "merge_weight_sign": ("double c = exp(m[pi] - M);", "double c = exp(M - m[pi]);"),
    "append_row_zero": ("int32_t r = (int32_t)(slot % block_size);", "int32_t r = 0;"),
    "copy_k_only": ("memcpy((char*)v_cache + dst * block_bytes, (const char*)v_cache + src * block_bytes, block_bytes);", ""),
    "half_exponent_bias": ("v = ldexp((double)(f | 0x400), e - 25);", "v = ldexp((double)(f | 0x400), e - 24);"),
    "bf16_low_half": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    before, after = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(before) >= 1, f"mutation anchor not found: {before}"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(before, after, 1))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", str(mutant_src), "-o",
                    str(lib), "-lm"], check=True, capture_output=True)
    env = dict(os.environ, PKV_ORACLE_LIB=str(lib))
    pins = [os.path.join(HERE, f) for f in ("test_oracle_pins.py", "test_oracle_prefill_pins.py")]
    r = subprocess.run([sys.executable, "-m", "pytest", *pins, "-x", "-q", "-p", "no:cacheprovider"], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"the pins did not notice the '{name}' mutation:\n{r.stdout[-2000:]}"
