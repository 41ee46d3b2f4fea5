"""Plants plausible mistakes in copies of the oracle's C source (on the CPU)
and checks that the pin tests catch every one of them.  Each mutant is compiled
separately and the pin suite runs against it in a child process."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PIN_TESTS = [os.path.join(ROOT, "tests", f) for f in
             ("test_oracle_quant.py", "test_oracle_logits.py", "test_oracle_next.py")]

# (name, original text, mutated text): each must occur exactly once.
MUTATIONS = [
    ("scale_boundary", "if (amax <= ldexp(6.0, e))", "if (amax < ldexp(6.0, e))"),
    ("scale_off_by_one", "return (uint8_t)(e + 127);", "return (uint8_t)(e + 128);"),
    ("tie_not_even", "(dist == best_dist && (c % 2 == 0) && (best % 2 != 0))", "0"),
    ("saturate_wrong", "if (a > 6.0) return (uint8_t)(sign | 7);", "if (a > 6.0) return (uint8_t)(sign | 6);"),
    ("zero_sign_dropped", "uint8_t sign = signbit(y) ? 0x8 : 0x0;", "uint8_t sign = (y < 0) ? 0x8 : 0x0;"),
    ("nibbles_swapped", "vals[i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));",
     "vals[i] = (uint8_t)((codes[2 * i] << 4) | codes[2 * i + 1]);"),
    ("dequant_nibble", "uint8_t code = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);",
     "uint8_t code = (d % 2 == 0) ? (byte >> 4) : (byte & 0xF);"),
    ("dequant_block_index", "int e = (int)scales[d / BLOCK] - 127;", "int e = (int)scales[d % 4] - 127;"),
    ("scale_area_offset", "uint8_t* sdst = cache + page * page_bytes + (int64_t)page_size * VAL_BYTES + off * SCALE_BYTES;",
     "uint8_t* sdst = cache + page * page_bytes + (int64_t)page_size * VAL_BYTES + (page_size - 1 - off) * SCALE_BYTES;"),
    ("relu_dropped", "double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    ("relu_sign", "double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot < 0.0 ? -dot : 0.0;"),
    ("weight_index", "acc += (double)w[h] * relu;", "acc += (double)w[0] * relu;"),
    ("mag_abs_w", "m += fabs((double)w[h]) * adot;", "m += (double)w[h] * adot;"),
    ("mag_abs_dot", "adot += fabs(p);", "adot += p;"),
    ("decode_window", "int64_t len = (int64_t)context_lens[b] - next_n + j + 1;",
     "int64_t len = (int64_t)context_lens[b] - next_n + j;"),
    ("page_index", "int64_t page = block_table[b * max_blocks + s / page_size];",
     "int64_t page = block_table[b * max_blocks + s % page_size];"),
    ("topk_tie_order", "return (x->i < y->i) ? -1 : (x->i > y->i);", "return (x->i > y->i) ? -1 : (x->i < y->i);"),
    ("topk_not_relative", "tmp[i].i = i; }", "tmp[i].i = i + st; }"),
    ("q_head_stride", "oracle_dequant_vec128(q_vals + (t * H + h) * VAL_BYTES, q_scales + (t * H + h) * SCALE_BYTES,",
     "oracle_dequant_vec128(q_vals + (t + h) * VAL_BYTES, q_scales + (t + h) * SCALE_BYTES,"),
    ("rope_sign", "x[2 * i] = fmaf(a, c, -bs);", "x[2 * i] = fmaf(a, c, bs);"),
    ("rope_sin_for_cos", "x[2 * i + 1] = fmaf(a, s, bc);", "x[2 * i + 1] = fmaf(a, c, bc);"),
    ("rope_half_split_pairs", "const float a = x[2 * i], b = x[2 * i + 1],",
     "const float a = x[i], b = x[i + half],"),
    ("rope_token_not_position", "const float* c_row = cs + (int64_t)pos[t] * half;",
     "const float* c_row = cs + (int64_t)t * half;"),
    ("kpool_mask_late", "const int write = (n >= P) && slots[p] >= 0 && p >= P - 1;",
     "const int write = (n >= P) && slots[p] >= 0 && p >= P;"),
    ("kpool_window_shift", "const int64_t r0 = p - P + 1; /* the pool's first row */",
     "const int64_t r0 = p - P + 2; /* the pool's first row */"),
    ("kpool_ape_reversed", "+ (double)ape[(int64_t)j * D_HEAD + d];",
     "+ (double)ape[(int64_t)(P - 1 - j) * D_HEAD + d];"),
    ("kpool_mag_abs", "am += e * fabs(kv);", "am += e * kv;"),
    ("quant_f32_nibbles", "vals[i] = (uint8_t)((codes[2 * i + 1] << 4) | codes[2 * i]); /* element 2i low */",
     "vals[i] = (uint8_t)((codes[2 * i] << 4) | codes[2 * i + 1]);"),
    ("kpool_insert_from_zero", "for (int64_t p = P - 1; p < n; ++p) {", "for (int64_t p = 0; p < n; ++p) {"),
    ("quant_f32_scale_block", "uint8_t s = oracle_ue8m0_scale(x + b * BLOCK, BLOCK);\n    scales[b] = s;\n    for (int i = 0; i < BLOCK; ++i)\n      codes[b * BLOCK + i] = oracle_e2m1_code(ldexp(x[b * BLOCK + i], 127 - (int)s));",
     "uint8_t s = oracle_ue8m0_scale(x, BLOCK);\n    scales[b] = s;\n    for (int i = 0; i < BLOCK; ++i)\n      codes[b * BLOCK + i] = oracle_e2m1_code(ldexp(x[b * BLOCK + i], 127 - (int)s));"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutation(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = src.replace(old, new)
    c_path = tmp_path / "oracle_mut.c"
    so_path = tmp_path / "liboracle_mut.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(so_path),
                    str(c_path), "-lm"], check=True)
    env = dict(os.environ, IDX_ORACLE_LIB_OVERRIDE=str(so_path), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *PIN_TESTS], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"mutation {name} survived the pins:\n{r.stdout[-2000:]}"
