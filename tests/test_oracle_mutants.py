"""Plant plausible mistakes in copies of the oracle's C source and show that
the pins catch every one (CPU only; the real oracle is never modified)."""
import os
import subprocess

import pytest

import oracle
from oracle_pins import ALL_CHECKS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement, replace-count)
MUTANTS = [
    ("causal_top_left", "int64_t lim = off + i + 1;", "int64_t lim = i + 1;", 1),
    ("causal_off_by_one", "int64_t lim = off + i + 1;", "int64_t lim = off + i;", 1),
    ("no_causal_mask", "if (causal) {", "if (0) {", 1),
    ("gqa_modulo_heads", "int32_t kvh = h / g;", "int32_t kvh = h % Hkv;", 1),
    ("scale_dropped", "s_row[j] = scale * acc;", "s_row[j] = acc;", 1),
    ("page_offset_swapped", "int64_t row = page * P + j % P;", "int64_t row = page * P + j / P;", 1),
    ("page_index_transposed", "page_table[b * pt_stride + j / P]", "page_table[b * pt_stride + j % P]", 1),
    ("no_normalisation", "for (int c = 0; c < d; ++c) o[c] /= l;", "", 1),
    ("lse_missing_max", "*lse = m + log(l);", "*lse = log(l);", 1),
    ("values_from_k_cache", "o[c] += p * kv_value(kv->v,", "o[c] += p * kv_value(kv->k,", 1),
    ("exp_sign_flipped", "double p = exp(s_row[j] - m);", "double p = exp(m - s_row[j]);", 1),
    ("last_key_dropped", "for (int64_t j = j_lo; j < n_vis; ++j) {\n        double p", "for (int64_t j = j_lo; j + 1 < n_vis; ++j) {\n        double p", 1),
    ("cu_k_prefix_wrong", "cu_k[b + 1] = (int32_t)sk;", "cu_k[b + 1] = (int32_t)sq;", 1),
    ("page_table_no_divide", "int64_t q = slot / page_size;", "int64_t q = slot;", 1),
    ("store_swaps_k_v", "memcpy(k_cache + slot * row_elems, k + t * row_elems", "memcpy(k_cache + slot * row_elems, v + t * row_elems", 1),
    ("e4m3_bias_8", "else mag = ldexp(1.0 + (double)m / 8.0, e - 7);", "else mag = ldexp(1.0 + (double)m / 8.0, e - 8);", 1),
    ("e4m3_subnormal_scale", "if (e == 0) mag = ldexp((double)m / 8.0, -6);", "if (e == 0) mag = ldexp((double)m / 8.0, -7);", 1),
    ("e4m3_ties_up", "else c = (lo & 1) ? hi : lo;", "else c = hi;", 1),
    ("e4m3_truncates", "if (dlo < dhi) c = lo;", "if (1) c = lo;", 1),
    ("fp8_scale_head_0", "* (double)scale[kvh];", "* (double)scale[0];", 1),
    ("fp8_store_multiplies", "widen_bf16_f32(k[src]) / k_scale[h]", "widen_bf16_f32(k[src]) * k_scale[h]", 1),
    ("fp8_k_read_with_v_scale", "kv_value(kv->k, kv->fp8, kv->k_scale,", "kv_value(kv->k, kv->fp8, kv->v_scale,", 1),
    ("rope_sign", "o[ia] = a * cs - b * sn;", "o[ia] = a * cs + b * sn;", 1),
    ("rope_pairs_adjacent", "int32_t ib = interleaved ? 2 * i + 1 : i + h;", "int32_t ib = interleaved ? 2 * i + 1 : i + 1;", 1),
    ("rope_frequency_halved", "pow(base, -2.0 * (double)i / (double)r)", "pow(base, -1.0 * (double)i / (double)r)", 1),
    ("rope_cos_sin_swapped", "cos_t[(int64_t)p * h + i] = cos(ang);", "cos_t[(int64_t)p * h + i] = sin(ang);", 1),
    ("bf16_ties_away", "double rr = nearbyint(scaled);", "double rr = round(scaled);", 1),
    ("window_off_by_one", "j_lo = off + i - window_left;", "j_lo = off + i - window_left + 1;", 1),
    ("window_from_query_index", "j_lo = off + i - window_left;", "j_lo = i - window_left;", 1),
    ("window_ignored", "if (window_left >= 0) {\n        j_lo", "if (0) {\n        j_lo", 1),
    ("block_mask_ignored", "if (mrow && mrow[j / ORACLE_MASK_BLOCK] == 0) { s_row[j] = -INFINITY; continue; }", "", 1),
    ("block_mask_key_blocks_of_64", "mrow[j / ORACLE_MASK_BLOCK] == 0", "mrow[j / 64] == 0", 1),
    ("block_mask_query_by_position", "+ i / ORACLE_MASK_BLOCK) * (int64_t)bm->nk;", "+ (off + i) / ORACLE_MASK_BLOCK) * (int64_t)bm->nk;", 1),
    ("block_mask_empty_row_nan", "if (m == -INFINITY) { *lse = -INFINITY; return ORACLE_OK; }   /* every key hidden */", "", 1),
]


def _build_mutant(tmp_path, name, old, new, count):
    src = open(SRC).read()
    assert src.count(old) >= count, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, count)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", str(c), "-o", str(so), "-lm"],
                   check=True)
    return oracle.load_variant(str(so))


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m[0])
def test_pins_catch_mutant(tmp_path, mutant):
    name, old, new, count = mutant
    lib = _build_mutant(tmp_path, name, old, new, count)
    caught = []
    for check in ALL_CHECKS:
        try:
            check(lib=lib)
        except (AssertionError, oracle.OracleError):
            caught.append(check.__name__)
    assert caught, f"no pin caught the planted mistake '{name}'"
