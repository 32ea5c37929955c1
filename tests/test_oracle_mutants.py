"""Planted mistakes in the oracle must trip at least one pin.

Each case copies oracle/mla_oracle.c, applies one small textual change of the
kind a careless restatement could make (a dropped term, a wrong sign, a wrong
index or operand), builds the copy into a temporary library and runs every
quick pin against it. The real oracle passes all pins (test_oracle_pins.py);
each mutant must fail at least one. Every mutant keeps its reads in bounds.
"""
import os

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "mla_oracle.c")

# (id, original text, replacement, occurrence index)
MUTANTS = [
    ("absorb_drops_q_pe", "memcpy(dst + kv_rank, q_pe + rh * d_rope,",
     "memset(dst + kv_rank, 0,", 0),
    ("absorb_head0_weights", "const float* w_h = w_uk + (int64_t)h * d_nope * kv_rank;",
     "const float* w_h = w_uk;", 0),
    ("absorb_head0_query", "const float* q = q_nope + rh * d_nope;",
     "const float* q = q_nope + (rh - h) * d_nope;", 0),
    ("decode_drops_rope_term", "dot_elem(q_f, kv_cache, kv_dtype, off, W)",
     "dot_elem(q_f, kv_cache, kv_dtype, off, kv_rank)", 0),
    ("decode_no_scale", "off, W) * scale;", "off, W) * 1.0f;", 0),
    ("decode_rescale_sign", "expf(st->top - top)", "expf(top - st->top)", 0),
    ("decode_acc_not_rescaled", "st->acc[d] * carry + w *", "st->acc[d] + w *", 0),
    ("decode_l_not_rescaled", "st->mass = st->mass * carry + w;", "st->mass = st->mass + w;", 0),
    ("decode_v_reversed", "w * load_elem(base, dtype, off + d)",
     "w * load_elem(base, dtype, off + st->n - 1 - d)", 0),
    ("decode_horizon_off_by_one", "horizon = seq_len - t_q + t + 1;",
     "horizon = seq_len - t_q + t;", 0),
    ("decode_horizon_from_chunk_start", "horizon = seq_len - t_q + t + 1;",
     "horizon = t + 1;", 0),
    ("decode_row_in_block_reversed", "+ j % block_size) * W;",
     "+ (block_size - 1 - j % block_size)) * W;", 0),
    ("decode_lse_no_log", "st->top + logf(st->mass)", "st->top + st->mass", 0),
    ("decode_wrong_table_row", "block_table + (int64_t)b * max_blocks", "block_table", 0),
    ("bf16_wrong_shift", "[i] << 16;", "[i] << 15;", 0),
    ("combine_weight_sign", "expf(lse_parts[s] - M)", "expf(M - lse_parts[s])", 0),
    ("combine_lse_no_log", "*lse_out = M + logf(wsum);", "*lse_out = M;", 0),
    ("decompress_reversed", "1, o, 1, kv_rank);", "1, o + kv_rank - 1, -1, kv_rank);", 0),
    ("naive_drops_rope_term", "k_pe + (int64_t)t * dr, 1, dr)", "k_pe + (int64_t)t * dr, 1, 0)", 0),
    ("absorbed_form_drops_rope_term", "k_pe + (int64_t)t * dr, 1, dr)",
     "k_pe + (int64_t)t * dr, 1, 0)", 1),
    ("naive_v_uses_w_uk", "dot_from(0.0f, wv + (int64_t)j * r, 1, c, 1, r)",
     "dot_from(0.0f, wk + (int64_t)(j % dn) * r, 1, c, 1, r)", 0),
    ("rope_neox_sign", "x[v] = xu * sn + xv * cs;", "x[v] = xu * sn - xv * cs;", 0),
    ("rope_interleaved_pair", "turn_plane(x, 2 * k, 2 * k + 1, angle)",
     "turn_plane(x, 2 * k, (2 * k + 2) % n_dims, angle)", 0),
    ("perm_wrong", "(i >> 1) + n_dims / 2 :", "n_dims - 1 - (i >> 1) :", 0),
    ("append_ties_away", "return (uint16_t)((u + 0x7fffu + lsb) >> 16);",
     "return (uint16_t)((u + 0x8000u) >> 16);", 0),
    ("append_truncates", "return (uint16_t)((u + 0x7fffu + lsb) >> 16);",
     "return (uint16_t)(u >> 16);", 0),
    ("append_writes_padding", "const int64_t s = slots[n];\n        if (s < 0) continue;",
     "const int64_t s = slots[n] < 0 ? 0 : slots[n];", 0),
    ("append_rope_from_kv", "(int64_t)n * d_rope + (j - kv_rank));",
     "(int64_t)n * kv_rank + (j - kv_rank));", 0),
    ("q_prolog_rope_skipped", "(float)positions[r], rope_base);", "(float)0, rope_base);", 0),
    ("q_prolog_row0_position", "(float)positions[r], rope_base);",
     "(float)positions[0], rope_base);", 0),
    ("q_prolog_head0_rope", "oracle_rope_neox(q_abs + ((int64_t)r * n_head + h) * W + kv_rank,",
     "oracle_rope_neox(q_abs + ((int64_t)r * n_head) * W + kv_rank,", 0),
    ("prolog_norm_sum_not_mean", "sqrt(ss / (double)kv_rank + eps)", "sqrt(ss + eps)", 0),
    ("prolog_norm_drops_eps", "sqrt(ss / (double)kv_rank + eps)", "sqrt(ss / (double)kv_rank)", 0),
    ("prolog_norm_no_gamma", "row[i] = g * x / rms;", "row[i] = x / rms;", 0),
    ("prolog_norm_no_sqrt", "const double rms = sqrt(ss / (double)kv_rank + eps);",
     "const double rms = ss / (double)kv_rank + eps;", 0),
    ("prolog_rope_interleaved", "oracle_rope_neox(pe, d_rope,", "oracle_rope_interleaved(pe, d_rope,", 0),
    ("prolog_rope_skipped", "oracle_rope_neox(pe, d_rope, (float)position, rope_base);", ";", 0),
    ("prolog_position_of_token0", "d_rope > 0 ? positions[n] : 0", "d_rope > 0 ? positions[0] : 0", 0),
    ("prolog_writes_padding", "const int64_t s = slots[n];\n        if (s < 0) continue;",
     "const int64_t s = slots[n] < 0 ? 0 : slots[n];", 1),
    ("q_norm_sum_not_mean", "sqrt(ss / (double)n + eps)", "sqrt(ss + eps)", 0),
    ("q_norm_no_gamma", "out[(int64_t)r * n + i] = (float)(g * x / rms);",
     "out[(int64_t)r * n + i] = (float)(x / rms);", 0),
    ("q_norm_eps_outside", "sqrt(ss / (double)n + eps)", "(sqrt(ss / (double)n) + eps)", 0),
    ("q_norm_row0_stats", "const double x = load_elem(xin, src_dtype, (int64_t)r * n + k);",
     "const double x = load_elem(xin, src_dtype, k);", 0),
    ("project_transposed", "dot_from(0.0f, x + (int64_t)r * k, 1, w + j, n, k)",
     "dot_from(0.0f, x + (int64_t)r * k, 1, w + (int64_t)j * k % ((int64_t)k * n), 1, k)", 0),
    ("project_drops_last_term", "dot_from(0.0f, x + (int64_t)r * k, 1, w + j, n, k)",
     "dot_from(0.0f, x + (int64_t)r * k, 1, w + j, n, k - 1)", 0),
]


def _mutate(text, old, new, occurrence):
    idx = -1
    for _ in range(occurrence + 1):
        idx = text.find(old, idx + 1)
        assert idx >= 0, f"mutation anchor not found: {old!r}"
    return text[:idx] + new + text[idx + len(old):]


@pytest.mark.parametrize("mid,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, mid, old, new, occ):
    with open(SRC) as f:
        text = f.read()
    mutated = _mutate(text, old, new, occ)
    assert mutated != text
    src = tmp_path / f"{mid}.c"
    src.write_text(mutated)
    lib = oracle.load(oracle.build(str(src), str(tmp_path / f"lib{mid}.so")))
    failed = []
    for check in pins.QUICK_CHECKS:
        try:
            check(lib)
        except (AssertionError, oracle.OracleError):
            failed.append(check.__name__)
    assert failed, f"mutant {mid} passed every pin"
