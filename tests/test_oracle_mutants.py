"""Each plausible slip planted in a copy of the oracle must fail at least one pin.

The mutants are made on the CPU from the oracle's source text at test time:
a dropped term, a wrong index, a transposed operand, a wrong sign, a wrong
rounding, a broken tie-break.  The committed oracle itself is never changed.
"""
import os
import subprocess

import pytest

import oracle
import oracle_pins as pins

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "hss_oracle.c")).read()

# (name, text to replace, replacement, which occurrence (0-based)).
# Not listed: the sign of a NaN's bf16 pattern (IEEE 754 leaves a NaN's sign unspecified
# for conversions and PyTorch itself gives 0xFFFF for both signs, so nothing outside the
# oracle fixes it), and, because they are equivalent mutants (no input tells them apart):
# loosening the explicit overflow test in the bf16 rounding (the binary32
# conversion of 2^128 is +inf anyway), and dropping the -0 -> +0 step of the
# per-row selection (its comparator already orders -0 and +0 as equal).
MUTANTS = [
    ("q_drops_first_term", "for (int d = 0; d < k->hd; ++d) {\n            acc +=",
     "for (int d = 1; d < k->hd; ++d) {\n            acc +=", 0),
    ("kv_drops_last_term", "for (int d = 0; d < k->hd; ++d) {\n                    acc +=",
     "for (int d = 0; d + 1 < k->hd; ++d) {\n                    acc +=", 0),
    ("q_transposed_P", "k->P[(int64_t)d * k->r + j]", "k->P[(int64_t)j * k->hd + d]", 0),
    ("kv_transposed_P", "k->P[(int64_t)d * k->r + j]", "k->P[(int64_t)j * k->hd + d]", 1),
    ("slot_not_transposed", "slot[((int64_t)h * k->bs + t) * k->r + j]",
     "slot[((int64_t)t * k->nkv + h) * k->r + j]", 0),
    ("kv_input_head_major", "kb + ((int64_t)t * k->nkv + h) * k->hd",
     "kb + ((int64_t)h * k->bs + t) * k->hd", 0),
    ("gqa_modulo", "int c_kv = h / g;", "int c_kv = h % k->nkv;", 0),
    ("score_ignores_layer", "k->A + (k->layer * k->max_blocks + id) * slot_elems;\n    double best",
     "k->A + (id) * slot_elems;\n    double best", 0),
    ("kv_ignores_layer", "k->A + (k->layer * k->max_blocks + id) * slot_elems;\n    const uint16_t* kb",
     "k->A + (id) * slot_elems;\n    const uint16_t* kb", 0),
    ("score_wrong_row_index", "((s * k->rows + row) * (int64_t)k->nq + h)",
     "((s + row) * (int64_t)k->nq + h)", 0),
    ("score_max_floor_zero", "double best = -INFINITY;", "double best = 0.0;", 0),
    ("score_min_not_max", "if (dot > best) {", "if (-dot > -best || best == -INFINITY) {", 0),
    ("score_abs_dot", "dot += term;", "dot += fabs(term);", 0),
    ("round_toward_zero", "double q = nearbyint(ldexp(x, -qexp));",
     "double q = trunc(ldexp(x, -qexp));", 0),
    ("round_half_away", "double q = nearbyint(ldexp(x, -qexp));",
     "double q = round(ldexp(x, -qexp));", 0),
    ("double_rounding", "double q = nearbyint(ldexp(x, -qexp));",
     "double q = nearbyint(ldexp((double)(float)x, -qexp));", 0),
    ("seven_bits_only", "int qexp = e - 8;", "int qexp = e - 7;", 0),
    ("no_subnormal_floor", "if (qexp < -133) {\n            qexp = -133;",
     "if (qexp < -149) {\n            qexp = -149;", 0),
    ("tie_break_reversed", "return (x->idx > y->idx) - (x->idx < y->idx);",
     "return (x->idx < y->idx) - (x->idx > y->idx);", 0),
    ("descending_victims", "if (x->v < y->v) {\n        return -1;",
     "if (x->v > y->v) {\n        return -1;", 0),
    ("nan_not_mapped", "if (isnan(v)) {\n                v = INFINITY;",
     "if (isnan(v)) {\n                v = -INFINITY;", 0),
    ("no_minus_one_pad", "victims[s * (int64_t)k + j] = j < n ? keyed[j].idx : -1;",
     "victims[s * (int64_t)k + j] = j < n ? keyed[j].idx : 0;", 0),
    ("bad_id_scored_zero", "*score = INFINITY;\n        *tsum = 0.0;",
     "*score = 0.0;\n        *tsum = 0.0;", 0),
    ("length_mask_off_by_one", "if (ctx_len != NULL && pos >= ctx_len[s]) {",
     "if (ctx_len != NULL && pos > ctx_len[s]) {", 0),
    ("causal_mask_off_by_one", "if (row_pos0 != NULL && pos > row_pos0[s] + row) {",
     "if (row_pos0 != NULL && pos >= row_pos0[s] + row) {", 0),
    ("causal_ignores_row", "if (row_pos0 != NULL && pos > row_pos0[s] + row) {",
     "if (row_pos0 != NULL && pos > row_pos0[s]) {", 0),
    ("position_not_per_sequence", "i - k->seq_offsets[s], k->ctx_len",
     "i, k->ctx_len", 0),
    ("token_block_and_position_swapped", "int64_t blk = s / k->bs;\n    int t = (int)(s % k->bs);",
     "int64_t blk = s % k->bs;\n    int t = (int)(s / k->bs);", 0),
    ("token_cache_head_major", "((blk * k->bs + t) * k->nkv + h) * (int64_t)k->hd",
     "((blk * k->nkv + h) * k->bs + t) * (int64_t)k->hd", 0),
    ("token_a_g_token_major", "((k->layer * k->max_blocks + blk) * k->nkv + h) * k->bs + t)",
     "((k->layer * k->max_blocks + blk) * k->bs + t) * k->nkv + h)", 0),
    ("token_ignores_layer", "(((k->layer * k->max_blocks + blk) * k->nkv",
     "(((0 * k->max_blocks + blk) * k->nkv", 0),
    ("token_drops_last_term", "for (int d = 0; d < k->hd; ++d) {\n                acc +=",
     "for (int d = 0; d + 1 < k->hd; ++d) {\n                acc +=", 0),
    ("token_transposed_P", "k->P[(int64_t)d * k->r + j]", "k->P[(int64_t)j * k->hd + d]", 2),
    ("rows_max_over_all_rows", "    one.rows = 1;\n    orc_score_one(&one, row, id,",
     "    one.rows = 1;\n    orc_score_one(&one, 0, id,", 0),
    ("rows_bad_id_plus_inf", "        k->score[i] = -INFINITY;", "        k->score[i] = INFINITY;", 0),
    ("select_complete_off_by_one", "int64_t complete = (first_pos + r + 1) / block_size;",
     "int64_t complete = (first_pos + r) / block_size;", 0),
    ("select_ascending", "v = isnan(v) ? INFINITY : -v;", "v = isnan(v) ? INFINITY : v;", 0),
    ("select_nan_first", "v = isnan(v) ? INFINITY : -v;", "v = isnan(v) ? -INFINITY : -v;", 0),
    ("token_status_counts_padding", "if (slots[i] >= max_blocks * block_size) {",
     "if (slots[i] < 0 || slots[i] >= max_blocks * block_size) {", 0),
    ("victims_global_index", "keyed[i].idx = (int32_t)i;\n        }\n        qsort(keyed, (size_t)n,",
     "keyed[i].idx = (int32_t)(base + i);\n        }\n        qsort(keyed, (size_t)n,", 0),
    ("select_no_minus_one_pad", "lists[r * (int64_t)topk + i] = i < complete ? keyed[i].idx : -1;",
     "lists[r * (int64_t)topk + i] = i < complete ? keyed[i].idx : 0;", 0),
    ("select_ignores_first_pos", "int64_t complete = (first_pos + r + 1) / block_size;",
     "int64_t complete = (r + 1) / block_size;", 0),
    ("select_row_stride_is_n", "double v = (double)scores[r * stride + j];",
     "double v = (double)scores[r * n + j];", 0),
    ("score_drops_last_token", "for (int t = 0; t < k->bs; ++t) {\n                const uint16_t* a",
     "for (int t = 0; t + 1 < k->bs; ++t) {\n                const uint16_t* a", 0),
    ("score_drops_last_head", "for (int h = 0; h < k->nq; ++h) {", "for (int h = 0; h + 1 < k->nq; ++h) {",
     0),
    ("score_drops_last_row", "for (int row = 0; row < k->rows; ++row) {",
     "for (int row = 0; row + 1 < k->rows; ++row) {", 0),
    ("tsum_signed", "mag += fabs(term);", "mag += term;", 0),
    ("masked_max_floor_zero", "double best = -INFINITY;", "double best = 0.0;", 1),
    ("masked_drops_last_head", "for (int h = 0; h < k->nq; ++h) {", "for (int h = 0; h + 1 < k->nq; ++h) {",
     1),
    ("overflow_saturates", "y = copysign(INFINITY, x);", "y = copysign(0x1.FEp127, x);", 0),
    ("bf16_widen_wrong_shift", "uint32_t u = ((uint32_t)b) << 16;", "uint32_t u = ((uint32_t)b) << 15;", 0),
    ("kv_bad_position_zero_based", "            return i + 1;", "            return i;", 0),
    ("token_cache_not_written", "memcpy(crow, krow, (size_t)k->hd * sizeof(uint16_t));",
     "(void)crow;", 0),
    ("q_float_accumulator", "double acc = 0.0;\n        for (int d = 0; d < k->hd; ++d) {\n            acc +=",
     "float acc = 0.0;\n        for (int d = 0; d < k->hd; ++d) {\n            acc +=", 0),
    ("kv_float_accumulator", "double acc = 0.0;\n                for (int d = 0; d < k->hd; ++d) {\n                    acc +=",
     "float acc = 0.0;\n                for (int d = 0; d < k->hd; ++d) {\n                    acc +=", 0),
    ("token_float_accumulator", "double acc = 0.0;\n            for (int d = 0; d < k->hd; ++d) {\n                acc +=",
     "float acc = 0.0;\n            for (int d = 0; d < k->hd; ++d) {\n                acc +=", 0),
    ("q_rounds_through_float", "k->Qp[v * k->r + j] = orc_bf16_from_double(acc);",
     "k->Qp[v * k->r + j] = orc_bf16_from_double((double)(float)acc);", 0),
    ("kv_rounds_through_float", "slot[((int64_t)h * k->bs + t) * k->r + j] = orc_bf16_from_double(acc);",
     "slot[((int64_t)h * k->bs + t) * k->r + j] = orc_bf16_from_double((double)(float)acc);", 0),
    ("token_rounds_through_float", "arow[j] = orc_bf16_from_double(acc);",
     "arow[j] = orc_bf16_from_double((double)(float)acc);", 0),
]


def _mutate(text, old, new, occurrence):
    pos = -1
    for _ in range(occurrence + 1):
        pos = text.find(old, pos + 1)
        assert pos >= 0, f"mutation site not found: {old!r}"
    return text[:pos] + new + text[pos + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, occ, tmp_path):
    src = tmp_path / f"{name}.c"
    src.write_text(_mutate(SRC, old, new, occ))
    so = oracle.build(force=True, src=str(src), out=str(tmp_path / f"lib{name}.so"))
    L = oracle.load_from(so)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(L)
        except Exception as e:  # an assertion, or a crash-free error raised by the pin
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"mutant {name} passed every pin"


def test_unmutated_copy_passes(tmp_path):
    src = tmp_path / "same.c"
    src.write_text(SRC)
    L = oracle.load_from(oracle.build(force=True, src=str(src), out=str(tmp_path / "libsame.so")))
    for pin in pins.ALL_PINS:
        pin(L)
