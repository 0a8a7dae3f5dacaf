"""Planted mistakes: each mutant of oracle.c must fail at least one pin.

The mutants are built from a copy of the oracle source on the CPU; the real
oracle is never changed.  This shows the pins would catch a dropped term, a
wrong sign or index, or a transposed operand anywhere in the oracle.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_backward_pins as bpins
from tests import test_oracle_chunked_pins as cpins
from tests import test_oracle_pages_pins as ppins
from tests import test_oracle_rope_pins as rpins
from tests import test_oracle_rope_q_pins as rqpins
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "oracle.c")

MUTANTS = {
    "gqa_map_modulo": ("hq / group, pre + n, pre + i", "hq % g->num_kv_heads, pre + n, pre + i"),
    "causal_off_by_one": ("if (j > last_key) {", "if (j >= last_key && j > 0) {"),
    "log2_lse": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "token_stride_head_dim": ("token_in_block * kv_dim(g) * 2 +\n", "token_in_block * g->head_dim * 2 +\n"),
    "v_offset_wrong": ("memcpy(&vb, pool + addr + v_offset(g), 2);", "memcpy(&vb, pool + addr + v_offset(g) / 2, 2);"),
    "scale_dropped": ("s_buf[j] = scale * dot;", "s_buf[j] = dot;"),
    "table_index_transposed": ("(int64_t)slot * g->n_layers * g->max_blocks_per_seq +\n                  (int64_t)layer * g->max_blocks_per_seq",
                               "(int64_t)layer * g->num_slots * g->max_blocks_per_seq +\n                  (int64_t)slot * g->max_blocks_per_seq"),
    "merge_without_rescale": ("ls += l[i] * c;", "ls += l[i];"),
    "normaliser_off": ("o[k] = acc / l;", "o[k] = acc / (l + 1e-3);"),
    "write_v_at_k": ("uint8_t* v_dst = k_dst + v_offset(g);", "uint8_t* v_dst = k_dst + v_offset(g) + 2;"),
    "prefix_ignored": ("int32_t pre = c->prefix ? c->prefix[b] : 0;", "int32_t pre = 0;"),
    "prefix_last_key_off_by_one": ("pre + n, pre + i, c->scale", "pre + n, pre + i - 1, c->scale"),
    "prefix_not_in_position": ("pre + n, pre + i, c->scale", "pre + n, i, c->scale"),
    "rope_signs_swapped": ("const float y1 = a - b, y2 = e + f;", "const float y1 = a + b, y2 = e - f;"),
    "rope_interleaved_pairs": ("const float x1 = bf16_to_float(x[i]), x2 = bf16_to_float(x[i + half]);",
                               "const float x1 = bf16_to_float(x[2 * i]), x2 = bf16_to_float(x[2 * i + 1]);"),
    "rope_next_table_row": ("rope_row(g, g->num_kv_heads, k_new + t * kv_dim(g), cos_tab + (int64_t)tok_pos[t] * half,",
                            "rope_row(g, g->num_kv_heads, k_new + t * kv_dim(g), cos_tab + (int64_t)(tok_pos[t] + 1 < max_pos ? tok_pos[t] + 1 : tok_pos[t]) * half,"),
    "rope_truncating_round": ("u += 0x7FFFu + lsb;", "u += 0u * lsb;"),
    "ropeq_position_without_prefix": ("const int64_t pos = (int64_t)pre + (t - cu_seqlens[b]);",
                                      "const int64_t pos = (t - cu_seqlens[b]);"),
    "ropeq_packed_row_as_position": ("const int64_t pos = (int64_t)pre + (t - cu_seqlens[b]);",
                                     "const int64_t pos = (int64_t)pre + t;"),
    "ropeq_kv_head_count": ("rope_row(g, g->num_q_heads, q + t * row,", "rope_row(g, g->num_kv_heads, q + t * row,"),
    "alloc_pop_order": ("*e = free_pages[--top]; /* pop_back */", "*e = free_pages[(--top) ^ 1]; /* pop_back */"),
    "alloc_last_block_missing": ("const int32_t hi = (len + TOKENS_PER_BLOCK - 1) / TOKENS_PER_BLOCK;",
                                 "const int32_t hi = len / TOKENS_PER_BLOCK;"),
    "alloc_sequences_reversed": ("        for (int32_t b = 0; b < batch; ++b) {\n            const int32_t slot = slots[b], len = seq_lens[b];",
                          "        for (int32_t b = batch - 1; b >= 0; --b) {\n            const int32_t slot = slots[b], len = seq_lens[b];"),
    "release_keeps_entry": ("                free_pages[top++] = *e; /* push_back */\n                *e = -1;",
                            "                free_pages[top++] = *e; /* push_back */"),
    "bwd_D_dropped": ("ds[j] = p[j] * (ds[j] - D);", "ds[j] = p[j] * ds[j];"),
    "bwd_dk_unscaled": ("dkj[k] += c->scale * ds[j] * qv[k];", "dkj[k] += ds[j] * qv[k];"),
    "bwd_dv_uses_ds": ("dvj[k] += p[j] * dov[k];", "dvj[k] += ds[j] * dov[k];"),
    "bwd_first_head_only": ("    for (int32_t r = 0; r < group; ++r) {\n        const int32_t h = hk * group + r;\n        for (int32_t i = 0; i < n; ++i) {",
                            "    for (int32_t r = 0; r < 1; ++r) {\n        const int32_t h = hk * group + r;\n        for (int32_t i = 0; i < n; ++i) {"),
    "bwd_rows_skips_diagonal": ("        for (int32_t i = j; i < n; ++i) {\n            const int64_t qrow = r0 + i;",
                                "        for (int32_t i = j + 1; i < n; ++i) {\n            const int64_t qrow = r0 + i;"),
    "bwd_rows_stats_of_next_row": ("const double pij = exp(bc->scale * dot - st[3 * i]) / st[3 * i + 1];",
                                   "const double pij = exp(bc->scale * dot - st[3 * (i + (i + 1 < n))]) / st[3 * i + 1];"),
    "max_not_subtracted": ("for (int32_t j = 0; j < n; ++j) l += exp(s[j] - m);",
                           "for (int32_t j = 0; j < n; ++j) l += exp(s[j] - m) * (1 + 1e-9 * m);"),
}

PIN_TESTS = [
    lambda gd: pins.test_worked_example_decode(gd),
    lambda gd: pins.test_worked_example_prefill_rows(gd),
    lambda gd: pins.test_worked_example_blocks_and_merge(gd),
    lambda gd: pins.test_softmax_stress_rows(gd),
    lambda gd: pins.test_layout_constants_and_offsets(gd),
    lambda gd: pins.test_layout_as_array_shape(),
    lambda gd: pins.test_zero_query_gives_running_mean(),
    lambda gd: pins.test_causal_row0_is_first_value(),
    lambda gd: pins.test_lse_split_merge_identity(),
    lambda gd: pins.test_prefill_matches_library_sdpa(8, 2, 64, [40]),
    lambda gd: pins.test_decode_matches_library_sdpa(),
    lambda gd: cpins.test_chunked_matches_library_sdpa(8, 2, 64, [0, 16, 23], [40, 17, 1]),
    lambda gd: cpins.test_chunk_of_one_is_decode(),
    lambda gd: rpins.test_worked_example_pairing(gd),
    lambda gd: rpins.test_special_angles(),
    lambda gd: rpins.test_matches_torch_fp32_ops_byte_for_byte(),
    lambda gd: rqpins.test_identity_table_changes_nothing(),
    lambda gd: rqpins.test_quarter_turns_by_position(8, 2, 64),
    lambda gd: rqpins.test_prefill_rope_matches_library_sdpa_on_complex_turns(),
    lambda gd: ppins.test_worked_example(gd),
    lambda gd: ppins.test_decode_takes_a_page_only_at_a_new_block(),
    lambda gd: bpins.test_matches_torch_autograd(8, 2, 64, [40, 17]),
    lambda gd: bpins.test_identities(),
    lambda gd: bpins.test_sampled_rows_equal_the_full_backward(8, 2, 64, [40, 17, 1]),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, golden_dir):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor missing: " + name
    mutated = src.replace(old, new)
    c_path = tmp_path / "oracle.c"
    c_path.write_text(mutated)
    hdr = os.path.join(os.path.dirname(SRC), "oracle.h")
    (tmp_path / "oracle.h").write_text(open(hdr).read())
    so = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-o", str(so),
                    str(c_path), "-lm"], check=True)
    caught = []
    with oracle.use_library(str(so)):
        for i, t in enumerate(PIN_TESTS):
            try:
                t(golden_dir)
            except AssertionError:
                caught.append(i)
    assert caught, "no pin caught mutant " + name
