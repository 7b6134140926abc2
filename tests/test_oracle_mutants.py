"""Plant plausible mistakes in a copy of the C oracle and check that the pins catch them.

Each mutant is a textual edit of ``oracle/kv_oracle.c`` compiled into a
temporary library; a compact battery of the pins in ``test_oracle_pins.py``
runs against it in a child process (a mutant may read out of bounds and
crash, which also counts as caught). The unmodified source must pass the same
battery.
"""
import os
import subprocess
import sys
import textwrap

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kv_oracle.c")

MUTANTS = {
    "src_shard_by_dst_heads": ("const int64_t sp = (h / src_heads) * src_copies;",
                               "const int64_t sp = (h / dst_heads) * src_copies;"),
    "dst_local_head_by_src_heads": ("const int64_t dh = h % dst_heads;",
                                    "const int64_t dh = h % src_heads;"),
    "src_table_index_by_dst_block": ("src_bt[src_off[r] + t / src_block]",
                                     "src_bt[src_off[r] + t / dst_block]"),
    "dst_offset_by_src_block": ("const int64_t doff = t % dst_block;",
                                "const int64_t doff = t % src_block;"),
    "src_row_stride_by_dst_block": ("* src_block + soff)", "* dst_block + soff)"),
    "dropped_local_head": ("* src_heads + sh) * D + e;", "* src_heads) * D + e;"),
    "layer_component_transposed": ("((((l * C + c) * dst_num_blocks",
                                   "((((c * C + l) * dst_num_blocks"),
    "last_token_dropped": ("for (int64_t t = 0; t < n; ++t)",
                           "for (int64_t t = 0; t + 1 < n; ++t)"),
    "low_byte_only": ("for (int32_t b = 0; b < elem_bytes; ++b)",
                      "for (int32_t b = 0; b < 1; ++b)"),
    "count_without_components": ("return (int64_t)num_layers * num_components * kv_heads",
                                 "return (int64_t)num_layers * kv_heads"),
    "first_request_only": ("for (int32_t r = 0; r < num_requests; ++r) {",
                           "for (int32_t r = 0; r < 1 && r < num_requests; ++r) {"),
}

CONVERT_MUTANTS = {
    "e4m3_ties_to_lower": ("code = (lo & 1) ? lo + 1 : lo;", "code = lo;"),
    "e4m3_no_saturation": ("if (a >= 448.0)", "if (a >= 1e30)"),
    "e4m3_subnormal_exponent": ("return ldexp((double)m, -9);", "return ldexp((double)m, -10);"),
    "scale_not_inverted": ("const float y = x * inv;", "const float y = x * s;"),
    "per_head_scale_ignores_head": ("scales[(l * C + c) * kv_heads + h]",
                                    "scales[(l * C + c) * kv_heads]"),
    "bf16_ties_always_up": ("pick = ((lo >> 16) & 1) ? lo + 0x10000u : lo;",
                            "pick = lo + 0x10000u;"),
    "bf16_high_byte_dropped": ("to[1] = (uint8_t)(b >> 8);", "to[1] = 0;"),
    "nan_sign_from_nowhere": ("to[0] = (uint8_t)(((xb >> 24) & 0x80) | 0x7F);",
                              "to[0] = (uint8_t)0x7F;"),
    "nan_code_sign_dropped": ("b = (uint16_t)(((from[0] & 0x80) << 8) | 0x7FC0);",
                              "b = (uint16_t)0x7FC0;"),
}

CONVERT_BATTERY = textwrap.dedent("""
    import sys
    sys.path[:0] = [{root!r}, {tests!r}]
    import oracle, test_oracle_convert_pins as P
    lib = oracle.load({lib!r})
    P.test_e4m3_decode_fixed_points(lib)
    P.test_e4m3_decode_matches_torch(lib)
    P.test_e4m3_round_trip(lib)
    P.test_e4m3_encode_matches_torch_in_range(lib)
    P.test_e4m3_encode_saturates_and_keeps_nan(lib)
    P.test_bf16_encode_matches_torch(lib)
    for per_head in (0, 1):
        P.test_quantize_placement_reduces_to_a_copy_of_codes(lib, per_head)
        P.test_dequantize_placement_reduces_to_a_copy_of_values(lib, per_head)
    P.test_quantize_then_dequantize_stays_within_e4m3_precision(lib)
    P.test_nan_keeps_its_sign_through_both_conversions(lib)
""")

LAYOUT_MUTANTS = {
    "token_and_head_strides_swapped": ("soff * s_token_stride + sh * s_head_stride;",
                                       "soff * s_head_stride + sh * s_token_stride;"),
    "base_ignores_shard": ("dst_base[(dp * L + l) * C + c]", "dst_base[(0 * L + l) * C + c]"),
    "base_layer_component_swapped": ("src_base[(sp * L + l) * C + c]",
                                     "src_base[(sp * L + c) * C + l]"),
    "dst_block_stride_dropped": ("dblk * d_block_stride +", "dblk * d_token_stride +"),
    "generic_quant_scale_not_inverted": ("to[0] = kvo_e4m3_encode(x * inv);",
                                         "to[0] = kvo_e4m3_encode(x * s);"),
    "generic_dequant_sign_dropped": ("b = kvo_bf16_encode(kvo_e4m3_decode(from[0]) * s);",
                                     "b = kvo_bf16_encode(fabsf(kvo_e4m3_decode(from[0])) * s);"),
}

LAYOUT_BATTERY = textwrap.dedent("""
    import sys
    sys.path[:0] = [{root!r}, {tests!r}]
    import oracle, test_oracle_layout_pins as P
    lib = oracle.load({lib!r})
    P.test_standard_views_reduce_to_the_standard_oracle(lib)
    P.test_head_major_blocks_are_a_transpose(lib)
    P.test_head_major_prefill_side_too(lib)
    P.test_separate_buffers_per_layer_and_component(lib)
    P.test_k_and_v_interleaved_per_block(lib)
    P.test_staging_buffer_holds_pd_py_gather(lib)
    P.test_pack_then_unpack_equals_the_direct_relayout(lib)
    P.test_standard_views_reduce_to_the_converting_oracle(lib, "quant")
    P.test_standard_views_reduce_to_the_converting_oracle(lib, "dequant")
""")

REPLICA_MUTANTS = {
    "read_from_the_last_copy": ("const int64_t sp = (h / src_heads) * src_copies;",
                                "const int64_t sp = (h / src_heads) * src_copies + "
                                "(src_copies - 1);"),
    "only_the_first_copy_written": ("for (int64_t k = 0; k < dst_copies; ++k) {",
                                    "for (int64_t k = 0; k < 1; ++k) {"),
    "copy_index_dropped": ("const int64_t dp = (h / dst_heads) * dst_copies + k;",
                           "const int64_t dp = (h / dst_heads) * dst_copies;"),
    "copies_counted_on_the_wrong_side": (
        "const int64_t dst_copies = cards_per_head(kv_heads, dst_tp);",
        "const int64_t dst_copies = cards_per_head(kv_heads, src_tp);"),
    "copies_ignored": ("return tp <= kv_heads ? 1 : tp / kv_heads;", "return 1;"),
    "copies_as_extra_heads": ("return tp <= kv_heads ? kv_heads / tp : 1;",
                              "return tp <= kv_heads ? kv_heads / tp : tp / kv_heads;"),
}

REPLICA_BATTERY = textwrap.dedent("""
    import sys
    sys.path[:0] = [{root!r}, {tests!r}]
    import oracle, test_oracle_replica_pins as P
    lib = oracle.load({lib!r})
    for H in (1, 2):
        for tp in P.REPLICATED_TP:
            P.test_tagged_heads_reach_every_decode_copy_from_the_first_prefill_copy(lib, H, tp)
    for H, tp in [(1, (1, 8)), (2, (8, 2)), (8, (4, 16))]:
        P.test_pd_py_restatement_agrees_with_replication(lib, H, tp)
    for H, tp_d in [(1, 4), (2, 4)]:
        P.test_decode_copies_equal_the_unreplicated_relayout(lib, H, tp_d)
    for H, tp_s in [(1, 4), (2, 8)]:
        P.test_prefill_copies_reduce_to_the_first_copy(lib, H, tp_s)
    P.test_replication_in_the_converting_and_layout_nests(lib)
""")

BATTERY = textwrap.dedent("""
    import sys
    sys.path[:0] = [{root!r}, {tests!r}]
    import oracle, test_oracle_pins as P
    lib = oracle.load({lib!r})
    P.test_llama70b_4k_prompt_is_1_34_gb_and_27_ms(lib)
    P.test_deepseek_mla_4k_prompt_is_0_29_gb_and_6_ms(lib)
    P.test_relayout_moves_exactly_the_counted_bytes(lib)
    P.test_tiny_tagged_every_tag_lands_once_in_its_decode_slot(lib)
    for tp in [(1, 1), (1, 2), (2, 1), (2, 2)]:
        P.test_enumerate_block_sizes_and_tp(lib, tp)
    for case in ["tp4_to_tp8", "tp4_to_tp2_ragged", "tp3_to_tp2_odd_blocks"]:
        P.test_relayout_then_inverse_is_identity(lib, case)
""")


def _battery(lib_path, battery=None):
    code = (battery or BATTERY).format(root=ROOT, tests=os.path.join(ROOT, "tests"),
                                       lib=lib_path)
    return subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                          timeout=300)


def _build(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    return oracle.build(force=True, src=str(src), out=str(tmp_path / f"lib{name}.so"))


def test_unmutated_oracle_passes_the_battery(tmp_path):
    with open(SRC) as f:
        lib = _build(tmp_path, "control", f.read())
    res = _battery(lib)
    assert res.returncode == 0, res.stderr[-3000:]
    res = _battery(lib, CONVERT_BATTERY)
    assert res.returncode == 0, res.stderr[-3000:]
    res = _battery(lib, LAYOUT_BATTERY)
    assert res.returncode == 0, res.stderr[-3000:]
    res = _battery(lib, REPLICA_BATTERY)
    assert res.returncode == 0, res.stderr[-3000:]


@pytest.mark.parametrize("name", sorted(REPLICA_MUTANTS))
def test_replica_mutant_is_caught(tmp_path, name):
    """Head-replication mistakes, planted in every loop nest, fail the replica pins."""
    old, new = REPLICA_MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) >= 1, f"mutation site for {name} not in the oracle"
    lib = _build(tmp_path, name, text.replace(old, new))
    res = _battery(lib, REPLICA_BATTERY)
    assert res.returncode != 0, f"mutant {name} survived the replica pins"


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) >= 1, f"mutation site for {name} not in the oracle"
    lib = _build(tmp_path, name, text.replace(old, new))
    res = _battery(lib)
    assert res.returncode != 0, f"mutant {name} survived the pins"


INDEX_MUTANTS = ["src_shard_by_dst_heads", "dst_local_head_by_src_heads",
                 "src_table_index_by_dst_block", "dst_offset_by_src_block",
                 "src_row_stride_by_dst_block", "dropped_local_head",
                 "layer_component_transposed", "last_token_dropped"]


@pytest.mark.parametrize("name", INDEX_MUTANTS)
def test_conversion_index_mutant_is_caught(tmp_path, name):
    """The same indexing mistakes planted only in the converting loop nest (the
    second occurrence of each site; the layout-generic nest is the third) must fail
    the conversion pins."""
    old, new = MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) >= 2, f"{name}: expected a site in each loop nest"
    first = text.index(old) + len(old)
    lib = _build(tmp_path, name, text[:first] + text[first:].replace(old, new, 1))
    res = _battery(lib, CONVERT_BATTERY)
    assert res.returncode != 0, f"mutant {name} survived the conversion pins"


@pytest.mark.parametrize("name", sorted(CONVERT_MUTANTS))
def test_conversion_mutant_is_caught(tmp_path, name):
    old, new = CONVERT_MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) >= 1, f"mutation site for {name} not in the oracle"
    lib = _build(tmp_path, name, text.replace(old, new))
    res = _battery(lib, CONVERT_BATTERY)
    assert res.returncode != 0, f"mutant {name} survived the pins"


@pytest.mark.parametrize("name", sorted(LAYOUT_MUTANTS))
def test_layout_mutant_is_caught(tmp_path, name):
    old, new = LAYOUT_MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) == 1, f"mutation site for {name} not unique in the oracle"
    lib = _build(tmp_path, name, text.replace(old, new))
    res = _battery(lib, LAYOUT_BATTERY)
    assert res.returncode != 0, f"mutant {name} survived the layout pins"
