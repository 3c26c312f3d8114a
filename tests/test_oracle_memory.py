"""Pins of the KV memory arithmetic against the page's own tables.

"Context Optimization", Memory Savings, Memory with Sliding Window and Memory Budget
Calculator; "Per-Head Attention as a Scoring Signal", Scoring granularity (block of 16
tokens = 5.00 MiB at 320 KiB per token); "Context views at marginal cost", Fact 1
(one head's n x n matrix at n = 100k is about 1e10 entries)."""
import json
import math
import os

from oracle import memory

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")))
KiB, MiB = 1024, 1024 * 1024


def test_memory_savings_table_consistent_rows():
    for row in GOLD["memory_savings_table"]["rows"]:
        shape = (row["layers"], row["kv_heads"], row["head_dim"])
        if not row["consistent_with_formula"]:
            # the page's own calculator disagrees with this row: recorded, not pinned
            assert memory.kv_payload_bytes_per_position(*shape, "f32") != row["f32_per_position_KiB"] * KiB
            continue
        assert memory.kv_payload_bytes_per_position(*shape, "f32") == row["f32_per_position_KiB"] * KiB
        assert memory.kv_payload_bytes_per_position(*shape, "e4m3") == row["fp8_per_position_KiB"] * KiB
        assert memory.kv_cache_bytes(*shape, "f32", 4096) == row["at_4k_f32_MiB"] * MiB
        assert memory.kv_cache_bytes(*shape, "e4m3", 4096) == row["at_4k_fp8_MiB"] * MiB
        assert memory.kv_cache_bytes(*shape, "f32", 32768) == row["at_32k_f32_MiB"] * MiB
        assert memory.kv_cache_bytes(*shape, "e4m3", 32768) == row["at_32k_fp8_MiB"] * MiB


def test_sliding_window_table():
    for row in GOLD["sliding_window_table"]["rows_35B"]:
        got = memory.kv_cache_bytes(10, 4, 128, row["format"], context=10 ** 6, window=row["window"])
        assert got == row["MiB"] * MiB


def test_budget_calculator():
    c = GOLD["budget_calculator"]
    assert memory.kv_elements_per_position(10, 4, 128) == c["elements_per_position_35B"]
    assert memory.kv_bytes_per_position(10, 4, 128, "f32") == c["f32_per_position_KiB_35B"] * KiB
    fp8 = memory.kv_bytes_per_position(10, 4, 128, "e4m3")
    assert fp8 == 10240 + 10 * 2 * c["scale_bytes_per_position_per_cache"]
    assert abs(fp8 / KiB - c["fp8_per_position_KiB_35B_approx"]) / c["fp8_per_position_KiB_35B_approx"] < 0.05
    assert memory.kv_elements_per_position(15, 8, 128) == c["elements_per_position_397B"]
    assert memory.kv_bytes_per_position(15, 8, 128, "f32") == c["f32_per_position_KiB_397B"] * KiB
    at8k = memory.kv_cache_bytes(10, 4, 128, "e4m3", 8192, with_scales=True) / 1e6
    assert abs(at8k - c["fp8_8k_context_35B_MB_approx"]) / c["fp8_8k_context_35B_MB_approx"] < 0.05


def test_block_unit():
    b = GOLD["block_unit"]
    s = b["shape_from_figure"]
    per_token = s["layers"] * 2 * s["kv_heads"] * s["head_dim"] * s["bytes_per_elem"]
    assert per_token == b["per_token_KiB"] * KiB
    assert per_token * b["block_tokens"] == b["per_block_MiB"] * MiB


def test_attention_matrix_size():
    a = GOLD["attention_matrix_size"]
    assert round(math.log10(a["n"] ** 2)) == a["entries_order_of_magnitude"]
