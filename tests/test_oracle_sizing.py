"""Pins for the closed forms: every value here is one the pages print."""
import math

import numpy as np
import pytest

from oracle import sizing

GiB = 2 ** 30
MiB = 2 ** 20


def test_block_counts_at_1000_tokens(golden):
    g = golden("block_counts.json")
    for row in g["rows"]:
        b = row["block_size"]
        assert sizing.blocks_needed(g["tokens"], b) == row["blocks"] == row["table_entries"]
        # the table's waste column is the worst case over lengths: B - 1 tokens
        worst = max(sizing.tail_waste(s, b) for s in range(1, 4 * b + 1))
        assert worst == row["worst_waste_tokens"]


def test_ceil_example(golden):
    e = golden("block_counts.json")["ceil_example"]
    assert sizing.blocks_needed(e["tokens"], e["block_size"]) == e["blocks"]


def test_tail_waste_bound_brute_force(golden):
    e = golden("block_counts.json")["tail_bound"]
    assert max(sizing.tail_waste(s, e["block_size"]) for s in range(1, 5000)) == e["max_waste_slots"]
    for b in (8, 16, 32):
        w = [sizing.tail_waste(s, b) for s in range(1, 20 * b)]
        assert min(w) == 0 and max(w) == b - 1
        # waste is zero exactly at multiples of B
        assert all((sizing.tail_waste(s, b) == 0) == (s % b == 0) for s in range(1, 20 * b))


def test_example_1(golden):
    e = golden("block_counts.json")["example_1"]
    per = sizing.blocks_needed(e["tokens"], e["block_size"])
    assert per == e["blocks_per_seq"]
    assert per * e["seqs"] == e["paged_blocks"]
    assert e["seqs"] * sizing.blocks_needed(e["s_max"], e["block_size"]) == e["contiguous_blocks"]


def test_engineering_capacity_example(golden):
    e = golden("capacity.json")["engineering_example"]
    bb = sizing.kv_bytes_per_block(e["layers"], e["block_size"], e["kv_heads"], e["head_dim"],
                                   e["elem_bytes"])
    assert bb == e["block_bytes"] == 2 * MiB
    blocks = sizing.pool_blocks(e["pool_gib"] * GiB, bb)
    assert blocks == e["blocks"]
    assert sizing.blocks_needed(e["tokens_per_request"], e["block_size"]) == e["blocks_per_request"]
    assert sizing.max_concurrency(blocks, e["tokens_per_request"], e["block_size"]) == e["concurrency"]
    assert sizing.blocks_needed(e["contiguous_s_max"], e["block_size"]) == e["contiguous_blocks_per_request"]
    cont = sizing.max_concurrency(blocks, e["contiguous_s_max"], e["block_size"])
    assert cont == e["contiguous_concurrency"]
    assert e["concurrency"] // cont == e["ratio"]


def test_try_it_example(golden):
    e = golden("capacity.json")["try_it"]
    # 128 KiB per token is the 8B shape: 2 x 32 layers x 8 kv heads x 128 x 2 bytes
    assert sizing.kv_bytes_per_sequence(32, 1, 8, 128, 2) == e["bytes_per_token"]
    assert e["block_size"] * e["bytes_per_token"] == e["block_bytes"]
    blocks = sizing.pool_blocks(e["pool_gib"] * GiB, e["block_bytes"])
    assert blocks == e["blocks"]
    assert sizing.blocks_needed(e["tokens_per_seq"], e["block_size"]) == e["blocks_per_seq"]
    assert sizing.max_concurrency(blocks, e["tokens_per_seq"], e["block_size"]) == e["concurrency"]


def test_llama7b_kv_bytes(golden):
    e = golden("capacity.json")["llama7b"]
    b = sizing.kv_bytes_per_sequence(e["layers"], e["tokens"], e["heads"], e["head_dim"],
                                     e["elem_bytes"], batch=e["batch"])
    assert b == GiB                                   # exactly 2^30 bytes
    assert round(b / 1e9) == e["approx_gb"]


def test_llama13b_kv_bytes(golden):
    e = golden("capacity.json")["llama13b"]
    b = sizing.kv_bytes_per_sequence(e["layers"], e["tokens"], e["heads"], e["head_dim"],
                                     e["elem_bytes"])
    per = b / GiB
    assert per == 3.125
    assert round(per, 1) == e["approx_gib_per_seq"]
    assert round(round(per, 1) * e["seqs"], 1) == e["approx_total_gib"]


def test_contiguous_utilisation(golden):
    e = golden("capacity.json")["contiguous_utilisation"]
    util = sizing.effective_utilisation([e["avg_tokens"]], [e["s_max"]])
    assert round(100 * util, 1) == e["approx_percent"]
    assert sizing.fragmentation([e["avg_tokens"]], [e["s_max"]]) == pytest.approx(1 - util)


def test_paged_utilisation_above_90_percent_at_typical_lengths():
    # daiw.org 'Paged Attention', section 定义 table: paged utilisation usually > 90%,
    # waste at most the last block, so utilisation >= s / (s + B - 1), which exceeds 0.9
    # once s > 9 (B - 1).  Brute force at B = 16.
    for s in range(1, 4096):
        alloc = sizing.blocks_needed(s, 16) * 16
        u = sizing.effective_utilisation([s], [alloc])
        assert u >= s / (s + 15) - 1e-15
        if s > 9 * 15:
            assert u > 0.9


def test_planted_floor_instead_of_ceil_is_caught(golden):
    g = golden("block_counts.json")
    floor_blocks = lambda t, b: t // b
    assert floor_blocks(g["ceil_example"]["tokens"], 16) != g["ceil_example"]["blocks"]
