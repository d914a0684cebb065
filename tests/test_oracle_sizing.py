"""Pins of ``oracle.sizing`` against the numbers the pages print."""

from fractions import Fraction

import pytest

from oracle import sizing

KIB, MIB, GIB = 1 << 10, 1 << 20, 1 << 30


def test_m_token_printed_values(golden):
    for case in golden("sizing_examples.json")["m_token"]:
        assert sizing.m_token(case["L"], case["H_kv"], case["D_h"], case["b"]) == case["bytes"], case["cite"]


def test_request_bytes_8k(golden):
    g = golden("sizing_examples.json")["request_bytes_8k_gib"]
    assert g["tokens"] * sizing.m_token(32, 8, 128, 2) == g["gib"] * GIB


def test_trajectory_sizes_and_concurrency(golden):
    g = golden("sizing_examples.json")["trajectory_gb"]
    m = sizing.m_token(80, 8, 128, 2)
    assert m == g["m_token"]
    for s, gb, conc in zip(g["tokens"], g["gb_1dp"], g["concurrent"]):
        assert round(s * m / 1e9, 1) == gb
        assert int(g["pool_gb"] * 1e9 // (s * m)) == conc


def test_b_max(golden):
    g = golden("sizing_examples.json")["b_max"]
    for s, b in zip(g["tokens"], g["b_max"]):
        assert (g["kv_gib"] * GIB) // (s * g["kib_per_token"] * KIB) == b


def test_block_bytes_and_pool_70b_tp8(golden):
    g = golden("sizing_examples.json")["block_70b_tp8"]
    m_gpu = sizing.m_token(80, 1, 128, 2)
    assert m_gpu == g["m_token_gpu"]
    for b, kib in g["block_kib"].items():
        assert sizing.m_block(80, 1, 128, 2, int(b)) == kib * KIB
    n_blocks = (g["pool_gib"] * GIB) // sizing.m_block(80, 1, 128, 2, 16)
    assert n_blocks == g["n_blocks_b16"]
    assert n_blocks * 16 == g["tokens_b16"]
    for b, mean in g["mean_waste_tokens"].items():
        assert sizing.mean_tail_waste(int(b)) == Fraction(mean)
        waste = g["n_seq"] * sizing.mean_tail_waste(int(b)) * m_gpu
        assert waste == g["node_waste_mib"][b] * MIB


def test_qwen_capacity_table(golden):
    g = golden("sizing_examples.json")["qwen_capacity"]
    m = sizing.m_token(36, 8, 128, 2)
    assert m == g["m_token"]
    for tok, mib in g["prefill_tokens_mib"]:
        assert tok * m == mib * MIB
    per_req = []
    for tok, mib in g["total_tokens_alloc_mib"]:
        slots = g["block_size"] * sizing.blocks_for(tok, g["block_size"])
        assert slots * m == mib * MIB
        per_req.append(mib)
    assert [g["pool_mib"] // r for r in per_req] == g["fits"]


def test_paging_example_without_sharing(golden):
    g = golden("sizing_examples.json")["paging_example"]
    L, B = g["lengths"], g["block_size"]
    assert [B * sizing.blocks_for(s, B) for s in L] == g["paged_slots"]
    assert sizing.paged_slots(L, B) == g["paged_total"]
    assert sum(L) == g["used"]
    assert sum(sizing.tail_waste(s, B) for s in L) == g["paged_unused"]
    assert len(L) * g["reserved_each"] == g["reserved_total"]
    assert g["reserved_total"] - sum(L) == g["reserved_unused"]


@pytest.mark.parametrize("B", [1, 2, 3, 4, 7, 8, 16, 32, 64])
def test_tail_waste_two_forms_and_bound(B):
    # "KV 缓存管理": (B - S mod B) mod B ; "第 8 章 推理优化" §8.3.1: p*ceil(L/p) - L
    for s in range(0, 5 * B + 3):
        w = sizing.tail_waste(s, B)
        assert w == B * sizing.blocks_for(s, B) - s
        assert 0 <= w <= B - 1  # "PagedAttention 的块表与碎片控制" §04
    assert sizing.mean_tail_waste(B) == Fraction(B - 1, 2)  # the Russian page states (B-1)/2
