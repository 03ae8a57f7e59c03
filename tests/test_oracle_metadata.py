"""Pins for the oracle's metadata builder (CPU only).

Sources: "3.6 ModelRunner, CUDA Graph, and benchmarks", section 2 (worked
block_size = 4 example, decode slot rule) and section 4 (cache layout sizes);
"Warmup Guide -- Inference Serving Internals", chapter 3 (block counts, append
rule).
"""

import json
import os

import numpy as np
import pytest

from oracle import metadata as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_worked_example_prefill_matches_page():
    g = _load("worked_example_prefill.json")
    seq = dict(block_table=g["block_table"], num_cached_tokens=g["num_cached_tokens"],
               num_scheduled_tokens=g["num_scheduled_tokens"])
    md = om.prepare_prefill([seq], g["block_size"])
    exp = g["expected"]
    assert md["slot_mapping"].tolist() == exp["slot_mapping"]
    assert md["cu_seqlens_q"].tolist() == exp["cu_seqlens_q"]
    assert md["cu_seqlens_k"].tolist() == exp["cu_seqlens_k"]
    assert md["max_seqlen_q"] == exp["max_seqlen_q"]
    assert md["max_seqlen_k"] == exp["max_seqlen_k"]
    assert md["need_block_tables"] is exp["need_block_tables"]
    assert md["positions"].tolist() == exp["positions"]
    assert md["block_tables"].tolist() == [g["block_table"]]


def test_no_history_needs_no_block_tables():
    # Q and K the same length: the kernel uses this step's k/v directly (section 2)
    seqs = [dict(block_table=[3, 1], num_cached_tokens=0, num_scheduled_tokens=6),
            dict(block_table=[0], num_cached_tokens=0, num_scheduled_tokens=2)]
    md = om.prepare_prefill(seqs, 4)
    assert md["need_block_tables"] is False
    assert md["block_tables"] is None
    assert md["cu_seqlens_q"].tolist() == md["cu_seqlens_k"].tolist() == [0, 6, 8]
    assert md["slot_mapping"].tolist() == [12, 13, 14, 15, 4, 5, 0, 1]


def test_sequence_without_blocks_writes_nothing():
    # warm-up sequences have no block table: they add rows but no slots (section 2)
    seqs = [dict(block_table=[], num_cached_tokens=0, num_scheduled_tokens=5)]
    md = om.prepare_prefill(seqs, 4)
    assert md["slot_mapping"].tolist() == []
    assert md["cu_seqlens_q"].tolist() == [0, 5]


def test_block_rules():
    g = _load("block_rules.json")
    for n, bs, want in g["blocks_needed"]:
        assert om.blocks_needed(n, bs) == want
    for n, bs, want in g["append_needs_block"]:
        assert om.append_needs_block(n, bs) is want


def test_blocks_needed_brute_force():
    # the count is the smallest k with k * bs >= n
    for bs in (1, 2, 3, 4, 16, 256):
        for n in range(0, 600, 7):
            k = om.blocks_needed(n, bs)
            assert k * bs >= n and (k == 0 or (k - 1) * bs < n)


def test_decode_slot_derived_case():
    d = _load("block_rules.json")["decode_slot_derived"]
    md = om.prepare_decode([dict(block_table=d["block_table"], length=d["length"])], d["block_size"])
    assert md["slot_mapping"].tolist() == [d["slot"]]
    assert md["context_lens"].tolist() == [d["length"]]
    assert md["positions"].tolist() == [d["length"] - 1]


def test_decode_slot_is_position_of_last_token():
    # the decode slot equals the prefill slot rule applied to position len - 1
    rng = np.random.default_rng(0)
    for bs in (1, 2, 4, 16):
        for length in range(1, 70):
            table = rng.permutation(200)[: om.blocks_needed(length, bs)].tolist()
            dec = om.prepare_decode([dict(block_table=table, length=length)], bs)
            pre = om.prepare_prefill([dict(block_table=table, num_cached_tokens=length - 1,
                                           num_scheduled_tokens=1)], bs)
            assert dec["slot_mapping"].tolist() == pre["slot_mapping"].tolist()


def test_decode_padding_rows():
    tables = [[4, 9], [1]]
    md = om.prepare_decode([dict(block_table=t, length=n) for t, n in zip(tables, [5, 3])], 4)
    assert md["block_tables"].tolist() == [[4, 9], [1, -1]]
    assert md["slot_mapping"].tolist() == [9 * 4 + 0, 1 * 4 + 2]


def test_decode_rejects_wrong_table_length():
    with pytest.raises(ValueError):
        om.prepare_decode([dict(block_table=[1, 2], length=4)], 4)


def test_qwen3_layout_sizes():
    g = _load("kv_layout_qwen3.json")
    shape = (2, g["num_layers"], 1, g["block_size"], g["num_kv_heads"], g["head_dim"])
    block_bytes = int(np.prod(shape)) * g["itemsize"]
    assert block_bytes == g["block_bytes"]
    assert block_bytes // g["block_size"] == g["bytes_per_token"]
    per_layer_token = 2 * g["num_kv_heads"] * g["head_dim"] * g["itemsize"]
    assert per_layer_token == g["bytes_per_token_per_layer"]
