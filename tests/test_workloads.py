"""The seeded synthetic workloads follow the stated recipe (CPU only): sizes, head
shapes, length ranges, prefix-hit rules and disjoint block tables drawn from the pool."""

import math

import pytest
import torch

from pagedattention_kv_cache_gb300 import workloads as wl


def _check_tables(w, lengths):
    used = [b for t in w.block_tables for b in t]
    assert len(used) == len(set(used)), "a physical block is shared between sequences"
    assert all(0 <= b < w.num_blocks for b in used)
    for t, n in zip(w.block_tables, lengths):
        assert len(t) == math.ceil(n / w.block_size)
    return used


def test_tiny_decode():
    w = wl.tiny_decode()
    assert w.context_lens == [10, 17, 33, 64]
    assert (w.block_size, w.num_blocks, w.num_q_heads, w.num_kv_heads, w.head_dim) == (4, 64, 8, 2, 64)
    assert w.dtype == torch.float32
    _check_tables(w, w.context_lens)


def test_qwen3_decode_batch32():
    w = wl.qwen3_decode_b32()
    assert len(w.context_lens) == 32 and all(128 <= n <= 2048 for n in w.context_lens)
    assert (w.block_size, w.num_blocks, w.num_q_heads, w.num_kv_heads, w.head_dim) == (256, 512, 16, 8, 128)
    assert w.dtype == torch.bfloat16
    _check_tables(w, w.context_lens)


def test_qwen3_decode_batch256_28_layers():
    w = wl.qwen3_decode_b256_28l()
    assert w.num_layers == 28 and len(w.context_lens) == 256
    assert all(1024 <= n <= 8192 for n in w.context_lens)
    assert (w.block_size, w.num_q_heads, w.num_kv_heads, w.head_dim) == (256, 16, 8, 128)
    used = _check_tables(w, w.context_lens)
    assert sorted(used) == list(range(w.num_blocks))  # the pool holds exactly the needed blocks, permuted
    assert used != sorted(used)


def test_long_context_decode():
    w = wl.long_context_decode()
    assert w.context_lens == [32768, 65536, 100000, 131072]
    assert (w.block_size, w.num_blocks, w.num_q_heads, w.num_kv_heads, w.head_dim) == (16, 40000, 32, 8, 128)
    assert w.big_key_fraction == pytest.approx(0.01) and w.big_key_scale == 8.0
    _check_tables(w, w.context_lens)


def test_qwen3_prefill_with_prefix_hits():
    w = wl.qwen3_prefill_prefix()
    assert w.batch == 16 and w.block_size == 256
    assert (w.num_q_heads, w.num_kv_heads, w.head_dim) == (16, 8, 128)
    for c, m in zip(w.num_cached, w.num_new):
        assert c % 256 == 0
        assert 1 <= m <= 512
    # the drawn total length n satisfies 256 <= n <= 4096 and c <= n / 2; new = min(512, n - c)
    assert any(c > 0 for c in w.num_cached) and any(m == 512 for m in w.num_new)
    assert all(c + m <= 4096 for c, m in zip(w.num_cached, w.num_new))
    _check_tables(w, [c + m for c, m in zip(w.num_cached, w.num_new)])


def test_long_history_prefill():
    w = wl.long_history_prefill()
    assert w.num_cached == [16384] and w.num_new == [512]
    _check_tables(w, [16896])


def test_seeded_and_reproducible():
    a, b = wl.qwen3_decode_b32(), wl.qwen3_decode_b32()
    assert a.context_lens == b.context_lens and a.block_tables == b.block_tables
    c = wl.qwen3_decode_b32(seed=7)
    assert c.context_lens != a.context_lens


def test_tiny_decode_tensors_on_cpu():
    w = wl.tiny_decode()
    t = wl.decode_tensors(w, "cpu")
    assert t["q"].shape == (4, 8, 64)
    assert t["k_cache"].shape == (64, 4, 2, 64) and t["v_cache"].shape == (64, 4, 2, 64)
    again = wl.decode_tensors(w, "cpu")
    assert torch.equal(t["q"], again["q"]) and torch.equal(t["k_cache"], again["k_cache"])
