"""bench.py's algorithmic work per launch (the roofline numerators), CPU only: the stated
figures for the bench workloads, and brute-force counts on small cases."""

import bench
from pagedattention_kv_cache_gb300 import workloads as wl


def test_decode_bytes_of_the_bench_launch():
    w = wl.qwen3_decode_b256_28l()
    ctx = sum(w.context_lens)
    assert ctx == 1_174_899
    per_token = 8 * 128 * 2 * 2  # K and V rows of all KV heads, bf16
    assert per_token == 4096
    q_out = 2 * 256 * 16 * 128 * 2
    table_entries = sum(-(-n // 256) for n in w.context_lens)
    assert bench.decode_alg_bytes(w) == ctx * per_token + q_out + 4 * table_entries + 4 * 256
    assert bench.decode_alg_bytes(w) == 4_814_503_340


def test_fp8_decode_bytes_are_one_byte_per_element():
    w = wl.qwen3_decode_b256_28l()
    assert bench.decode_alg_bytes(w) - bench.decode_alg_bytes_fp8(w) == sum(w.context_lens) * 8 * 128 * 2


def test_store_bytes_per_token():
    w = wl.qwen3_decode_b256_28l()
    assert bench.store_alg_bytes(1, w) == 8196  # K and V rows read and written, plus the slot


def test_prefill_flops_brute_force():
    p = wl.random_prefill(3, batch=5, max_new=40, max_cached_blocks=3, block_size=16, num_q_heads=4,
                          num_kv_heads=2, head_dim=64)
    pairs = 0
    for c, n in zip(p.num_cached, p.num_new):
        for r in range(n):  # query row r sits at position c + r and sees keys 0 .. c + r
            for t in range(c + n):
                pairs += t <= c + r
    assert bench.prefill_flops(p) == 4 * 64 * 4 * pairs  # QK^T and PV: 2 FLOPs each per (row, key, dim)


def test_prefill_flops_of_the_bench_batch():
    assert bench.prefill_flops(wl.qwen3_prefill_prefix()) == 34_667_020_288
