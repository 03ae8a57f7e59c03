"""Seeded synthetic inputs for the paged KV-cache kernels.

This module only draws inputs: sequence lengths, physical block assignments
and the K/V/q values.  It holds none of the method's arithmetic (no slot
computation, no attention); the product's metadata builder and the oracle's
each derive slot_mapping / cu_seqlens from what is drawn here.  Both the GPU
tests and the oracle consume the exact tensors drawn here.

Workload shapes follow a Qwen3-0.6B-sized decoder layer (16 query heads,
8 KV heads, head_dim 128, bf16), the model of the benchmark table in
"3.6 ModelRunner, CUDA Graph, and benchmarks", section 7; the random token
streams of that benchmark are replaced by N(0, 1) activations.

Block assignment: a random permutation of the pool's block ids is drawn and
each sequence takes the next ceil(len / block_size) ids of it in order, so
sequences own disjoint, scattered blocks.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

QWEN3_06B = dict(num_q_heads=16, num_kv_heads=8, head_dim=128, num_layers=28)


@dataclasses.dataclass
class DecodeWorkload:
    """Structure of one decode batch (host-side lists, no tensors)."""

    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    dtype: torch.dtype
    context_lens: list[int]
    block_tables: list[list[int]]  # physical ids, exactly the blocks each context covers
    num_layers: int = 1
    big_key_fraction: float = 0.0  # fraction of (slot, kv head) key vectors scaled by big_key_scale
    big_key_scale: float = 8.0

    @property
    def batch(self) -> int:
        return len(self.context_lens)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def max_blocks_per_seq(self) -> int:
        return max((len(t) for t in self.block_tables), default=0)


@dataclasses.dataclass
class PrefillWorkload:
    """Structure of one varlen prefill / chunked-prefill batch."""

    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    dtype: torch.dtype
    num_cached: list[int]  # tokens already in the cache per sequence (prefix hit / earlier chunks)
    num_new: list[int]  # tokens computed in this scheduler step per sequence
    block_tables: list[list[int]]  # covers num_cached + num_new tokens

    @property
    def batch(self) -> int:
        return len(self.num_new)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def max_blocks_per_seq(self) -> int:
        return max((len(t) for t in self.block_tables), default=0)


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def _assign_blocks(rng: np.random.Generator, lengths: list[int], block_size: int,
                   num_blocks: int) -> list[list[int]]:
    perm = rng.permutation(num_blocks).tolist()
    tables = []
    pos = 0
    for n in lengths:
        k = _ceil_div(n, block_size)
        if pos + k > num_blocks:
            raise ValueError("pool too small for the drawn lengths")
        tables.append(perm[pos:pos + k])
        pos += k
    return tables


# ---------------------------------------------------------------- decode configs

def tiny_decode(seed: int = 1001) -> DecodeWorkload:
    """4 sequences, contexts [10, 17, 33, 64], block_size 4, 8q/2kv heads, d=64, fp32, 64-block pool."""
    rng = np.random.default_rng(seed)
    lens = [10, 17, 33, 64]
    tables = _assign_blocks(rng, lens, 4, 64)
    return DecodeWorkload("tiny-decode-b4-bs4-fp32", seed, 8, 2, 64, 4, 64, torch.float32, lens, tables)


def qwen3_decode_b32(seed: int = 1002) -> DecodeWorkload:
    """Batch 32, contexts uniform in [128, 2048], block_size 256, 512-block pool, bf16."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(128, 2048, size=32, endpoint=True).tolist()
    tables = _assign_blocks(rng, lens, 256, 512)
    return DecodeWorkload("qwen3-0.6b-decode-b32-ctx128-2048", seed, 16, 8, 128, 256, 512,
                          torch.bfloat16, lens, tables)


def qwen3_decode_b256_28l(seed: int = 1003, batch: int = 256, num_layers: int = 28) -> DecodeWorkload:
    """Batch 256, contexts uniform in [1024, 8192], block_size 256, 28 layers of separate pools.

    Each layer's pool holds exactly the blocks the batch needs; one block
    table per sequence indexes every layer's pool, as in the pages' per-layer
    slices of one cache tensor ("3.6 ModelRunner ...", section 4).
    """
    rng = np.random.default_rng(seed)
    lens = rng.integers(1024, 8192, size=batch, endpoint=True).tolist()
    num_blocks = sum(_ceil_div(n, 256) for n in lens)
    tables = _assign_blocks(rng, lens, 256, num_blocks)
    return DecodeWorkload(f"qwen3-0.6b-decode-b{batch}-ctx1k-8k-{num_layers}layers", seed, 16, 8, 128, 256,
                          num_blocks, torch.bfloat16, lens, tables, num_layers=num_layers)


def long_context_decode(seed: int = 1005) -> DecodeWorkload:
    """Batch 4, contexts [32768, 65536, 100000, 131072], block_size 16, 32q/8kv, 40000-block pool,
    1% of key vectors scaled x8."""
    rng = np.random.default_rng(seed)
    lens = [32768, 65536, 100000, 131072]
    tables = _assign_blocks(rng, lens, 16, 40000)
    return DecodeWorkload("long-context-decode-b4-ctx32k-131k-bs16", seed, 32, 8, 128, 16, 40000,
                          torch.bfloat16, lens, tables, big_key_fraction=0.01)


def random_decode(seed: int, *, batch: int, max_ctx: int, block_size: int, num_q_heads: int,
                  num_kv_heads: int, head_dim: int, dtype: torch.dtype, min_ctx: int = 0,
                  spare_blocks: int = 8) -> DecodeWorkload:
    """Small randomised decode batch for sweeps (contexts uniform in [min_ctx, max_ctx])."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(min_ctx, max_ctx, size=batch, endpoint=True).tolist()
    num_blocks = sum(_ceil_div(n, block_size) for n in lens) + spare_blocks
    tables = _assign_blocks(rng, lens, block_size, num_blocks)
    return DecodeWorkload(f"random-decode-s{seed}", seed, num_q_heads, num_kv_heads, head_dim,
                          block_size, num_blocks, dtype, lens, tables)


# ---------------------------------------------------------------- prefill configs

def qwen3_prefill_prefix(seed: int = 1004, batch: int = 16, chunk: int = 512) -> PrefillWorkload:
    """16 sequences of total length uniform in [256, 4096]; a random multiple of the block size
    (0 to half the length) is already cached; up to ``chunk`` new tokens per sequence in this step."""
    rng = np.random.default_rng(seed)
    bs = 256
    lens = rng.integers(256, 4096, size=batch, endpoint=True).tolist()
    cached = [bs * int(rng.integers(0, (n // 2) // bs, endpoint=True)) for n in lens]
    new = [min(chunk, n - c) for n, c in zip(lens, cached)]
    covered = [c + m for c, m in zip(cached, new)]
    num_blocks = 2 * sum(_ceil_div(n, bs) for n in covered)
    tables = _assign_blocks(rng, covered, bs, num_blocks)
    return PrefillWorkload(f"qwen3-0.6b-prefill-b{batch}-prefix-chunk{chunk}", seed, 16, 8, 128, bs,
                           num_blocks, torch.bfloat16, cached, new, tables)


def long_history_prefill(seed: int = 1006, history: int = 16384, chunk: int = 512) -> PrefillWorkload:
    """One sequence resuming after a long cached history (chunked prefill of a long document):
    ``history`` tokens cached (a multiple of 256), ``chunk`` new tokens, Qwen3-0.6B heads, block size 256."""
    rng = np.random.default_rng(seed)
    bs = 256
    n = history + chunk
    num_blocks = 2 * _ceil_div(n, bs)
    tables = _assign_blocks(rng, [n], bs, num_blocks)
    return PrefillWorkload(f"qwen3-0.6b-prefill-b1-history{history // 1024}k-chunk{chunk}", seed, 16, 8, 128, bs,
                           num_blocks, torch.bfloat16, [history], [chunk], tables)


def random_prefill(seed: int, *, batch: int, max_new: int, max_cached_blocks: int, block_size: int,
                   num_q_heads: int, num_kv_heads: int, head_dim: int, dtype: torch.dtype = torch.bfloat16,
                   min_new: int = 0, spare_blocks: int = 4) -> PrefillWorkload:
    """Small randomised prefill batch: cached = block_size * U{0..max_cached_blocks}, new = U{min_new..max_new}."""
    rng = np.random.default_rng(seed)
    cached = [block_size * int(rng.integers(0, max_cached_blocks, endpoint=True)) for _ in range(batch)]
    new = rng.integers(min_new, max_new, size=batch, endpoint=True).tolist()
    covered = [c + m for c, m in zip(cached, new)]
    num_blocks = sum(_ceil_div(n, block_size) for n in covered) + spare_blocks
    tables = _assign_blocks(rng, covered, block_size, num_blocks)
    return PrefillWorkload(f"random-prefill-s{seed}", seed, num_q_heads, num_kv_heads, head_dim, block_size,
                           num_blocks, dtype, cached, new, tables)


# ---------------------------------------------------------------- tensors

def _randn(gen: torch.Generator, shape, device, dtype) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def _poison_unused(pool: torch.Tensor, tables: list[list[int]], valid: list[int], block_size: int) -> None:
    """NaN into every block no table references and into every slot of a sequence's
    blocks at a logical position >= valid[b]."""
    used = torch.zeros(pool.shape[0], dtype=torch.bool)
    for table in tables:
        used[table] = True
    pool[(~used).to(pool.device)] = float("nan")
    for table, n in zip(tables, valid):
        for j, block in enumerate(table):
            first = j * block_size
            if first >= n:
                pool[block] = float("nan")
            elif first + block_size > n:
                pool[block, n - first:] = float("nan")


def decode_tensors(wl: DecodeWorkload, device="cpu", layer: int = 0, poison: bool = False) -> dict:
    """Draw q, the new token's k/v and the K/V pools of one layer.

    Returns q [B, Hq, D], k_new / v_new [B, Hkv, D] (the token at position
    context_len - 1 of each sequence, to be stored before attention), and
    k_cache / v_cache [num_blocks, block_size, Hkv, D] holding the history.
    With ``poison`` every cache entry outside the sequences' contexts is NaN.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed * 1000 + layer)
    B, Hq, Hkv, D = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    pool_shape = (wl.num_blocks, wl.block_size, Hkv, D)
    q = _randn(gen, (B, Hq, D), device, wl.dtype)
    k_new = _randn(gen, (B, Hkv, D), device, wl.dtype)
    v_new = _randn(gen, (B, Hkv, D), device, wl.dtype)
    if wl.big_key_fraction > 0:
        k32 = torch.randn(pool_shape, generator=gen, device=device, dtype=torch.float32)
        big = torch.rand((wl.num_blocks, wl.block_size, Hkv, 1), generator=gen, device=device) < wl.big_key_fraction
        k32 = torch.where(big, k32 * wl.big_key_scale, k32)
        k_cache = k32.to(wl.dtype)
        del k32
        kn32 = torch.randn((B, Hkv, D), generator=gen, device=device)
        bign = torch.rand((B, Hkv, 1), generator=gen, device=device) < wl.big_key_fraction
        k_new = torch.where(bign, kn32 * wl.big_key_scale, kn32).to(wl.dtype)
    else:
        k_cache = _randn(gen, pool_shape, device, wl.dtype)
    v_cache = _randn(gen, pool_shape, device, wl.dtype)
    if poison:
        _poison_unused(k_cache, wl.block_tables, wl.context_lens, wl.block_size)
        _poison_unused(v_cache, wl.block_tables, wl.context_lens, wl.block_size)
    return dict(q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache)


def prefill_tensors(wl: PrefillWorkload, device="cpu", poison: bool = False) -> dict:
    """Draw q / k / v for this step's tokens (packed [total_q, H, D]) and the cache pools.

    The cache holds N(0, 1) history for every sequence's cached prefix; the
    new rows k, v are to be stored through slot_mapping before attention.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed * 1000)
    total_q = sum(wl.num_new)
    Hq, Hkv, D = wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    q = _randn(gen, (total_q, Hq, D), device, wl.dtype)
    k = _randn(gen, (total_q, Hkv, D), device, wl.dtype)
    v = _randn(gen, (total_q, Hkv, D), device, wl.dtype)
    pool_shape = (wl.num_blocks, wl.block_size, Hkv, D)
    k_cache = _randn(gen, pool_shape, device, wl.dtype)
    v_cache = _randn(gen, pool_shape, device, wl.dtype)
    if poison:
        # positions from num_cached on are written by the store: poison them so a missing store shows
        _poison_unused(k_cache, wl.block_tables, wl.num_cached, wl.block_size)
        _poison_unused(v_cache, wl.block_tables, wl.num_cached, wl.block_size)
    return dict(q=q, k=k, v=v, k_cache=k_cache, v_cache=v_cache)


def verify_tensors(wl: DecodeWorkload, q_len: int, device="cpu", layer: int = 0) -> dict:
    """Draw the inputs of one speculative-decoding verify pass.

    q [B, q_len, Hq, D] holds the last q_len positions of each context; k_new /
    v_new [B * q_len, Hkv, D] are their K/V rows (sequence-major), to be stored
    before attention; the caches hold the history as in decode_tensors.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed * 1000 + 500 + layer)
    B, Hq, Hkv, D = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    pool_shape = (wl.num_blocks, wl.block_size, Hkv, D)
    return dict(q=_randn(gen, (B, q_len, Hq, D), device, wl.dtype),
                k_new=_randn(gen, (B * q_len, Hkv, D), device, wl.dtype),
                v_new=_randn(gen, (B * q_len, Hkv, D), device, wl.dtype),
                k_cache=_randn(gen, pool_shape, device, wl.dtype),
                v_cache=_randn(gen, pool_shape, device, wl.dtype))
