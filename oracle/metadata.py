"""Oracle for the host-side metadata the paged kernels consume.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources:
* "3.6 ModelRunner, CUDA Graph, and benchmarks", section 2 "Turning sequences
  into tensors": prefill packs each sequence's tokens [start, end) with
  start = num_cached_tokens and end = start + num_scheduled_tokens; positions
  continue from start; cu_seqlens_q grows by end - start, cu_seqlens_k by end;
  each computed token i gets slot block_table[i // block_size] * block_size
  + i % block_size; block_tables are needed iff the K side is longer than the
  Q side.  Decode takes one token per sequence at position len - 1, its slot
  is in the last block of the table at offset last_block_num_tokens - 1, and
  context_lens counts the new token.  Block tables are right-padded with -1.
* "Warmup Guide -- Inference Serving Internals", chapter 3 "PagedAttention":
  blocks_needed is ceil division, and growing a sequence by one token takes a
  new block iff its length is an exact multiple of block_size.
"""

from __future__ import annotations

import numpy as np


def blocks_needed(num_tokens: int, block_size: int) -> int:
    """Number of fixed-size blocks that hold ``num_tokens`` tokens (ceil division).

    Warmup Guide, chapter 3: 8 tokens in blocks of 4 need 2 blocks; the 9th
    token needs a third.
    """
    if block_size <= 0 or num_tokens < 0:
        raise ValueError("block_size must be positive and num_tokens non-negative")
    count = 0
    covered = 0
    while covered < num_tokens:  # one block at a time: no arithmetic shortcut
        count += 1
        covered += block_size
    return count


def append_needs_block(length: int, block_size: int) -> bool:
    """Whether appending one token to a sequence of ``length`` tokens takes a new block.

    Warmup Guide, chapter 3: a new block is needed iff the last block is
    exactly full, i.e. the current length is a multiple of the block size.
    """
    return length % block_size == 0


def padded_block_tables(tables: list[list[int]], width: int | None = None) -> np.ndarray:
    """Stack per-sequence block tables into an int32 matrix right-padded with -1.

    "3.6 ModelRunner ...", section 2: the -1 padding only aligns the matrix;
    kernels read the leading blocks that context_lens (or cu_seqlens_k) cover.
    """
    if width is None:
        width = max((len(t) for t in tables), default=0)
    out = np.full((len(tables), width), -1, dtype=np.int32)
    for b, table in enumerate(tables):
        out[b, : len(table)] = table
    return out


def prepare_prefill(seqs: list[dict], block_size: int) -> dict:
    """Prefill metadata for packed variable-length sequences.

    Each ``seq`` is a dict with ``block_table`` (list of physical block ids),
    ``num_cached_tokens`` and ``num_scheduled_tokens``.  Follows section 2 of
    "3.6 ModelRunner, CUDA Graph, and benchmarks", token by token.

    Returns slot_mapping (int32 [total_q]), positions (int64 [total_q]),
    cu_seqlens_q / cu_seqlens_k (int32 [B+1]), max_seqlen_q, max_seqlen_k,
    need_block_tables (bool) and block_tables (int32 [B, W], -1 padded, or None).
    """
    slot_mapping: list[int] = []
    positions: list[int] = []
    cu_q = [0]
    cu_k = [0]
    max_q = 0
    max_k = 0
    for seq in seqs:
        start = seq["num_cached_tokens"]
        end = start + seq["num_scheduled_tokens"]
        positions.extend(range(start, end))
        cu_q.append(cu_q[-1] + (end - start))
        cu_k.append(cu_k[-1] + end)
        max_q = max(max_q, end - start)
        max_k = max(max_k, end)
        table = seq["block_table"]
        if not table:
            continue  # a sequence with no blocks writes nothing to the cache
        for i in range(start, end):
            block_id = table[i // block_size]
            slot_mapping.append(block_id * block_size + i % block_size)
    need_tables = cu_k[-1] > cu_q[-1]
    tables = padded_block_tables([s["block_table"] for s in seqs]) if need_tables else None
    return {
        "slot_mapping": np.asarray(slot_mapping, dtype=np.int32),
        "positions": np.asarray(positions, dtype=np.int64),
        "cu_seqlens_q": np.asarray(cu_q, dtype=np.int32),
        "cu_seqlens_k": np.asarray(cu_k, dtype=np.int32),
        "max_seqlen_q": max_q,
        "max_seqlen_k": max_k,
        "need_block_tables": bool(need_tables),
        "block_tables": tables,
    }


def prepare_decode(seqs: list[dict], block_size: int) -> dict:
    """Decode metadata: one new token per sequence, already counted in its length.

    Each ``seq`` is a dict with ``block_table`` and ``length`` (tokens including
    the new one).  Section 2 of "3.6 ModelRunner ...": the new token sits in
    the last block of the table, at offset last_block_num_tokens - 1, where
    last_block_num_tokens is how many of the sequence's tokens fall in that
    last block; context_lens is the full length.
    """
    slot_mapping = []
    positions = []
    context_lens = []
    for seq in seqs:
        length = seq["length"]
        table = seq["block_table"]
        if len(table) != blocks_needed(length, block_size):
            raise ValueError("decode expects exactly blocks_needed(length) blocks in the table")
        if length == 0:
            slot_mapping.append(-1)  # padding row (section 5): nothing stored, nothing read
        else:
            last_block_num_tokens = length - (len(table) - 1) * block_size
            slot_mapping.append(table[-1] * block_size + last_block_num_tokens - 1)
        positions.append(length - 1)
        context_lens.append(length)
    return {
        "slot_mapping": np.asarray(slot_mapping, dtype=np.int32),
        "positions": np.asarray(positions, dtype=np.int64),
        "context_lens": np.asarray(context_lens, dtype=np.int32),
        "block_tables": padded_block_tables([s["block_table"] for s in seqs]),
    }
