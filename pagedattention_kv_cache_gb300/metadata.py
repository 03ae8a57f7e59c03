"""Host-side metadata the kernels consume, built from per-sequence block tables.

The product's own builder (the engine-side step of "3.6 ModelRunner, CUDA
Graph, and benchmarks", section 2): it turns sequences into the int32 arrays
kv_store / paged_decode_attn / paged_varlen_prefill_attn take, vectorised
with numpy.  Section 5's graph-replay padding (slot -1, context length 0)
is available through ``pad_decode``.
"""

from __future__ import annotations

import numpy as np
import torch


def table_matrix(tables: list[list[int]], width: int | None = None) -> np.ndarray:
    """Stack block tables into an int32 [B, W] matrix right-padded with -1."""
    w = max((len(t) for t in tables), default=0) if width is None else width
    mat = np.full((len(tables), max(w, 1)), -1, dtype=np.int32)
    for i, t in enumerate(tables):
        mat[i, :len(t)] = t
    return mat


def prefill_metadata(block_tables: list[list[int]], num_cached: list[int], num_new: list[int],
                     block_size: int, table_width: int | None = None, always_tables: bool = False) -> dict:
    """slot_mapping / cu_seqlens_q / cu_seqlens_k / max_seqlen_* / block_tables for a packed prefill.

    Tokens [num_cached[i], num_cached[i] + num_new[i]) of sequence i are
    computed in this scheduler step; the K side runs from 0.  block_tables is None when
    no sequence has history (then the kernel reads this step's k, v), unless
    ``always_tables`` asks for it anyway (attention then reads the stored rows).
    """
    cached = np.asarray(num_cached, dtype=np.int64)
    new = np.asarray(num_new, dtype=np.int64)
    cu_q = np.zeros(len(new) + 1, dtype=np.int32)
    cu_k = np.zeros(len(new) + 1, dtype=np.int32)
    np.cumsum(new, out=cu_q[1:])
    np.cumsum(cached + new, out=cu_k[1:])
    slots = []
    for table, c, n in zip(block_tables, cached, new):
        if not table:
            continue
        pos = np.arange(c, c + n, dtype=np.int64)
        tab = np.asarray(table, dtype=np.int64)
        slots.append(tab[pos // block_size] * block_size + pos % block_size)
    slot_mapping = np.concatenate(slots).astype(np.int32) if slots else np.zeros(0, dtype=np.int32)
    need = bool(cu_k[-1] > cu_q[-1])
    return {
        "slot_mapping": slot_mapping,
        "cu_seqlens_q": cu_q,
        "cu_seqlens_k": cu_k,
        "max_seqlen_q": int(new.max()) if len(new) else 0,
        "max_seqlen_k": int((cached + new).max()) if len(new) else 0,
        "need_block_tables": need,
        "block_tables": table_matrix(block_tables, table_width) if (need or always_tables) else None,
    }


def decode_metadata(block_tables: list[list[int]], lengths: list[int], block_size: int,
                    table_width: int | None = None) -> dict:
    """slot_mapping / context_lens / block_tables for one decode step.

    ``lengths`` count the new token.  Its slot is at position length - 1, in
    the last block of the table, so every table must hold exactly
    ceil(length / block_size) blocks (none for a length-0 padding row): with a
    longer table the last entry would not be the block of position length - 1.
    A table of another length raises ValueError.
    """
    if block_size <= 0:
        raise ValueError("block_size must be positive")
    if len(block_tables) != len(lengths):
        raise ValueError("one block table per sequence is required")
    lens = np.asarray(lengths, dtype=np.int64)
    if lens.size and lens.min() < 0:
        raise ValueError("lengths must be non-negative")
    n_blocks = np.array([len(t) for t in block_tables], dtype=np.int64)
    bad = np.flatnonzero(n_blocks != -(-lens // block_size))
    if bad.size:
        b = int(bad[0])
        raise ValueError(f"sequence {b}: length {int(lens[b])} needs {-(-int(lens[b]) // block_size)} blocks of "
                         f"{block_size}, its table has {int(n_blocks[b])}")
    last = np.array([t[-1] if t else -1 for t in block_tables], dtype=np.int64)
    in_last = lens - (n_blocks - 1) * block_size
    slots = np.where(lens > 0, last * block_size + in_last - 1, -1).astype(np.int32)
    return {
        "slot_mapping": slots,
        "context_lens": lens.astype(np.int32),
        "block_tables": table_matrix(block_tables, table_width),
    }


def pad_decode(md: dict, batch: int) -> dict:
    """Pad decode metadata to ``batch`` rows: slot -1 (no write) and context length 0 (no read)."""
    n = len(md["context_lens"])
    if batch < n:
        raise ValueError("cannot pad to a smaller batch")
    slots = np.full(batch, -1, dtype=np.int32)
    slots[:n] = md["slot_mapping"]
    lens = np.zeros(batch, dtype=np.int32)
    lens[:n] = md["context_lens"]
    tables = np.full((batch, md["block_tables"].shape[1]), -1, dtype=np.int32)
    tables[:n] = md["block_tables"]
    return {"slot_mapping": slots, "context_lens": lens, "block_tables": tables}


def to_device(md: dict, device) -> dict:
    """Copy every numpy array of a metadata dict to an int32 tensor on ``device``."""
    return {k: (torch.from_numpy(np.ascontiguousarray(v)).to(device) if isinstance(v, np.ndarray) else v)
            for k, v in md.items()}
