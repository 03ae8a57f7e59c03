"""Oracle for the paged KV-cache kernels, in float64 numpy.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Paging moves K/V rows around, it does not change the result: attention over a
paged cache equals attention over the same tokens stored contiguously
("Warmup Guide -- Inference Serving Internals", chapter 3: reads gather
through the block table in logical order).  So every function here gathers
the logical K/V rows explicitly, then computes plain softmax attention
softmax(scale * q K^T) V with query head h reading KV head h // (Hq / Hkv).

Cache layout for one layer ("3.6 ModelRunner, CUDA Graph, and benchmarks",
section 4): k_cache and v_cache are [num_blocks, block_size, num_kv_heads,
head_dim]; logical token t of a sequence lives in physical block
block_table[t // block_size] at offset t % block_size.
"""

from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def kv_store(k_cache, v_cache, k, v, slot_mapping):
    """Scatter new K/V rows into the paged cache; returns updated copies.

    "3.6 ModelRunner ...", sections 2 and 5: row i goes to slot
    slot_mapping[i] = block_id * block_size + offset, and a slot of -1 (batch
    padding) writes nothing.  A pure element copy in the arrays' own dtype,
    so bf16 data passed as raw 16-bit integers is copied bit for bit.

    k_cache, v_cache: [num_blocks, block_size, Hkv, D]; k, v: [N, Hkv, D].
    """
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    block_size = k_out.shape[1]
    num_slots = k_out.shape[0] * block_size
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot == -1:
            continue
        if not 0 <= slot < num_slots:
            raise IndexError(f"slot {slot} outside the cache ({num_slots} slots)")
        block, offset = divmod(slot, block_size)
        k_out[block, offset] = k[i]
        v_out[block, offset] = v[i]
    return k_out, v_out


def gather_tokens(cache, block_table, num_tokens: int) -> np.ndarray:
    """Logical rows 0..num_tokens-1 of one sequence: [num_tokens, Hkv, D].

    Only the first blocks_needed(num_tokens) table entries are dereferenced;
    padding (-1) or stale ids further right are never touched.
    """
    block_size = cache.shape[1]
    rows = []
    for t in range(num_tokens):
        block = int(block_table[t // block_size])
        if not 0 <= block < cache.shape[0]:
            raise IndexError(f"block id {block} outside the pool")
        rows.append(cache[block, t % block_size])
    if not rows:
        return np.zeros((0,) + tuple(cache.shape[2:]), dtype=np.float64)
    return _f64(np.stack(rows))


def softmax_attention_rows(q_rows, keys, values, scale: float, visible=None):
    """Plain attention for a block of query rows against one head's keys.

    q_rows: [R, D]; keys, values: [T, D]; visible: optional bool [R, T] mask
    (True = the query row may attend that key).  Each row's scores are
    s = scale * q . k; the row's output is sum_t softmax(s)_t v_t, computed
    with the row maximum subtracted before exp (exact in real arithmetic).
    """
    q_rows = _f64(q_rows)
    keys = _f64(keys)
    values = _f64(values)
    scores = scale * (q_rows @ keys.T)
    if visible is not None:
        scores = np.where(visible, scores, -np.inf)
    m = scores.max(axis=1, keepdims=True)
    p = np.exp(scores - m)
    return (p @ values) / p.sum(axis=1, keepdims=True)


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale: float):
    """Decode attention through block tables (one query token per sequence).

    q: [B, Hq, D]; block_tables: [B, W]; context_lens: [B] counts the token just
    stored ("3.6 ModelRunner ...", section 2).  A sequence with context length
    0 (graph-replay padding, section 5) reads nothing; its output is defined
    as 0.  Returns float64 [B, Hq, D].
    """
    q = _f64(q)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    group = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        ctx = int(context_lens[b])
        if ctx == 0:
            continue
        keys = gather_tokens(k_cache, block_tables[b], ctx)
        values = gather_tokens(v_cache, block_tables[b], ctx)
        for h in range(Hq):
            g = h // group
            out[b, h] = softmax_attention_rows(q[b, h][None, :], keys[:, g], values[:, g], scale)[0]
    return out


def decode_partials(q, k_cache, v_cache, block_tables, context_lens, scale: float, bounds):
    """Per-partition softmax state for split-K decode.

    bounds[b] is a list of token boundaries 0 = t_0 < t_1 < ... < t_S = ctx_b.
    For each partition j and head h returns (o_j, m_j, l_j): m_j the maximum
    score over the partition, l_j = sum exp(s - m_j) and o_j = sum exp(s - m_j) v
    (not yet divided by l_j).  Returns a list over b of lists over j of tuples
    of arrays shaped [Hq, D], [Hq], [Hq].
    """
    q = _f64(q)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    group = Hq // Hkv
    result = []
    for b in range(B):
        ctx = int(context_lens[b])
        keys = gather_tokens(k_cache, block_tables[b], ctx)
        values = gather_tokens(v_cache, block_tables[b], ctx)
        parts = []
        edges = list(bounds[b])
        for lo, hi in zip(edges[:-1], edges[1:]):
            o = np.zeros((Hq, D))
            m = np.full(Hq, -np.inf)
            l = np.zeros(Hq)
            for h in range(Hq):
                g = h // group
                s = scale * (keys[lo:hi, g] @ q[b, h])
                m[h] = s.max()
                p = np.exp(s - m[h])
                l[h] = p.sum()
                o[h] = p @ values[lo:hi, g]
            parts.append((o, m, l))
        result.append(parts)
    return result


def combine_partials(parts):
    """Merge partition states of one sequence by log-sum-exp rescaling.

    With M = max_j m_j and w_j = exp(m_j - M):  L = sum_j w_j l_j and the
    output is sum_j w_j o_j / L.  Returns float64 [Hq, D].
    """
    ms = np.stack([p[1] for p in parts])  # [S, Hq]
    big_m = ms.max(axis=0)
    w = np.exp(ms - big_m)  # [S, Hq]
    total_l = sum(w[j] * parts[j][2] for j in range(len(parts)))
    total_o = sum(w[j][:, None] * parts[j][0] for j in range(len(parts)))
    return total_o / total_l[:, None]


def paged_prefill_attention(q, cu_seqlens_q, cu_seqlens_k, scale: float, *, k_cache=None,
                            v_cache=None, block_tables=None, k=None, v=None, causal: bool = True):
    """Varlen (packed) prefill / chunked-prefill attention.

    "3.6 ModelRunner ...", section 2: sequence i owns query rows
    cu_seqlens_q[i]..cu_seqlens_q[i+1]-1 (the tokens computed in this scheduler step) and
    its keys span positions 0..nk-1 with nk = cu_seqlens_k[i+1] - cu_seqlens_k[i].
    The first c = nk - nq keys are history (prefix-cache hit or an earlier
    chunk); query row r sits at absolute position c + r and, when causal,
    attends keys 0..c + r.

    With block_tables given, all nk keys are gathered from the paged cache
    (the new rows having been stored there first).  Without, keys come from
    the packed k, v arrays at rows cu_seqlens_k[i]..cu_seqlens_k[i+1]-1.

    q: [total_q, Hq, D]; returns float64 [total_q, Hq, D].
    """
    q = _f64(q)
    total_q, Hq, D = q.shape
    B = len(cu_seqlens_q) - 1
    out = np.zeros((total_q, Hq, D), dtype=np.float64)
    for i in range(B):
        q0, q1 = int(cu_seqlens_q[i]), int(cu_seqlens_q[i + 1])
        k0, k1 = int(cu_seqlens_k[i]), int(cu_seqlens_k[i + 1])
        nq, nk = q1 - q0, k1 - k0
        if nq == 0:
            continue
        cached = nk - nq
        if cached < 0:
            raise ValueError("a sequence cannot have more query rows than keys")
        if block_tables is not None:
            keys = gather_tokens(k_cache, block_tables[i], nk)
            values = gather_tokens(v_cache, block_tables[i], nk)
        else:
            keys = _f64(k[k0:k1])
            values = _f64(v[k0:k1])
        Hkv = keys.shape[1]
        group = Hq // Hkv
        visible = None
        if causal:
            rows = np.arange(nq)[:, None]
            cols = np.arange(nk)[None, :]
            visible = cols <= cached + rows
        for h in range(Hq):
            g = h // group
            out[q0:q1, h] = softmax_attention_rows(q[q0:q1, h], keys[:, g], values[:, g], scale, visible)
    return out


def copy_blocks(caches, pairs):
    """Copy-on-write block copy: for every (src, dst) pair, block dst of every cache
    becomes a copy of block src; returns updated copies.

    "Warmup Guide -- Inference Serving Internals", chapter 4: a sequence about
    to write into a block it shares copies that one block first and writes
    into its private copy.  caches: list of [num_blocks, ...] arrays (K and V
    of every layer); pairs: [n, 2] with no destination also used as a source.
    """
    out = [np.array(c, copy=True) for c in caches]
    for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
        for c, orig in zip(out, caches):
            c[dst] = orig[src]
    return out
