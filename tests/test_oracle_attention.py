"""Pins for the attention oracle (CPU only).

Each check ties the oracle to something other than itself: hand-computed
values, closed forms, a textbook contiguous attention built from
scipy.special.softmax, brute-force float64 loops, and invariants that hold by
the mathematics (block placement, prefix hits, chunking, split/combine).
"""

import json
import math
import os

import numpy as np
import pytest
from scipy.special import softmax

from oracle import attention as oa
from oracle import metadata as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _hand():
    with open(os.path.join(GOLDEN, "hand_attention.json")) as f:
        return json.load(f)


def _place(rng, contexts, block_size, hkv, d, spare=3, values=None):
    """Draw contiguous K/V per sequence and scatter them into a randomly permuted pool.

    Placement walks blocks in table order and fills offsets 0..block_size-1 (no
    slot formula), so it checks the oracle's gather by an independent route.
    """
    nblocks = [math.ceil(n / block_size) for n in contexts]
    num_blocks = sum(nblocks) + spare
    perm = rng.permutation(num_blocks)
    kc = rng.standard_normal((num_blocks, block_size, hkv, d)) if values is None else values(num_blocks)
    vc = rng.standard_normal((num_blocks, block_size, hkv, d))
    k_seq, v_seq, tables = [], [], []
    pos = 0
    for n, nb in zip(contexts, nblocks):
        ks = rng.standard_normal((n, hkv, d))
        vs = rng.standard_normal((n, hkv, d))
        table = perm[pos:pos + nb].tolist()
        pos += nb
        t = 0
        for blk in table:
            for off in range(block_size):
                if t < n:
                    kc[blk, off] = ks[t]
                    vc[blk, off] = vs[t]
                t += 1
        k_seq.append(ks)
        v_seq.append(vs)
        tables.append(table)
    return kc, vc, om.padded_block_tables(tables, max(nblocks) + 2), k_seq, v_seq


def _textbook(q, k, v, scale, causal_offset=None):
    """Contiguous attention with scipy's softmax; causal_offset c lets row r see keys <= c + r."""
    s = scale * q @ k.T
    if causal_offset is not None:
        r = np.arange(q.shape[0])[:, None]
        t = np.arange(k.shape[0])[None, :]
        s = np.where(t <= causal_offset + r, s, -np.inf)
    return softmax(s, axis=-1) @ v


# ------------------------------------------------------------------ hand values

def test_decode_hand_value():
    g = _hand()["decode_two_keys"]
    kc = np.zeros((2, 1, 1, 2))
    vc = np.zeros((2, 1, 1, 2))
    # block_size 1, the two tokens placed in reverse physical order
    kc[1, 0, 0], kc[0, 0, 0] = g["keys"]
    vc[1, 0, 0], vc[0, 0, 0] = g["values"]
    out = oa.paged_decode_attention(np.array(g["q"])[None, None], kc, vc, np.array([[1, 0]]),
                                    np.array([2]), g["scale"])
    np.testing.assert_allclose(out[0, 0], g["out"], rtol=0, atol=1e-12)


def test_prefill_hand_value_bottom_right_causal():
    g = _hand()["prefill_causal_bottom_right"]
    keys = np.array(g["keys"])[:, None, :]
    values = np.array(g["values"])[:, None, :]
    q = np.array(g["q"])[:, None, :]
    # paged: block_size 2, table [1, 0]
    kc = np.full((2, 2, 1, 2), np.nan)
    vc = np.full((2, 2, 1, 2), np.nan)
    kc[1, 0], kc[1, 1], kc[0, 0] = keys
    vc[1, 0], vc[1, 1], vc[0, 0] = values
    out = oa.paged_prefill_attention(q, [0, 2], [0, 3], g["scale"], k_cache=kc, v_cache=vc,
                                     block_tables=np.array([[1, 0]]))
    np.testing.assert_allclose(out[:, 0], g["out"], rtol=0, atol=1e-12)


def test_combine_hand_value():
    g = _hand()["combine_two_partitions"]
    parts = [(np.array([p["o"]]), np.array([p["m"]]), np.array([p["l"]])) for p in g["parts"]]
    np.testing.assert_allclose(oa.combine_partials(parts)[0], g["out"], rtol=0, atol=1e-12)


# ------------------------------------------------------------------ closed forms

def test_single_token_returns_its_value():
    rng = np.random.default_rng(1)
    kc, vc, bt, ks, vs = _place(rng, [1, 1], 4, 2, 8)
    q = rng.standard_normal((2, 4, 8))
    out = oa.paged_decode_attention(q, kc, vc, bt, np.array([1, 1]), 0.3)
    for b in range(2):
        for h in range(4):
            np.testing.assert_allclose(out[b, h], vs[b][0, h // 2], atol=1e-12)


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    kc, vc, bt, ks, vs = _place(rng, [13], 4, 1, 8)
    row = rng.standard_normal(8)
    for t in range(13):
        kc[bt[0, t // 4], t % 4, 0] = row
    q = rng.standard_normal((1, 1, 8))
    out = oa.paged_decode_attention(q, kc, vc, bt, np.array([13]), 0.7)
    np.testing.assert_allclose(out[0, 0], vs[0][:, 0].mean(axis=0), atol=1e-12)


def test_constant_values_pass_through():
    rng = np.random.default_rng(3)
    kc, vc, bt, ks, vs = _place(rng, [9, 30], 8, 2, 16)
    vc[:] = 2.5
    q = rng.standard_normal((2, 2, 16))
    out = oa.paged_decode_attention(q, kc, vc, bt, np.array([9, 30]), 0.25)
    np.testing.assert_allclose(out, 2.5, atol=1e-12)


def test_dominant_logit_selects_its_row():
    rng = np.random.default_rng(4)
    kc, vc, bt, ks, vs = _place(rng, [20], 4, 1, 8)
    q = np.zeros((1, 1, 8))
    q[0, 0, 0] = 1.0
    kc[..., 0] = 0.0
    kc[bt[0, 11 // 4], 11 % 4, 0, 0] = 100.0  # token 11 dominates by e^100
    out = oa.paged_decode_attention(q, kc, vc, bt, np.array([20]), 1.0)
    np.testing.assert_allclose(out[0, 0], vc[bt[0, 11 // 4], 11 % 4, 0], atol=1e-12)


def test_zero_context_gives_zero_and_reads_nothing():
    kc = np.full((2, 4, 1, 8), np.nan)
    out = oa.paged_decode_attention(np.ones((1, 1, 8)), kc, kc, np.array([[-1, -1]]), np.array([0]), 1.0)
    assert np.all(out == 0)


def test_gqa_contiguous_grouping():
    # 4 query heads over 2 KV heads: heads 0,1 read KV head 0 and heads 2,3 read KV head 1
    rng = np.random.default_rng(5)
    kc, vc, bt, ks, vs = _place(rng, [6], 2, 2, 4)
    vc[..., 0, :] = 1.0
    vc[..., 1, :] = -3.0
    q = rng.standard_normal((1, 4, 4))
    out = oa.paged_decode_attention(q, kc, vc, bt, np.array([6]), 1.0)
    np.testing.assert_allclose(out[0, :2], 1.0, atol=1e-12)
    np.testing.assert_allclose(out[0, 2:], -3.0, atol=1e-12)


# ------------------------------------------------------------------ textbook + brute force

@pytest.mark.parametrize("block_size", [1, 3, 4, 16])
@pytest.mark.parametrize("group", [1, 2, 4])
def test_decode_matches_textbook_contiguous(block_size, group):
    rng = np.random.default_rng(10 * block_size + group)
    hkv, d = 2, 8
    contexts = [1, 5, 17, 40]
    kc, vc, bt, ks, vs = _place(rng, contexts, block_size, hkv, d)
    q = rng.standard_normal((4, hkv * group, d))
    out = oa.paged_decode_attention(q, kc, vc, bt, np.array(contexts), 0.35)
    for b in range(4):
        for h in range(hkv * group):
            ref = _textbook(q[b, h][None], ks[b][:, h // group], vs[b][:, h // group], 0.35)[0]
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-12, atol=1e-12)


def _brute_force_row(qv, keys, values, scale):
    """float64 loops, no max subtraction (tiny inputs only)."""
    weights = []
    for kv in keys:
        dot = 0.0
        for a, b in zip(qv, kv):
            dot += a * b
        weights.append(math.exp(scale * dot))
    total = sum(weights)
    out = [0.0] * len(values[0])
    for w, vv in zip(weights, values):
        for j, x in enumerate(vv):
            out[j] += w * x
    return [x / total for x in out]


@pytest.mark.parametrize("block_size", [1, 2, 4, 16])
@pytest.mark.parametrize("group", [1, 2, 4])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_brute_force_tiny(block_size, group, d):
    rng = np.random.default_rng(block_size * 100 + group * 10 + d)
    contexts = list(range(1, 21, 3))
    kc, vc, bt, ks, vs = _place(rng, contexts, block_size, 1, d)
    q = rng.standard_normal((len(contexts), group, d))
    scale = 1 / math.sqrt(d)
    out = oa.paged_decode_attention(q, kc, vc, bt, np.array(contexts), scale)
    for b, n in enumerate(contexts):
        for h in range(group):
            ref = _brute_force_row(q[b, h].tolist(), ks[b][:, 0].tolist(), vs[b][:, 0].tolist(), scale)
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-10, atol=1e-12)


def test_prefill_matches_textbook_causal():
    rng = np.random.default_rng(20)
    cached = [0, 4, 8, 12]
    new = [5, 1, 7, 4]
    full = [c + n for c, n in zip(cached, new)]
    kc, vc, bt, ks, vs = _place(rng, full, 4, 2, 16)
    total = sum(new)
    q = rng.standard_normal((total, 4, 16))
    cu_q = np.concatenate([[0], np.cumsum(new)])
    cu_k = np.concatenate([[0], np.cumsum(full)])
    out = oa.paged_prefill_attention(q, cu_q, cu_k, 0.5, k_cache=kc, v_cache=vc, block_tables=bt)
    for i in range(4):
        for h in range(4):
            ref = _textbook(q[cu_q[i]:cu_q[i + 1], h], ks[i][:, h // 2], vs[i][:, h // 2], 0.5,
                            causal_offset=cached[i])
            np.testing.assert_allclose(out[cu_q[i]:cu_q[i + 1], h], ref, rtol=1e-12, atol=1e-12)


def test_prefill_no_history_packed_path():
    rng = np.random.default_rng(21)
    new = [3, 9, 1]
    total = sum(new)
    q = rng.standard_normal((total, 2, 8))
    k = rng.standard_normal((total, 1, 8))
    v = rng.standard_normal((total, 1, 8))
    cu = np.concatenate([[0], np.cumsum(new)])
    out = oa.paged_prefill_attention(q, cu, cu, 0.4, k=k, v=v)
    for i in range(3):
        sl = slice(cu[i], cu[i + 1])
        for h in range(2):
            ref = _textbook(q[sl, h], k[sl, 0], v[sl, 0], 0.4, causal_offset=0)
            np.testing.assert_allclose(out[sl, h], ref, rtol=1e-12, atol=1e-12)


def test_prefill_non_causal_matches_textbook_full():
    # causal=False: every query row of a sequence attends all nk keys, history and new alike
    rng = np.random.default_rng(22)
    cached = [0, 4, 9]
    new = [6, 3, 2]
    full = [c + n for c, n in zip(cached, new)]
    kc, vc, bt, ks, vs = _place(rng, full, 4, 2, 8)
    q = rng.standard_normal((sum(new), 4, 8))
    cu_q = np.concatenate([[0], np.cumsum(new)])
    cu_k = np.concatenate([[0], np.cumsum(full)])
    paged = oa.paged_prefill_attention(q, cu_q, cu_k, 0.3, k_cache=kc, v_cache=vc, block_tables=bt, causal=False)
    k_packed = np.concatenate(ks)
    v_packed = np.concatenate(vs)
    packed = oa.paged_prefill_attention(q, cu_q, cu_k, 0.3, k=k_packed, v=v_packed, causal=False)
    for i in range(3):
        rows = slice(cu_q[i], cu_q[i + 1])
        for h in range(4):
            ref = _textbook(q[rows, h], ks[i][:, h // 2], vs[i][:, h // 2], 0.3)
            np.testing.assert_allclose(paged[rows, h], ref, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(packed[rows, h], ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ invariants

def test_block_permutation_invariance():
    rng = np.random.default_rng(30)
    contexts = [7, 33, 64]
    kc, vc, bt, ks, vs = _place(rng, contexts, 4, 2, 8)
    q = rng.standard_normal((3, 4, 8))
    base = oa.paged_decode_attention(q, kc, vc, bt, np.array(contexts), 0.3)
    # move every block to a new physical id
    perm = rng.permutation(kc.shape[0])
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1)
    moved = oa.paged_decode_attention(q, kc2, vc2, bt2, np.array(contexts), 0.3)
    np.testing.assert_array_equal(base, moved)


def test_stale_table_entries_are_not_read():
    rng = np.random.default_rng(31)
    kc, vc, bt, ks, vs = _place(rng, [6], 4, 1, 8)
    bt2 = bt.copy()
    bt2[0, 2:] = 10**6  # beyond ceil(6/4) = 2 entries: never dereferenced
    q = rng.standard_normal((1, 1, 8))
    a = oa.paged_decode_attention(q, kc, vc, bt, np.array([6]), 0.3)
    b = oa.paged_decode_attention(q, kc, vc, bt2, np.array([6]), 0.3)
    np.testing.assert_array_equal(a, b)


def test_prefix_hit_equals_full_recompute():
    rng = np.random.default_rng(32)
    n, c = 23, 8
    kc, vc, bt, ks, vs = _place(rng, [n], 4, 2, 16)
    q_all = rng.standard_normal((n, 4, 16))
    full = oa.paged_prefill_attention(q_all, [0, n], [0, n], 0.3, k_cache=kc, v_cache=vc, block_tables=bt)
    hit = oa.paged_prefill_attention(q_all[c:], [0, n - c], [0, n], 0.3, k_cache=kc, v_cache=vc,
                                     block_tables=bt)
    np.testing.assert_allclose(hit, full[c:], rtol=1e-13, atol=1e-13)


def test_chunked_prefill_equals_one_chunk():
    rng = np.random.default_rng(33)
    n = 16
    kc, vc, bt, ks, vs = _place(rng, [n], 4, 1, 8)
    q = rng.standard_normal((n, 2, 8))
    one = oa.paged_prefill_attention(q, [0, n], [0, n], 0.5, k_cache=kc, v_cache=vc, block_tables=bt)
    first = oa.paged_prefill_attention(q[:8], [0, 8], [0, 8], 0.5, k_cache=kc, v_cache=vc, block_tables=bt)
    second = oa.paged_prefill_attention(q[8:], [0, 8], [0, 16], 0.5, k_cache=kc, v_cache=vc, block_tables=bt)
    np.testing.assert_allclose(np.concatenate([first, second]), one, rtol=1e-13, atol=1e-13)


def test_decode_equals_prefill_last_row():
    rng = np.random.default_rng(34)
    contexts = [5, 12]
    kc, vc, bt, ks, vs = _place(rng, contexts, 4, 2, 8)
    q = rng.standard_normal((2, 4, 8))
    dec = oa.paged_decode_attention(q, kc, vc, bt, np.array(contexts), 0.3)
    pre = oa.paged_prefill_attention(q, [0, 1, 2], [0, 5, 17], 0.3, k_cache=kc, v_cache=vc, block_tables=bt)
    np.testing.assert_allclose(pre, dec, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("splits", [1, 2, 7])
def test_split_and_combine_equals_whole(splits):
    rng = np.random.default_rng(40 + splits)
    contexts = [9, 50, 131]
    kc, vc, bt, ks, vs = _place(rng, contexts, 16, 2, 8)
    q = rng.standard_normal((3, 4, 8))
    whole = oa.paged_decode_attention(q, kc, vc, bt, np.array(contexts), 0.6)
    bounds = []
    for n in contexts:
        edges = sorted(set([0, n] + rng.integers(1, n, size=splits - 1).tolist())) if n > 1 else [0, n]
        bounds.append(edges)
    parts = oa.decode_partials(q, kc, vc, bt, np.array(contexts), 0.6, bounds)
    for b in range(3):
        np.testing.assert_allclose(oa.combine_partials(parts[b]), whole[b], rtol=1e-12, atol=1e-12)


def test_kv_store_closed_form():
    rng = np.random.default_rng(50)
    kc = rng.integers(-2**15, 2**15, size=(6, 4, 2, 8), dtype=np.int16)
    vc = rng.integers(-2**15, 2**15, size=(6, 4, 2, 8), dtype=np.int16)
    k = rng.integers(-2**15, 2**15, size=(5, 2, 8), dtype=np.int16)
    v = rng.integers(-2**15, 2**15, size=(5, 2, 8), dtype=np.int16)
    slots = np.array([3, -1, 17, 0, 23], dtype=np.int32)
    k2, v2 = oa.kv_store(kc, vc, k, v, slots)
    flat_k = kc.reshape(24, 2, 8).copy()
    flat_v = vc.reshape(24, 2, 8).copy()
    for i, s in enumerate(slots):
        if s >= 0:
            flat_k[s] = k[i]
            flat_v[s] = v[i]
    np.testing.assert_array_equal(k2.reshape(24, 2, 8), flat_k)
    np.testing.assert_array_equal(v2.reshape(24, 2, 8), flat_v)
    # untouched slots are unchanged, including those of the skipped row
    untouched = [s for s in range(24) if s not in (3, 17, 0, 23)]
    np.testing.assert_array_equal(k2.reshape(24, 2, 8)[untouched], kc.reshape(24, 2, 8)[untouched])


def test_kv_store_rejects_out_of_pool_slot():
    kc = np.zeros((2, 4, 1, 8))
    with pytest.raises(IndexError):
        oa.kv_store(kc, kc, np.zeros((1, 1, 8)), np.zeros((1, 1, 8)), np.array([8]))


def test_copy_blocks_closed_form_and_sharing():
    rng = np.random.default_rng(60)
    k = rng.integers(0, 255, size=(6, 4, 2, 8), dtype=np.uint8)
    v = rng.integers(0, 255, size=(6, 4, 2, 8), dtype=np.uint8)
    k2, v2 = oa.copy_blocks([k, v], [[1, 4], [2, 5]])
    np.testing.assert_array_equal(k2[4], k[1])
    np.testing.assert_array_equal(v2[5], v[2])
    np.testing.assert_array_equal(k2[[0, 1, 2, 3]], k[[0, 1, 2, 3]])
    # a sequence that shares a prefix block and then copies it reads the same history
    kc, vc, bt, ks, vs = _place(rng, [10], 4, 1, 8)
    q = rng.standard_normal((1, 2, 8))
    base = oa.paged_decode_attention(q, kc, vc, bt, np.array([10]), 0.5)
    free = kc.shape[0] - 1
    kc2, vc2 = oa.copy_blocks([kc, vc], [[bt[0, 1], free]])
    bt2 = bt.copy()
    bt2[0, 1] = free
    np.testing.assert_array_equal(oa.paged_decode_attention(q, kc2, vc2, bt2, np.array([10]), 0.5), base)


def test_parallel_driver_reproduces_the_serial_oracle():
    # the process-pool driver only fans the loop over sequences out: every row must be the
    # serial oracle's, bit for bit (decode through shared files, and prefill per sequence)
    from oracle.parallel import OraclePool

    rng = np.random.default_rng(21)
    bs, hq, hkv, d = 4, 4, 2, 64
    lens = [0, 1, 5, 9, 13]
    nb = sum(-(-n // bs) for n in lens) + 2
    perm = rng.permutation(nb).tolist()
    tables, pos = [], 0
    for n in lens:
        k = -(-n // bs)
        tables.append(perm[pos:pos + k])
        pos += k
    kc = rng.standard_normal((nb, bs, hkv, d)).astype(np.float32)
    vc = rng.standard_normal((nb, bs, hkv, d)).astype(np.float32)
    q = rng.standard_normal((len(lens), hq, d)).astype(np.float32)
    bt = om.padded_block_tables(tables)
    cl = np.asarray(lens, dtype=np.int32)
    want = oa.paged_decode_attention(q, kc, vc, bt, cl, 0.3)
    with OraclePool(2) as pool:
        views, specs = pool.shared({"k_cache": (kc.shape, np.float32), "v_cache": (vc.shape, np.float32)})
        views["k_cache"][:] = kc
        views["v_cache"][:] = vc
        specs.update(q=q, block_tables=bt, context_lens=cl, scale=0.3)
        for chunk in (1, 2):
            assert np.array_equal(pool.decode(specs, len(lens), chunk=chunk), want)
        cached, new = [0, 4, 8], [3, 2, 5]
        tabs = [perm[:1], perm[1:3], perm[3:7]]
        meta = om.prepare_prefill([dict(block_table=t, num_cached_tokens=c, num_scheduled_tokens=n)
                                   for t, c, n in zip(tabs, cached, new)], bs)
        qp = rng.standard_normal((sum(new), hq, d)).astype(np.float32)
        want_p = oa.paged_prefill_attention(qp, meta["cu_seqlens_q"], meta["cu_seqlens_k"], 0.2, k_cache=kc,
                                            v_cache=vc, block_tables=meta["block_tables"])
        specs.update(q=qp, cu_seqlens_q=meta["cu_seqlens_q"], cu_seqlens_k=meta["cu_seqlens_k"],
                     block_tables=meta["block_tables"], scale=0.2, causal=True)
        assert np.array_equal(pool.prefill(specs, 3, sum(new)), want_p)
