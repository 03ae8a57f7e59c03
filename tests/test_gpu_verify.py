"""GPU parity of kv_store + paged_verify_attn (speculative-decoding target pass) against the oracle.

The oracle for a verify pass is varlen prefill attention with q_len query rows
per sequence whose keys are the whole context: row i sits at position
T - q_len + i (bottom-right causal alignment).
"""

import numpy as np
import pytest
import torch

import pagedattention_kv_cache_gb300 as pkv
from pagedattention_kv_cache_gb300 import _lib
from pagedattention_kv_cache_gb300 import metadata as md
from pagedattention_kv_cache_gb300 import workloads as wl
from oracle import attention as oa
from oracle import metadata as om

from _harness import as_np, assert_close, bits, widen_bf16_bits

pytestmark = pytest.mark.gpu


def run_verify(w, q_len, num_splits=0):
    t = wl.verify_tensors(w, q_len, "cpu")
    g = {k: v.cuda() for k, v in t.items()}
    # the q_len newest positions of every context are stored first
    pm = md.prefill_metadata(w.block_tables, [n - q_len for n in w.context_lens], [q_len] * w.batch, w.block_size)
    dm = md.to_device(md.decode_metadata(w.block_tables, w.context_lens, w.block_size), "cuda")
    pkv.kv_store(g["k_new"], g["v_new"], g["k_cache"], g["v_cache"], torch.from_numpy(pm["slot_mapping"]).cuda())
    out = pkv.paged_verify_attn(g["q"], g["k_cache"], g["v_cache"], dm["block_tables"], dm["context_lens"], w.scale,
                                num_splits=num_splits)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    seqs = [dict(block_table=tb, num_cached_tokens=n - q_len, num_scheduled_tokens=q_len)
            for tb, n in zip(w.block_tables, w.context_lens)]
    om_ = om.prepare_prefill(seqs, w.block_size)
    assert np.array_equal(om_["slot_mapping"], pm["slot_mapping"])
    kcb, vcb = oa.kv_store(bits(t["k_cache"]), bits(t["v_cache"]), bits(t["k_new"]), bits(t["v_new"]),
                           om_["slot_mapping"])
    assert np.array_equal(bits(g["k_cache"]), kcb) and np.array_equal(bits(g["v_cache"]), vcb)
    kc, vc = oa.kv_store(as_np(t["k_cache"]), as_np(t["v_cache"]), as_np(t["k_new"]), as_np(t["v_new"]),
                         om_["slot_mapping"])
    B, ql, hq, d = t["q"].shape
    ref = oa.paged_prefill_attention(as_np(t["q"]).reshape(B * ql, hq, d), om_["cu_seqlens_q"], om_["cu_seqlens_k"],
                                     w.scale, k_cache=kc, v_cache=vc, block_tables=om.padded_block_tables(w.block_tables))
    assert_close(out.reshape(B * ql, hq, d), ref, w.dtype, f"verify q_len={q_len}")
    return out, g, dm


@pytest.mark.parametrize("q_len,group", [(2, 2), (3, 2), (4, 2), (8, 1), (2, 4), (5, 1), (8, 2), (4, 4)])
def test_verify_matches_oracle(q_len, group):
    w = wl.random_decode(40 + q_len, batch=7, max_ctx=700, min_ctx=q_len, block_size=16, num_q_heads=4 * group,
                         num_kv_heads=4, head_dim=128, dtype=torch.bfloat16)
    for splits in (0, 1, 3):
        run_verify(w, q_len, splits)


@pytest.mark.parametrize("block_size", [8, 48, 3])
def test_verify_block_sizes(block_size):
    # 48: 16-token tensor copies inside a block; 8 and 3: one copy per token row
    w = wl.random_decode(70 + block_size, batch=6, max_ctx=500, min_ctx=4, block_size=block_size, num_q_heads=8,
                         num_kv_heads=4, head_dim=128, dtype=torch.bfloat16)
    for splits in (0, 2):
        run_verify(w, 4, splits)


@pytest.mark.parametrize("group", [2, 4])
def test_verify_split_part_that_sees_no_key(group):
    # context 1153 in 9 fixed parts of 144 tokens: the last part is token 1152 alone, a
    # merge group of its own, and query rows 0-2 (positions 1149-1151) see none of its
    # keys, so that group's maxima for those rows are -inf
    lens = [1153, 300, 1153]
    bs = 16
    nb = sum(-(-n // bs) for n in lens) + 3
    perm = np.random.default_rng(12).permutation(nb).tolist()
    tables, pos = [], 0
    for n in lens:
        k = -(-n // bs)
        tables.append(perm[pos:pos + k])
        pos += k
    w = wl.DecodeWorkload("lone-last-part", 13, 4 * group, 4, 128, bs, nb, torch.bfloat16, lens, tables)
    run_verify(w, 4, num_splits=9)


def test_verify_batch256_q4_full_size_every_sequence(oracle_pool):
    # the bench's verify case at full size (batch 256, one layer, q_len 4) in the launch it times:
    # the whole pool against the oracle's store, and all 256 sequences' four query rows against the
    # oracle's varlen prefill definition
    q_len = 4
    w = wl.qwen3_decode_b256_28l(num_layers=1)
    t = wl.verify_tensors(w, q_len, "cuda")
    pm = md.prefill_metadata(w.block_tables, [n - q_len for n in w.context_lens], [q_len] * w.batch, w.block_size)
    dm = md.to_device(md.decode_metadata(w.block_tables, w.context_lens, w.block_size), "cuda")
    kb_pre, vb_pre = bits(t["k_cache"]), bits(t["v_cache"])
    pkv.kv_store(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], torch.from_numpy(pm["slot_mapping"]).cuda())
    out = pkv.paged_verify_attn(t["q"], t["k_cache"], t["v_cache"], dm["block_tables"], dm["context_lens"], w.scale)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    seqs = [dict(block_table=tb, num_cached_tokens=n - q_len, num_scheduled_tokens=q_len)
            for tb, n in zip(w.block_tables, w.context_lens)]
    om_ = om.prepare_prefill(seqs, w.block_size)
    assert np.array_equal(om_["slot_mapping"], pm["slot_mapping"])
    kcb, vcb = oa.kv_store(kb_pre, vb_pre, bits(t["k_new"]), bits(t["v_new"]), om_["slot_mapping"])
    del kb_pre, vb_pre
    assert np.array_equal(bits(t["k_cache"]), kcb) and np.array_equal(bits(t["v_cache"]), vcb)
    B, ql, hq, d = t["q"].shape
    q = as_np(t["q"]).reshape(B * ql, hq, d)
    del t
    views, specs = oracle_pool.shared({"k_cache": (kcb.shape, np.float32), "v_cache": (vcb.shape, np.float32),
                                       "q": (q.shape, np.float32)})
    widen_bf16_bits(kcb, views["k_cache"])
    widen_bf16_bits(vcb, views["v_cache"])
    views["q"][:] = q
    del views, kcb, vcb
    specs.update(cu_seqlens_q=om_["cu_seqlens_q"], cu_seqlens_k=om_["cu_seqlens_k"],
                 block_tables=om.padded_block_tables(w.block_tables), scale=w.scale, causal=True)
    ref = oracle_pool.prefill(specs, B, B * ql)
    oracle_pool.release()
    assert_close(out.reshape(B * ql, hq, d), ref, w.dtype, "verify batch-256 q_len 4")


def test_verify_qwen3_batch32_q4():
    w = wl.qwen3_decode_b32()
    run_verify(w, 4)


def test_verify_single_token_is_decode():
    w = wl.random_decode(50, batch=9, max_ctx=900, min_ctx=1, block_size=32, num_q_heads=16, num_kv_heads=8,
                         head_dim=128, dtype=torch.bfloat16)
    out, g, dm = run_verify(w, 1)
    dec = pkv.paged_decode_attn(g["q"][:, 0].contiguous(), g["k_cache"], g["v_cache"], dm["block_tables"],
                                dm["context_lens"], w.scale)
    torch.cuda.synchronize()
    assert torch.equal(dec, out[:, 0])


def test_verify_rejects_context_shorter_than_q_len():
    q = torch.ones(2, 4, 2, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 16, 1, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.tensor([[0], [1]], dtype=torch.int32, device="cuda")
    out = pkv.paged_verify_attn(q, kc, kc, bt, torch.tensor([3, 5], dtype=torch.int32, device="cuda"), 0.1,
                                num_splits=1)
    assert pkv.device_error() & _lib.DERR_LEN_RANGE
    assert torch.all(out[0] == 0)  # the short row reads nothing and writes zeros
    with pytest.raises(_lib.PagedKVError):
        pkv.paged_verify_attn(torch.ones(2, 9, 1, 128, dtype=torch.bfloat16, device="cuda"), kc, kc, bt,
                              torch.tensor([9, 9], dtype=torch.int32, device="cuda"), 0.1)
