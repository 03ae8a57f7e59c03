"""GPU parity of kv_store + paged_varlen_prefill_attn against the oracle (through the C-ABI)."""

import numpy as np
import pytest
import torch

import pagedattention_kv_cache_gb300 as pkv
from pagedattention_kv_cache_gb300 import metadata as md
from pagedattention_kv_cache_gb300 import workloads as wl

from _harness import assert_close, run_prefill

pytestmark = pytest.mark.gpu


def test_qwen3_prefill_prefix_chunk():
    run_prefill(wl.qwen3_prefill_prefix())


def test_qwen3_prefill_prefix_chunk_poisoned():
    run_prefill(wl.qwen3_prefill_prefix(), poison=True)


@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("block_size", [4, 8, 16, 24, 32, 48, 64, 96, 256])
def test_prefill_groups_and_block_sizes(group, block_size):
    w = wl.random_prefill(group * 10 + block_size, batch=5, max_new=150, min_new=1, max_cached_blocks=3,
                          block_size=block_size, num_q_heads=2 * group, num_kv_heads=2, head_dim=128)
    run_prefill(w)


@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("block_size", [8, 16, 64, 256])
def test_prefill_head_dim_64(group, block_size):
    # one 64-wide slab per Q / K / V tile, O of 64 columns in TMEM, 128-byte staged output rows
    w = wl.random_prefill(700 + group * 10 + block_size, batch=5, max_new=300, min_new=1, max_cached_blocks=4,
                          block_size=block_size, num_q_heads=2 * group, num_kv_heads=2, head_dim=64)
    run_prefill(w)


def test_prefill_head_dim_64_packed_and_non_causal():
    w = wl.random_prefill(731, batch=6, max_new=200, min_new=1, max_cached_blocks=0, block_size=16,
                          num_q_heads=8, num_kv_heads=4, head_dim=64)
    r_packed = run_prefill(w, use_tables=False)
    r_paged = run_prefill(w, use_tables=True)
    assert torch.equal(r_packed["out"], r_paged["out"])
    w = wl.random_prefill(732, batch=4, max_new=90, min_new=1, max_cached_blocks=2, block_size=16,
                          num_q_heads=8, num_kv_heads=4, head_dim=64)
    run_prefill(w, causal=False)


def test_prefill_edge_lengths():
    # empty sequences, single-row sequences, tile-boundary lengths
    news = [0, 1, 63, 64, 65, 128, 129, 31, 33]
    cached = [0, 16, 0, 32, 16, 0, 64, 48, 0]
    tables, pos = [], 0
    perm = np.random.default_rng(4).permutation(200).tolist()
    for n, c in zip(news, cached):
        k = -(-(n + c) // 16)
        tables.append(perm[pos:pos + k])
        pos += k
    w = wl.PrefillWorkload("edges", 5, 4, 2, 128, 16, 200, torch.bfloat16, cached, news, tables)
    run_prefill(w)


def test_prefill_no_history_packed_path():
    w = wl.random_prefill(21, batch=6, max_new=200, min_new=1, max_cached_blocks=0, block_size=16,
                          num_q_heads=16, num_kv_heads=8, head_dim=128)
    assert sum(w.num_cached) == 0
    r_packed = run_prefill(w, use_tables=False)
    r_paged = run_prefill(w, use_tables=True)
    assert torch.equal(r_packed["out"], r_paged["out"])


def test_prefill_non_causal():
    w = wl.random_prefill(22, batch=4, max_new=90, min_new=1, max_cached_blocks=2, block_size=16,
                          num_q_heads=8, num_kv_heads=4, head_dim=128)
    run_prefill(w, causal=False)


def test_prefix_hit_equals_full_recompute():
    # same tokens: a prefill with a prefix-cache hit gives the last rows of a full recompute
    bs, hq, hkv, d = 16, 8, 4, 128
    n, c = 300, 96
    gen = torch.Generator().manual_seed(12)
    table = torch.randperm(40, generator=gen)[: -(-n // bs)].tolist()
    kc = torch.randn(40, bs, hkv, d, generator=gen).to(torch.bfloat16).cuda()
    vc = torch.randn(40, bs, hkv, d, generator=gen).to(torch.bfloat16).cuda()
    q = torch.randn(n, hq, d, generator=gen).to(torch.bfloat16).cuda()
    full_md = md.to_device(md.prefill_metadata([table], [0], [n], bs, always_tables=True), "cuda")
    hit_md = md.to_device(md.prefill_metadata([table], [c], [n - c], bs, always_tables=True), "cuda")
    scale = d ** -0.5
    full = pkv.paged_varlen_prefill_attn(q, full_md["cu_seqlens_q"], full_md["cu_seqlens_k"], n, n, scale,
                                         k_cache=kc, v_cache=vc, block_tables=full_md["block_tables"])
    hit = pkv.paged_varlen_prefill_attn(q[c:].contiguous(), hit_md["cu_seqlens_q"], hit_md["cu_seqlens_k"], n - c, n,
                                        scale, k_cache=kc, v_cache=vc, block_tables=hit_md["block_tables"])
    torch.cuda.synchronize()
    diff = (hit.float() - full[c:].float()).abs().max().item()
    assert diff <= 1e-2


def test_decode_equals_prefill_single_row():
    w = wl.random_decode(31, batch=7, max_ctx=500, min_ctx=1, block_size=16, num_q_heads=8, num_kv_heads=4,
                         head_dim=128, dtype=torch.bfloat16)
    t = wl.decode_tensors(w, "cpu")
    g = {k: v.cuda() for k, v in t.items()}
    dm = md.to_device(md.decode_metadata(w.block_tables, w.context_lens, w.block_size), "cuda")
    dec = pkv.paged_decode_attn(g["q"], g["k_cache"], g["v_cache"], dm["block_tables"], dm["context_lens"], w.scale)
    pm = md.prefill_metadata(w.block_tables, [n - 1 for n in w.context_lens], [1] * w.batch, w.block_size,
                             always_tables=True)
    gp = md.to_device(pm, "cuda")
    pre = pkv.paged_varlen_prefill_attn(g["q"], gp["cu_seqlens_q"], gp["cu_seqlens_k"], 1, pm["max_seqlen_k"],
                                        w.scale, k_cache=g["k_cache"], v_cache=g["v_cache"],
                                        block_tables=gp["block_tables"])
    torch.cuda.synchronize()
    assert (dec.float() - pre.float()).abs().max().item() <= 1e-2


def test_prefill_many_short_sequences_repeated():
    # hundreds of CTAs, two per SM: the tensor pipe runs behind the softmax, which is
    # when a premature completion wait would read O before its last P.V landed
    bs, nq, cached, B = 256, 64, 64, 400
    rng = np.random.default_rng(17)
    perm = rng.permutation(B + 8).tolist()
    tables = [[perm[i]] for i in range(B)]
    w = wl.PrefillWorkload("many-short", 23, 4, 2, 128, bs, B + 8, torch.bfloat16, [cached] * B, [nq] * B, tables)
    for _ in range(3):
        run_prefill(w)


def _long_history(seed: int, group: int = 2, block_size: int = 256) -> wl.PrefillWorkload:
    # histories of up to 12 blocks of 256: the last query tiles need ~25 key tiles of 128,
    # far past the 8 above which a tile runs as several parts
    return wl.random_prefill(seed, batch=3, max_new=300, min_new=40, max_cached_blocks=12, block_size=block_size,
                             num_q_heads=8 * group, num_kv_heads=8, head_dim=128)


@pytest.mark.parametrize("group", [2, 4])
def test_long_items_split_and_unsplit_match_oracle(group):
    w = _long_history(31 + group, group)
    split = run_prefill(w)                   # cached workspace: long tiles run as two parts
    whole = run_prefill(w, workspace=False)  # never split
    # the two paths differ only in rounding order
    d = (split["out"].float() - whole["out"].float()).abs().max().item()
    assert d <= 1.6e-2, d


def test_long_items_split_non_causal():
    w = _long_history(35)
    run_prefill(w, causal=False)


def test_split_workspace_reused_and_left_zeroed():
    w = _long_history(36)
    hq, hkv = w.num_q_heads, w.num_kv_heads
    ws = pkv.prefill_workspace(w.batch, hq, hkv, w.head_dim, max(w.num_new))
    assert ws is not None
    outs = [run_prefill(w, workspace=ws)["out"] for _ in range(3)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    items = w.batch * hkv * -(-max(w.num_new) // (128 // (hq // hkv)))
    assert items * 4 <= 32768
    assert int(ws[:65536].count_nonzero()) == 0  # the counter area (tickets, ready counts) back at zero


def test_long_items_split_head_dim_64():
    # the split records hold 64 fp32 columns per row
    w = wl.random_prefill(38, batch=3, max_new=300, min_new=40, max_cached_blocks=12, block_size=256,
                          num_q_heads=16, num_kv_heads=8, head_dim=64)
    assert pkv.prefill_workspace_bytes(3, 16, 8, 64, max(w.num_new)) > 0
    split = run_prefill(w)
    whole = run_prefill(w, workspace=False)
    d = (split["out"].float() - whole["out"].float()).abs().max().item()
    assert d <= 1.6e-2, d


def test_split_workspace_shared_by_calls_of_growing_size():
    # one workspace: a one-sequence split (few tickets, large records), then three sequences (more
    # tickets), then one again; the tickets stay in the fixed counter area, clear of every call's
    # records.  Each call against the unsplit kernel
    one = wl.random_prefill(40, batch=1, max_new=120, min_new=120, max_cached_blocks=16, block_size=256,
                            num_q_heads=16, num_kv_heads=8, head_dim=128)
    one.num_cached[0] = 16 * 256
    one.block_tables[0] = list(range(-(-(16 * 256 + 120) // 256)))
    one.num_blocks = max(one.num_blocks, len(one.block_tables[0]) + 4)
    three = wl.random_prefill(41, batch=3, max_new=140, min_new=40, max_cached_blocks=10, block_size=256,
                              num_q_heads=16, num_kv_heads=8, head_dim=128)
    sizes = [pkv.prefill_workspace_bytes(w.batch, 16, 8, 128, max(w.num_new)) for w in (one, three)]
    assert min(sizes) > 0
    ws = torch.zeros(max(sizes), dtype=torch.uint8, device="cuda")
    for w in (one, three, one, three):
        t = wl.prefill_tensors(w, "cuda")
        meta = md.prefill_metadata(w.block_tables, w.num_cached, w.num_new, w.block_size, always_tables=True)
        gm = md.to_device(meta, "cuda")
        pkv.kv_store(t["k"], t["v"], t["k_cache"], t["v_cache"], gm["slot_mapping"])
        outs = [pkv.paged_varlen_prefill_attn(t["q"], gm["cu_seqlens_q"], gm["cu_seqlens_k"], meta["max_seqlen_q"],
                                              meta["max_seqlen_k"], w.scale, k_cache=t["k_cache"],
                                              v_cache=t["v_cache"], block_tables=gm["block_tables"], workspace=ws_arg)
                for ws_arg in (ws, False)]
        torch.cuda.synchronize()
        assert pkv.device_error() == 0
        d = (outs[0].float() - outs[1].float()).abs().max().item()
        assert d <= 1.6e-2, (w.batch, d)


def test_single_long_history_runs_as_eight_parts():
    # one sequence, a 16k-token history and 200 new tokens: 16 pairs of query tiles for a GPU of ~150 SMs,
    # so each pair (130 key tiles of 128) runs as eight parts
    w = wl.random_prefill(37, batch=1, max_new=200, min_new=200, max_cached_blocks=64, block_size=256,
                          num_q_heads=16, num_kv_heads=8, head_dim=128)
    w.num_cached[0] = 64 * 256
    w.block_tables[0] = list(range(-(-(64 * 256 + 200) // 256)))
    w.num_blocks = max(w.num_blocks, len(w.block_tables[0]) + 4)
    assert pkv.prefill_workspace_bytes(1, 16, 8, 128, 200) > 0
    split = run_prefill(w)
    whole = run_prefill(w, workspace=False)
    d = (split["out"].float() - whole["out"].float()).abs().max().item()
    assert d <= 1.6e-2, d
