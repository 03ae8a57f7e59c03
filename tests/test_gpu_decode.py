"""GPU parity of kv_store + paged_decode_attn against the oracle (through the C-ABI)."""

import math

import numpy as np
import pytest
import torch

import pagedattention_kv_cache_gb300 as pkv
from pagedattention_kv_cache_gb300 import metadata as md
from pagedattention_kv_cache_gb300 import workloads as wl
from oracle import attention as oa

from _harness import as_np, assert_close, decode_layer_full, run_decode

pytestmark = pytest.mark.gpu


def test_tiny_decode_fp32():
    r = run_decode(wl.tiny_decode())
    assert r["stats"]["max_abs"] < 1e-5


def test_tiny_decode_fp32_poisoned():
    run_decode(wl.tiny_decode(), poison=True)


def test_qwen3_decode_b32_bf16():
    run_decode(wl.qwen3_decode_b32())


def test_qwen3_decode_b32_poisoned():
    run_decode(wl.qwen3_decode_b32(), poison=True)


@pytest.mark.parametrize("splits", [1, 2, 7, 0])
def test_split_invariance_fp32(splits):
    w = wl.random_decode(11, batch=6, max_ctx=300, min_ctx=1, block_size=16, num_q_heads=8, num_kv_heads=2,
                         head_dim=128, dtype=torch.float32)
    r = run_decode(w, num_splits=splits)
    base = run_decode(w, num_splits=1)
    np.testing.assert_allclose(r["out"].cpu().numpy(), base["out"].cpu().numpy(), rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("block_size", [1, 2, 4, 16])
@pytest.mark.parametrize("group", [1, 2, 4])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_brute_force_grid(block_size, group, d, dtype):
    # every context length 1..20 in one batch
    rng = np.random.default_rng(block_size * 1000 + group * 100 + d)
    lens = list(range(1, 21))
    nb = sum(math.ceil(n / block_size) for n in lens) + 3
    perm = rng.permutation(nb).tolist()
    tables, pos = [], 0
    for n in lens:
        k = math.ceil(n / block_size)
        tables.append(perm[pos:pos + k])
        pos += k
    w = wl.DecodeWorkload("grid", 77, 2 * group, 2, d, block_size, nb, dtype, lens, tables)
    for splits in (0, 1, 3):
        run_decode(w, num_splits=splits)


@pytest.mark.parametrize("kv_heads", [1, 2, 4, 8])
def test_kv_head_counts(kv_heads):
    w = wl.random_decode(5, batch=9, max_ctx=700, min_ctx=1, block_size=32, num_q_heads=2 * kv_heads,
                         num_kv_heads=kv_heads, head_dim=128, dtype=torch.bfloat16)
    run_decode(w)


def test_group_8():
    w = wl.random_decode(6, batch=5, max_ctx=400, min_ctx=1, block_size=16, num_q_heads=16, num_kv_heads=2,
                         head_dim=128, dtype=torch.bfloat16)
    run_decode(w)


# G = 4 runs the tensor-core kernel: block sizes that are multiples of 16 fill
# its stages with 16-token tensor copies (split points on multiples of 16),
# others with one copy per token row.  Poisoned caches put NaN in every slot
# no sequence owns, including the tail of a sequence's last block that a
# 16-token copy brings in.
@pytest.mark.parametrize("kv_heads,block_size", [(1, 16), (2, 32), (3, 48), (4, 16), (8, 16), (8, 64), (2, 8),
                                                 (4, 24), (8, 1)])
@pytest.mark.parametrize("splits", [0, 1, 4])
def test_mma_kernel_stage_layouts(kv_heads, block_size, splits):
    w = wl.random_decode(60 + kv_heads * 7 + block_size, batch=7, max_ctx=900, min_ctx=1, block_size=block_size,
                         num_q_heads=4 * kv_heads, num_kv_heads=kv_heads, head_dim=128, dtype=torch.bfloat16)
    run_decode(w, num_splits=splits, poison=True)


# Many parts per sequence: the parts merge in groups of 8 (the last arrival of a
# group merges it), then the last group merger merges the groups.  Covers one
# group, a partial last group, and ~150 automatic parts; the fp32 case runs the
# CUDA-core kernel, the bf16 one the tensor-core kernel.
@pytest.mark.parametrize("group,dtype", [(2, torch.float32), (4, torch.bfloat16)])
@pytest.mark.parametrize("lens,splits", [([60000], 0), ([20000, 3, 40000], 0), ([9000, 700], 9), ([5000], 8),
                                         ([30000, 1], 23)])
def test_grouped_merge_of_many_parts(group, dtype, lens, splits):
    rng = np.random.default_rng(sum(lens) + splits + group)
    bs = 16
    nb = sum(math.ceil(n / bs) for n in lens) + 5
    perm = rng.permutation(nb).tolist()
    tables, pos = [], 0
    for n in lens:
        k = math.ceil(n / bs)
        tables.append(perm[pos:pos + k])
        pos += k
    w = wl.DecodeWorkload("many-parts", 91, 2 * group, 2, 128, bs, nb, dtype, lens, tables)
    run_decode(w, num_splits=splits)


def test_qwen3_b256_one_layer_full_size_every_sequence(oracle_pool):
    # one layer of the 28-layer bench step at full size (batch 256, 4.8 GB of K/V) in the launch the
    # bench times (automatic split): the whole pool against the oracle's store, and all 256
    # sequences against the oracle's attention
    decode_layer_full(oracle_pool, wl.qwen3_decode_b256_28l(num_layers=1), 0, "batch-256 layer 0")


def test_qwen3_b256_all_28_layers_every_sequence(oracle_pool):
    # the bench step's other 27 layers, each drawn from its own seed as in the bench
    w = wl.qwen3_decode_b256_28l()
    for layer in range(1, w.num_layers):
        decode_layer_full(oracle_pool, w, layer, f"batch-256 layer {layer}")


def test_long_context_split_decode_full_size():
    r = run_decode(wl.long_context_decode(), gen_device="cuda", check_store=True)
    assert r["stats"]["mean_abs"] < 1e-3


def test_zero_context_rows_and_padding():
    # graph-replay padding: rows with slot -1 and context length 0 read and write nothing
    w = wl.random_decode(8, batch=5, max_ctx=90, min_ctx=1, block_size=8, num_q_heads=4, num_kv_heads=2,
                         head_dim=64, dtype=torch.float32)
    t = wl.decode_tensors(w, "cpu")
    meta = md.pad_decode(md.decode_metadata(w.block_tables, w.context_lens, w.block_size), 8)
    dev = "cuda"
    q = torch.randn(8, 4, 64, generator=torch.Generator().manual_seed(3)).to(dev)
    q[:5] = t["q"].to(dev)
    kn = torch.zeros(8, 2, 64, device=dev)
    vn = torch.zeros(8, 2, 64, device=dev)
    kn[:5] = t["k_new"].to(dev)
    vn[:5] = t["v_new"].to(dev)
    kc, vc = t["k_cache"].to(dev), t["v_cache"].to(dev)
    gm = md.to_device(meta, dev)
    gm["block_tables"][5:, :] = 10 ** 6  # stale ids on padded rows: never read
    pkv.kv_store(kn, vn, kc, vc, gm["slot_mapping"])
    out = torch.full((8, 4, 64), float("nan"), device=dev)
    for splits in (0, 1, 4):
        pkv.paged_decode_attn(q, kc, vc, gm["block_tables"], gm["context_lens"], w.scale, num_splits=splits, out=out)
        torch.cuda.synchronize()
        assert pkv.device_error() == 0
        assert torch.all(out[5:] == 0)
        kco, vco = oa.kv_store(as_np(t["k_cache"]), as_np(t["v_cache"]), as_np(t["k_new"]), as_np(t["v_new"]),
                               meta["slot_mapping"][:5])
        ref = oa.paged_decode_attention(as_np(t["q"]), kco, vco, meta["block_tables"][:5], meta["context_lens"][:5],
                                        w.scale)
        assert_close(out[:5], ref, torch.float32, "padded")
    assert torch.equal(kc.cpu(), torch.from_numpy(kco)) and torch.equal(vc.cpu(), torch.from_numpy(vco))


def test_block_permutation_bit_identical():
    w = wl.qwen3_decode_b32()
    r = run_decode(w)
    g = r["tensors"]
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(9))
    kc2 = torch.empty_like(g["k_cache"])
    vc2 = torch.empty_like(g["v_cache"])
    kc2[perm.cuda()] = g["k_cache"]
    vc2[perm.cuda()] = g["v_cache"]
    bt = r["meta"]["block_tables"]
    bt2 = torch.where(bt >= 0, perm.cuda()[bt.clamp(min=0).long()].int(), bt)
    out2 = pkv.paged_decode_attn(g["q"], kc2, vc2, bt2, r["meta"]["context_lens"], w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out2, r["out"])


def test_repeated_calls_reuse_workspace():
    w = wl.qwen3_decode_b32()
    r = run_decode(w)
    g = r["tensors"]
    ws = pkv.decode_workspace(w.batch, w.num_q_heads, w.head_dim, 0)
    outs = [pkv.paged_decode_attn(g["q"], g["k_cache"], g["v_cache"], r["meta"]["block_tables"],
                                  r["meta"]["context_lens"], w.scale, workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, r["out"])
    # the workspace's ticket counters are back at zero
    assert torch.count_nonzero(ws[: 4 * w.batch]) == 0


def test_workspace_shared_by_calls_of_growing_batch():
    # one workspace for a small batch, then larger ones: every call's ticket counters sit in the fixed
    # counter area at the start, which no call's partial results reach
    ws_calls = []
    for seed, batch in ((61, 2), (62, 40), (63, 3), (64, 90)):
        w = wl.random_decode(seed, batch=batch, max_ctx=4000, min_ctx=1500, block_size=16, num_q_heads=16,
                             num_kv_heads=8, head_dim=128, dtype=torch.bfloat16)
        t = {k: v.cuda() for k, v in wl.decode_tensors(w, "cpu").items()}
        m = md.to_device(md.decode_metadata(w.block_tables, w.context_lens, w.block_size), "cuda")
        ws_calls.append((w, t, m))
    need = max(pkv.decode_workspace_bytes(w.batch, 16, 128) for w, _, _ in ws_calls)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for w, t, m in ws_calls:
        shared = pkv.paged_decode_attn(t["q"], t["k_cache"], t["v_cache"], m["block_tables"], m["context_lens"],
                                       w.scale, workspace=ws)
        fresh = pkv.paged_decode_attn(t["q"], t["k_cache"], t["v_cache"], m["block_tables"], m["context_lens"],
                                      w.scale)
        torch.cuda.synchronize()
        assert pkv.device_error() == 0
        assert torch.equal(shared, fresh), w.batch
