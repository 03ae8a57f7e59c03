"""GPU tests of prefix-shared block tables with copy-on-write block copies, and
of store + decode captured once in a CUDA graph and replayed with new data
(batch padded to a bucket with slot -1 / context 0 rows)."""

import numpy as np
import pytest
import torch

import pagedattention_kv_cache_gb300 as pkv
from pagedattention_kv_cache_gb300 import _lib
from pagedattention_kv_cache_gb300 import metadata as md
from oracle import attention as oa
from oracle import metadata as om

from _harness import as_np, assert_close, bits

pytestmark = pytest.mark.gpu


def test_copy_blocks_bit_exact_all_layers():
    gen = torch.Generator().manual_seed(1)
    L, nb = 3, 10
    ks = [torch.randn(nb, 16, 2, 128, generator=gen).bfloat16() for _ in range(L)]
    vs = [torch.randn(nb, 16, 2, 128, generator=gen).bfloat16() for _ in range(L)]
    pairs = torch.tensor([[1, 7], [4, 8], [2, 2]], dtype=torch.int32)
    gk = [t.cuda() for t in ks]
    gv = [t.cuda() for t in vs]
    pkv.copy_blocks(gk, gv, pairs.cuda())
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    want = oa.copy_blocks([bits(t) for t in ks + vs], pairs.numpy())
    for got, w in zip(gk + gv, want):
        assert np.array_equal(bits(got), w)
    pkv.copy_blocks(gk, gv, torch.tensor([[0, 99]], dtype=torch.int32, device="cuda"))
    assert pkv.device_error() == _lib.DERR_BLOCK_RANGE


def test_shared_prefix_then_copy_on_write():
    # sequence B forks from A after 37 tokens (block size 16: blocks a0, a1 full, a2 holds 5);
    # before B writes token 37 into the shared partial block a2 it copies a2 to a free block
    bs, hkv, hq, d, L = 16, 2, 4, 128, 2
    gen = torch.Generator().manual_seed(2)
    nb = 8
    kc = [torch.randn(nb, bs, hkv, d, generator=gen).bfloat16() for _ in range(L)]
    vc = [torch.randn(nb, bs, hkv, d, generator=gen).bfloat16() for _ in range(L)]
    table_a = [5, 1, 6]
    table_b = [5, 1, 3]  # a2 = 6 copied to the free block 3
    pairs = torch.tensor([[6, 3]], dtype=torch.int32)
    lens = [38, 38]
    q = torch.randn(L, 2, hq, d, generator=gen).bfloat16()
    kn = torch.randn(L, 2, hkv, d, generator=gen).bfloat16()
    vn = torch.randn(L, 2, hkv, d, generator=gen).bfloat16()
    meta = md.decode_metadata([table_a, table_b], lens, bs)
    gm = md.to_device(meta, "cuda")
    gk = [t.cuda() for t in kc]
    gv = [t.cuda() for t in vc]
    pkv.copy_blocks(gk, gv, pairs.cuda())
    outs = []
    for layer in range(L):
        pkv.kv_store(kn[layer].cuda(), vn[layer].cuda(), gk[layer], gv[layer], gm["slot_mapping"])
        outs.append(pkv.paged_decode_attn(q[layer].cuda(), gk[layer], gv[layer], gm["block_tables"],
                                          gm["context_lens"], d ** -0.5))
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    ometa = om.prepare_decode([dict(block_table=table_a, length=38), dict(block_table=table_b, length=38)], bs)
    assert ometa["slot_mapping"].tolist() == [6 * 16 + 5, 3 * 16 + 5]
    copied = oa.copy_blocks([as_np(t) for t in kc + vc], pairs.numpy())
    for layer in range(L):
        k2, v2 = oa.kv_store(copied[layer], copied[L + layer], as_np(kn[layer]), as_np(vn[layer]),
                             ometa["slot_mapping"])
        assert np.array_equal(gk[layer].float().cpu().numpy(), k2)
        ref = oa.paged_decode_attention(as_np(q[layer]), k2, v2, ometa["block_tables"], ometa["context_lens"],
                                        d ** -0.5)
        assert_close(outs[layer], ref, torch.bfloat16, "cow decode")
        # the shared prefix blocks 5 and 1 were read by both sequences; a2 keeps A's history
        assert np.array_equal(k2[6, :5], as_np(kc[layer])[6, :5])


def test_store_and_decode_captured_in_a_cuda_graph():
    bs, hkv, hq, d, L, bucket = 16, 2, 4, 128, 3, 8
    gen = torch.Generator().manual_seed(3)
    nb = 64
    kc = [torch.randn(nb, bs, hkv, d, generator=gen).bfloat16().cuda() for _ in range(L)]
    vc = [torch.randn(nb, bs, hkv, d, generator=gen).bfloat16().cuda() for _ in range(L)]
    width = 10
    # static buffers of the captured step (the bucket's fixed addresses)
    s_q = torch.zeros(L, bucket, hq, d, dtype=torch.bfloat16, device="cuda")
    s_k = torch.zeros(L, bucket, hkv, d, dtype=torch.bfloat16, device="cuda")
    s_v = torch.zeros(L, bucket, hkv, d, dtype=torch.bfloat16, device="cuda")
    s_slot = torch.full((bucket,), -1, dtype=torch.int32, device="cuda")
    s_len = torch.zeros(bucket, dtype=torch.int32, device="cuda")
    s_tab = torch.full((bucket, width), -1, dtype=torch.int32, device="cuda")
    s_out = torch.zeros(L, bucket, hq, d, dtype=torch.bfloat16, device="cuda")
    ws = pkv.decode_workspace(bucket, hq, d, 0)

    def step():
        for layer in range(L):
            pkv.kv_store(s_k[layer], s_v[layer], kc[layer], vc[layer], s_slot)
            pkv.paged_decode_attn(s_q[layer], kc[layer], vc[layer], s_tab, s_len, d ** -0.5, workspace=ws,
                                  out=s_out[layer])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    rng = np.random.default_rng(4)
    perm = rng.permutation(nb).tolist()
    tables = [perm[i * 10:i * 10 + 10] for i in range(5)]
    for replay in range(2):
        lens = rng.integers(1, 150, size=5).tolist()
        tabs = [t[: -(-n // bs)] for t, n in zip(tables, lens)]
        meta = md.pad_decode(md.decode_metadata(tabs, lens, bs, table_width=width), bucket)
        before = [(as_np(kc[layer]), as_np(vc[layer])) for layer in range(L)]
        s_slot.copy_(torch.from_numpy(meta["slot_mapping"]))
        s_len.copy_(torch.from_numpy(meta["context_lens"]))
        s_tab.copy_(torch.from_numpy(meta["block_tables"]))
        for buf in (s_q, s_k, s_v):
            buf.copy_(torch.randn(buf.shape, generator=gen).bfloat16())
        s_out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pkv.device_error() == 0
        assert torch.all(s_out[:, 5:] == 0)  # padded rows read nothing and write zeros
        for layer in range(L):
            k2, v2 = oa.kv_store(before[layer][0], before[layer][1], as_np(s_k[layer][:5]), as_np(s_v[layer][:5]),
                                 meta["slot_mapping"][:5])
            assert np.array_equal(as_np(kc[layer]), k2)
            ref = oa.paged_decode_attention(as_np(s_q[layer][:5]), k2, v2, meta["block_tables"][:5],
                                            meta["context_lens"][:5], d ** -0.5)
            assert_close(s_out[layer][:5], ref, torch.bfloat16, f"graph replay {replay} layer {layer}")
