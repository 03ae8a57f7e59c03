"""GPU parity of the FP8 (E4M3) KV cache: the quantizing store is bit-exact
against the oracle's codec, and decode over the one-byte cache matches the
oracle's attention over the dequantized cache."""

import numpy as np
import pytest
import torch

import pagedattention_kv_cache_gb300 as pkv
from pagedattention_kv_cache_gb300 import _lib
from pagedattention_kv_cache_gb300 import metadata as md
from pagedattention_kv_cache_gb300 import workloads as wl
from oracle import attention as oa
from oracle import fp8 as of8
from oracle import metadata as om

from _harness import as_np, assert_close

pytestmark = pytest.mark.gpu

K_SCALE, V_SCALE = 1.0 / 64, 3.0 / 256


def test_kv_store_fp8_bit_exact_with_saturation():
    gen = torch.Generator().manual_seed(0)
    N, nb, bs, hkv, d = 50, 12, 8, 2, 128
    k = (torch.randn(N, hkv, d, generator=gen) * 3).to(torch.bfloat16)
    v = (torch.randn(N, hkv, d, generator=gen) * 3).to(torch.bfloat16)
    k[0, 0, :4] = torch.tensor([1e6, -1e6, 448 * K_SCALE * 1.02, 0.0])  # saturation and zero
    kc = torch.randint(0, 256, (nb, bs, hkv, d), generator=gen, dtype=torch.uint8)
    vc = torch.randint(0, 256, (nb, bs, hkv, d), generator=gen, dtype=torch.uint8)
    slots = torch.randperm(nb * bs, generator=gen)[:N].int()
    slots[3] = -1
    gk, gv = kc.cuda(), vc.cuda()
    pkv.kv_store_fp8(k.cuda(), v.cuda(), gk, gv, slots.cuda(), K_SCALE, V_SCALE)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    wk, wv = of8.kv_store_fp8(kc.numpy(), vc.numpy(), as_np(k), as_np(v), slots.numpy(), K_SCALE, V_SCALE)
    assert np.array_equal(gk.cpu().numpy(), wk)
    assert np.array_equal(gv.cpu().numpy(), wv)


def _quantized_pool(shape, gen, scale):
    x = torch.randn(shape, generator=gen).to(torch.bfloat16)
    return torch.from_numpy(of8.quantize(as_np(x), scale))


@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("splits", [0, 1, 5])
def test_fp8_decode_matches_oracle_on_dequantized_cache(group, splits):
    _fp8_decode_case(group, splits, 1.0)


# q far outside f16's range either way: both kernels carry q in f16 after a
# per-row power-of-two scaling, which must leave the scores unchanged
@pytest.mark.parametrize("group", [2, 4])
@pytest.mark.parametrize("q_scale", [1e-6, 3e4, 1e9])
def test_fp8_decode_q_magnitudes(group, q_scale):
    _fp8_decode_case(group, 0, q_scale)


# G = 4 runs the tensor-core kernel: 16-token tensor copies when the block size
# is a multiple of 16, one copy per token row otherwise.  Every code outside
# the contexts is the E4M3 NaN (0x7f), including the tail of a sequence's last
# block that a 16-token copy brings in.
@pytest.mark.parametrize("kv_heads,block_size", [(1, 16), (2, 8), (3, 48), (8, 16), (8, 32), (4, 5)])
@pytest.mark.parametrize("splits", [0, 1, 4])
def test_fp8_decode_group4_layouts(kv_heads, block_size, splits):
    _fp8_decode_case(4, splits, 1.0, kv_heads=kv_heads, block_size=block_size, poison=True)


def _poison_codes(pool, tables, lens, block_size):
    used = torch.zeros(pool.shape[0], block_size, dtype=torch.bool)
    for table, n in zip(tables, lens):
        for j, block in enumerate(table):
            used[block, : max(0, min(block_size, n - j * block_size))] = True
    pool[~used] = 0x7F


def _fp8_decode_case(group, splits, q_scale, kv_heads=4, block_size=16, poison=False):
    w = wl.random_decode(60 + group + 7 * kv_heads + block_size, batch=12, max_ctx=1200, min_ctx=0,
                         block_size=block_size, num_q_heads=group * kv_heads, num_kv_heads=kv_heads, head_dim=128,
                         dtype=torch.bfloat16)
    gen = torch.Generator().manual_seed(group)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc, vc = _quantized_pool(shape, gen, K_SCALE), _quantized_pool(shape, gen, V_SCALE)
    if poison:
        # the new token's slot (position len - 1) is written by the store below
        for pool in (kc, vc):
            _poison_codes(pool, w.block_tables, [max(0, n - 1) for n in w.context_lens], w.block_size)
    q = (torch.randn(w.batch, w.num_q_heads, w.head_dim, generator=gen) * q_scale).to(torch.bfloat16)
    kn = torch.randn(w.batch, w.num_kv_heads, w.head_dim, generator=gen).to(torch.bfloat16)
    vn = torch.randn(w.batch, w.num_kv_heads, w.head_dim, generator=gen).to(torch.bfloat16)
    meta = md.decode_metadata(w.block_tables, w.context_lens, w.block_size)
    gm = md.to_device(meta, "cuda")
    gk, gv = kc.cuda(), vc.cuda()
    pkv.kv_store_fp8(kn.cuda(), vn.cuda(), gk, gv, gm["slot_mapping"], K_SCALE, V_SCALE)
    out = pkv.paged_decode_attn_fp8(q.cuda(), gk, gv, gm["block_tables"], gm["context_lens"], w.scale, K_SCALE,
                                    V_SCALE, num_splits=splits)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    om_ = om.prepare_decode([dict(block_table=t, length=n) for t, n in zip(w.block_tables, w.context_lens)],
                            w.block_size)
    wk, wv = of8.kv_store_fp8(kc.numpy(), vc.numpy(), as_np(kn), as_np(vn), om_["slot_mapping"], K_SCALE, V_SCALE)
    assert np.array_equal(gk.cpu().numpy(), wk) and np.array_equal(gv.cpu().numpy(), wv)
    ref = oa.paged_decode_attention(as_np(q), of8.dequantize(wk, K_SCALE), of8.dequantize(wv, V_SCALE),
                                    om_["block_tables"], om_["context_lens"], w.scale)
    assert_close(out, ref, torch.bfloat16, f"fp8 decode G={group} splits={splits}")


def test_fp8_decode_batch256_full_size_every_sequence(oracle_pool):
    # one layer of the bench's FP8 step at full size (batch 256, 2.4 GB of codes) in the launch it
    # times: the quantizing store of the new tokens bit for bit against the oracle's codec over the
    # whole pool, then all 256 sequences against the oracle on the dequantized blocks
    w = wl.qwen3_decode_b256_28l(num_layers=1)
    dev = "cuda"
    gen = torch.Generator(device=dev).manual_seed(11)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc, vc = [(torch.randn(shape, generator=gen, device=dev) / s).clamp_(-448, 448).to(torch.float8_e4m3fn)
              .view(torch.uint8) for s in (K_SCALE, V_SCALE)]
    q = torch.randn(w.batch, w.num_q_heads, w.head_dim, generator=gen, device=dev).bfloat16()
    kn = torch.randn(w.batch, w.num_kv_heads, w.head_dim, generator=gen, device=dev).bfloat16()
    vn = torch.randn(w.batch, w.num_kv_heads, w.head_dim, generator=gen, device=dev).bfloat16()
    meta = md.decode_metadata(w.block_tables, w.context_lens, w.block_size)
    gm = md.to_device(meta, dev)
    kc_pre, vc_pre = kc.cpu().numpy(), vc.cpu().numpy()
    pkv.kv_store_fp8(kn, vn, kc, vc, gm["slot_mapping"], K_SCALE, V_SCALE)
    out = pkv.paged_decode_attn_fp8(q, kc, vc, gm["block_tables"], gm["context_lens"], w.scale, K_SCALE, V_SCALE)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    om_ = om.prepare_decode([dict(block_table=t, length=n) for t, n in zip(w.block_tables, w.context_lens)],
                            w.block_size)
    wk, wv = of8.kv_store_fp8(kc_pre, vc_pre, as_np(kn), as_np(vn), om_["slot_mapping"], K_SCALE, V_SCALE)
    del kc_pre, vc_pre
    assert np.array_equal(kc.cpu().numpy(), wk) and np.array_equal(vc.cpu().numpy(), wv)
    del kc, vc
    views, specs = oracle_pool.shared({"k_codes": (wk.shape, np.uint8), "v_codes": (wv.shape, np.uint8)})
    views["k_codes"][:] = wk
    views["v_codes"][:] = wv
    del views, wk, wv
    specs.update(q=as_np(q), block_tables=om_["block_tables"], context_lens=om_["context_lens"], scale=w.scale,
                 k_scale=K_SCALE, v_scale=V_SCALE)
    ref = oracle_pool.decode_fp8(specs, w.batch)
    oracle_pool.release()
    assert_close(out, ref, torch.bfloat16, "fp8 batch-256 layer 0")


def test_fp8_argument_errors():
    q = torch.zeros(1, 2, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(2, 16, 1, 128, dtype=torch.uint8, device="cuda")
    bt = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
    cl = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(_lib.PagedKVError):
        pkv.paged_decode_attn_fp8(q, kc, kc, bt, cl, 0.1, 0.0, 1.0)  # scale must be > 0
    with pytest.raises(_lib.PagedKVError):
        pkv.paged_decode_attn_fp8(torch.zeros(1, 6, 128, dtype=torch.bfloat16, device="cuda"), kc, kc, bt, cl, 0.1,
                                  1.0, 1.0)  # G = 6 is not a supported group size
