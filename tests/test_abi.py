"""The C ABI: the library loads and exports every declared symbol (CPU), and
argument errors come back as status codes without launching (GPU)."""

import ctypes
import os
import re

import numpy as np
import pytest
import torch

import pagedattention_kv_cache_gb300 as pkv
from pagedattention_kv_cache_gb300 import _lib
from pagedattention_kv_cache_gb300 import metadata as md
from oracle import metadata as om

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def _built():
    if not os.path.exists(_lib.LIB_PATH):
        pytest.skip("libpagedkv.so not built (run __graft_entry__.build())")


def test_library_exports_every_declared_symbol():
    _built()
    lib = ctypes.CDLL(_lib.LIB_PATH)
    names = _declared()
    assert {"pkv_kv_store", "pkv_paged_decode_attn", "pkv_paged_varlen_prefill_attn"} <= set(names)
    for name in names:
        assert hasattr(lib, name), f"{name} declared in pagedkv.h but not exported"
    assert {n for n, _, _ in _lib.SIGNATURES} == set(names)


def test_version_and_status_strings():
    _built()
    lib = _lib.load()
    assert lib.pkv_version() >= 10000
    assert lib.pkv_status_string(0) == b"ok"
    assert lib.pkv_status_string(_lib.EWORKSPACE) == b"workspace missing or too small"


def test_prefill_workspace_is_zero_when_nothing_splits():
    # shapes without a tensor-core path, empty batches and (without a GPU) any shape never split
    _built()
    lib = _lib.load()
    assert lib.pkv_paged_varlen_prefill_workspace_bytes(16, 16, 8, 96, 512) == 0  # head_dim 96
    assert lib.pkv_paged_varlen_prefill_workspace_bytes(16, 48, 8, 128, 512) == 0  # G = 6 unsupported
    assert lib.pkv_paged_varlen_prefill_workspace_bytes(0, 16, 8, 128, 512) == 0
    if not torch.cuda.is_available():
        assert lib.pkv_paged_varlen_prefill_workspace_bytes(1, 16, 8, 128, 512) == 0


@pytest.mark.gpu
def test_prefill_workspace_size_rule():
    # work items are pairs of query tiles of 128 / G tokens, one CTA per SM: P = floor(SMs / pairs) parts
    # (at most 8, one wave) when at most half the SMs have a pair; then one int ticket and one int ready
    # count per (sequence, KV head, query tile), each array in a 32 KiB half of the 64 KiB counter
    # area, and P records of 128 rows x (128 fp32 + m + l) per query tile
    lib = _lib.load()
    sms = torch.cuda.get_device_properties(0).multi_processor_count

    def expect(batch, hq, hkv, max_q):
        tq = 128 // (hq // hkv)
        pairs = batch * hkv * (-(-max_q // (2 * tq)))
        if 2 * pairs > sms:
            return 0
        parts = min(8, sms // pairs)
        items = 2 * pairs
        flags = max(32768, -(-items * 4 // 256) * 256)
        return 2 * flags + items * parts * (128 * 128 * 4 + 128 * 8)

    for batch, hq, hkv, max_q in [(16, 16, 8, 512), (1, 8, 8, 1), (3, 32, 4, 1000), (1, 16, 8, 512), (2, 32, 8, 300)]:
        assert lib.pkv_paged_varlen_prefill_workspace_bytes(batch, hq, hkv, 128, max_q) == expect(batch, hq, hkv, max_q)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(_lib.LibraryMissing):
        _lib.load()


def test_host_metadata_matches_oracle():
    rng = np.random.default_rng(0)
    for bs in (1, 4, 16, 256):
        lens = rng.integers(1, 700, size=9).tolist()
        cached = [bs * int(rng.integers(0, n // (2 * bs) + 1)) for n in lens]
        new = [n - c for n, c in zip(lens, cached)]
        tables = [rng.permutation(5000)[: -(-n // bs)].tolist() for n in lens]
        got = md.prefill_metadata(tables, cached, new, bs)
        want = om.prepare_prefill([dict(block_table=t, num_cached_tokens=c, num_scheduled_tokens=n)
                                   for t, c, n in zip(tables, cached, new)], bs)
        for key in ("slot_mapping", "cu_seqlens_q", "cu_seqlens_k"):
            assert np.array_equal(got[key], want[key]), key
        assert got["max_seqlen_q"] == want["max_seqlen_q"] and got["max_seqlen_k"] == want["max_seqlen_k"]
        assert (got["block_tables"] is None) == (want["block_tables"] is None)
        dgot = md.decode_metadata(tables, lens, bs)
        dwant = om.prepare_decode([dict(block_table=t, length=n) for t, n in zip(tables, lens)], bs)
        for key in ("slot_mapping", "context_lens", "block_tables"):
            assert np.array_equal(dgot[key], dwant[key]), key


def test_decode_metadata_refuses_tables_of_the_wrong_length():
    # the new token's slot comes from the last table entry, so the table must hold exactly
    # ceil(length / block_size) blocks, as the oracle requires
    assert md.decode_metadata([[3, 1], []], [6, 0], 4)["slot_mapping"].tolist() == [5, -1]
    for tables, lens in (([[3, 1, 9]], [6]), ([[3]], [6]), ([[2]], [0]), ([[]], [1])):
        with pytest.raises(ValueError, match="table has"):
            md.decode_metadata(tables, lens, 4)
        with pytest.raises(ValueError):
            om.prepare_decode([dict(block_table=t, length=n) for t, n in zip(tables, lens)], 4)
    with pytest.raises(ValueError):
        md.decode_metadata([[1]], [-1], 4)


def test_noalloc_rejects_bad_arguments_on_the_host():
    # argument errors come back before any CUDA call (and so before its scratch memset is queued):
    # these pointers are never dereferenced
    _built()
    lib = _lib.load()
    f = lib.pkv_paged_decode_attn_noalloc
    ok_ptr = 4096
    args = dict(out=ok_ptr, q=ok_ptr, kc=ok_ptr, vc=ok_ptr, bt=ok_ptr, mb=4, cl=ok_ptr, batch=2, hq=4, hkv=2, d=128,
                bs=16, nb=8, scale=ctypes.c_float(0.1), splits=0, dtype=_lib.BF16, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["out"], a["q"], a["kc"], a["vc"], a["bt"], a["mb"], a["cl"], a["batch"], a["hq"], a["hkv"], a["d"],
                 a["bs"], a["nb"], a["scale"], a["splits"], a["dtype"], a["stream"])

    assert call(out=None) == _lib.EINVAL
    assert call(hq=3) == _lib.EINVAL
    assert call(d=96) == _lib.EUNSUPPORTED
    assert call(dtype=7) == _lib.EUNSUPPORTED
    assert call(q=ok_ptr + 8) == _lib.EALIGN
    assert call(batch=0) == _lib.OK


def test_pad_decode_rows():
    m = md.pad_decode(md.decode_metadata([[3, 1]], [6], 4), 4)
    assert m["slot_mapping"].tolist() == [5, -1, -1, -1]
    assert m["context_lens"].tolist() == [6, 0, 0, 0]
    assert m["block_tables"][1:].tolist() == [[-1, -1]] * 3


# ---------------------------------------------------------------- GPU: argument validation

@pytest.mark.gpu
def test_argument_errors_return_status():
    lib = _lib.load()
    dev = "cuda"
    q = torch.zeros(2, 4, 128, dtype=torch.bfloat16, device=dev)
    kc = torch.zeros(4, 16, 2, 128, dtype=torch.bfloat16, device=dev)
    bt = torch.zeros(2, 3, dtype=torch.int32, device=dev)
    cl = torch.ones(2, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    s = torch.cuda.current_stream().cuda_stream

    def dec(**kw):
        a = dict(out=out.data_ptr(), q=q.data_ptr(), k=kc.data_ptr(), v=kc.data_ptr(), bt=bt.data_ptr(), mb=3,
                 cl=cl.data_ptr(), B=2, hq=4, hkv=2, d=128, bs=16, nb=4, scale=ctypes.c_float(0.1), splits=1,
                 ws=None, wsb=0, dt=_lib.BF16)
        a.update(kw)
        return lib.pkv_paged_decode_attn(a["out"], a["q"], a["k"], a["v"], a["bt"], a["mb"], a["cl"], a["B"],
                                         a["hq"], a["hkv"], a["d"], a["bs"], a["nb"], a["scale"], a["splits"],
                                         a["ws"], a["wsb"], a["dt"], s)

    assert dec() == _lib.OK
    assert dec(hq=3) == _lib.EINVAL
    assert dec(d=96) == _lib.EUNSUPPORTED
    assert dec(q=None) == _lib.EINVAL
    assert dec(q=q.data_ptr() + 2) == _lib.EALIGN
    assert dec(splits=0) == _lib.EWORKSPACE
    assert dec(splits=4, ws=None) == _lib.EWORKSPACE
    assert dec(bs=0) == _lib.EINVAL
    assert dec(dt=7) == _lib.EUNSUPPORTED
    assert dec(B=0) == _lib.OK
    assert lib.pkv_paged_decode_workspace_bytes(2, 4, 128, 1) == 0
    assert lib.pkv_paged_decode_workspace_bytes(2, 4, 128, 3) > 0
    with pytest.raises(_lib.PagedKVError):
        pkv.paged_decode_attn(q, kc, kc, bt, cl, 0.1, num_splits=2, workspace=torch.zeros(8, dtype=torch.uint8,
                                                                                           device=dev))
    k = torch.zeros(3, 2, 128, dtype=torch.bfloat16, device=dev)
    slots = torch.zeros(3, dtype=torch.int32, device=dev)
    st = lib.pkv_kv_store(k.data_ptr(), k.data_ptr(), kc.data_ptr(), kc.data_ptr(), slots.data_ptr(), -1, 4, 16, 2,
                          128, _lib.BF16, s)
    assert st == _lib.EINVAL
    st = lib.pkv_kv_store(k.data_ptr() + 4, k.data_ptr(), kc.data_ptr(), kc.data_ptr(), slots.data_ptr(), 3, 4, 16,
                          2, 128, _lib.BF16, s)
    assert st == _lib.EALIGN
    st = lib.pkv_paged_varlen_prefill_attn(q.data_ptr(), q.data_ptr(), None, None, None, None, bt.data_ptr(),
                                           bt.data_ptr(), 1, 1, None, 0, 1, 2, 0, 4, 2, 96, 16, 4,
                                           ctypes.c_float(0.1), 1, None, 0, _lib.BF16, s)
    assert st == _lib.EUNSUPPORTED
    for d in (64, 128):
        st = lib.pkv_paged_varlen_prefill_attn(q.data_ptr(), q.data_ptr(), None, None, None, None, bt.data_ptr(),
                                               bt.data_ptr(), 1, 1, None, 0, 1, 2, 0, 4, 2, d, 16, 4,
                                               ctypes.c_float(0.1), 1, None, 0, _lib.BF16, s)
        assert st == _lib.EINVAL  # no block tables and no packed k / v
    st = lib.pkv_paged_varlen_prefill_attn(q.data_ptr(), q.data_ptr(), None, None, None, None, bt.data_ptr(),
                                           bt.data_ptr(), 1, 1, None, 0, 1, -1, 0, 4, 2, 128, 16, 4,
                                           ctypes.c_float(0.1), 1, None, 0, _lib.BF16, s)
    assert st == _lib.EINVAL
    st = lib.pkv_paged_varlen_prefill_attn(q.data_ptr(), q.data_ptr(), None, None, kc.data_ptr(), kc.data_ptr(),
                                           bt.data_ptr(), bt.data_ptr(), 1, 1, bt.data_ptr(), 1, 1, 2, 0, 4, 2, 128,
                                           16, 4, ctypes.c_float(0.1), 1, q.data_ptr() + 16, 1 << 20, _lib.BF16, s)
    assert st == _lib.EALIGN  # the workspace must be 256-byte aligned
    torch.cuda.synchronize()
    assert pkv.device_error() == 0


@pytest.mark.gpu
def test_out_of_range_indices_raise_device_error_bits():
    # the kernels' own bounds checks turn these into error bits, never an access
    dev = "cuda"
    pkv.device_error(reset=True)
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.float32, device=dev)
    k = torch.ones(2, 2, 64, device=dev)
    pkv.kv_store(k, k, kc, kc, torch.tensor([64, -5], dtype=torch.int32, device=dev))
    assert pkv.device_error() == _lib.DERR_SLOT_RANGE
    assert torch.count_nonzero(kc) == 0
    q = torch.ones(1, 2, 64, device=dev)
    bt = torch.tensor([[7]], dtype=torch.int32, device=dev)  # block 7 of a 4-block pool
    pkv.paged_decode_attn(q, kc, kc, bt, torch.tensor([5], dtype=torch.int32, device=dev), 0.1, num_splits=1)
    assert pkv.device_error() & _lib.DERR_BLOCK_RANGE
    pkv.paged_decode_attn(q, kc, kc, bt, torch.tensor([17], dtype=torch.int32, device=dev), 0.1, num_splits=1)
    assert pkv.device_error() & _lib.DERR_LEN_RANGE
    assert pkv.device_error() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("block_size", [64, 24, None])  # tcgen05 paged, mma.sync paged, packed k/v
def test_bad_cu_seqlens_raise_the_range_bit_and_write_nothing(block_size):
    # a negative start, a negative row count and a sequence longer than max_seqlen_q are
    # skipped by the prefill kernels' own range checks: nothing is read or written there
    dev = "cuda"
    d, hq, hkv = 128, 4, 2
    q = torch.ones(8, hq, d, dtype=torch.bfloat16, device=dev)
    kv = torch.ones(8, hkv, d, dtype=torch.bfloat16, device=dev)
    cases = [([-5, 3], [0, 8], 8), ([0, 4, 2], [0, 4, 6], 8), ([0, 6], [0, 6], 4)]
    for cu_q, cu_k, max_q in cases:
        pkv.device_error(reset=True)
        out = torch.full_like(q, 7.0)
        kwargs = dict(k=kv, v=kv)
        if block_size is not None:
            kc = torch.ones(8, block_size, hkv, d, dtype=torch.bfloat16, device=dev)
            bt = torch.arange(len(cu_q) - 1, dtype=torch.int32, device=dev)[:, None].contiguous()
            kwargs = dict(k_cache=kc, v_cache=kc, block_tables=bt)
        pkv.paged_varlen_prefill_attn(q, torch.tensor(cu_q, dtype=torch.int32, device=dev),
                                      torch.tensor(cu_k, dtype=torch.int32, device=dev), max_q, 8, 0.1,
                                      out=out, workspace=False, **kwargs)
        torch.cuda.synchronize()
        assert pkv.device_error() & _lib.DERR_LEN_RANGE, (cu_q, cu_k, max_q)
        if cu_q[1] < 0 or cu_q[0] < 0 or max_q < cu_q[-1] - cu_q[0]:
            # the single sequence is skipped whole
            assert torch.all(out == 7.0), (cu_q, cu_k, max_q)
    assert pkv.device_error() == 0


@pytest.mark.gpu
def test_binding_rejects_mismatched_shapes_before_launch():
    # a wrong-sized out or a cache of another head_dim would make a kernel write or read
    # out of bounds: the binding refuses them on the host
    dev = "cuda"
    q = torch.zeros(2, 4, 128, dtype=torch.bfloat16, device=dev)
    kc = torch.zeros(4, 16, 2, 128, dtype=torch.bfloat16, device=dev)
    bt = torch.zeros(2, 3, dtype=torch.int32, device=dev)
    cl = torch.ones(2, dtype=torch.int32, device=dev)
    short = torch.empty(1, 4, 128, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError, match="out must have shape"):
        pkv.paged_decode_attn(q, kc, kc, bt, cl, 0.1, num_splits=1, out=short)
    with pytest.raises(ValueError, match="out must have shape"):
        pkv.paged_decode_attn_noalloc(q, kc, kc, bt, cl, 0.1, out=short)
    with pytest.raises(ValueError, match="inconsistent shapes"):
        pkv.paged_decode_attn_noalloc(q, kc[..., :64].contiguous(), kc[..., :64].contiguous(), bt, cl, 0.1)
    with pytest.raises(ValueError, match="out must have shape"):
        pkv.paged_verify_attn(q[:, None], kc, kc, bt, cl, 0.1, num_splits=1, out=short)
    cu = torch.tensor([0, 1], dtype=torch.int32, device=dev)
    with pytest.raises(ValueError, match="head_dim differs"):
        pkv.paged_varlen_prefill_attn(q[:1], cu, cu, 1, 1, 0.1, k_cache=kc[..., :64].contiguous(),
                                      v_cache=kc[..., :64].contiguous(), block_tables=bt[:1])
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        pkv.paged_decode_attn(q, kc, kc, bt.cpu(), cl, 0.1, num_splits=1)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
