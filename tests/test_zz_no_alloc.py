"""pkv_paged_decode_attn_noalloc: paged decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: hooks that run inside another engine's
execution step, runtimes whose device memory belongs to a pool this library
cannot reach, and latency-critical code that must not pay cudaMalloc's
implicit synchronisation.  The no-allocation entry point gives them decode
without a caller-provided workspace, using a fixed scratch array inside the
library.  These tests call it through the C ABI and check that it matches
pkv_paged_decode_attn (same tolerance as the parity tests), on two calls in a
row (the second reuses the array's leftover contents), and that sizes beyond
the array are rejected before anything is launched.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""

import ctypes

import pytest
import torch

import pagedattention_kv_cache_gb300 as pkv
from pagedattention_kv_cache_gb300 import _lib
from pagedattention_kv_cache_gb300 import metadata as md
from pagedattention_kv_cache_gb300 import workloads as wl

from _harness import assert_close

pytestmark = pytest.mark.gpu


def _inputs(w):
    t = wl.decode_tensors(w, "cpu")
    g = {k: v.cuda() for k, v in t.items()}
    meta = md.to_device(md.decode_metadata(w.block_tables, w.context_lens, w.block_size), "cuda")
    return g, meta


def _noalloc(w, g, meta, out, num_splits):
    nb, bs, hkv, d = g["k_cache"].shape
    return _lib.load().pkv_paged_decode_attn_noalloc(
        out.data_ptr(), g["q"].data_ptr(), g["k_cache"].data_ptr(), g["v_cache"].data_ptr(),
        meta["block_tables"].data_ptr(), meta["block_tables"].shape[1], meta["context_lens"].data_ptr(), w.batch,
        w.num_q_heads, hkv, d, bs, nb, ctypes.c_float(w.scale), num_splits,
        _lib.BF16 if w.dtype == torch.bfloat16 else _lib.F32, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("make,num_splits", [(wl.qwen3_decode_b32, 0), (wl.qwen3_decode_b32, 5),
                                             (wl.tiny_decode, 3), (wl.tiny_decode, 1)])
def test_noalloc_matches_workspace_entry_point_twice(make, num_splits):
    w = make()
    g, meta = _inputs(w)
    ref = pkv.paged_decode_attn(g["q"], g["k_cache"], g["v_cache"], meta["block_tables"], meta["context_lens"],
                                w.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    ref_np = ref.double().cpu().numpy()
    for _ in range(2):
        out = torch.full_like(g["q"], float("nan"))
        assert _noalloc(w, g, meta, out, num_splits) == _lib.OK
        torch.cuda.synchronize()
        assert_close(out, ref_np, w.dtype, f"noalloc {w.name} splits={num_splits}")
    assert pkv.device_error() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 4000 sequences with the automatic split need ~36 MB of workspace, more than the 8 MiB array
    B, hq, hkv, d, bs = 4000, 16, 8, 128, 16
    assert pkv.decode_workspace_bytes(B, hq, d, 0) > _lib.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(B, hq, d, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(2, bs, hkv, d, dtype=torch.bfloat16, device="cuda")
    w = wl.DecodeWorkload("oversize", 0, hq, hkv, d, bs, 2, torch.bfloat16, [0] * B, [[]] * B)
    g = {"q": q, "k_cache": kc, "v_cache": kc}
    meta = {"block_tables": torch.full((B, 1), -1, dtype=torch.int32, device="cuda"),
            "context_lens": torch.zeros(B, dtype=torch.int32, device="cuda")}
    out = torch.full_like(q, 7.0)
    assert _noalloc(w, g, meta, out, 0) == _lib.ESCRATCH
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)  # nothing was launched
    # a fixed split small enough for the array is accepted
    assert _noalloc(w, g, meta, out, 1) == _lib.OK
    torch.cuda.synchronize()
    assert torch.all(out == 0)
