"""Shared helpers for the parity tests: run a workload through the CUDA path
(via the C-ABI binding) and through the oracle, and compare.

Tolerances (attention outputs against the float64 oracle):
* bf16 in/out, fp32 accumulation: max-abs 1e-2 and mean-abs 1e-3.  Where the
  oracle value itself is >= 4 in magnitude, bf16 cannot represent it within
  1e-2 (its half-ulp there is 2^-6), so that element's bound is the bf16
  half-ulp of the value plus 2e-3.
* bf16 outputs are also compared with the oracle rounded to bf16 (round to
  nearest even): within 1e-2 where |oracle| < 2, and at most one bf16 ulp
  away (the correctly rounded value or a neighbour) where |oracle| >= 2, since
  one ulp there (2^-6 and up) is already wider than 1e-2.
* fp32: max-abs 1e-4.
Every bf16 comparison is recorded: how many elements have |oracle| >= 4 and
how many of those needed the widened bound (error above 1e-2).  The test
session prints the records that have any (tests/conftest.py).
The KV store is compared bit for bit over the whole pool.
"""

from __future__ import annotations

import numpy as np
import torch

import pagedattention_kv_cache_gb300 as pkv
from pagedattention_kv_cache_gb300 import metadata as md
from pagedattention_kv_cache_gb300 import workloads as wl
from oracle import attention as oa
from oracle import metadata as om

BF16_MAX, BF16_MEAN = 1e-2, 1e-3
F32_MAX = 1e-4


def as_np(t: torch.Tensor) -> np.ndarray:
    """Exact float view for the oracle (bf16 widens exactly to float32)."""
    t = t.detach().cpu()
    return (t.float() if t.dtype == torch.bfloat16 else t).numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    return (t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)).numpy()


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 8)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float64 values rounded to the nearest bf16 (8 significant bits, ties to even), in float64.

    One rounding step from float64, so no double rounding through float32.
    Normal range only (the outputs here are far from bf16's subnormals).
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)  # x = m * 2^e with 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0), e - 8)  # np.rint rounds halves to even


# every bf16 comparison of the session: (label, elements, |oracle| >= 4, widened bound used, max vs bf16(oracle))
BF16_RECORDS: list[tuple] = []


def assert_close(got: torch.Tensor, ref: np.ndarray, dtype: torch.dtype, label: str = "") -> dict:
    g = got.detach().double().cpu().numpy()
    assert np.all(np.isfinite(g)), f"{label}: non-finite output"
    err = np.abs(g - ref)
    stats = {"max_abs": float(err.max()) if err.size else 0.0, "mean_abs": float(err.mean()) if err.size else 0.0}
    if dtype == torch.float32:
        assert stats["max_abs"] <= F32_MAX, f"{label}: max abs {stats['max_abs']:.3e} > {F32_MAX}"
    else:
        bound = np.maximum(BF16_MAX, bf16_half_ulp(ref) + 2e-3)
        worst = float((err - bound).max()) if err.size else -1.0
        assert worst <= 0, f"{label}: max abs {stats['max_abs']:.3e} exceeds the bf16 bound"
        assert stats["mean_abs"] <= BF16_MEAN, f"{label}: mean abs {stats['mean_abs']:.3e} > {BF16_MEAN}"
        # against the oracle rounded to bf16: 1e-2 below |oracle| = 2, one ulp (2 half-ulps) above
        rb = bf16_round(ref)
        err_b = np.abs(g - rb)
        big = np.abs(ref) >= 2.0
        bound_b = np.where(big, 2.0 * bf16_half_ulp(rb), BF16_MAX)
        worst_b = float((err_b - bound_b).max()) if err.size else -1.0
        assert worst_b <= 1e-12, f"{label}: {int((err_b > bound_b).sum())} elements beyond the bf16-rounded bound"
        stats["max_abs_vs_bf16_oracle"] = float(err_b.max()) if err.size else 0.0
        stats["mean_abs_vs_bf16_oracle"] = float(err_b.mean()) if err.size else 0.0
        stats["abs_ge_4"] = int((np.abs(ref) >= 4.0).sum())
        stats["widened"] = int(((np.abs(ref) >= 4.0) & (err > BF16_MAX)).sum())
        BF16_RECORDS.append((label, int(err.size), stats["abs_ge_4"], stats["widened"],
                             stats["max_abs_vs_bf16_oracle"]))
    return stats


def oracle_decode_tables(w: wl.DecodeWorkload) -> dict:
    seqs = [dict(block_table=t, length=n) for t, n in zip(w.block_tables, w.context_lens)]
    return om.prepare_decode(seqs, w.block_size)


def run_decode(w: wl.DecodeWorkload, *, num_splits: int = 0, poison: bool = False, layer: int = 0,
               device="cuda", check_store: bool = True, gen_device="cpu") -> dict:
    """Store the new tokens and run decode on the GPU; compare store and output with the oracle."""
    t = wl.decode_tensors(w, gen_device, layer=layer, poison=poison)
    meta = md.decode_metadata(w.block_tables, w.context_lens, w.block_size)
    g = {k: v.to(device, copy=True) for k, v in t.items()}
    gm = md.to_device(meta, device)
    pkv.kv_store(g["k_new"], g["v_new"], g["k_cache"], g["v_cache"], gm["slot_mapping"])
    out = pkv.paged_decode_attn(g["q"], g["k_cache"], g["v_cache"], gm["block_tables"], gm["context_lens"],
                                w.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    err = pkv.device_error()
    assert err == 0, f"device error bits {err:#x}"

    ometa = oracle_decode_tables(w)
    assert np.array_equal(ometa["slot_mapping"], meta["slot_mapping"])
    if check_store:
        kc_bits, vc_bits = oa.kv_store(bits(t["k_cache"]), bits(t["v_cache"]), bits(t["k_new"]), bits(t["v_new"]),
                                       ometa["slot_mapping"])
        assert np.array_equal(bits(g["k_cache"]), kc_bits), "k_cache differs from the oracle store"
        assert np.array_equal(bits(g["v_cache"]), vc_bits), "v_cache differs from the oracle store"
    kc, vc = oa.kv_store(as_np(t["k_cache"]), as_np(t["v_cache"]), as_np(t["k_new"]), as_np(t["v_new"]),
                         ometa["slot_mapping"])
    ref = oa.paged_decode_attention(as_np(t["q"]), kc, vc, ometa["block_tables"], ometa["context_lens"], w.scale)
    stats = assert_close(out, ref, w.dtype, w.name)
    return {"out": out, "ref": ref, "stats": stats, "tensors": g, "meta": gm}


def run_prefill(w: wl.PrefillWorkload, *, use_tables: bool = True, poison: bool = False, device="cuda",
                causal: bool = True, workspace=None) -> dict:
    """Store this step's rows and run varlen prefill on the GPU; compare with the oracle."""
    t = wl.prefill_tensors(w, "cpu", poison=poison)
    meta = md.prefill_metadata(w.block_tables, w.num_cached, w.num_new, w.block_size, always_tables=use_tables)
    g = {k: v.to(device, copy=True) for k, v in t.items()}
    gm = md.to_device(meta, device)
    if use_tables:
        pkv.kv_store(g["k"], g["v"], g["k_cache"], g["v_cache"], gm["slot_mapping"])
        out = pkv.paged_varlen_prefill_attn(g["q"], gm["cu_seqlens_q"], gm["cu_seqlens_k"], meta["max_seqlen_q"],
                                            meta["max_seqlen_k"], w.scale, k_cache=g["k_cache"],
                                            v_cache=g["v_cache"], block_tables=gm["block_tables"], causal=causal,
                                            workspace=workspace)
    else:
        out = pkv.paged_varlen_prefill_attn(g["q"], gm["cu_seqlens_q"], gm["cu_seqlens_k"], meta["max_seqlen_q"],
                                            meta["max_seqlen_k"], w.scale, k=g["k"], v=g["v"], causal=causal,
                                            workspace=workspace)
    torch.cuda.synchronize()
    err = pkv.device_error()
    assert err == 0, f"device error bits {err:#x}"

    seqs = [dict(block_table=tb, num_cached_tokens=c, num_scheduled_tokens=n)
            for tb, c, n in zip(w.block_tables, w.num_cached, w.num_new)]
    ometa = om.prepare_prefill(seqs, w.block_size)
    assert np.array_equal(ometa["slot_mapping"], meta["slot_mapping"])
    assert np.array_equal(ometa["cu_seqlens_q"], meta["cu_seqlens_q"])
    assert np.array_equal(ometa["cu_seqlens_k"], meta["cu_seqlens_k"])
    if use_tables:
        kc_bits, vc_bits = oa.kv_store(bits(t["k_cache"]), bits(t["v_cache"]), bits(t["k"]), bits(t["v"]),
                                       ometa["slot_mapping"])
        assert np.array_equal(bits(g["k_cache"]), kc_bits), "k_cache differs from the oracle store"
        assert np.array_equal(bits(g["v_cache"]), vc_bits), "v_cache differs from the oracle store"
        kc, vc = oa.kv_store(as_np(t["k_cache"]), as_np(t["v_cache"]), as_np(t["k"]), as_np(t["v"]),
                             ometa["slot_mapping"])
        ref = oa.paged_prefill_attention(as_np(t["q"]), ometa["cu_seqlens_q"], ometa["cu_seqlens_k"], w.scale,
                                         k_cache=kc, v_cache=vc, block_tables=om.padded_block_tables(w.block_tables),
                                         causal=causal)
    else:
        ref = oa.paged_prefill_attention(as_np(t["q"]), ometa["cu_seqlens_q"], ometa["cu_seqlens_k"], w.scale,
                                         k=as_np(t["k"]), v=as_np(t["v"]), causal=causal)
    stats = assert_close(out, ref, w.dtype, w.name)
    return {"out": out, "ref": ref, "stats": stats, "tensors": g, "meta": gm}


# ---------------------------------------------------------------- full-size checks on every sequence

def widen_bf16_bits(src: np.ndarray, dst: np.ndarray, chunk: int = 64) -> None:
    """Exact bf16 -> float32 widening of raw 16-bit patterns (int16) into dst, ``chunk`` rows at a time."""
    for i in range(0, src.shape[0], chunk):
        dst[i:i + chunk] = (src[i:i + chunk].view(np.uint16).astype(np.uint32) << 16).view(np.float32)


def decode_layer_full(pool, w: wl.DecodeWorkload, layer: int, label: str) -> dict:
    """One layer of a full-size decode batch in the launch the benchmark times (automatic split,
    caller workspace): store the new tokens, decode, then compare the whole pool bit for bit with
    the oracle's store and every sequence's output with the oracle's attention (run on every
    host core by ``pool``)."""
    t = wl.decode_tensors(w, "cuda", layer=layer)
    meta = md.decode_metadata(w.block_tables, w.context_lens, w.block_size)
    gm = md.to_device(meta, "cuda")
    kb_pre, vb_pre = bits(t["k_cache"]), bits(t["v_cache"])
    ws = pkv.decode_workspace(w.batch, w.num_q_heads, w.head_dim, 0)
    pkv.kv_store(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], gm["slot_mapping"])
    out = pkv.paged_decode_attn(t["q"], t["k_cache"], t["v_cache"], gm["block_tables"], gm["context_lens"], w.scale,
                                workspace=ws)
    torch.cuda.synchronize()
    err = pkv.device_error()
    assert err == 0, f"device error bits {err:#x}"
    ometa = oracle_decode_tables(w)
    assert np.array_equal(ometa["slot_mapping"], meta["slot_mapping"])
    kc_bits, vc_bits = oa.kv_store(kb_pre, vb_pre, bits(t["k_new"]), bits(t["v_new"]), ometa["slot_mapping"])
    del kb_pre, vb_pre
    assert np.array_equal(bits(t["k_cache"]), kc_bits), f"{label}: k_cache differs from the oracle store"
    assert np.array_equal(bits(t["v_cache"]), vc_bits), f"{label}: v_cache differs from the oracle store"
    q = as_np(t["q"])
    del t
    views, specs = pool.shared({"k_cache": (kc_bits.shape, np.float32), "v_cache": (vc_bits.shape, np.float32),
                                "q": (q.shape, np.float32)})
    widen_bf16_bits(kc_bits, views["k_cache"])
    widen_bf16_bits(vc_bits, views["v_cache"])
    views["q"][:] = q
    del kc_bits, vc_bits, views
    specs.update(block_tables=ometa["block_tables"], context_lens=ometa["context_lens"], scale=w.scale)
    ref = pool.decode(specs, w.batch)
    pool.release()
    return assert_close(out, ref, w.dtype, label)
