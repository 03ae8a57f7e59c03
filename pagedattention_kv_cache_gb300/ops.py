"""Python binding of the C ABI: argument marshalling only.

Each function takes torch tensors that already live on the current CUDA
device, checks device, dtype, shape and contiguity (a mismatch that would let
a kernel read or write out of bounds is a host-side error, raised before any
launch), and passes raw pointers and sizes to libpagedkv.so on the current
torch stream.  Every step of the path runs
in the library's CUDA kernels; nothing here computes.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib

_DTYPES = {torch.float32: _lib.F32, torch.bfloat16: _lib.BF16}


def _dtype_code(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}; expected float32 or bfloat16") from None


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype=None, ndim=None, device=None, shape=None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the other arguments on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _device(t: torch.Tensor, name: str) -> torch.device:
    """The device every argument of a call must be on: the current CUDA device, where the
    library launches its kernels."""
    _need(t, name)
    cur = torch.cuda.current_device()
    if t.device.index != cur:
        raise ValueError(f"{name} is on {t.device} but the current CUDA device is cuda:{cur}")
    return t.device


def _stream(stream, device: torch.device) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if stream.device != device:
        raise ValueError(f"stream belongs to {stream.device}, the tensors to {device}")
    return stream.cuda_stream


def kv_store(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
             slot_mapping: torch.Tensor, stream=None) -> None:
    """Write k/v rows [N, Hkv, D] into k_cache/v_cache [blocks, bs, Hkv, D] at slot_mapping (-1 skips)."""
    dev = _device(k, "k")
    for name, t in (("k", k), ("v", v), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need(t, name, dtype=k.dtype, device=dev)
    _need(slot_mapping, "slot_mapping", dtype=torch.int32, ndim=1, device=dev)
    if k.dim() != 3 or v.shape != k.shape or k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("expected k, v [N, Hkv, D] and caches [blocks, bs, Hkv, D]")
    if k_cache.shape[2:] != k.shape[1:] or slot_mapping.shape[0] != k.shape[0]:
        raise ValueError("k/v rows and the cache disagree on (Hkv, D), or slot_mapping length differs")
    nb, bs, hkv, d = k_cache.shape
    st = _lib.load().pkv_kv_store(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
                                  k.shape[0], nb, bs, hkv, d, _dtype_code(k), _stream(stream, dev))
    _lib.check("pkv_kv_store", st)


def copy_blocks(k_caches: list[torch.Tensor], v_caches: list[torch.Tensor], block_pairs: torch.Tensor,
                stream=None) -> None:
    """Copy-on-write block copies: for each (src, dst) row of block_pairs (int32 [n, 2]),
    block dst of every layer's K and V pool becomes a copy of block src."""
    if len(k_caches) != len(v_caches) or not k_caches:
        raise ValueError("need one K and one V pool per layer")
    shape = k_caches[0].shape
    dev = _device(k_caches[0], "k_caches[0]")
    for t in list(k_caches) + list(v_caches):
        _need(t, "cache", device=dev)
        if t.shape != shape or t.dtype != k_caches[0].dtype:
            raise ValueError("every pool must have the same shape and dtype")
    _need(block_pairs, "block_pairs", dtype=torch.int32, ndim=2, device=dev)
    if block_pairs.shape[1] != 2:
        raise ValueError("block_pairs must be [n, 2]")
    L = len(k_caches)
    kp = (ctypes.c_void_p * L)(*[t.data_ptr() for t in k_caches])
    vp = (ctypes.c_void_p * L)(*[t.data_ptr() for t in v_caches])
    block_bytes = k_caches[0][0].numel() * k_caches[0].element_size()
    st = _lib.load().pkv_copy_blocks(kp, vp, L, _ptr(block_pairs), block_pairs.shape[0], shape[0], block_bytes,
                                     _stream(stream, dev))
    _lib.check("pkv_copy_blocks", st)


def kv_store_fp8(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 slot_mapping: torch.Tensor, k_scale: float, v_scale: float, stream=None) -> None:
    """Quantizing store: bf16 rows [N, Hkv, D] into E4M3 caches [blocks, bs, Hkv, D] (uint8 or
    float8_e4m3fn tensors) as e4m3(x / scale); slot -1 skips."""
    dev = _device(k, "k")
    _need(k, "k", dtype=torch.bfloat16, ndim=3)
    _need(v, "v", dtype=torch.bfloat16, ndim=3, device=dev)
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _need(t, name, ndim=4, device=dev)
        if t.element_size() != 1:
            raise TypeError(f"{name} must be a one-byte (E4M3) tensor")
    _need(slot_mapping, "slot_mapping", dtype=torch.int32, ndim=1, device=dev)
    if v.shape != k.shape or v_cache.shape != k_cache.shape or k_cache.shape[2:] != k.shape[1:]:
        raise ValueError("expected k, v [N, Hkv, D] and caches [blocks, bs, Hkv, D]")
    if slot_mapping.shape[0] != k.shape[0]:
        raise ValueError("slot_mapping length differs from the number of rows")
    nb, bs, hkv, d = k_cache.shape
    st = _lib.load().pkv_kv_store_fp8(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
                                      k.shape[0], nb, bs, hkv, d, ctypes.c_float(k_scale),
                                      ctypes.c_float(v_scale), _stream(stream, dev))
    _lib.check("pkv_kv_store_fp8", st)


def paged_decode_attn_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                          block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                          k_scale: float, v_scale: float, *, num_splits: int = 0,
                          workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                          stream=None) -> torch.Tensor:
    """Decode attention over an E4M3 cache with per-tensor scales; q / out bf16 [B, Hq, D]."""
    dev = _device(q, "q")
    _need(q, "q", dtype=torch.bfloat16, ndim=3)
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _need(t, name, ndim=4, device=dev)
        if t.element_size() != 1:
            raise TypeError(f"{name} must be a one-byte (E4M3) tensor")
    _need(block_tables, "block_tables", dtype=torch.int32, ndim=2, device=dev)
    _need(context_lens, "context_lens", dtype=torch.int32, ndim=1, device=dev)
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("inconsistent shapes between q, caches, block_tables and context_lens")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", dtype=torch.bfloat16, device=dev, shape=q.shape)
    if workspace is None:
        workspace = decode_workspace(B, hq, d, num_splits, device=dev)
    else:
        _need(workspace, "workspace", device=dev)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib.load().pkv_paged_decode_attn_fp8(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), B, hq, hkv, d, bs, nb, ctypes.c_float(scale), ctypes.c_float(k_scale),
        ctypes.c_float(v_scale), num_splits, ws_ptr, ws_bytes, _stream(stream, dev))
    _lib.check("pkv_paged_decode_attn_fp8", st)
    return out


def decode_workspace_bytes(batch: int, num_q_heads: int, head_dim: int, num_splits: int = 0) -> int:
    """Bytes of split workspace paged_decode_attn needs on the current device."""
    return int(_lib.load().pkv_paged_decode_workspace_bytes(batch, num_q_heads, head_dim, num_splits))


def decode_workspace(batch: int, num_q_heads: int, head_dim: int, num_splits: int = 0,
                     device=None) -> torch.Tensor | None:
    """Allocate a zero-filled workspace (uint8) for paged_decode_attn, or None when none is needed."""
    n = decode_workspace_bytes(batch, num_q_heads, head_dim, num_splits)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device or torch.cuda.current_device())


def paged_decode_attn(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, *,
                      num_splits: int = 0, workspace: torch.Tensor | None = None,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Decode attention through block tables; returns out [B, Hq, D] (same dtype as q).

    num_splits: 0 = automatic split over the context, S >= 1 = S equal parts.
    workspace: from decode_workspace(); allocated (zero-filled) when None.
    """
    dev = _device(q, "q")
    _need(q, "q", ndim=3)
    _need(k_cache, "k_cache", dtype=q.dtype, ndim=4, device=dev)
    _need(v_cache, "v_cache", dtype=q.dtype, ndim=4, device=dev)
    _need(block_tables, "block_tables", dtype=torch.int32, ndim=2, device=dev)
    _need(context_lens, "context_lens", dtype=torch.int32, ndim=1, device=dev)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("inconsistent shapes between q, caches, block_tables and context_lens")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", dtype=q.dtype, device=dev, shape=q.shape)
    if workspace is None:
        workspace = decode_workspace(B, hq, d, num_splits, device=dev)
    else:
        _need(workspace, "workspace", device=dev)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib.load().pkv_paged_decode_attn(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), B, hq, hkv, d, bs, nb, ctypes.c_float(scale), num_splits, ws_ptr, ws_bytes,
        _dtype_code(q), _stream(stream, dev))
    _lib.check("pkv_paged_decode_attn", st)
    return out


def paged_verify_attn(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, *,
                      num_splits: int = 0, workspace: torch.Tensor | None = None,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Speculative-decoding verify attention: q [B, q_len, Hq, D], the last q_len context
    tokens of each sequence, each causally limited to its own position."""
    dev = _device(q, "q")
    _need(q, "q", ndim=4)
    _need(k_cache, "k_cache", dtype=q.dtype, ndim=4, device=dev)
    _need(v_cache, "v_cache", dtype=q.dtype, ndim=4, device=dev, shape=k_cache.shape)
    _need(block_tables, "block_tables", dtype=torch.int32, ndim=2, device=dev)
    _need(context_lens, "context_lens", dtype=torch.int32, ndim=1, device=dev)
    B, ql, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("inconsistent shapes between q, caches, block_tables and context_lens")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", dtype=q.dtype, device=dev, shape=q.shape)
    if workspace is None:
        workspace = decode_workspace(B, ql * hq, d, num_splits, device=dev)
    else:
        _need(workspace, "workspace", device=dev)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib.load().pkv_paged_verify_attn(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), B, ql, hq, hkv, d, bs, nb, ctypes.c_float(scale), num_splits, ws_ptr, ws_bytes,
        _dtype_code(q), _stream(stream, dev))
    _lib.check("pkv_paged_verify_attn", st)
    return out


def paged_decode_attn_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                              block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, *,
                              num_splits: int = 0, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """paged_decode_attn for callers that cannot allocate: the split workspace is the
    library's fixed 8 MiB device array (calls on one device must not overlap)."""
    dev = _device(q, "q")
    _need(q, "q", ndim=3)
    _need(k_cache, "k_cache", dtype=q.dtype, ndim=4, device=dev)
    _need(v_cache, "v_cache", dtype=q.dtype, ndim=4, device=dev, shape=k_cache.shape)
    _need(block_tables, "block_tables", dtype=torch.int32, ndim=2, device=dev)
    _need(context_lens, "context_lens", dtype=torch.int32, ndim=1, device=dev)
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("inconsistent shapes between q, caches, block_tables and context_lens")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", dtype=q.dtype, device=dev, shape=q.shape)
    st = _lib.load().pkv_paged_decode_attn_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), B, hq, hkv, d, bs, nb, ctypes.c_float(scale), num_splits, _dtype_code(q),
        _stream(stream, dev))
    _lib.check("pkv_paged_decode_attn_noalloc", st)
    return out


def prefill_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                            max_seqlen_q: int) -> int:
    """Bytes of the optional split workspace of paged_varlen_prefill_attn (0: never splits)."""
    return int(_lib.load().pkv_paged_varlen_prefill_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim,
                                                                     max_seqlen_q))


def prefill_workspace(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, max_seqlen_q: int,
                      device=None) -> torch.Tensor | None:
    """A zero-filled workspace (uint8) for paged_varlen_prefill_attn, or None when none is needed."""
    n = prefill_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_seqlen_q)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device or torch.cuda.current_device())


_prefill_ws: dict[int, torch.Tensor] = {}


def _cached_prefill_workspace(nbytes: int, device: torch.device) -> torch.Tensor:
    """One zero-filled workspace per device, grown on demand; the kernel leaves it zeroed."""
    idx = device.index if device.index is not None else torch.cuda.current_device()
    ws = _prefill_ws.get(idx)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        _prefill_ws[idx] = ws
    return ws


def paged_varlen_prefill_attn(q: torch.Tensor, cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor,
                              max_seqlen_q: int, max_seqlen_k: int, scale: float, *,
                              k: torch.Tensor | None = None, v: torch.Tensor | None = None,
                              k_cache: torch.Tensor | None = None, v_cache: torch.Tensor | None = None,
                              block_tables: torch.Tensor | None = None, causal: bool = True,
                              workspace: torch.Tensor | bool | None = None,
                              out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Packed varlen prefill attention; keys through block_tables (cache) or from packed k/v.

    workspace: None = a zero-filled workspace cached per device (calls that may
    overlap on different streams must pass their own); False = never split long
    query tiles; or a tensor from prefill_workspace().
    """
    dev = _device(q, "q")
    _need(q, "q", ndim=3)
    _need(cu_seqlens_q, "cu_seqlens_q", dtype=torch.int32, ndim=1, device=dev)
    _need(cu_seqlens_k, "cu_seqlens_k", dtype=torch.int32, ndim=1, device=dev)
    if cu_seqlens_k.shape != cu_seqlens_q.shape:
        raise ValueError("cu_seqlens_q and cu_seqlens_k lengths differ")
    B = cu_seqlens_q.shape[0] - 1
    total_q, hq, d = q.shape
    if block_tables is not None:
        _need(block_tables, "block_tables", dtype=torch.int32, ndim=2, device=dev)
        _need(k_cache, "k_cache", dtype=q.dtype, ndim=4, device=dev)
        _need(v_cache, "v_cache", dtype=q.dtype, ndim=4, device=dev, shape=k_cache.shape)
        nb, bs, hkv, d2 = k_cache.shape
        if d2 != d:
            raise ValueError("k_cache head_dim differs from q's")
        mb = block_tables.shape[1]
        total_k = 0
        if block_tables.shape[0] != B:
            raise ValueError("block_tables rows must equal the batch")
    else:
        if k is None or v is None:
            raise ValueError("without block_tables the packed k and v are required")
        _need(k, "k", dtype=q.dtype, ndim=3, device=dev)
        _need(v, "v", dtype=q.dtype, ndim=3, device=dev)
        hkv = k.shape[1]
        if k.shape[2] != d:
            raise ValueError("k head_dim differs from q's")
        nb = bs = mb = 0
        total_k = k.shape[0]
        if v.shape != k.shape:
            raise ValueError("k and v shapes differ")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", dtype=q.dtype, device=dev, shape=q.shape)
    ws_bytes = 0
    if workspace is None:
        ws_bytes = prefill_workspace_bytes(B, hq, hkv, d, int(max_seqlen_q))
        workspace = _cached_prefill_workspace(ws_bytes, dev) if ws_bytes > 0 else None
    elif workspace is False:
        workspace = None
    else:
        _need(workspace, "workspace", dtype=torch.uint8, device=dev)
        ws_bytes = workspace.numel()
    st = _lib.load().pkv_paged_varlen_prefill_attn(
        _ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(cu_seqlens_q),
        _ptr(cu_seqlens_k), int(max_seqlen_q), int(max_seqlen_k), _ptr(block_tables), mb, B, total_q,
        total_k, hq, hkv, d, bs, nb, ctypes.c_float(scale), 1 if causal else 0, _ptr(workspace), ws_bytes,
        _dtype_code(q), _stream(stream, dev))
    _lib.check("pkv_paged_varlen_prefill_attn", st)
    return out


def device_error(reset: bool = True) -> int:
    """Read (and by default clear) the current device's error word; synchronises the device."""
    flags = ctypes.c_uint32(0)
    _lib.check("pkv_get_device_error", _lib.load().pkv_get_device_error(ctypes.byref(flags), 1 if reset else 0))
    return int(flags.value)
