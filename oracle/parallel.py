"""Runs the oracle's per-sequence attention on every host core.

TEST INFRASTRUCTURE ONLY (see the package docstring).

This module holds none of the method's arithmetic.  Each worker process calls
the unchanged oracle functions of ``oracle.attention`` (and ``oracle.fp8``)
on some of a batch's sequences; only the loop over sequences is fanned out.

Large inputs (a layer's K/V pools) are written once into files (in /dev/shm
when it has room, else in the temporary directory).  A worker reads the
blocks that a sequence's block table names, in table order, and gives the
oracle those blocks with a table that numbers them 0, 1, 2, ...: the oracle
gathers the sequence's tokens through that table exactly as it would through
the original one, so each output row is what the single-process oracle
computes on the whole pool.  Workers are started with the ``spawn`` method: a
process forked after the parent initialised CUDA can hang.
"""

from __future__ import annotations

import multiprocessing as mp
import os
import shutil
import tempfile

import numpy as np

_FILES: dict = {}  # worker side: path -> open file


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux
        return os.cpu_count() or 1


def _worker_init() -> None:
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"


def _is_file_spec(spec) -> bool:
    return isinstance(spec, tuple) and len(spec) == 3 and isinstance(spec[0], str)


def _read_rows(spec, index) -> np.ndarray:
    """Rows ``index`` (along the first axis) of a shared file, read into private memory.

    One read per row (a cache block is contiguous), so a worker never maps the
    whole file."""
    path, shape, dtype = spec
    f = _FILES.get(path)
    if f is None:
        for old in list(_FILES):  # files of earlier batches: removed or no longer used
            _FILES.pop(old).close()
        f = _FILES[path] = open(path, "rb", buffering=0)
    dt = np.dtype(dtype)
    row = int(np.prod(shape[1:], dtype=np.int64)) * dt.itemsize
    index = np.asarray(index, dtype=np.int64).reshape(-1)
    out = np.empty((len(index),) + tuple(shape[1:]), dtype=dt)
    if len(index) == 0:
        return out
    flat = out.reshape(len(index), -1).view(np.uint8)
    for j, r in enumerate(index.tolist()):
        if not 0 <= r < shape[0]:
            raise IndexError(f"row {r} outside a shared array of {shape[0]} rows")
        f.seek(r * row)
        if f.readinto(memoryview(flat[j])) != row:
            raise IOError(f"short read from {path}")
    return out


def _arg(specs: dict, name: str, index):
    """Rows ``index`` of an argument: read from its shared file, or taken from the array passed."""
    spec = specs[name]
    if _is_file_spec(spec):
        return _read_rows(spec, index)
    return np.asarray(spec)[np.asarray(index, dtype=np.int64)]


def _block_size(spec) -> int:
    return int(spec[1][1]) if _is_file_spec(spec) else int(np.asarray(spec).shape[1])


def _own_blocks(table_row, num_tokens: int, block_size: int):
    """The blocks holding a sequence's first num_tokens tokens, in table order, and the table that
    numbers them 0, 1, 2, ..."""
    nblk = -(-num_tokens // block_size)
    return np.asarray(table_row[:nblk], dtype=np.int64), np.arange(nblk, dtype=np.int64)[None, :]


def _decode_rows(specs: dict, rows: list[int]):
    """oracle.attention.paged_decode_attention for each of ``rows`` over its own blocks."""
    from oracle import attention as oa

    bt = np.asarray(specs["block_tables"])
    cl = np.asarray(specs["context_lens"])
    bs = _block_size(specs["k_cache"])
    outs = []
    for b in rows:
        blocks, local = _own_blocks(bt[b], int(cl[b]), bs)
        kb, vb = _arg(specs, "k_cache", blocks), _arg(specs, "v_cache", blocks)
        outs.append(oa.paged_decode_attention(_arg(specs, "q", [b]), kb, vb, local, cl[b:b + 1], specs["scale"]))
    return rows, np.concatenate(outs)


def _decode_fp8_rows(specs: dict, rows: list[int]):
    """Decode over an E4M3 cache: each row's blocks read back with oracle.fp8.dequantize, then
    oracle.attention.paged_decode_attention over them."""
    from oracle import attention as oa
    from oracle import fp8 as of8

    bt = np.asarray(specs["block_tables"])
    cl = np.asarray(specs["context_lens"])
    bs = _block_size(specs["k_codes"])
    outs = []
    for b in rows:
        blocks, local = _own_blocks(bt[b], int(cl[b]), bs)
        kb = of8.dequantize(_arg(specs, "k_codes", blocks), specs["k_scale"])
        vb = of8.dequantize(_arg(specs, "v_codes", blocks), specs["v_scale"])
        outs.append(oa.paged_decode_attention(_arg(specs, "q", [b]), kb, vb, local, cl[b:b + 1], specs["scale"]))
    return rows, np.concatenate(outs)


def _prefill_seq(specs: dict, i: int):
    """oracle.attention.paged_prefill_attention of sequence i alone: its own cu_seqlens pair, and
    its blocks (or its rows of the packed k, v)."""
    from oracle import attention as oa

    cu_q = np.asarray(specs["cu_seqlens_q"])
    cu_k = np.asarray(specs["cu_seqlens_k"])
    q0, q1 = int(cu_q[i]), int(cu_q[i + 1])
    k0, k1 = int(cu_k[i]), int(cu_k[i + 1])
    cu_q1 = np.array([0, q1 - q0])
    cu_k1 = np.array([0, k1 - k0])
    q = _arg(specs, "q", range(q0, q1))
    if specs.get("block_tables") is not None:
        blocks, local = _own_blocks(np.asarray(specs["block_tables"])[i], k1 - k0, _block_size(specs["k_cache"]))
        out = oa.paged_prefill_attention(q, cu_q1, cu_k1, specs["scale"], k_cache=_arg(specs, "k_cache", blocks),
                                         v_cache=_arg(specs, "v_cache", blocks), block_tables=local,
                                         causal=specs["causal"])
    else:
        out = oa.paged_prefill_attention(q, cu_q1, cu_k1, specs["scale"], k=_arg(specs, "k", range(k0, k1)),
                                         v=_arg(specs, "v", range(k0, k1)), causal=specs["causal"])
    return i, out


class OraclePool:
    """A pool of ``workers`` spawned processes running the oracle, and the shared files they read."""

    def __init__(self, workers: int | None = None):
        self.workers = workers or host_cores()
        self._pool = mp.get_context("spawn").Pool(self.workers, initializer=_worker_init)
        self._dirs: list[str] = []

    # ------------------------------------------------------------ shared inputs
    def _new_dir(self, nbytes: int) -> str:
        for base in ("/dev/shm", tempfile.gettempdir()):
            try:
                if os.path.isdir(base) and shutil.disk_usage(base).free > nbytes + (1 << 30):
                    d = tempfile.mkdtemp(prefix="oracle-", dir=base)
                    self._dirs.append(d)
                    return d
            except OSError:
                continue
        raise RuntimeError(f"no room for {nbytes / 1e9:.1f} GB of shared oracle inputs")

    def shared(self, arrays: dict) -> tuple[dict, dict]:
        """Writable shared files for ``arrays`` {name: (shape, dtype)}.

        Returns (views, specs): fill the views in the parent (then drop them),
        pass the specs to the run functions.  Files from earlier calls are
        removed first.
        """
        self.release()
        total = sum(int(np.prod(shape)) * np.dtype(dt).itemsize for shape, dt in arrays.values())
        d = self._new_dir(total)
        views, specs = {}, {}
        for name, (shape, dt) in arrays.items():
            path = os.path.join(d, name + ".bin")
            views[name] = np.memmap(path, dtype=np.dtype(dt), mode="w+", shape=tuple(shape))
            specs[name] = (path, tuple(int(x) for x in shape), np.dtype(dt).str)
        return views, specs

    def release(self) -> None:
        for d in self._dirs:
            shutil.rmtree(d, ignore_errors=True)
        self._dirs = []

    # ------------------------------------------------------------ runs
    def _rows(self, fn, specs: dict, batch: int, chunk: int) -> np.ndarray:
        tasks = [(specs, list(range(b, min(batch, b + chunk)))) for b in range(0, batch, chunk)]
        out = None
        for rows, o in self._pool.starmap(fn, tasks, chunksize=1):
            if out is None:
                out = np.zeros((batch,) + o.shape[1:], dtype=np.float64)
            out[rows] = o
        return out if out is not None else np.zeros((0,), dtype=np.float64)

    def decode(self, specs: dict, batch: int, chunk: int = 1) -> np.ndarray:
        """oracle.attention.paged_decode_attention over the whole batch, ``chunk`` rows per task.

        ``specs``: k_cache, v_cache, q (shared-file specs or arrays), block_tables,
        context_lens (arrays) and the float ``scale``.
        """
        return self._rows(_decode_rows, specs, batch, chunk)

    def decode_fp8(self, specs: dict, batch: int, chunk: int = 1) -> np.ndarray:
        """Decode over an E4M3 cache: ``specs`` as for decode with k_codes, v_codes in place of the
        caches, plus k_scale and v_scale."""
        return self._rows(_decode_fp8_rows, specs, batch, chunk)

    def prefill(self, specs: dict, batch: int, total_q: int) -> np.ndarray:
        """oracle.attention.paged_prefill_attention, one task per sequence.

        ``specs``: q, cu_seqlens_q/k, scale, causal, and either k_cache, v_cache,
        block_tables or the packed k, v.
        """
        out = np.zeros((0,), dtype=np.float64)
        cu_q = np.asarray(specs["cu_seqlens_q"])
        for i, o in self._pool.starmap(_prefill_seq, [(specs, i) for i in range(batch)], chunksize=1):
            if out.shape[0] != total_q:
                out = np.zeros((total_q,) + o.shape[1:], dtype=np.float64)
            out[int(cu_q[i]):int(cu_q[i]) + o.shape[0]] = o
        return out

    def close(self) -> None:
        self._pool.terminate()
        self._pool.join()
        self.release()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
