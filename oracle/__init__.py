"""CPU oracle for paged-KV-cache attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
its Python binding) may import, call or execute anything in this package; only
the test suite, the smoke check and the CPU-baseline leg of the benchmark do.

The oracle is a plain, slow, obviously correct restatement of what the hot
path computes, in float64 numpy:

* ``metadata``  -- the host-side tensors the kernels consume: ``slot_mapping``,
  ``cu_seqlens_q/k``, ``max_seqlen_q/k``, ``context_lens`` and the padded
  ``block_tables`` matrix ("3.6 ModelRunner, CUDA Graph, and benchmarks",
  section 2 "Turning sequences into tensors"), and the block-count rules of
  "Warmup Guide -- Inference Serving Internals", chapter 3.
* ``attention`` -- the slot scatter (``kv_store``), paged decode attention,
  its split partitions and log-sum-exp combine, and varlen / chunked prefill
  attention through ``block_tables``.

It shares no code, header, table or helper with the CUDA path.

Pin status of each function (what fixes it other than itself; the tests under
``tests/test_oracle_*.py`` hold the pins):

* metadata.prepare_prefill / prepare_decode / blocks_needed / append_needs_block:
  pinned to the worked example printed in section 2 of "3.6 ModelRunner ..."
  (golden fixture) and to the boundary cases of chapter 3 of the Warmup Guide.
* attention.kv_store: pinned by the byte-copy closed form (every written slot
  equals its source row, every other byte unchanged, slot -1 skipped).
* attention.paged_decode_attention / paged_prefill_attention: pinned to
  hand-computed golden values, closed forms (ctx=1, equal keys, constant V,
  dominant logit), a textbook contiguous attention built from
  ``scipy.special.softmax`` and brute-force float64 loops on tiny shapes,
  and the block-permutation and prefix-hit invariants.
* fp8.e4m3_encode / e4m3_decode / quantize / kv_store_fp8 (the reduced-precision
  KV cache, a reading: OCP E4M3 with a per-tensor scale): pinned to code values
  fixed by the format definition, round trips of every finite code, torch's
  float8_e4m3fn conversion inside the finite range, saturation and ties to even.
* attention.decode_partials / combine_partials: pinned by the identity that
  merging the partitions of a context reproduces attention over the whole
  context, and by a hand-computed two-partition example.
* The float32 rounding of the GPU path itself is not modelled: the oracle is
  float64 and the comparison uses the stated tolerances (parity of the last
  bits of float arithmetic is unpinned by design).
"""

from . import attention, fp8, metadata  # noqa: F401
