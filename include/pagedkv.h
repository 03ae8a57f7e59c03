/*
 * pagedkv.h -- C ABI of the paged KV-cache attention library (libpagedkv.so).
 *
 * Three operations, each the kernel-level step named in "3.6 ModelRunner,
 * CUDA Graph, and benchmarks" (a walk through nano-vllm's engine loop):
 *
 *   pkv_kv_store                  writes each new token's K/V row into its cache slot
 *                                 (section 2, "Turning sequences into tensors": slot =
 *                                 physical_block_id * block_size + offset_in_block;
 *                                 section 5: slot -1 writes nothing)
 *   pkv_paged_decode_attn         one query token per sequence, attention over
 *                                 context_lens[b] cached tokens gathered through the
 *                                 block table (section 2, decode; section 5, padding
 *                                 rows with context_lens 0), split over the context with
 *                                 a log-sum-exp combine
 *   pkv_paged_varlen_prefill_attn packed variable-length (chunked) prefill with
 *                                 cu_seqlens_q / cu_seqlens_k, reading prefix-cached
 *                                 history through block_tables when K is longer than Q
 *                                 (section 2, prepare_prefill)
 *
 * Attention is softmax(scale * q K^T) V per query head; query head h reads KV
 * head h / (num_q_heads / num_kv_heads) (grouped-query attention, contiguous
 * groups).  Call order is the caller's: store first, then attend, so the new
 * token is part of its own context (section 2: context_lens counts it).
 *
 * Cache layout for one layer (section 4, "How KV Cache GPU memory is carved
 * out"): k_cache and v_cache are each [num_blocks, block_size, num_kv_heads,
 * head_dim], row-major and contiguous, in the element type given by `dtype`.
 * A whole-model cache (2, layers, blocks, block_size, kv_heads, head_dim)
 * is passed one layer slice at a time.
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" must be device memory (or managed memory)
 *    of the current CUDA device; the library dereferences them only on the
 *    GPU.  Tensor pointers must be 16-byte aligned.
 *  - The caller owns every buffer.  The library allocates no device memory
 *    (pkv_paged_decode_attn_noalloc's fixed scratch is part of the library's
 *    device image, not an allocation).
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream);
 *    nothing synchronises.  Argument errors are detected on the host and
 *    returned as a negative pkv_status before anything is launched.
 *  - Kernels are launched with programmatic dependent launch: each one waits
 *    for every earlier kernel in the stream to complete before touching
 *    memory, and releases the next kernel for scheduling at its start.  A
 *    caller's own kernel launched with programmatic stream serialization
 *    after one of these must therefore execute griddepcontrol.wait (or
 *    cudaGridDependencySynchronize) before reading this library's outputs,
 *    as that launch mode requires anyway.
 *  - Indices read on the device (slots, block ids, context lengths, cu_seqlens)
 *    are range-checked by the kernels: an out-of-range value skips the access
 *    and raises a bit in the per-device error word (pkv_get_device_error);
 *    the kernels never trap.
 *  - Element offsets are computed in 64-bit; counts are int32.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* pkv_stream_t;

typedef enum {
  PKV_F32 = 0,  /* float32 K/V/q/out */
  PKV_BF16 = 1  /* bfloat16 K/V/q/out; arithmetic in float32 */
} pkv_dtype;

typedef enum {
  PKV_OK = 0,
  PKV_EINVAL = -1,       /* null pointer, negative or inconsistent size */
  PKV_EUNSUPPORTED = -2, /* head_dim / head grouping / dtype combination not built */
  PKV_EALIGN = -3,       /* a tensor pointer is not 16-byte aligned */
  PKV_ECUDA = -4,        /* the CUDA runtime reported an error (query or launch) */
  PKV_EWORKSPACE = -5,   /* split workspace missing or smaller than required */
  PKV_ESCRATCH = -6      /* pkv_paged_decode_attn_noalloc: sizes exceed its fixed scratch */
} pkv_status;

/* Size of the fixed scratch array behind pkv_paged_decode_attn_noalloc. */
#define PKV_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

/* Device error word bits (pkv_get_device_error). */
#define PKV_DERR_SLOT_RANGE 0x1u     /* kv_store: slot >= num_blocks * block_size or < -1 */
#define PKV_DERR_BLOCK_RANGE 0x2u    /* a block table entry that must be read is outside [0, num_blocks) */
#define PKV_DERR_LEN_RANGE 0x4u      /* context_lens / cu_seqlens inconsistent with the table width or the batch */
#define PKV_DERR_WAIT_TIMEOUT 0x8u   /* a pipeline wait gave up (about 1 s); the results are invalid */

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int pkv_version(void);

/* Static string for a pkv_status value. */
const char* pkv_status_string(int status);

/*
 * Reads (and with reset != 0 clears) the current device's error word.
 * Synchronises the device.  Returns PKV_OK or PKV_ECUDA.
 */
int pkv_get_device_error(uint32_t* flags, int reset);

/*
 * kv_store: for every i in [0, num_tokens) with slot_mapping[i] >= 0,
 *   k_cache[slot / block_size, slot % block_size, :, :] = k[i, :, :]   and the same for v.
 * slot_mapping[i] == -1 (batch padding) writes nothing.  A byte copy: the
 * result is bit-exact, and cache bytes of other slots are untouched.
 *
 *   k, v            device, [num_tokens, num_kv_heads, head_dim], contiguous
 *   k_cache, v_cache device, [num_blocks, block_size, num_kv_heads, head_dim]
 *   slot_mapping    device, int32 [num_tokens]
 *   num_tokens >= 0 (0 launches nothing); num_kv_heads * head_dim * element size
 *   must be a multiple of 16 bytes.
 * Duplicate slots among rows are a caller error (which row lands is unspecified).
 */
int pkv_kv_store(const void* k, const void* v, void* k_cache, void* v_cache,
                 const int32_t* slot_mapping, int32_t num_tokens, int32_t num_blocks,
                 int32_t block_size, int32_t num_kv_heads, int32_t head_dim, pkv_dtype dtype,
                 pkv_stream_t stream);

/*
 * Bytes of split workspace pkv_paged_decode_attn needs on the current device
 * for these sizes (0 when num_splits == 1).  num_splits: 0 = automatic
 * (the context tokens of the whole batch are divided evenly over a grid sized
 * to the GPU), S >= 1 = every sequence's context cut into S equal parts (on
 * the tensor-core path, split points are rounded up to multiples of 16 tokens).
 * Returns 0 and sets nothing on invalid sizes; a CUDA query failure also returns 0.
 */
size_t pkv_paged_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t head_dim,
                                        int32_t num_splits);

/*
 * paged_decode_attn: for each sequence b and query head h (kv head g = h / G,
 * G = num_q_heads / num_kv_heads), with T = context_lens[b]:
 *   s_t = scale * q[b, h, :] . K_t,    K_t = k_cache[block_tables[b, t / block_size], t % block_size, g, :]
 *   out[b, h, :] = sum_{t < T} softmax(s)_t V_t       (V_t likewise from v_cache)
 * T == 0 (padding row) reads nothing and writes zeros.  Only the first
 * ceil(T / block_size) entries of row b of block_tables are read; -1 padding
 * or stale ids to their right are never touched.
 *
 *   out             device, [batch, num_q_heads, head_dim]
 *   q               device, [batch, num_q_heads, head_dim]
 *   k_cache,v_cache device, [num_blocks, block_size, num_kv_heads, head_dim]
 *   block_tables    device, int32 [batch, max_blocks_per_seq]
 *   context_lens    device, int32 [batch], each in [0, max_blocks_per_seq * block_size]
 *   num_splits      0 = automatic, S >= 1 = S equal parts per sequence (1 = no split)
 *   workspace       device, >= pkv_paged_decode_workspace_bytes(...) bytes, 256-byte
 *                   aligned; may be NULL when that is 0.  It must be zero-filled once
 *                   after allocation.  Its first 64 KiB hold ticket counters only, which
 *                   every call leaves at zero again; partial results follow them.  So
 *                   calls of any sizes, eager or replayed from CUDA graphs, may share it
 *                   (and share it with pkv_paged_varlen_prefill_attn, whose workspace
 *                   starts with the same counter area); only batches whose batch + parts
 *                   exceed 16,384 counters extend the area.  A call that raised
 *                   PKV_DERR_WAIT_TIMEOUT may leave counters set: zero the workspace again
 *                   after one.  Calls sharing a workspace must not overlap in time.
 * Supported: head_dim in {64, 128}; G in {1, 2, 4, 8}; num_kv_heads in [1, 8];
 * dtype F32 or BF16.
 */
int pkv_paged_decode_attn(void* out, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                          const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t num_blocks, float scale, int32_t num_splits, void* workspace,
                          size_t workspace_bytes, pkv_dtype dtype, pkv_stream_t stream);

/*
 * paged_verify_attn: the target pass of speculative decoding ("Warmup Guide --
 * Inference Serving Internals", chapter 7: the target scores all drafted
 * positions in one parallel pass).  Each sequence b has q_len query tokens,
 * the last q_len positions of its context (their K/V stored first with
 * pkv_kv_store, as decode stores its one new token).  Query token i of
 * sequence b sits at position T - q_len + i (T = context_lens[b]) and attends
 * cached tokens 0 .. T - q_len + i:
 *   out[b, i, h, :] = sum_{t <= T - q_len + i} softmax(scale * q[b, i, h, :] . K_t) V_t
 * with K_t / V_t gathered through block_tables as in paged_decode_attn.
 * q_len == 1 is paged_decode_attn.
 *
 *   out, q          device, [batch, q_len, num_q_heads, head_dim]
 *   context_lens    device, int32 [batch]; each is 0 (padding row: zeros, nothing
 *                   read) or in [q_len, max_blocks_per_seq * block_size]; a value
 *                   in [1, q_len) raises PKV_DERR_LEN_RANGE and the row reads nothing
 *   workspace       as for paged_decode_attn, sized by
 *                   pkv_paged_decode_workspace_bytes(batch, q_len * num_q_heads,
 *                   head_dim, num_splits)
 *   other arguments as for paged_decode_attn.
 * Supported: BF16, head_dim 128, G in {1, 2, 4, 8}, q_len <= 8 with
 * G * q_len <= 16, num_kv_heads in [1, 8].
 */
int pkv_paged_verify_attn(void* out, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                          const int32_t* context_lens, int32_t batch, int32_t q_len,
                          int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, int32_t num_blocks, float scale, int32_t num_splits,
                          void* workspace, size_t workspace_bytes, pkv_dtype dtype,
                          pkv_stream_t stream);

/*
 * copy_blocks: the copy of copy-on-write prefix sharing ("Warmup Guide --
 * Inference Serving Internals", chapter 4: a sequence about to write into a
 * block it shares copies that block first and writes into the copy).  For
 * every pair (src, dst) of block_pairs and every layer l, block dst of
 * k_caches[l] and of v_caches[l] becomes a byte copy of block src.
 *
 *   k_caches, v_caches HOST arrays of num_layers device pointers (<= 128 layers),
 *                   each a pool of num_blocks blocks of block_bytes bytes
 *                   (block_size * num_kv_heads * head_dim * element size)
 *   block_pairs     device, int32 [num_pairs, 2]: (src, dst); a pair with an id
 *                   outside [0, num_blocks) is skipped and raises
 *                   PKV_DERR_BLOCK_RANGE; src == dst copies nothing
 *   block_bytes     multiple of 16
 * A destination that is also a source in the same call, or two pairs with the
 * same destination, is a caller error (the result is unspecified).
 */
int pkv_copy_blocks(void* const* k_caches, void* const* v_caches, int32_t num_layers,
                    const int32_t* block_pairs, int32_t num_pairs, int32_t num_blocks,
                    int64_t block_bytes, pkv_stream_t stream);

/*
 * FP8 KV cache.  The pages name a reduced-precision cache ("10 Serving
 * Engines", 10.2.2, --kv-cache-dtype) without a format; this library stores
 * OCP FP8 E4M3 with one float scale for K and one for V (per layer): an
 * element x is stored as e4m3(x / scale), rounded to nearest even and
 * saturated to +-448, and read back as value(code) * scale.  The cache layout
 * is the bf16 one with one byte per element.
 *
 * kv_store_fp8: pkv_kv_store's slot scatter, quantizing bf16 rows.
 *   k, v            device, bf16 [num_tokens, num_kv_heads, head_dim]
 *   k_cache, v_cache device, E4M3 bytes [num_blocks, block_size, num_kv_heads, head_dim]
 *   k_scale, v_scale finite and > 0
 * The division x / scale is an IEEE float32 division, so the stored codes are
 * exactly determined.  num_kv_heads * head_dim must be a multiple of 16.
 */
int pkv_kv_store_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                     const int32_t* slot_mapping, int32_t num_tokens, int32_t num_blocks,
                     int32_t block_size, int32_t num_kv_heads, int32_t head_dim, float k_scale,
                     float v_scale, pkv_stream_t stream);

/*
 * paged_decode_attn over an FP8 E4M3 cache: the same result as
 * pkv_paged_decode_attn on the dequantized cache (value(code) * scale).
 *   q, out          device, bf16 [batch, num_q_heads, head_dim]
 *   k_cache,v_cache device, E4M3 bytes, layout as above
 *   workspace       as for pkv_paged_decode_attn (same size function)
 * Supported: head_dim 128; G in {1, 2, 4, 8}; num_kv_heads in [1, 8].
 */
int pkv_paged_decode_attn_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int32_t num_blocks, float scale, float k_scale, float v_scale,
                              int32_t num_splits, void* workspace, size_t workspace_bytes,
                              pkv_stream_t stream);

/*
 * paged_decode_attn without a caller-provided workspace (no counterpart in the
 * pages: it is an addition of this library).
 *
 * For callers that cannot allocate device memory -- hooks running inside
 * another engine's execution step where the allocator is off limits,
 * runtimes whose device memory belongs to a pool this library cannot reach,
 * and latency-critical code that must not pay cudaMalloc's implicit
 * synchronisation.  It computes exactly what pkv_paged_decode_attn computes,
 * with the same arguments minus the workspace, and allocates nothing: no
 * cudaMalloc, cudaFree or allocating library call.
 *
 * The split workspace is a fixed array of PKV_NOALLOC_SCRATCH_BYTES bytes
 * (8 MiB) inside the library's device image, held by every GPU that
 * loads the library until the process exits.  Sizes whose workspace
 * (pkv_paged_decode_workspace_bytes) exceeds it return PKV_ESCRATCH without
 * launching; with 152 SMs, 16 query heads and head_dim 128 the automatic
 * split fits batches up to about 700.  Every argument is checked first, as
 * for pkv_paged_decode_attn: a call that returns an error has queued nothing
 * on `stream`.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call clears the array's ticket counters
 * (cudaMemsetAsync on `stream`) and then reuses the array, which keeps the
 * previous call's contents otherwise.  All calls on a device share the one
 * array: calls that overlap on the GPU (different streams without ordering)
 * race and give wrong results.
 */
int pkv_paged_decode_attn_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int32_t num_blocks, float scale, int32_t num_splits, pkv_dtype dtype,
                                  pkv_stream_t stream);

/*
 * paged_varlen_prefill_attn: sequence i owns query rows cu_seqlens_q[i] ..
 * cu_seqlens_q[i+1]-1 (nq rows, the tokens computed in this scheduler step) and nk =
 * cu_seqlens_k[i+1] - cu_seqlens_k[i] keys; the first c = nk - nq keys are
 * history.  Query row r is at absolute position c + r and, when causal, attends
 * keys 0 .. c + r (bottom-right aligned); otherwise all nk keys.
 *
 * Keys/values come from the paged cache through block_tables when
 * block_tables != NULL (the new rows must have been stored first with
 * pkv_kv_store), else from the packed k, v rows cu_seqlens_k[i] .. cu_seqlens_k[i+1]-1.
 *
 *   out             device, [total_q, num_q_heads, head_dim]
 *   q               device, [total_q, num_q_heads, head_dim]
 *   k, v            device, [total_k, num_kv_heads, head_dim]; read only when block_tables == NULL
 *   k_cache,v_cache device, cache layout above; read only when block_tables != NULL
 *   cu_seqlens_q/k  device, int32 [batch + 1], non-decreasing, starting at 0.  A
 *                   sequence whose rows fall outside q / out (cu_seqlens_q[i] < 0 or
 *                   cu_seqlens_q[i+1] > total_q), with nq < 0 or nk < nq, with nq >
 *                   max_seqlen_q, with more keys than its table row covers, or, without
 *                   block_tables, with key rows outside [0, total_k), is skipped (its
 *                   output rows are not written) and raises PKV_DERR_LEN_RANGE
 *   max_seqlen_q    >= every nq (sizes the grid); max_seqlen_k >= every nk
 *   block_tables    device, int32 [batch, max_blocks_per_seq] or NULL
 *   total_q, total_k rows of q/out and of the packed k/v (total_k is ignored with block_tables)
 *   causal          1 = causal (bottom-right), 0 = full
 *   workspace       device, 256-byte aligned, or NULL.  When the work items (pairs of
 *                   query tiles of 128 / G tokens x KV heads x sequences) fill at most
 *                   half the SMs and the workspace holds at least
 *                   pkv_paged_varlen_prefill_workspace_bytes(...) bytes, the tensor-core
 *                   kernel runs each pair with more than 8 key tiles of 128 as up to
 *                   P = min(8, SMs / pairs) parts over consecutive key ranges
 *                   and merges them (log-sum-exp, in part order, so results do not depend
 *                   on timing).  Otherwise nothing is split.  It must be zero-filled once
 *                   after allocation; its first 64 KiB are the same counter area as in
 *                   pkv_paged_decode_attn's workspace (calls of any sizes may share it).
 *                   Calls sharing a workspace must not overlap in time.
 * Supported: BF16 only; head_dim 64 or 128; G in {1, 2, 4, 8}.  Block sizes that
 * are a multiple of 128, or a divisor of 128 of at least 8, and the packed path run
 * on the tcgen05 tensor-core kernel; other block sizes on an mma.sync kernel (which
 * ignores the workspace, and takes head_dim 128 only: head_dim 64 with such a block
 * size returns PKV_EUNSUPPORTED).
 */
int pkv_paged_varlen_prefill_attn(void* out, const void* q, const void* k, const void* v,
                                  const void* k_cache, const void* v_cache,
                                  const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                  int32_t max_seqlen_q, int32_t max_seqlen_k,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  int32_t batch, int32_t total_q, int32_t total_k,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t block_size, int32_t num_blocks, float scale,
                                  int32_t causal, void* workspace, size_t workspace_bytes,
                                  pkv_dtype dtype, pkv_stream_t stream);

/*
 * Bytes of the optional workspace of pkv_paged_varlen_prefill_attn for these
 * sizes on the current device: a ticket and a ready count per (sequence, KV
 * head, query tile; the tiles rounded up to whole pairs), each array in one
 * 32 KiB half of the 64 KiB counter area, then P records of 66,560 bytes
 * (head_dim 128; 33,792 for 64) per query tile, P as above.  0 when nothing
 * would be split (the items fill the GPU, the shape has no tensor-core path,
 * or no device is present).  This
 * sizing rule is the library's own (the pages' flash-attn call has no
 * workspace); it follows the split-decode workspace above.
 */
size_t pkv_paged_varlen_prefill_workspace_bytes(int32_t batch, int32_t num_q_heads,
                                                int32_t num_kv_heads, int32_t head_dim,
                                                int32_t max_seqlen_q);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
