// paged_decode_attn: one query token per sequence, attention over the
// sequence's cached tokens gathered through its block table.
//
// What is computed ("3.6 ModelRunner, CUDA Graph, and benchmarks", section 2,
// decode; section 5, padding rows): for sequence b and query head h reading
// KV head g = h / G, over t < context_lens[b],
//     s_t = scale * q[b, h] . K_t,  out[b, h] = sum_t softmax(s)_t V_t,
// with K_t / V_t at physical block block_tables[b, t / bs], offset t % bs.
// context_lens 0 writes zeros and reads nothing.
//
// How (GB300 design; the kernels are in decode_mma.cuh and decode_simt.cuh,
// launched from decode_launch.cuh):
//  * A CTA covers every KV head of a token range, so each token's K (or V)
//    row of all heads, [Hkv, D], is contiguous in the [blocks, bs, Hkv, D]
//    pool.  A producer warp streams the range into a ring of shared-memory
//    stages with TMA copies completed on mbarriers; every K/V byte is read
//    from HBM once, and all G query heads of a KV head reuse it on chip.
//  * bf16 caches with head_dim 128 run on paged_decode_mma_kernel: each
//    consumer warp takes 16-token chunks and computes S = Q K^T and
//    O^T = V^T P^T with mma.sync, with an online softmax in the exp2 domain on
//    the accumulator fragments.  fp32 caches and head_dim 64 run on
//    paged_decode_kernel (CUDA-core dot products and shuffle reductions).
//  * Split over the context: the batch's context tokens, flattened, are
//    divided evenly over one persistent CTA per SM (automatic mode) or each
//    sequence into S equal parts.  A sequence covered by one CTA is written
//    directly; otherwise each part writes (o, m, l) to the workspace and
//    atomic tickets (no waiting) elect the CTAs that merge the parts by
//    log-sum-exp, in groups of eight consecutive parts and then the groups.
#include "decode_launch.cuh"

extern "C" size_t pkv_paged_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t head_dim,
                                                   int32_t num_splits) {
  if (batch < 0 || num_q_heads <= 0 || head_dim <= 0 || num_splits < 0) return 0;
  pkv::DeviceInfo info;
  if (pkv::device_info(&info) != PKV_OK) return 0;
  size_t a, b;
  return workspace_layout(batch, num_q_heads, head_dim, num_splits, info.sms, &a, &b);
}

namespace {

// Host-side argument checks of pkv_paged_decode_attn (everything but the
// workspace): PKV_OK when a launch may follow, 1 when batch is 0 (nothing to
// do), else the negative status to return.
int check_decode_args(const void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
                      int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int32_t num_blocks, int32_t num_splits, pkv_dtype dtype) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_blocks < 0 || max_blocks_per_seq < 0 || num_splits < 0)
    return PKV_EINVAL;
  if (num_q_heads % num_kv_heads != 0) return PKV_EINVAL;
  if (dtype != PKV_F32 && dtype != PKV_BF16) return PKV_EUNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PKV_EUNSUPPORTED;
  if (num_kv_heads > 8) return PKV_EUNSUPPORTED;
  if (static_cast<long long>(max_blocks_per_seq) * block_size > INT32_MAX) return PKV_EINVAL;
  if (batch == 0) return 1;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_EINVAL;
  if (!pkv::aligned16(out) || !pkv::aligned16(q) || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
    return PKV_EALIGN;
  return PKV_OK;
}

}  // namespace

extern "C" int pkv_paged_decode_attn(void* out, const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                                     int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                     int32_t num_blocks, float scale, int32_t num_splits, void* workspace,
                                     size_t workspace_bytes, pkv_dtype dtype, pkv_stream_t stream) {
  const int chk = check_decode_args(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch,
                                    num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, num_splits, dtype);
  if (chk != PKV_OK) return chk > 0 ? PKV_OK : chk;

  pkv::DeviceInfo info;
  if (pkv::device_info(&info) != PKV_OK) return PKV_ECUDA;
  int st = PKV_OK;
  unsigned int* err = pkv::device_error_word(&st);
  if (st != PKV_OK) return st;

  Params p{};
  size_t off_o = 0, off_ml = 0;
  const size_t need = workspace_layout(batch, num_q_heads, head_dim, num_splits, info.sms, &off_o, &off_ml);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return PKV_EWORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PKV_EALIGN;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    p.counters = reinterpret_cast<int32_t*>(ws);
    p.part_o = reinterpret_cast<float*>(ws + off_o);
    p.part_ml = reinterpret_cast<float*>(ws + off_ml);
  }
  p.out = out;
  p.q = q;
  p.k_cache = static_cast<const unsigned char*>(k_cache);
  p.v_cache = static_cast<const unsigned char*>(v_cache);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.err = err;
  p.max_blocks = max_blocks_per_seq;
  p.batch = batch;
  p.hq = num_q_heads;
  p.ql = 1;
  p.hkv = num_kv_heads;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.v_scale = 1.f;
  p.num_splits = num_splits;
  const int group = num_q_heads / num_kv_heads;
  if (dtype == PKV_BF16) {
    if (head_dim == 128) return dispatch_g<__nv_bfloat16, 128>(p, group, info.sms, stream);
    return dispatch_g<__nv_bfloat16, 64>(p, group, info.sms, stream);
  }
  if (head_dim == 128) return dispatch_g<float, 128>(p, group, info.sms, stream);
  return dispatch_g<float, 64>(p, group, info.sms, stream);
}

// ------------------------------------------------------------------ no-allocation variant
//
// Some callers cannot allocate device memory for the split workspace: code
// running inside another engine's execution hook that must not touch the
// allocator, runtimes whose memory is owned by a pool this library cannot
// see, and latency-critical paths that must avoid cudaMalloc's implicit
// device synchronisation.  pkv_paged_decode_attn_noalloc serves them with a
// fixed-size scratch array that lives in the library's own device image.

namespace {

constexpr size_t kNoAllocScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;  // 8 MiB per device

// Device-side scratch.  In host code this name is only a host stand-in; its
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of this device's scratch array, looked up once per device
// with that device current.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return PKV_ECUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PKV_ECUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" int pkv_paged_decode_attn_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                                             const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                             int32_t num_blocks, float scale, int32_t num_splits, pkv_dtype dtype,
                                             pkv_stream_t stream) {
  // every argument is checked before anything is queued on the stream (the
  // memset below included)
  const int chk = check_decode_args(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch,
                                    num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, num_splits, dtype);
  if (chk != PKV_OK) return chk > 0 ? PKV_OK : chk;
  pkv::DeviceInfo info;
  if (pkv::device_info(&info) != PKV_OK) return PKV_ECUDA;
  size_t off_o = 0, off_ml = 0;
  const size_t need = workspace_layout(batch, num_q_heads, head_dim, num_splits, info.sms, &off_o, &off_ml);
  if (need > kNoAllocScratchBytes) return PKV_ESCRATCH;
  void* scratch = nullptr;
  if (need > 0) {
    const int st = noalloc_scratch(&scratch);
    if (st != PKV_OK) return st;
    // the ticket counters must start at zero; the array keeps the previous call's contents
    if (cudaMemsetAsync(scratch, 0, off_o, stream) != cudaSuccess) return PKV_ECUDA;
  }
  return pkv_paged_decode_attn(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch,
                               num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, num_splits, scratch,
                               need > 0 ? kNoAllocScratchBytes : 0, dtype, stream);
}
