// paged_verify_attn: the target-model pass of speculative decoding over a
// paged KV cache ("Warmup Guide -- Inference Serving Internals", chapter 7:
// one target pass scores every drafted position in parallel).  Each sequence
// has q_len query tokens, the last q_len tokens of its context (stored first,
// like decode's new token); query token i attends the cache up to its own
// position context_lens[b] - q_len + i.  It is decode with q_len query rows
// per sequence and runs on the same kernel (decode_mma.cuh): K and V are
// streamed once per KV head for all q_len x G rows, with the same split over
// the context and log-sum-exp combine.
#include "decode_launch.cuh"

namespace {

// Rows per KV head R = G * q_len <= 16: the tensor-core (mma.sync) kernel,
// the same one bf16 decode with head_dim 128 runs on (so q_len 1 is decode).
template <int G, int QL>
int launch_rows(Params& p, int sms, cudaStream_t stream) {
  return launch_mma<G, QL>(p, sms, stream);
}

template <int G>
int dispatch_ql(Params& p, int ql, int sms, cudaStream_t stream) {
  switch (ql) {
    case 1: return launch_rows<G, 1>(p, sms, stream);
    case 2: if constexpr (G * 2 <= 16) return launch_rows<G, 2>(p, sms, stream); break;
    case 3: if constexpr (G * 3 <= 16) return launch_rows<G, 3>(p, sms, stream); break;
    case 4: if constexpr (G * 4 <= 16) return launch_rows<G, 4>(p, sms, stream); break;
    case 5: if constexpr (G * 5 <= 16) return launch_rows<G, 5>(p, sms, stream); break;
    case 6: if constexpr (G * 6 <= 16) return launch_rows<G, 6>(p, sms, stream); break;
    case 7: if constexpr (G * 7 <= 16) return launch_rows<G, 7>(p, sms, stream); break;
    case 8: if constexpr (G * 8 <= 16) return launch_rows<G, 8>(p, sms, stream); break;
    default: break;
  }
  return PKV_EUNSUPPORTED;
}

}  // namespace

extern "C" int pkv_paged_verify_attn(void* out, const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, int32_t batch, int32_t q_len, int32_t num_q_heads,
                                     int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                     float scale, int32_t num_splits, void* workspace, size_t workspace_bytes,
                                     pkv_dtype dtype, pkv_stream_t stream) {
  if (batch < 0 || q_len <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_blocks < 0 || max_blocks_per_seq < 0 || num_splits < 0)
    return PKV_EINVAL;
  if (num_q_heads % num_kv_heads != 0) return PKV_EINVAL;
  if (dtype != PKV_BF16 || head_dim != 128) return PKV_EUNSUPPORTED;
  if (num_kv_heads > 8) return PKV_EUNSUPPORTED;
  const int group = num_q_heads / num_kv_heads;
  if ((group != 1 && group != 2 && group != 4 && group != 8) || group * q_len > 16 || q_len > 8)
    return PKV_EUNSUPPORTED;
  if (static_cast<long long>(max_blocks_per_seq) * block_size > INT32_MAX) return PKV_EINVAL;
  if (batch == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_EINVAL;
  if (!pkv::aligned16(out) || !pkv::aligned16(q) || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
    return PKV_EALIGN;

  pkv::DeviceInfo info;
  if (pkv::device_info(&info) != PKV_OK) return PKV_ECUDA;
  int st = PKV_OK;
  unsigned int* err = pkv::device_error_word(&st);
  if (st != PKV_OK) return st;

  Params p{};
  size_t off_o = 0, off_ml = 0;
  const size_t need =
      workspace_layout(batch, q_len * num_q_heads, head_dim, num_splits, info.sms, &off_o, &off_ml);
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
  p.ql = q_len;
  p.hkv = num_kv_heads;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.v_scale = 1.f;
  p.num_splits = num_splits;
  switch (group) {
    case 1: return dispatch_ql<1>(p, q_len, info.sms, stream);
    case 2: return dispatch_ql<2>(p, q_len, info.sms, stream);
    case 4: return dispatch_ql<4>(p, q_len, info.sms, stream);
    default: return dispatch_ql<8>(p, q_len, info.sms, stream);
  }
}
