// FP8 (E4M3) KV cache: a quantizing slot scatter and paged decode reading the
// one-byte cache.
//
// The pages name a reduced-precision KV cache ("10 Serving Engines", 10.2.2:
// --kv-cache-dtype; "3.6 ModelRunner, CUDA Graph, and benchmarks", section 4:
// nano-vllm has none) without a format.  This library takes OCP E4M3 with a
// per-tensor scale per K and per V: an element x is stored as
// e4m3(x / scale), rounded to nearest even and saturated to +-448, and read
// back as value(code) * scale.  Decode streams half the bytes of bf16.
#include "decode_launch.cuh"

namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Two floats to two E4M3 codes (x0 in the low byte), round to nearest even, saturating.
__device__ __forceinline__ uint32_t to_e4m3x2(float x0, float x1) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(x1), "f"(x0));
  return r;
}

// 16 bf16 -> 16 E4M3 codes of x / scale (IEEE division, as the stored value is defined).
__device__ __forceinline__ uint4 quantize16(const uint4& a, const uint4& b, float scale) {
  float f[16];
  pkv::Chunk<__nv_bfloat16>::unpack(a, f);
  pkv::Chunk<__nv_bfloat16>::unpack(b, f + 8);
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = to_e4m3x2(__fdiv_rn(f[4 * i], scale), __fdiv_rn(f[4 * i + 1], scale));
    const uint32_t hi = to_e4m3x2(__fdiv_rn(f[4 * i + 2], scale), __fdiv_rn(f[4 * i + 3], scale));
    w[i] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// One thread per 16 output codes of a token row (all KV heads of the token).
__global__ void __launch_bounds__(256) kv_store_fp8_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                           uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                           const int32_t* __restrict__ slot_mapping,
                                                           int64_t total_chunks, int32_t chunks_per_row,
                                                           int64_t num_slots, float k_scale, float v_scale,
                                                           unsigned int* err) {
  pkv::pdl_enter();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total_chunks;
       idx += stride) {
    const int64_t token = idx / chunks_per_row;
    const int32_t chunk = static_cast<int32_t>(idx - token * chunks_per_row);
    const int32_t slot = __ldg(slot_mapping + token);
    if (slot == -1) continue;
    if (slot < 0 || slot >= num_slots) {
      if (chunk == 0) pkv::raise_error(err, PKV_DERR_SLOT_RANGE);
      continue;
    }
    const int64_t dst = static_cast<int64_t>(slot) * chunks_per_row + chunk;
    k_cache[dst] = quantize16(ld_stream(k + 2 * idx), ld_stream(k + 2 * idx + 1), k_scale);
    v_cache[dst] = quantize16(ld_stream(v + 2 * idx), ld_stream(v + 2 * idx + 1), v_scale);
  }
}

// Every group size runs on the tensor-core kernel, codes widened to f16 in
// registers, two 16-key chunks per warp per stage.
template <int G>
int launch_fp8(Params& p, int sms, cudaStream_t stream) {
  return launch_mma<G, 1, __nv_fp8_e4m3>(p, sms, stream);
}

}  // namespace

extern "C" int pkv_kv_store_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                                const int32_t* slot_mapping, int32_t num_tokens, int32_t num_blocks,
                                int32_t block_size, int32_t num_kv_heads, int32_t head_dim, float k_scale,
                                float v_scale, pkv_stream_t stream) {
  if (num_tokens < 0 || num_blocks < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PKV_EINVAL;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || isinf(k_scale) || isinf(v_scale)) return PKV_EINVAL;
  const int64_t row_codes = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (row_codes % 16 != 0) return PKV_EUNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_EINVAL;
  if (!pkv::aligned16(k) || !pkv::aligned16(v) || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
    return PKV_EALIGN;
  int st = PKV_OK;
  unsigned int* err = pkv::device_error_word(&st);
  if (st != PKV_OK) return st;
  pkv::DeviceInfo info;
  if (pkv::device_info(&info) != PKV_OK) return PKV_ECUDA;
  const int32_t chunks_per_row = static_cast<int32_t>(row_codes / 16);
  const int64_t total = static_cast<int64_t>(num_tokens) * chunks_per_row;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(info.sms) * 8;
  if (blocks > cap) blocks = cap;
  const cudaError_t e = pkv::launch_pdl(
      kv_store_fp8_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, static_cast<const uint4*>(k),
      static_cast<const uint4*>(v), static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slot_mapping, total,
      chunks_per_row, static_cast<int64_t>(num_blocks) * block_size, k_scale, v_scale, err);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

extern "C" int pkv_paged_decode_attn_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                         int32_t num_blocks, float scale, float k_scale, float v_scale,
                                         int32_t num_splits, void* workspace, size_t workspace_bytes,
                                         pkv_stream_t stream) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_blocks < 0 || max_blocks_per_seq < 0 || num_splits < 0)
    return PKV_EINVAL;
  if (num_q_heads % num_kv_heads != 0) return PKV_EINVAL;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || isinf(k_scale) || isinf(v_scale)) return PKV_EINVAL;
  if (head_dim != 128 || num_kv_heads > 8) return PKV_EUNSUPPORTED;
  const int group = num_q_heads / num_kv_heads;
  if (group != 1 && group != 2 && group != 4 && group != 8) return PKV_EUNSUPPORTED;
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
  p.scale_log2 = scale * 1.4426950408889634f * k_scale;
  p.v_scale = v_scale;
  p.num_splits = num_splits;
  switch (group) {
    case 1: return launch_fp8<1>(p, info.sms, stream);
    case 2: return launch_fp8<2>(p, info.sms, stream);
    case 4: return launch_fp8<4>(p, info.sms, stream);
    default: return launch_fp8<8>(p, info.sms, stream);
  }
}
