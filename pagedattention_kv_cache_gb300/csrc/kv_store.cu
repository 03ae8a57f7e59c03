// kv_store: scatter each new token's K and V rows into its paged-cache slot.
//
// "3.6 ModelRunner, CUDA Graph, and benchmarks", section 2: slot =
// physical_block_id * block_size + offset_in_block, so the row of slot s
// starts at element s * num_kv_heads * head_dim of the [num_blocks,
// block_size, Hkv, D] cache; section 5: slot -1 (batch padding) writes
// nothing.  The copy moves 16-byte chunks, so it is bit-exact for any dtype.
#include "common.cuh"

namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// One thread per 16-byte chunk of a token row (all KV heads of the token).
__global__ void __launch_bounds__(256) kv_store_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                       uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                       const int32_t* __restrict__ slot_mapping, int64_t total_chunks,
                                                       int32_t chunks_per_row, int64_t num_slots,
                                                       unsigned int* err) {
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
    const uint4 kv = ld_stream(k + idx);
    const uint4 vv = ld_stream(v + idx);
    k_cache[dst] = kv;
    v_cache[dst] = vv;
  }
}

}  // namespace

extern "C" int pkv_kv_store(const void* k, const void* v, void* k_cache, void* v_cache,
                            const int32_t* slot_mapping, int32_t num_tokens, int32_t num_blocks,
                            int32_t block_size, int32_t num_kv_heads, int32_t head_dim, pkv_dtype dtype,
                            pkv_stream_t stream) {
  if (num_tokens < 0 || num_blocks < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PKV_EINVAL;
  if (dtype != PKV_F32 && dtype != PKV_BF16) return PKV_EUNSUPPORTED;
  const int64_t elt = dtype == PKV_F32 ? 4 : 2;
  const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * elt;
  if (row_bytes % 16 != 0) return PKV_EUNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_EINVAL;
  if (!pkv::aligned16(k) || !pkv::aligned16(v) || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
    return PKV_EALIGN;
  int st = PKV_OK;
  unsigned int* err = pkv::device_error_word(&st);
  if (st != PKV_OK) return st;
  pkv::DeviceInfo info;
  if (pkv::device_info(&info) != PKV_OK) return PKV_ECUDA;

  const int32_t chunks_per_row = static_cast<int32_t>(row_bytes / 16);
  const int64_t total_chunks = static_cast<int64_t>(num_tokens) * chunks_per_row;
  const int threads = 256;
  int64_t blocks = (total_chunks + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(info.sms) * 8;
  if (blocks > cap) blocks = cap;
  kv_store_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), slot_mapping, total_chunks, chunks_per_row,
      static_cast<int64_t>(num_blocks) * block_size, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}
