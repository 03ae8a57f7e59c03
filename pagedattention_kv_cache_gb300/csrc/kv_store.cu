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

// A token row (all KV heads of the token) is cpr 16-byte chunks, and the
// rows of k and v are consecutive, so the batch is one flat run of
// num_tokens * cpr chunks: chunk c belongs to token c / cpr, at chunk c % cpr
// of its row.  Thread t of T takes chunks t, t + T, t + 2T, ..., kBatch at a
// time: their K and V loads (and the slots) go out before any store, so one
// round trip to memory covers them.  Every thread's share differs from the
// others' by at most one chunk, whatever the batch size, and consecutive
// threads take consecutive chunks, so loads and stores stay coalesced (a
// warp's 512 bytes cross at most one row boundary when cpr >= 32).
constexpr int kBatch = 4;
constexpr int kBlocksPerSm = 4;  // resident blocks of 256 threads at this kernel's register count

__global__ void __launch_bounds__(256, kBlocksPerSm) kv_store_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                       uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                       const int32_t* __restrict__ slot_mapping, int64_t chunks,
                                                       int32_t cpr, int32_t cpr_shift, int64_t num_slots,
                                                       unsigned int* err) {
  pkv::pdl_enter();
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // token of chunk c: a shift when cpr is a power of two (cpr_shift >= 0)
  auto token_of = [&](int64_t c) { return cpr_shift >= 0 ? c >> cpr_shift : c / cpr; };
  for (int64_t c0 = t; c0 < chunks; c0 += kBatch * nthreads) {
    uint4 kr[kBatch], vr[kBatch];
    int32_t slot[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t c = c0 + u * nthreads;
      if (c < chunks) {
        slot[u] = __ldg(slot_mapping + token_of(c));
        kr[u] = ld_stream(k + c);
        vr[u] = ld_stream(v + c);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t c = c0 + u * nthreads;
      if (c >= chunks || slot[u] == -1) continue;
      const int64_t within = c - token_of(c) * cpr;
      if (slot[u] < 0 || slot[u] >= num_slots) {
        if (within == 0) pkv::raise_error(err, PKV_DERR_SLOT_RANGE);  // once per token
        continue;
      }
      const int64_t dst = static_cast<int64_t>(slot[u]) * cpr + within;
      k_cache[dst] = kr[u];
      v_cache[dst] = vr[u];
    }
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

  if (row_bytes / 16 > INT32_MAX) return PKV_EUNSUPPORTED;
  const int32_t cpr = static_cast<int32_t>(row_bytes / 16);
  int32_t cpr_shift = -1;
  if ((cpr & (cpr - 1)) == 0) {
    cpr_shift = 0;
    while ((1 << cpr_shift) < cpr) ++cpr_shift;
  }
  const int64_t chunks = static_cast<int64_t>(num_tokens) * cpr;
  const int threads = 256;
  // one chunk per thread until every resident block is in use, then more per thread
  const int64_t cap = static_cast<int64_t>(info.sms) * kBlocksPerSm;
  int64_t blocks = (chunks + threads - 1) / threads;
  if (blocks > cap) blocks = cap;
  const cudaError_t e = pkv::launch_pdl(
      kv_store_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream, static_cast<const uint4*>(k),
      static_cast<const uint4*>(v), static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slot_mapping, chunks,
      cpr, cpr_shift, static_cast<int64_t>(num_blocks) * block_size, err);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}
