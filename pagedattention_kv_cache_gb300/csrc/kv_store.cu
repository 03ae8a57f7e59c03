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

// A token row (all KV heads of the token) is cpr 16-byte chunks.  Lanes are
// grouped per token: a group of lpt lanes (cpr rounded up to a power of two,
// at most 32) takes one piece of kb * lpt chunks of a token, each lane kb
// (<= kBatch) of them.  The slot and every chunk of the piece are loaded
// before anything is stored, so one round trip to memory covers it.  Small
// batches (a decode step's few hundred tokens) take kb = 1 and several pieces
// per row, so they still spread over the SMs.
constexpr int kBatch = 4;
constexpr int kBlocksPerSm = 4;  // resident blocks of 256 threads at this kernel's register count

__global__ void __launch_bounds__(256, kBlocksPerSm) kv_store_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                       uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                       const int32_t* __restrict__ slot_mapping, int64_t units,
                                                       int32_t pieces, int32_t cpr, int32_t lpt, int32_t kb,
                                                       int64_t num_slots, unsigned int* err) {
  pkv::pdl_enter();
  const int lane = threadIdx.x % 32;
  const int sub = lane / lpt;  // unit of this lane inside the warp's group
  const int cl = lane % lpt;
  const int upw = 32 / lpt;    // units per warp pass
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * blockDim.x / 32;
  for (int64_t u0 = warp * upw; u0 < units; u0 += nwarps * upw) {
    const int64_t unit = u0 + sub;
    if (unit >= units) continue;
    const int64_t token = unit / pieces;
    const int c0 = static_cast<int>(unit - token * pieces) * kb * lpt + cl;  // this lane's first chunk
    const int32_t slot = __ldg(slot_mapping + token);
    const uint4* ks = k + token * cpr;
    const uint4* vs = v + token * cpr;
    uint4 kr[kBatch], vr[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int c = c0 + u * lpt;
      if (u < kb && c < cpr) {
        kr[u] = ld_stream(ks + c);
        vr[u] = ld_stream(vs + c);
      }
    }
    if (slot == -1) continue;
    if (slot < 0 || slot >= num_slots) {
      if (c0 == 0) pkv::raise_error(err, PKV_DERR_SLOT_RANGE);
      continue;
    }
    uint4* kd = k_cache + static_cast<int64_t>(slot) * cpr;
    uint4* vd = v_cache + static_cast<int64_t>(slot) * cpr;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int c = c0 + u * lpt;
      if (u < kb && c < cpr) {
        kd[c] = kr[u];
        vd[c] = vr[u];
      }
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
  int32_t lpt = 1;
  while (lpt < cpr && lpt < 32) lpt *= 2;
  const int threads = 256;
  const int64_t cap = static_cast<int64_t>(info.sms) * kBlocksPerSm;
  // kBatch chunks per lane once the batch fills every resident warp, else one
  const int64_t units_full = static_cast<int64_t>(num_tokens) * ((cpr + kBatch * lpt - 1) / (kBatch * lpt));
  const int32_t kb = units_full * lpt / 32 >= cap * (threads / 32) ? kBatch : 1;
  const int32_t pieces = (cpr + kb * lpt - 1) / (kb * lpt);
  const int64_t units = static_cast<int64_t>(num_tokens) * pieces;
  const int64_t units_per_block = (threads / 32) * (32 / lpt);
  int64_t blocks = (units + units_per_block - 1) / units_per_block;
  if (blocks > cap) blocks = cap;
  const cudaError_t e = pkv::launch_pdl(
      kv_store_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream, static_cast<const uint4*>(k),
      static_cast<const uint4*>(v), static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slot_mapping, units,
      pieces, cpr, lpt, kb, static_cast<int64_t>(num_blocks) * block_size, err);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}
