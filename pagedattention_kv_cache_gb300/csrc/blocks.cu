// copy_blocks: the copy half of copy-on-write block sharing.
//
// "Warmup Guide -- Inference Serving Internals", chapter 4: sequences that
// share a prefix point their block tables at the same physical blocks; a
// sequence about to write into a shared block first copies that one block
// and writes into its private copy.  This kernel performs those copies for
// every layer's K and V pool in one launch: block dst of each pool becomes a
// byte copy of block src.
#include "common.cuh"

namespace {

constexpr int kMaxLayers = 128;

struct LayerPointers {
  uint4* k[kMaxLayers];
  uint4* v[kMaxLayers];
};

__global__ void __launch_bounds__(256) copy_blocks_kernel(const __grid_constant__ LayerPointers pools,
                                                          const int32_t* __restrict__ pairs, int32_t num_pairs,
                                                          int32_t num_layers, int32_t num_blocks,
                                                          int64_t chunks_per_block, unsigned int* err) {
  pkv::pdl_enter();
  const int64_t per_pair = chunks_per_block * 2 * num_layers;
  const int64_t total = per_pair * num_pairs;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int32_t pair = static_cast<int32_t>(idx / per_pair);
    int64_t rest = idx - pair * per_pair;
    const int32_t pool = static_cast<int32_t>(rest / chunks_per_block);  // 2 * layer + (0: K, 1: V)
    const int64_t chunk = rest - pool * chunks_per_block;
    const int32_t src = __ldg(pairs + 2 * pair);
    const int32_t dst = __ldg(pairs + 2 * pair + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (chunk == 0 && pool == 0) pkv::raise_error(err, PKV_DERR_BLOCK_RANGE);
      continue;
    }
    if (src == dst) continue;
    uint4* base = (pool & 1) ? pools.v[pool >> 1] : pools.k[pool >> 1];
    base[static_cast<int64_t>(dst) * chunks_per_block + chunk] = base[static_cast<int64_t>(src) * chunks_per_block + chunk];
  }
}

}  // namespace

extern "C" int pkv_copy_blocks(void* const* k_caches, void* const* v_caches, int32_t num_layers,
                               const int32_t* block_pairs, int32_t num_pairs, int32_t num_blocks,
                               int64_t block_bytes, pkv_stream_t stream) {
  if (num_layers < 0 || num_layers > kMaxLayers || num_pairs < 0 || num_blocks < 0 || block_bytes <= 0)
    return PKV_EINVAL;
  if (block_bytes % 16 != 0) return PKV_EUNSUPPORTED;
  if (num_layers == 0 || num_pairs == 0) return PKV_OK;
  if (!k_caches || !v_caches || !block_pairs) return PKV_EINVAL;
  LayerPointers pools{};
  for (int l = 0; l < num_layers; ++l) {
    if (!k_caches[l] || !v_caches[l]) return PKV_EINVAL;
    if (!pkv::aligned16(k_caches[l]) || !pkv::aligned16(v_caches[l])) return PKV_EALIGN;
    pools.k[l] = static_cast<uint4*>(k_caches[l]);
    pools.v[l] = static_cast<uint4*>(v_caches[l]);
  }
  int st = PKV_OK;
  unsigned int* err = pkv::device_error_word(&st);
  if (st != PKV_OK) return st;
  pkv::DeviceInfo info;
  if (pkv::device_info(&info) != PKV_OK) return PKV_ECUDA;
  const int64_t chunks_per_block = block_bytes / 16;
  const int64_t total = chunks_per_block * 2 * num_layers * num_pairs;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(info.sms) * 8;
  if (blocks > cap) blocks = cap;
  const cudaError_t e = pkv::launch_pdl(copy_blocks_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                                        pools, block_pairs, num_pairs, num_layers, num_blocks, chunks_per_block, err);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}
