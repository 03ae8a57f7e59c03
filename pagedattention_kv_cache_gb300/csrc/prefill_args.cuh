// Arguments shared by the two prefill kernels (tcgen05 and mma.sync) and the
// C entry point that chooses between them.
#pragma once

#include "common.cuh"

namespace pkv {

struct PrefillArgs {
  void* out;
  const void* q;
  const void* k;
  const void* v;
  const void* k_cache;
  const void* v_cache;
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* block_tables;  // null: keys from the packed k, v
  unsigned int* err;
  int total_q;  // rows of q / out
  int total_k;  // rows of the packed k / v (0 when block_tables is used)
  int max_seqlen_q;
  int max_blocks;
  int batch;
  int hq;
  int hkv;
  int block_size;
  int num_blocks;
  float scale;
  int causal;
  int group;     // hq / hkv
  int head_dim;  // 64 or 128 (the mma.sync kernel: 128 only)
  void* workspace;         // split of long items (tcgen05 path), or null
  size_t workspace_bytes;
};

// Tensor-core (tcgen05 + TMEM + TMA) path; requires head_dim 64 or 128, bf16, and
// for the paged case a block size that is a multiple of 128 or a divisor of
// 128 of at least 8.
bool prefill_tc_supported(const PrefillArgs& a);
int prefill_tc_launch(const PrefillArgs& a, cudaStream_t stream);
// Workspace bytes that let the tcgen05 path split long items (0: never splits).
size_t prefill_tc_workspace_bytes(int batch, int num_kv_heads, int group, int head_dim, int max_seqlen_q);

}  // namespace pkv
