// Paged decode / verify attention kernel shared by the decode entry points
// (one query token per sequence, decode.cu) and the verify entry point (QL
// query tokens per sequence, verify.cu).
//
//
// What is computed ("3.6 ModelRunner, CUDA Graph, and benchmarks", section 2,
// decode; section 5, padding rows): for sequence b and query head h reading
// KV head g = h / G, over t < context_lens[b],
//     s_t = scale * q[b, h] . K_t,  out[b, h] = sum_t softmax(s)_t V_t,
// with K_t / V_t at physical block block_tables[b, t / bs], offset t % bs.
// context_lens 0 writes zeros and reads nothing.
//
// How (GB300 design), shared by both kernels:
//  * A CTA covers every KV head of a token range, so each token's K (or V)
//    row of all heads, [Hkv, D], is contiguous in the [blocks, bs, Hkv, D]
//    pool.  A producer warp streams the range into a ring of shared-memory
//    stages with TMA copies completed on mbarriers; every K/V byte is read from
//    HBM once, and all G query heads of a KV head reuse it on chip.
//  * Consumer warps, one per (KV head, token phase), fold each stage into a
//    running online softmax (exp2 domain) and accumulate P.V.
//  * Split over the context: the batch's context tokens, flattened, are
//    divided evenly over the grid (automatic mode) or each sequence into S
//    equal parts.  A sequence covered by one CTA is written directly; otherwise
//    each part writes (o, m, l) to the workspace and atomic tickets (no
//    waiting) elect the CTAs that merge the parts by log-sum-exp.
// paged_decode_mma_kernel (mma.sync tensor cores, 16-token tensor copies)
// runs every bf16 or FP8 cache with head_dim 128; paged_decode_kernel (CUDA
// cores, 1-D bulk copies of token spans) runs fp32 caches and head_dim 64.
//
// Verify (speculative-decoding target pass, QL > 1): query token i of
// sequence b sits at position context_lens[b] - QL + i and attends keys up to
// it, so the QL tokens just stored are causally masked among themselves.  The
// warp's rows become (query token, head) pairs; K/V are still read once.
//
// Files: decode_plan.cuh (parameters, split plan, merge), decode_simt.cuh
// and decode_mma.cuh (the two kernels), this file (host side: launch shapes,
// the split workspace layout and the dispatch over group sizes).  The entry
// points that include it are decode.cu, verify.cu and fp8.cu.
#pragma once

#include <algorithm>

#include "decode_mma.cuh"
#include "decode_simt.cuh"

namespace {

// ------------------------------------------------------------------ host side

struct LaunchShape {
  int nw, wph, t_stage, stages;
  size_t stage_bytes, smem;
};

template <typename T, int D, int R>
LaunchShape launch_shape(int hkv) {
  using S = Shape<T, D, R>;
  LaunchShape ls;
  ls.wph = hkv >= 8 ? 1 : 8 / hkv;
  ls.nw = hkv * ls.wph;
  ls.t_stage = S::ROUNDS * S::TPW * ls.wph;
  ls.stage_bytes = static_cast<size_t>(ls.t_stage) * hkv * S::ROW_BYTES * 2;
  const size_t misc = 2 * kMaxStages * sizeof(uint64_t) + 64 * sizeof(long long) + 32 * sizeof(int) +
                      (ls.wph > 1 ? static_cast<size_t>(ls.nw) * R * (D + 2) * sizeof(float) : 0);
  int stages = static_cast<int>((kSmemBudget - misc) / ls.stage_bytes);
  ls.stages = stages > kMaxStages ? kMaxStages : stages;
  ls.smem = ls.stages * ls.stage_bytes + misc;
  return ls;
}

size_t slot_count(int batch, int num_splits, int sms) {
  if (num_splits == 1) return 0;
  if (num_splits > 1) return static_cast<size_t>(batch) * num_splits;
  return static_cast<size_t>(sms) * kWorkspaceCtasPerSm + batch;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

size_t workspace_layout(int batch, int hq, int d, int num_splits, int sms, size_t* off_o, size_t* off_ml) {
  const size_t slots = slot_count(batch, num_splits, sms);
  if (slots == 0) return 0;
  // tickets: one per sequence, then one per slot (the merge groups), in the
  // fixed counter area (larger only past 16,384 counters)
  const size_t counters =
      std::max(pkv::kWorkspaceCounterBytes, align256((static_cast<size_t>(batch) + slots) * sizeof(int32_t)));
  *off_o = counters;
  *off_ml = counters + align256(slots * hq * d * sizeof(float));
  return *off_ml + align256(slots * hq * 2 * sizeof(float));
}

template <typename T, typename TC, int D, int G, int QL>
int launch(Params& p, int sms, cudaStream_t stream) {
  const LaunchShape ls = launch_shape<TC, D, G * QL>(p.hkv);
  if (ls.stages < 2) return PKV_EUNSUPPORTED;
  p.nw = ls.nw;
  p.wph = ls.wph;
  p.t_stage = ls.t_stage;
  p.stages = ls.stages;
  p.stage_bytes = ls.stage_bytes;
  auto kernel = paged_decode_kernel<T, TC, D, G, QL>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ls.smem)) !=
      cudaSuccess)
    return PKV_ECUDA;
  unsigned grid;
  if (p.num_splits > 0)
    grid = static_cast<unsigned>(static_cast<long long>(p.batch) * p.num_splits);
  else
    grid = static_cast<unsigned>(sms * kAutoCtasPerSm);
  if (grid == 0) return PKV_OK;
  return pkv::launch_pdl(kernel, dim3(grid), dim3((ls.nw + 1) * 32), ls.smem, stream, p) == cudaSuccess ? PKV_OK
                                                                                                       : PKV_ECUDA;
}

template <int G, int QL, typename TC = __nv_bfloat16>
int launch_mma(Params& p, int sms, cudaStream_t stream) {
  constexpr int ES = static_cast<int>(sizeof(TC));
  constexpr int R = G * QL;
  LaunchShape ls;
  ls.wph = p.hkv >= 8 ? 1 : 8 / p.hkv;
  ls.nw = p.hkv * ls.wph;
  ls.t_stage = kMmaTokens * mma_chunks_per_warp<TC>() * ls.wph;
  // tensor-copy layout when every 16-token box lies in one block
  alignas(64) CUtensorMap maps[2];
  std::memset(maps, 0, sizeof(maps));
  p.tma = (p.block_size % kMmaTokens == 0 && p.num_blocks > 0) ? 1 : 0;
  if (p.tma) {
    if (pkv::encode_paged_kv(&maps[0], p.k_cache, p.block_size, p.hkv, p.num_blocks, ES) != PKV_OK ||
        pkv::encode_paged_kv(&maps[1], p.v_cache, p.block_size, p.hkv, p.num_blocks, ES) != PKV_OK)
      return PKV_ECUDA;
    p.align = kMmaTokens;
    ls.stage_bytes = static_cast<size_t>(ls.t_stage) * p.hkv * 128 * ES * 2;
  } else {
    p.align = 1;
    const size_t ts = static_cast<size_t>(p.hkv) * 128 * ES + kMmaPad;
    ls.stage_bytes = static_cast<size_t>(ls.t_stage) * ts * 2;
  }
  // 1024 bytes of slack put the stages on a swizzle-period boundary
  const size_t misc = 1024 + 2 * kMaxStages * sizeof(uint64_t) + 64 * sizeof(long long) + 32 * sizeof(int) +
                      (ls.wph > 1 ? static_cast<size_t>(ls.nw) * R * (128 + 2) * sizeof(float) : 0);
  const int stages = static_cast<int>((kSmemBudget - misc) / ls.stage_bytes);
  ls.stages = stages > kMaxStages ? kMaxStages : stages;
  if (ls.stages < 2) return PKV_EUNSUPPORTED;
  ls.smem = ls.stages * ls.stage_bytes + misc;
  p.nw = ls.nw;
  p.wph = ls.wph;
  p.t_stage = ls.t_stage;
  p.stages = ls.stages;
  p.stage_bytes = ls.stage_bytes;
  auto kernel = paged_decode_mma_kernel<G, QL, TC>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ls.smem)) !=
      cudaSuccess)
    return PKV_ECUDA;
  unsigned grid;
  if (p.num_splits > 0)
    grid = static_cast<unsigned>(static_cast<long long>(p.batch) * p.num_splits);
  else
    grid = static_cast<unsigned>(sms * kAutoCtasPerSm);
  if (grid == 0) return PKV_OK;
  return pkv::launch_pdl(kernel, dim3(grid), dim3((ls.nw + 1) * 32), ls.smem, stream, p, maps[0], maps[1]) ==
                 cudaSuccess
             ? PKV_OK
             : PKV_ECUDA;
}

template <typename T, int D>
int dispatch_g(Params& p, int group, int sms, cudaStream_t stream) {
  switch (group) {
    case 1:
      if constexpr (std::is_same<T, __nv_bfloat16>::value && D == 128) return launch_mma<1, 1>(p, sms, stream);
      return launch<T, T, D, 1, 1>(p, sms, stream);
    case 2:
      if constexpr (std::is_same<T, __nv_bfloat16>::value && D == 128) return launch_mma<2, 1>(p, sms, stream);
      return launch<T, T, D, 2, 1>(p, sms, stream);
    case 4:
      if constexpr (std::is_same<T, __nv_bfloat16>::value && D == 128) return launch_mma<4, 1>(p, sms, stream);
      return launch<T, T, D, 4, 1>(p, sms, stream);
    case 8:
      if constexpr (std::is_same<T, __nv_bfloat16>::value && D == 128) return launch_mma<8, 1>(p, sms, stream);
      return launch<T, T, D, 8, 1>(p, sms, stream);
    default: return PKV_EUNSUPPORTED;
  }
}

}  // namespace
