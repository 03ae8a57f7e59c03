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
// How (GB300 design), shared by both kernels below:
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
#pragma once

#include <cuda.h>

#include <cfloat>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "common.cuh"

namespace {

using pkv::Chunk;

constexpr int kMinTokensPerCta = 32;
constexpr int kAutoCtasPerSm = 1;      // grid of the automatic split
constexpr int kWorkspaceCtasPerSm = 2;  // workspace sized for up to this many CTAs per SM
constexpr int kMaxStages = 4;
constexpr int kSmemBudget = 200 * 1024;

// d0,d1 += (a0,a1) * (b0,b1) as one packed f32x2 fma (sm_100 family): half
// the issue slots of two scalar fmas, same rounding per lane.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %5};\n\t"
      "mov.b64 d, {%0, %1};\n\t"
      "fma.rn.f32x2 d, a, b, d;\n\t"
      "mov.b64 {%0, %1}, d;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Register shape of a consumer warp that holds R query rows (query heads x
// query tokens) of one KV head.
template <typename T, int D, int R>
struct Shape {
  static constexpr int EPC = Chunk<T>::N;                   // elements per 16-byte chunk
  static constexpr int ROW_BYTES = D * static_cast<int>(sizeof(T));  // one head's row
  static constexpr int CHUNKS = ROW_BYTES / 16;
  static constexpr int EPL8 = (CHUNKS / 8) * EPC;
  static constexpr int LPT = (R * EPL8 > 32 && CHUNKS >= 16) ? 16 : 8;  // lanes per token
  static constexpr int CPL = CHUNKS / LPT;                  // chunks per lane
  static constexpr int EPL = CPL * EPC;                     // elements per lane
  static constexpr int TPW = 32 / LPT;                      // tokens per warp round
  // rounds per stage per warp: short rows (bf16 with head_dim 64) take more
  // tokens per stage so a stage still moves a useful number of bytes
  static constexpr int ROUNDS = (ROW_BYTES >= 512 || R >= 5) ? 2 : ((ROW_BYTES <= 128 && R <= 2) ? 8 : 4);
  static_assert(CPL >= 1, "head row too short for the lane split");
};

struct Params {
  void* out;
  const void* q;
  const unsigned char* k_cache;
  const unsigned char* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* part_o;     // [slots, QL * Hq, D]
  float* part_ml;    // [slots, QL * Hq, 2]
  int32_t* counters; // [batch] sequence tickets, then [slots] merge-group tickets
  unsigned int* err;
  int max_blocks;
  int batch;
  int hq;  // query heads per query token
  int ql;  // query tokens per sequence (1 = decode)
  int hkv;
  int block_size;
  int num_blocks;
  float scale_log2;  // scale * log2(e) (times the K scale for an FP8 cache)
  float v_scale;     // V scale of an FP8 cache (1 otherwise)
  int num_splits;    // 0 = automatic
  int nw;            // consumer warps
  int wph;           // consumer warps per KV head
  int t_stage;       // tokens per stage
  int stages;
  size_t stage_bytes;
  int align;  // split points fall on multiples of this many tokens of a sequence (0 or 1: anywhere)
  int tma;    // mma kernel: stages filled by 4-D tensor copies of 16-token boxes (block_size % 16 == 0)
};

// One contiguous piece of work: tokens [t0, t1) of sequence b.
struct Segment {
  int b;
  int ctx;  // context length of sequence b
  int t0, t1;
  int nparts;      // CTAs sharing sequence b
  int first_slot;  // workspace slot of the sequence's first part
  int slot;        // this part's slot
};

// Bounded pipeline wait.  On a timeout the CTA raises PKV_DERR_WAIT_TIMEOUT,
// sets its abort flag and carries on (all later waits return at once), so
// every warp still reaches every named barrier and the kernel ends; the
// results of an aborted CTA are invalid.
__device__ __forceinline__ void wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              unsigned int* err) {
  if (*abort_flag) return;
  if (!pkv::mbar_wait(bar, parity)) {
    *abort_flag = 1;
    pkv::raise_error(err, PKV_DERR_WAIT_TIMEOUT);
  }
}

__device__ __forceinline__ int align_tokens(const Params& p) { return p.align > 1 ? p.align : 1; }

__device__ __forceinline__ long long round_up(long long n, int a) { return (n + a - 1) / a * a; }

__device__ __forceinline__ int context_len(const Params& p, int b) {
  const int n = __ldg(p.context_lens + b);
  if (n < 0 || n > p.max_blocks * p.block_size || (n > 0 && n < p.ql)) {
    pkv::raise_error(p.err, PKV_DERR_LEN_RANGE);
    return 0;
  }
  return n;
}

// Work plan of this CTA, computed identically by every thread.
struct Plan {
  // automatic mode
  long long start, end, per;
  int b_first;
  long long cu_first;
  // fixed-split mode
  Segment fixed;
  bool fixed_valid;
};

// Block-wide sum over context lengths and search for the first sequence
// overlapping this CTA's token range (automatic mode).
__device__ void plan_auto(const Params& p, Plan& plan, long long* sh) {
  const int tid = threadIdx.x;
  const int nthreads = blockDim.x;
  const int A = align_tokens(p);
  long long local = 0;
  for (int b = tid; b < p.batch; b += nthreads) local += round_up(context_len(p, b), A);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) local += __shfl_xor_sync(0xffffffffu, local, off);
  if (tid % 32 == 0) sh[tid / 32] = local;
  __syncthreads();
  long long total = 0;
  for (int w = 0; w < nthreads / 32; ++w) total += sh[w];
  __syncthreads();
  const long long grid = gridDim.x;
  long long per = round_up((total + grid - 1) / grid, A);
  if (per < kMinTokensPerCta) per = round_up(kMinTokensPerCta, A);
  plan.per = per;
  plan.start = per * blockIdx.x;
  plan.end = plan.start + per < total ? plan.start + per : total;
  plan.b_first = -1;
  plan.cu_first = 0;
  if (plan.start >= plan.end) return;
  // chunked exclusive scan to locate the sequence containing token `start`
  if (tid == 0) sh[32] = -1;
  long long running = 0;
  for (int base = 0; base < p.batch; base += nthreads) {
    const int b = base + tid;
    const long long n = b < p.batch ? round_up(context_len(p, b), A) : 0;
    long long incl = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, off);
      if (tid % 32 >= off) incl += y;
    }
    if (tid % 32 == 31) sh[tid / 32] = incl;
    __syncthreads();
    long long warp_prefix = 0;
    long long chunk_total = 0;
    for (int w = 0; w < nthreads / 32; ++w) {
      if (w < tid / 32) warp_prefix += sh[w];
      chunk_total += sh[w];
    }
    const long long excl = running + warp_prefix + incl - n;
    if (n > 0 && excl <= plan.start && plan.start < excl + n) {
      sh[32] = b;
      sh[33] = excl;
    }
    running += chunk_total;
    __syncthreads();
    if (sh[32] >= 0) break;
  }
  plan.b_first = static_cast<int>(sh[32]);
  plan.cu_first = sh[33];
  __syncthreads();
}

__device__ void plan_fixed(const Params& p, Plan& plan) {
  const int S = p.num_splits;
  const int b = blockIdx.x / S;
  const int j = blockIdx.x % S;
  plan.fixed_valid = false;
  if (b >= p.batch) return;
  const int n = context_len(p, b);
  if (n == 0) return;
  const int chunk = static_cast<int>(round_up((n + S - 1) / S, align_tokens(p)));
  const int t0 = j * chunk;
  if (t0 >= n) return;
  const int t1 = t0 + chunk < n ? t0 + chunk : n;
  plan.fixed = Segment{b, n, t0, t1, (n + chunk - 1) / chunk, b * S, b * S + j};
  plan.fixed_valid = true;
}

// Calls fn(segment) for every segment of this CTA, in order.
template <typename Fn>
__device__ __forceinline__ bool for_each_segment(const Params& p, const Plan& plan, Fn&& fn) {
  if (p.num_splits > 0) {
    if (plan.fixed_valid) return fn(plan.fixed);
    return true;
  }
  if (plan.b_first < 0) return true;
  // positions run over the flattened contexts, each rounded up to the split
  // alignment; a part's end is clipped to the sequence's real length
  const int A = align_tokens(p);
  long long cu = plan.cu_first;
  for (int b = plan.b_first; b < p.batch && cu < plan.end; ++b) {
    const int n = context_len(p, b);
    const long long np = round_up(n, A);
    if (n > 0) {
      const long long s0 = plan.start > cu ? plan.start : cu;
      const long long s1 = plan.end < cu + np ? plan.end : cu + np;
      const int c0 = static_cast<int>(cu / plan.per);
      const int c1 = static_cast<int>((cu + np - 1) / plan.per);
      Segment seg{b, n, static_cast<int>(s0 - cu), static_cast<int>(s1 - cu < n ? s1 - cu : n), c1 - c0 + 1,
                  c0 + b, static_cast<int>(blockIdx.x) + b};
      if (!fn(seg)) return false;
    }
    cu += np;
  }
  return true;
}

// Log-sum-exp merge of `count` partial states (o, m, l) of one sequence, at
// workspace slots first + i * step.  With `final` the normalized rows go to the
// output; otherwise the merged state is written over slot `first` (each row is
// read and written by one warp only, so the in-place write is safe).  A warp
// takes four rows at a time so their loads overlap: one pass over the parts
// folds each lane's share of (m, l) online and the lanes combine them by
// shuffles; a second pass sums the weighted rows, each lane owning D / 32
// columns, eight parts per step.
template <typename T, int D>
__device__ __forceinline__ void merge_parts(const Params& p, const Segment& seg, int rows_per_seq, int first,
                                            int step, int count, bool final, int nthreads_c) {
  constexpr int RW = 4;  // rows a warp merges together
  constexpr int PER = D / 32;
  const int tid = threadIdx.x;
  const int warp = tid / 32;
  const int lane = tid % 32;
  const int nwarps = nthreads_c / 32;
  T* out = static_cast<T*>(p.out) + static_cast<size_t>(seg.b) * rows_per_seq * D;
  const size_t ml_stride = static_cast<size_t>(step) * rows_per_seq * 2;
  const size_t o_stride = static_cast<size_t>(step) * rows_per_seq * D;
  float* ml_base = p.part_ml + static_cast<size_t>(first) * rows_per_seq * 2;
  float* o_base = p.part_o + static_cast<size_t>(first) * rows_per_seq * D + lane * PER;
  for (int row0 = warp * RW; row0 < rows_per_seq; row0 += nwarps * RW) {
    float mm[RW], ll[RW];
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      mm[r] = -INFINITY;
      ll[r] = 0.f;
    }
    // (m, l) of this lane's parts, folded online
    for (int j = lane; j < count; j += 32) {
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        if (row0 + r >= rows_per_seq) continue;
        const float2 v = __ldcg(reinterpret_cast<const float2*>(ml_base + j * ml_stride + (row0 + r) * 2));
        const float mn = fmaxf(mm[r], v.x);
        if (mn != -INFINITY) {
          ll[r] = ll[r] * exp2f(mm[r] - mn) + v.y * exp2f(v.x - mn);
          mm[r] = mn;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < RW; ++r) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, mm[r], off);
        const float lo = __shfl_xor_sync(0xffffffffu, ll[r], off);
        const float mn = fmaxf(mm[r], mo);
        if (mn != -INFINITY) {
          ll[r] = ll[r] * exp2f(mm[r] - mn) + lo * exp2f(mo - mn);
          mm[r] = mn;
        }
      }
    }
    float acc[RW][PER];
#pragma unroll
    for (int r = 0; r < RW; ++r)
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[r][e] = 0.f;
    // kJ parts at a time: every load of a batch is issued before the first is
    // used, so a batch costs one round trip to L2
    constexpr int kJ = 4;
    for (int j0 = 0; j0 < count; j0 += kJ) {
      float v[kJ][RW][PER];
      float mj[kJ][RW];
#pragma unroll
      for (int jj = 0; jj < kJ; ++jj)
#pragma unroll
        for (int r = 0; r < RW; ++r) {
          mj[jj][r] = -INFINITY;
#pragma unroll
          for (int e = 0; e < PER; ++e) v[jj][r][e] = 0.f;
          if (j0 + jj >= count || row0 + r >= rows_per_seq) continue;
          const size_t j = j0 + jj;
          mj[jj][r] = __ldcg(ml_base + j * ml_stride + (row0 + r) * 2);
          const float* src = o_base + j * o_stride + static_cast<size_t>(row0 + r) * D;
          if constexpr (PER == 4) {
            const float4 x = __ldcg(reinterpret_cast<const float4*>(src));
            v[jj][r][0] = x.x;
            v[jj][r][1] = x.y;
            v[jj][r][2] = x.z;
            v[jj][r][3] = x.w;
          } else {
            const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
            v[jj][r][0] = x.x;
            v[jj][r][1] = x.y;
          }
        }
#pragma unroll
      for (int jj = 0; jj < kJ; ++jj)
#pragma unroll
        for (int r = 0; r < RW; ++r) {
          // 0 for absent parts and rows, and for rows no merged part sees a key of
          // (a verify row whose group holds only keys past its position)
          const float w = mm[r] == -INFINITY ? 0.f : exp2f(mj[jj][r] - mm[r]);
#pragma unroll
          for (int e = 0; e < PER; ++e) acc[r][e] = fmaf(w, v[jj][r][e], acc[r][e]);
        }
    }
    __syncwarp();
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      if (row0 + r >= rows_per_seq) continue;
      if (final) {
        const float inv = 1.f / ll[r];
#pragma unroll
        for (int e = 0; e < PER; ++e)
          out[static_cast<size_t>(row0 + r) * D + lane * PER + e] = static_cast<T>(acc[r][e] * inv);
      } else {
        float* dst = o_base + static_cast<size_t>(row0 + r) * D;
#pragma unroll
        for (int e = 0; e < PER; ++e) dst[e] = acc[r][e];
        if (lane == 0) *reinterpret_cast<float2*>(ml_base + (row0 + r) * 2) = make_float2(mm[r], ll[r]);
      }
    }
  }
}

// Parts of a split sequence merged per group of this many consecutive parts.
constexpr int kMergeGroup = 8;

// Called by all consumer threads after this CTA wrote its part of a split
// sequence.  Nothing waits on another CTA: atomic tickets elect the mergers.
// The part that arrives last in its group of kMergeGroup consecutive parts
// merges the group into the group's first slot; the group merger that
// arrives last merges the groups and writes the output (a sequence of at most
// kMergeGroup parts is merged straight to the output).  A long context split
// over ~150 parts thus merges in two short steps spread over ~20 CTAs instead
// of one CTA reading every part.
template <typename T, int D>
__device__ __forceinline__ void combine_if_last(const Params& p, const Segment& seg, int rows_per_seq, int* sh_flag,
                                                int nthreads_c) {
  const int tid = threadIdx.x;
  const int np = seg.nparts;
  const int part = seg.slot - seg.first_slot;
  const int gfirst = part / kMergeGroup * kMergeGroup;
  const int gsize = min(kMergeGroup, np - gfirst);
  const int ng = (np + kMergeGroup - 1) / kMergeGroup;
  int* gcount = p.counters + p.batch + seg.first_slot + gfirst;
  pkv::named_barrier_sync(1, nthreads_c);
  if (tid == 0) {
    __threadfence();
    sh_flag[0] = atomicAdd(gcount, 1) == gsize - 1;
  }
  pkv::named_barrier_sync(1, nthreads_c);
  if (sh_flag[0]) {
    __threadfence();
    if (ng == 1) {
      merge_parts<T, D>(p, seg, rows_per_seq, seg.first_slot, 1, np, true, nthreads_c);
      if (tid == 0) *gcount = 0;
    } else {
      merge_parts<T, D>(p, seg, rows_per_seq, seg.first_slot + gfirst, 1, gsize, false, nthreads_c);
      pkv::named_barrier_sync(1, nthreads_c);
      if (tid == 0) {
        *gcount = 0;
        __threadfence();
        sh_flag[0] = atomicAdd(p.counters + seg.b, 1) == ng - 1;
      }
      pkv::named_barrier_sync(1, nthreads_c);
      if (sh_flag[0]) {
        __threadfence();
        merge_parts<T, D>(p, seg, rows_per_seq, seg.first_slot, kMergeGroup, ng, true, nthreads_c);
        if (tid == 0) p.counters[seg.b] = 0;
      }
    }
  }
  pkv::named_barrier_sync(1, nthreads_c);
}

// G query heads per KV head, QL query tokens per sequence.  A consumer warp
// holds R = G * QL rows: row rho is query token rho / G, head g * G + rho % G.
// T is the q / out element type, TC the cache's (T: an FP8 cache runs on the
// tensor-core kernel below).
template <typename T, typename TC, int D, int G, int QL>
__global__ void __launch_bounds__(288, 1) paged_decode_kernel(const Params p) {
  pkv::pdl_enter();
  constexpr int R = G * QL;
  using S = Shape<TC, D, R>;
  constexpr int NQ = S::EPC / Chunk<T>::N;  // q / out chunks per cache chunk
  const int rows_per_seq = QL * p.hq;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x;
  const int warp = tid / 32;
  const int lane = tid % 32;
  const int nw = p.nw;

  unsigned char* stage_base = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.stages * p.stage_bytes);
  uint64_t* empty = full + kMaxStages;
  long long* sh = reinterpret_cast<long long*>(empty + kMaxStages);  // 64 scratch words
  int* sh_flag = reinterpret_cast<int*>(sh + 64);
  float* merge = reinterpret_cast<float*>(sh_flag + 32);

  volatile int* abort_flag = sh_flag + 1;
  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < p.stages; ++s) {
      pkv::mbar_init(&full[s], 1);
      pkv::mbar_init(&empty[s], nw);
    }
    pkv::fence_mbar_init();
  }

  // context length 0 rows: zeros, nothing read (section 5 padding)
  for (int b = blockIdx.x; b < p.batch; b += gridDim.x) {
    if (context_len(p, b) != 0) continue;
    T* o = static_cast<T*>(p.out) + static_cast<size_t>(b) * rows_per_seq * D;
    for (int i = tid; i < rows_per_seq * D; i += blockDim.x) o[i] = static_cast<T>(0.0f);
  }

  Plan plan;
  if (p.num_splits > 0) {
    plan_fixed(p, plan);
    __syncthreads();
  } else {
    plan_auto(p, plan, sh);
  }

  if (warp == nw) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    const uint64_t policy = pkv::l2_evict_first_policy();
    const size_t head_row = static_cast<size_t>(p.hkv) * S::ROW_BYTES;  // bytes per token, all heads
    int it = 0;
    for_each_segment(p, plan, [&](const Segment& seg) -> bool {
      const int32_t* table = p.block_tables + static_cast<size_t>(seg.b) * p.max_blocks;
      for (int t = seg.t0; t < seg.t1; t += p.t_stage, ++it) {
        const int s = it % p.stages;
        const uint32_t use = it / p.stages;
        if (use > 0) wait_or_abort(&empty[s], (use & 1u) ^ 1u, abort_flag, p.err);
        const int nt = min(p.t_stage, seg.t1 - t);
        unsigned char* ks = stage_base + s * p.stage_bytes;
        unsigned char* vs = ks + p.stage_bytes / 2;
        for (int tt = t; tt < t + nt;) {
          const int blk = tt / p.block_size;
          const int off = tt - blk * p.block_size;
          const int n = min(p.block_size - off, t + nt - tt);
          const int phys = __ldg(table + blk);
          if (phys < 0 || phys >= p.num_blocks) {
            pkv::raise_error(p.err, PKV_DERR_BLOCK_RANGE);
          } else {
            const size_t src = (static_cast<size_t>(phys) * p.block_size + off) * head_row;
            const size_t dst = static_cast<size_t>(tt - t) * head_row;
            const uint32_t bytes = static_cast<uint32_t>(n * head_row);
            pkv::mbar_expect_tx(&full[s], 2 * bytes);
            pkv::bulk_g2s(ks + dst, p.k_cache + src, bytes, &full[s], policy);
            pkv::bulk_g2s(vs + dst, p.v_cache + src, bytes, &full[s], policy);
          }
          tt += n;
        }
        pkv::mbar_arrive(&full[s]);
      }
      return true;
    });
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = warp % p.hkv;
  const int phase = warp / p.hkv;
  const int tg = lane / S::LPT;   // token group inside the warp
  const int lig = lane % S::LPT;  // lane inside the token group
  const int nthreads_c = nw * 32;
  int it = 0;

  for_each_segment(p, plan, [&](const Segment& seg) -> bool {
    // q of the R rows sharing KV head g, pre-scaled into the exp2 domain
    float qr[R][S::EPL];
#pragma unroll
    for (int h = 0; h < R; ++h) {
      const T* qh =
          static_cast<const T*>(p.q) + ((static_cast<size_t>(seg.b) * QL + h / G) * p.hq + g * G + h % G) * D;
#pragma unroll
      for (int k = 0; k < S::CPL; ++k)
#pragma unroll
        for (int u = 0; u < NQ; ++u) {
          const uint4 c = __ldg(reinterpret_cast<const uint4*>(qh) + (lig + S::LPT * k) * NQ + u);
          Chunk<T>::unpack(c, &qr[h][k * S::EPC + u * Chunk<T>::N]);
        }
#pragma unroll
      for (int e = 0; e < S::EPL; ++e) qr[h][e] *= p.scale_log2;
    }
    float acc[R][S::EPL];
    float m[R], l[R];
#pragma unroll
    for (int h = 0; h < R; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int e = 0; e < S::EPL; ++e) acc[h][e] = 0.f;
    }

    for (int t = seg.t0; t < seg.t1; t += p.t_stage, ++it) {
      const int s = it % p.stages;
      const uint32_t use = it / p.stages;
      wait_or_abort(&full[s], use & 1u, abort_flag, p.err);
      const int nt = min(p.t_stage, seg.t1 - t);
      const unsigned char* ks = stage_base + s * p.stage_bytes;
      const unsigned char* vs = ks + p.stage_bytes / 2;

      float sc[S::ROUNDS][R];
#pragma unroll
      for (int r = 0; r < S::ROUNDS; ++r) {
        const int tt = (r * p.wph + phase) * S::TPW + tg;
        const bool valid = tt < nt;
        float dot[R];
#pragma unroll
        for (int h = 0; h < R; ++h) dot[h] = 0.f;
        if (valid) {
          const unsigned char* row = ks + (static_cast<size_t>(tt) * p.hkv + g) * S::ROW_BYTES;
          // even and odd elements accumulate in the two lanes of an f32x2 pair
          float odd[R];
#pragma unroll
          for (int h = 0; h < R; ++h) odd[h] = 0.f;
#pragma unroll
          for (int k = 0; k < S::CPL; ++k) {
            float f[S::EPC];
            Chunk<TC>::unpack(pkv::lds128(row + (lig + S::LPT * k) * 16), f);
#pragma unroll
            for (int h = 0; h < R; ++h)
#pragma unroll
              for (int e = 0; e < S::EPC; e += 2)
                fma2(dot[h], odd[h], qr[h][k * S::EPC + e], qr[h][k * S::EPC + e + 1], f[e], f[e + 1]);
          }
#pragma unroll
          for (int h = 0; h < R; ++h) dot[h] += odd[h];
        }
#pragma unroll
        for (int h = 0; h < R; ++h) {
#pragma unroll
          for (int off = 1; off < S::LPT; off <<= 1) dot[h] += __shfl_xor_sync(0xffffffffu, dot[h], off);
          // query token h / G sits at position ctx - QL + h / G and sees keys up to it
          const bool visible = QL == 1 || t + tt <= seg.ctx - QL + h / G;
          sc[r][h] = (valid && visible) ? dot[h] : -INFINITY;
        }
      }

      // fold the stage into the running softmax state
#pragma unroll
      for (int h = 0; h < R; ++h) {
        float mt = sc[0][h];
#pragma unroll
        for (int r = 1; r < S::ROUNDS; ++r) mt = fmaxf(mt, sc[r][h]);
#pragma unroll
        for (int off = S::LPT; off < 32; off <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
        const float mnew = fmaxf(m[h], mt);
        if (mnew == -INFINITY) {
#pragma unroll
          for (int r = 0; r < S::ROUNDS; ++r) sc[r][h] = 0.f;
          continue;
        }
        if (mnew != m[h]) {
          const float corr = exp2f(m[h] - mnew);
          l[h] *= corr;
#pragma unroll
          for (int e = 0; e < S::EPL; ++e) acc[h][e] *= corr;
          m[h] = mnew;
        }
#pragma unroll
        for (int r = 0; r < S::ROUNDS; ++r) {
          const float pr = exp2f(sc[r][h] - mnew);
          l[h] += pr;
          sc[r][h] = pr;
        }
      }

#pragma unroll
      for (int r = 0; r < S::ROUNDS; ++r) {
        const int tt = (r * p.wph + phase) * S::TPW + tg;
        if (tt < nt) {
          const unsigned char* row = vs + (static_cast<size_t>(tt) * p.hkv + g) * S::ROW_BYTES;
#pragma unroll
          for (int k = 0; k < S::CPL; ++k) {
            float f[S::EPC];
            Chunk<TC>::unpack(pkv::lds128(row + (lig + S::LPT * k) * 16), f);
#pragma unroll
            for (int h = 0; h < R; ++h)
#pragma unroll
              for (int e = 0; e < S::EPC; e += 2)
                fma2(acc[h][k * S::EPC + e], acc[h][k * S::EPC + e + 1], sc[r][h], sc[r][h], f[e], f[e + 1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) pkv::mbar_arrive(&empty[s]);
    }


    // reduce the token groups of the warp (m is already warp-uniform)
#pragma unroll
    for (int h = 0; h < R; ++h) {
#pragma unroll
      for (int off = S::LPT; off < 32; off <<= 1) {
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
#pragma unroll
        for (int e = 0; e < S::EPL; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], off);
      }
    }

    // merge the warps that share KV head g (token phases)
    if (p.wph > 1) {
      const int rec = D + 2;
      if (tg == 0) {
#pragma unroll
        for (int h = 0; h < R; ++h) {
          float* dstm = merge + (static_cast<size_t>(warp) * R + h) * rec;
#pragma unroll
          for (int k = 0; k < S::CPL; ++k)
#pragma unroll
            for (int e = 0; e < S::EPC; ++e) dstm[(lig + S::LPT * k) * S::EPC + e] = acc[h][k * S::EPC + e];
          if (lig == 0) {
            dstm[D] = m[h];
            dstm[D + 1] = l[h];
          }
        }
      }
      pkv::named_barrier_sync(1, nthreads_c);
      if (phase == 0) {
#pragma unroll
        for (int h = 0; h < R; ++h) {
          float mm = m[h];
          for (int ph = 1; ph < p.wph; ++ph)
            mm = fmaxf(mm, merge[(static_cast<size_t>(ph * p.hkv + g) * R + h) * rec + D]);
          const float w0 = mm == -INFINITY ? 0.f : exp2f(m[h] - mm);
          float ll = l[h] * w0;
#pragma unroll
          for (int e = 0; e < S::EPL; ++e) acc[h][e] *= w0;
          for (int ph = 1; ph < p.wph; ++ph) {
            const float* src = merge + (static_cast<size_t>(ph * p.hkv + g) * R + h) * rec;
            const float mw = src[D];
            const float w = mw == -INFINITY ? 0.f : exp2f(mw - mm);
            ll += w * src[D + 1];
#pragma unroll
            for (int k = 0; k < S::CPL; ++k)
#pragma unroll
              for (int e = 0; e < S::EPC; ++e)
                acc[h][k * S::EPC + e] += w * src[(lig + S::LPT * k) * S::EPC + e];
          }
          m[h] = mm;
          l[h] = ll;
        }
      }
      pkv::named_barrier_sync(1, nthreads_c);
    }

    // write the result (whole sequence) or this part's state
    if (phase == 0 && tg == 0) {
#pragma unroll
      for (int h = 0; h < R; ++h) {
        const int head = (h / G) * p.hq + g * G + h % G;  // row within the sequence's QL * Hq rows
        if (seg.nparts == 1) {
          const float inv = 1.f / l[h];
          T* o = static_cast<T*>(p.out) + (static_cast<size_t>(seg.b) * rows_per_seq + head) * D;
#pragma unroll
          for (int k = 0; k < S::CPL; ++k) {
            float f[S::EPC];
#pragma unroll
            for (int e = 0; e < S::EPC; ++e) f[e] = acc[h][k * S::EPC + e] * inv;
#pragma unroll
            for (int u = 0; u < NQ; ++u)
              reinterpret_cast<uint4*>(o)[(lig + S::LPT * k) * NQ + u] = Chunk<T>::pack(f + u * Chunk<T>::N);
          }
        } else {
          float* po = p.part_o + (static_cast<size_t>(seg.slot) * rows_per_seq + head) * D;
#pragma unroll
          for (int k = 0; k < S::CPL; ++k)
#pragma unroll
            for (int e = 0; e < S::EPC; e += 4)
              *reinterpret_cast<float4*>(po + (lig + S::LPT * k) * S::EPC + e) =
                  make_float4(acc[h][k * S::EPC + e], acc[h][k * S::EPC + e + 1], acc[h][k * S::EPC + e + 2],
                              acc[h][k * S::EPC + e + 3]);
          if (lig == 0)
            *reinterpret_cast<float2*>(p.part_ml + (static_cast<size_t>(seg.slot) * rows_per_seq + head) * 2) =
                make_float2(m[h], l[h]);
        }
      }
    }

    if (seg.nparts > 1) combine_if_last<T, D>(p, seg, rows_per_seq, sh_flag, nthreads_c);
    return true;
  });
}

// ------------------------------------------------------------------ tensor-core variant
//
// With R >= 3 rows per KV head (grouped-query heads x verify tokens) the
// CUDA-core loop above runs out of registers and issue slots before HBM is
// saturated.  This variant keeps the same CTA plan, producer, split and
// combine, but each consumer warp computes its 16-token chunk of a stage with
// mma.sync m16n8k16 (bf16 in, fp32 accumulate): S = Q K^T with the R rows in
// the M dimension (rows >= R are zero), online softmax on the accumulator
// fragments (O rescaled only when a row maximum grows by more than 2^8), and
// O += P V with P taken straight from the S fragments.  The eight keys an
// ldmatrix reads must sit in eight different bank groups; two stage layouts
// give that:
//  * block_size a multiple of 16 (p.tma): a warp's 16 keys lie in one block,
//    and four tensor copies (K and V, two halves of head_dim) of a 16-token box
//    of every KV head fill its chunk, 128-byte swizzled, rows of one head's
//    tokens 128 bytes apart (split points then fall on multiples of 16 tokens);
//  * otherwise each token's row of all KV heads is its own bulk copy, at a
//    stride padded by 16 bytes.

constexpr int kMmaTokens = 16;  // keys per consumer warp per stage
constexpr int kMmaPad = 16;     // bytes after each token row in shared memory (per-token layout)

__device__ __forceinline__ void tma_load_4d(void* smem_dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(pkv::smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(pkv::smem_u32(bar)),
      "l"(policy)
      : "memory");
}

// TC is the cache's element type: bf16, or FP8 E4M3 (one byte, with per-tensor
// K and V scales).  For FP8 the operands are widened in registers to f16,
// which holds every E4M3 value exactly, and the MMAs run on f16:
//  * S = Q K^T: an ldmatrix word of a K row is four consecutive codes,
//    widened to the pairs (4c, 4c+1) and (4c+2, 4c+3); the k index of each
//    m16n8k16 step is permuted that way on both operands, so Q's fragments are
//    loaded in the same order.  Q is f16 after a per-row power-of-two scaling
//    that puts its largest element in [2^14, 2^15).
//  * O += P V: P is f16 times 2^7 (the lazy rescale lets P reach 2^8, and
//    2^15 is f16's top binade); l sums the same rounded weights, so the
//    factor cancels.  V's B fragment
//    pairs two keys of one column, so each lane reads 16 consecutive codes of
//    four key rows and byte-permutes key pairs together; n-tile j, column n
//    then stands for head_dim index 16 n + j, and a lane's accumulators cover
//    32 consecutive outputs.
// 16-key chunks a consumer warp takes per stage: two for an FP8 cache (its
// stages hold twice the tokens in the same bytes, and the second chunk's
// scores overlap the first's latency), one for bf16.
template <typename TC>
__host__ __device__ constexpr int mma_chunks_per_warp() {
  return std::is_same<TC, __nv_fp8_e4m3>::value ? 2 : 1;
}

template <int G, int QL, typename TC = __nv_bfloat16>
__global__ void __launch_bounds__(288, 1)
    paged_decode_mma_kernel(const Params p, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v) {
  pkv::pdl_enter();
  using T = __nv_bfloat16;
  constexpr bool kFp8 = std::is_same<TC, __nv_fp8_e4m3>::value;
  constexpr int ES = static_cast<int>(sizeof(TC));  // bytes per cache element
  constexpr int NH = ES;                             // tensor copies per K (or V) box: 128-byte rows
  constexpr int NSUB = mma_chunks_per_warp<TC>();
  constexpr int D = 128;
  constexpr int R = G * QL;
  static_assert(R <= 16, "at most 16 rows per KV head");
  constexpr int HH = R <= 8 ? 1 : 2;  // fragment row halves (r0, r0 + 8) that hold query rows
  // R <= 8: O is accumulated transposed, O^T = V^T P^T, with head_dim in the
  // M dimension (8 m-tiles of 16) and the rows in N: half the MMAs and half
  // the accumulator registers of O = P V, whose M rows 8..15 would be empty
  constexpr bool kT = HH == 1;
  constexpr int NO = kT ? 8 : 16;
  constexpr float kRescale = 8.0f;
  const int rows_per_seq = QL * p.hq;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x;
  const int warp = tid / 32;
  const int lane = tid % 32;
  const int nw = p.nw;
  const int ts = p.hkv * D * ES + kMmaPad;  // shared-memory stride of one token's row (per-token layout)
  const int box_bytes = p.hkv * kMmaTokens * 128;  // one tensor copy: 128-byte rows, 16 tokens, all heads

  // stages start on a 1024-byte boundary (the period of the 128-byte swizzle)
  unsigned char* stage_base = smem + ((1024u - (pkv::smem_u32(smem) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(stage_base + p.stages * p.stage_bytes);
  uint64_t* empty = full + kMaxStages;
  long long* sh = reinterpret_cast<long long*>(empty + kMaxStages);
  int* sh_flag = reinterpret_cast<int*>(sh + 64);
  float* merge = reinterpret_cast<float*>(sh_flag + 32);
  volatile int* abort_flag = sh_flag + 1;
  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < p.stages; ++s) {
      pkv::mbar_init(&full[s], 1);
      pkv::mbar_init(&empty[s], nw);
    }
    pkv::fence_mbar_init();
  }
  for (int b = blockIdx.x; b < p.batch; b += gridDim.x) {
    if (context_len(p, b) != 0) continue;
    T* o = static_cast<T*>(p.out) + static_cast<size_t>(b) * rows_per_seq * D;
    for (int i = tid; i < rows_per_seq * D; i += blockDim.x) o[i] = static_cast<T>(0.0f);
  }
  Plan plan;
  if (p.num_splits > 0) {
    plan_fixed(p, plan);
    __syncthreads();
  } else {
    plan_auto(p, plan, sh);
  }

  if (warp == nw) {
    // ------------------------------------------------------------ producer
    // Every lane issues the copies of its tokens (stage position % 32 == lane):
    // each token's row is a copy of its own (rows sit at a padded stride), and a
    // single issuing thread would bound the stage rate for small blocks.
    const uint64_t policy = pkv::l2_evict_first_policy();
    const uint32_t head_row = static_cast<uint32_t>(p.hkv) * D * ES;
    int it = 0;
    if (p.tma) {
      // lane c < wph loads the c-th 16-token box of a stage: one block, one offset
      if (lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
      }
      for_each_segment(p, plan, [&](const Segment& seg) -> bool {
        const int32_t* table = p.block_tables + static_cast<size_t>(seg.b) * p.max_blocks;
        for (int t = seg.t0; t < seg.t1; t += p.t_stage, ++it) {
          const int s = it % p.stages;
          const uint32_t use = it / p.stages;
          const int tc = t + lane * kMmaTokens;
          const bool mine = lane < p.t_stage / kMmaTokens && tc < seg.t1;
          const int blk = tc / p.block_size;
          const int phys = mine ? __ldg(table + blk) : 0;
          if (lane == 0 && use > 0) wait_or_abort(&empty[s], (use & 1u) ^ 1u, abort_flag, p.err);
          __syncwarp();
          if (mine) {
            if (phys < 0 || phys >= p.num_blocks) {
              pkv::raise_error(p.err, PKV_DERR_BLOCK_RANGE);
            } else {
              unsigned char* kd = stage_base + s * p.stage_bytes + lane * NH * box_bytes;
              unsigned char* vd = kd + p.stage_bytes / 2;
              const int off = tc - blk * p.block_size;
              pkv::mbar_expect_tx(&full[s], 2u * NH * static_cast<uint32_t>(box_bytes));
#pragma unroll
              for (int hh = 0; hh < NH; ++hh) {
                tma_load_4d(kd + hh * box_bytes, &tm_k, 64 * hh, off, 0, phys, &full[s], policy);
                tma_load_4d(vd + hh * box_bytes, &tm_v, 64 * hh, off, 0, phys, &full[s], policy);
              }
            }
          }
          __syncwarp();
          if (lane == 0) pkv::mbar_arrive(&full[s]);
        }
        return true;
      });
      return;
    }
    for_each_segment(p, plan, [&](const Segment& seg) -> bool {
      const int32_t* table = p.block_tables + static_cast<size_t>(seg.b) * p.max_blocks;
      for (int t = seg.t0; t < seg.t1; t += p.t_stage, ++it) {
        const int s = it % p.stages;
        const uint32_t use = it / p.stages;
        if (lane == 0 && use > 0) wait_or_abort(&empty[s], (use & 1u) ^ 1u, abort_flag, p.err);
        __syncwarp();
        const int nt = min(p.t_stage, seg.t1 - t);
        unsigned char* ks = stage_base + s * p.stage_bytes;
        unsigned char* vs = ks + p.stage_bytes / 2;
        int valid = 0;
        for (int u = lane; u < nt; u += 32) {
          const int phys = __ldg(table + (t + u) / p.block_size);
          valid += (phys >= 0 && phys < p.num_blocks) ? 1 : 0;
        }
        if (valid > 0) pkv::mbar_expect_tx(&full[s], 2 * valid * head_row);
        for (int u = lane; u < nt; u += 32) {
          const int tt = t + u;
          const int blk = tt / p.block_size;
          const int phys = __ldg(table + blk);
          if (phys < 0 || phys >= p.num_blocks) {
            pkv::raise_error(p.err, PKV_DERR_BLOCK_RANGE);
            continue;
          }
          const size_t src = (static_cast<size_t>(phys) * p.block_size + (tt - blk * p.block_size)) * head_row;
          const size_t dst = static_cast<size_t>(u) * ts;
          pkv::bulk_g2s(ks + dst, p.k_cache + src, head_row, &full[s], policy);
          pkv::bulk_g2s(vs + dst, p.v_cache + src, head_row, &full[s], policy);
        }
        __syncwarp();
        if (lane == 0) pkv::mbar_arrive(&full[s]);
      }
      return true;
    });
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = warp % p.hkv;
  const int phase = warp / p.hkv;
  const int r0 = lane >> 2;  // fragment rows r0 and r0 + 8
  const int c = lane & 3;
  const int nthreads_c = nw * 32;
  const uint32_t stage_addr = pkv::smem_u32(stage_base);
  // Lane offsets of the ldmatrix rows inside a warp's chunk: row stride rs,
  // second half of head_dim at +hs, 16-byte column j at (j ^ x) * 16 where x is
  // the row's swizzle phase (tensor layout) or 0 (per-token layout).  Every
  // row an ldmatrix lane addresses has phase lane & 7 (row = 8k + (lane & 7)).
  const int rs = p.tma ? 128 : ts;
  const int hs = p.tma ? box_bytes : 128;
  const uint32_t xr = p.tma ? static_cast<uint32_t>(lane & 7) : 0u;
  // chunk base (K) of this warp in stage 0, relative to the stage
  const int csub = p.tma ? NH * box_bytes : kMmaTokens * ts;  // bytes from one 16-token chunk to the next
  const int cbase = phase * NSUB * csub + (p.tma ? g * kMmaTokens * 128 : g * D * ES);
  const uint32_t krow = cbase + (lane & 7) * rs;
  const uint32_t vrow = cbase + ((lane & 7) + ((lane >> 3) & 1) * 8) * rs;
  const uint32_t kj = static_cast<uint32_t>(lane >> 3);
  const uint32_t vj = static_cast<uint32_t>(lane >> 4);
  // transposed P V: matrices 0, 1 read keys 0-7, matrices 2, 3 keys 8-15; odd matrices the upper 8 columns
  const uint32_t vrowt = cbase + ((lane & 7) + ((lane >> 4) & 1) * 8) * rs;
  const uint32_t vjt = static_cast<uint32_t>((lane >> 3) & 1);
  // FP8 V: this lane reads 16 codes (chunk lane / 4) of key rows 2c, 2c + 1 and
  // the same + 8; a row's swizzle phase is key & 7
  const uint32_t vq = static_cast<uint32_t>(lane >> 2);
  const uint32_t v8a = cbase + (2 * c) * rs + ((vq ^ (p.tma ? 2u * c : 0u)) << 4);
  const uint32_t v8b = cbase + (2 * c + 1) * rs + ((vq ^ (p.tma ? 2u * c + 1u : 0u)) << 4);
  int it = 0;

  for_each_segment(p, plan, [&](const Segment& seg) -> bool {
    // Q as the A operand: rows r0 / r0 + 8, columns 16 kk + 2c (+1) and + 8
    // (bf16), or 16 kk + 4c (+1) and 16 kk + 4c + 2 (+3) as scaled f16 (FP8)
    uint32_t qf[8][4];
    float qmul[2] = {p.scale_log2, p.scale_log2};
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int rho = r0 + 8 * hh;
      const uint32_t* qrow =
          rho < R ? reinterpret_cast<const uint32_t*>(static_cast<const T*>(p.q) +
                                                      ((static_cast<size_t>(seg.b) * QL + rho / G) * p.hq + g * G +
                                                       rho % G) * D)
                  : nullptr;
      if constexpr (kFp8) {
        float amax = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          qf[kk][hh] = qrow ? __ldg(qrow + kk * 8 + 2 * c) : 0u;
          qf[kk][2 + hh] = qrow ? __ldg(qrow + kk * 8 + 2 * c + 1) : 0u;
          amax = fmaxf(amax, fmaxf(fmaxf(fabsf(__uint_as_float(qf[kk][hh] << 16)),
                                         fabsf(__uint_as_float(qf[kk][hh] & 0xffff0000u))),
                                   fmaxf(fabsf(__uint_as_float(qf[kk][2 + hh] << 16)),
                                         fabsf(__uint_as_float(qf[kk][2 + hh] & 0xffff0000u)))));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const int ex = amax > 0.f ? min(max(14 - ilogbf(amax), -100), 100) : 0;
        const float up = ldexpf(1.f, ex);
        qmul[hh] = p.scale_log2 * ldexpf(1.f, -ex);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            const uint32_t x = qf[kk][2 * w + hh];
            qf[kk][2 * w + hh] =
                pkv::pack_f16x2(__uint_as_float(x << 16) * up, __uint_as_float(x & 0xffff0000u) * up);
          }
      } else {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          qf[kk][hh] = qrow ? __ldg(qrow + kk * 8 + c) : 0u;
          qf[kk][2 + hh] = qrow ? __ldg(qrow + kk * 8 + 4 + c) : 0u;
        }
      }
    }
    // the A fragment of k16 step kk; with R <= 8 its rows r0 + 8 are zero
    // constants, so their registers are not kept
    struct QFrag {
      uint32_t r[4];
    };
    auto qa = [&](int kk) {
      QFrag f;
      f.r[0] = qf[kk][0];
      f.r[1] = kT ? 0u : qf[kk][1];
      f.r[2] = qf[kk][2];
      f.r[3] = kT ? 0u : qf[kk][3];
      return f;
    };
    const int lim0 = seg.ctx - QL + (r0 < R ? r0 / G : 0);
    const int lim1 = seg.ctx - QL + (r0 + 8 < R ? (r0 + 8) / G : 0);
    float o[NO][4];
#pragma unroll
    for (int j = 0; j < NO; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[j][e] = 0.f;
    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.f, 0.f};

    for (int t = seg.t0; t < seg.t1; t += p.t_stage, ++it) {
      const int s = it % p.stages;
      const uint32_t use = it / p.stages;
      wait_or_abort(&full[s], use & 1u, abort_flag, p.err);
      const int nt = min(p.t_stage, seg.t1 - t);
      // this warp's NSUB chunks of 16 keys are chunks phase * NSUB + sub of the stage;
      // their scores share one running maximum, so the rescale check runs once
      const int tw0 = phase * NSUB * kMmaTokens;
      if (nt > tw0) {
        float sacc[NSUB][2][4];
        float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int sub = 0; sub < NSUB; ++sub) {
          const int tt0 = tw0 + sub * kMmaTokens;
          const int nv = min(max(nt - tt0, 0), kMmaTokens);  // valid keys of this chunk
#pragma unroll
          for (int nb = 0; nb < 2; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[sub][nb][e] = nv > 0 ? 0.f : -INFINITY;
          if (nv == 0) continue;  // only a later chunk can be empty; its P is 0
          const uint32_t kbase = stage_addr + s * p.stage_bytes + sub * csub;
          if (nv < kMmaTokens) {
            // V rows past the last key hold stale bytes: zero them so 0 * stale never reaches O
            constexpr int CPR = 8 * NH;  // 16-byte chunks of one head's row
            unsigned char* vrows = stage_base + s * p.stage_bytes + p.stage_bytes / 2 + sub * csub + cbase;
            for (int idx = lane; idx < (kMmaTokens - nv) * CPR; idx += 32)
              *reinterpret_cast<uint4*>(vrows + (nv + idx / CPR) * rs + ((idx % CPR) / 8) * hs + (idx % 8) * 16) =
                  make_uint4(0, 0, 0, 0);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
          }
          // S = Q K^T for 16 keys (two n-tiles of 8)
          if constexpr (kFp8) {
            // a word of four codes widens to the B pairs of one k16 step
#pragma unroll
            for (int q4 = 0; q4 < 2; ++q4) {
#pragma unroll
              for (int nb = 0; nb < 2; ++nb) {
                uint32_t b[4];
                pkv::ldsm_x4(kbase + krow + nb * 8 * rs + (((q4 * 4 + kj) ^ xr) << 4), b);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  pkv::mma_f16_16816(sacc[sub][nb], qa(4 * q4 + i).r, pkv::e4m3x2_to_f16x2(b[i]),
                                     pkv::e4m3x2_to_f16x2(b[i] >> 16));
              }
            }
          } else {
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
#pragma unroll
              for (int nb = 0; nb < 2; ++nb) {
                uint32_t b[4];
                pkv::ldsm_x4(kbase + krow + nb * 8 * rs + (k4 >> 1) * hs + ((((k4 & 1) * 4 + kj) ^ xr) << 4), b);
                pkv::mma_bf16_16816(sacc[sub][nb], qa(2 * k4).r, b[0], b[1]);
                pkv::mma_bf16_16816(sacc[sub][nb], qa(2 * k4 + 1).r, b[2], b[3]);
              }
            }
          }
          // scale, mask; with R <= 8 the fragment rows r0 + 8 hold no query row and are skipped (P = 0)
#pragma unroll
          for (int nb = 0; nb < 2; ++nb)
#pragma unroll
            for (int e = 0; e < 2 * HH; ++e) {
              const int key = nb * 8 + 2 * c + (e & 1);
              float x = sacc[sub][nb][e] * qmul[e >> 1];
              const bool visible = key < nv && (QL == 1 || t + tt0 + key <= ((e < 2) ? lim0 : lim1));
              x = visible ? x : -INFINITY;
              sacc[sub][nb][e] = x;
              mt[e >> 1] = fmaxf(mt[e >> 1], x);
            }
        }
        // online softmax per row (lazy rescale of O)
#pragma unroll
        for (int hh = 0; hh < HH; ++hh) {
          mt[hh] = fmaxf(mt[hh], __shfl_xor_sync(0xffffffffu, mt[hh], 1));
          mt[hh] = fmaxf(mt[hh], __shfl_xor_sync(0xffffffffu, mt[hh], 2));
          const float mn = fmaxf(m[hh], mt[hh]);
          const bool need = mn > m[hh] + kRescale || (m[hh] == -INFINITY && mn != -INFINITY);
          if constexpr (kT) {
            // row r0's state lives in quad r0; the accumulators hold rows 2c and 2c + 1
            if (__any_sync(0xffffffffu, need)) {
              const float corr = need ? exp2f(m[0] - mn) : 1.f;  // 0 while nothing has been accumulated
              if (need) {
                l[0] *= corr;
                m[0] = mn;
              }
              const float c0 = __shfl_sync(0xffffffffu, corr, 8 * c);
              const float c1 = __shfl_sync(0xffffffffu, corr, 8 * c + 4);
#pragma unroll
              for (int j = 0; j < NO; ++j) {
                o[j][0] *= c0;
                o[j][2] *= c0;
                o[j][1] *= c1;
                o[j][3] *= c1;
              }
            }
          } else if (need) {
            const float corr = exp2f(m[hh] - mn);  // 0 while nothing has been accumulated
            l[hh] *= corr;
#pragma unroll
            for (int j = 0; j < NO; ++j) {
              o[j][2 * hh] *= corr;
              o[j][2 * hh + 1] *= corr;
            }
            m[hh] = mn;
          }
        }
        const float mu0 = m[0] == -INFINITY ? 0.f : m[0];
        const float mu1 = m[1] == -INFINITY ? 0.f : m[1];
#pragma unroll
        for (int sub = 0; sub < NSUB; ++sub) {
          if (nt <= tw0 + sub * kMmaTokens) continue;
          const uint32_t vbase = stage_addr + s * p.stage_bytes + p.stage_bytes / 2 + sub * csub;
          uint32_t pf[4];
          if constexpr (kFp8) {
            // P as f16 times 2^7; l sums the same rounded weights
            constexpr float kPs = 128.0f;
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
              const __half2 lo =
                  __floats2half2_rn(exp2f(sacc[sub][nb][0] - mu0) * kPs, exp2f(sacc[sub][nb][1] - mu0) * kPs);
              l[0] += __low2float(lo) + __high2float(lo);
              pf[2 * nb] = *reinterpret_cast<const uint32_t*>(&lo);
              pf[2 * nb + 1] = 0u;
              if constexpr (HH == 2) {
                const __half2 hi =
                    __floats2half2_rn(exp2f(sacc[sub][nb][2] - mu1) * kPs, exp2f(sacc[sub][nb][3] - mu1) * kPs);
                l[1] += __low2float(hi) + __high2float(hi);
                pf[2 * nb + 1] = *reinterpret_cast<const uint32_t*>(&hi);
              }
            }
            // O^T += V^T P^T: the A fragment pairs keys (2c, 2c+1) and (2c+8, 2c+9)
            // of one head_dim index by byte permutes of 16 codes of each key row;
            // m-tile t, row m stands for head_dim 16 m + 2t (m < 8) or 16 (m - 8) + 2t + 1
            const unsigned char* vstage = stage_base + s * p.stage_bytes + p.stage_bytes / 2 + sub * csub;
            const uint4 ra = pkv::lds128(vstage + v8a);
            const uint4 rb = pkv::lds128(vstage + v8b);
            const uint4 rc = pkv::lds128(vstage + v8a + 8 * rs);
            const uint4 rd = pkv::lds128(vstage + v8b + 8 * rs);
            const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
            const uint32_t wc[4] = {rc.x, rc.y, rc.z, rc.w}, wd[4] = {rd.x, rd.y, rd.z, rd.w};
#pragma unroll
            for (int tm = 0; tm < 8; ++tm) {
              const uint32_t sel = (tm & 1) ? 0x7362u : 0x5140u;
              const uint32_t x = pkv::prmt(wa[tm >> 1], wb[tm >> 1], sel);
              const uint32_t y = pkv::prmt(wc[tm >> 1], wd[tm >> 1], sel);
              const uint32_t a[4] = {pkv::e4m3x2_to_f16x2(x), pkv::e4m3x2_to_f16x2(x >> 16), pkv::e4m3x2_to_f16x2(y),
                                     pkv::e4m3x2_to_f16x2(y >> 16)};
              pkv::mma_f16_16816(o[tm], a, pf[0], pf[2]);
            }
          } else {
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
              const __nv_bfloat162 lo =
                  __floats2bfloat162_rn(exp2f(sacc[sub][nb][0] - mu0), exp2f(sacc[sub][nb][1] - mu0));
              l[0] += __low2float(lo) + __high2float(lo);
              pf[2 * nb] = *reinterpret_cast<const uint32_t*>(&lo);
              pf[2 * nb + 1] = 0u;
              if constexpr (HH == 2) {
                const __nv_bfloat162 hi =
                    __floats2bfloat162_rn(exp2f(sacc[sub][nb][2] - mu1), exp2f(sacc[sub][nb][3] - mu1));
                l[1] += __low2float(hi) + __high2float(hi);
                pf[2 * nb + 1] = *reinterpret_cast<const uint32_t*>(&hi);
              }
            }
            if constexpr (kT) {
              // O^T += V^T P^T: m-tile t covers head_dim 16t .. 16t + 15; the four
              // 8x8 matrices are (keys 0-7 | 8-15) x (head_dim 16t + 0-7 | + 8-15)
#pragma unroll
              for (int tm = 0; tm < 8; ++tm) {
                uint32_t a[4];
                pkv::ldsm_x4_trans(vbase + vrowt + (tm >> 2) * hs + (((2 * (tm & 3) + vjt) ^ xr) << 4), a);
                pkv::mma_bf16_16816(o[tm], a, pf[0], pf[2]);
              }
            } else {
              // O += P V over the 16 keys: 16 n-tiles of 8 columns
#pragma unroll
              for (int jp = 0; jp < 8; ++jp) {
                uint32_t b[4];
                pkv::ldsm_x4_trans(vbase + vrow + (jp >> 2) * hs + (((2 * (jp & 3) + vj) ^ xr) << 4), b);
                pkv::mma_bf16_16816(o[2 * jp], pf, b[0], b[1]);
                pkv::mma_bf16_16816(o[2 * jp + 1], pf, b[2], b[3]);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) pkv::mbar_arrive(&empty[s]);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 1);
      l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 2);
    }

    if constexpr (kT) {
      // this lane's accumulators hold rows 2c and 2c + 1 (columns of O^T); their
      // (m, l) come from the quads that own those rows.  Accumulator (tm, e)
      // is head_dim index dA(tm) (e < 2) or dA(tm) + dB (e >= 2).
      const float mr0 = __shfl_sync(0xffffffffu, m[0], 8 * c), mr1 = __shfl_sync(0xffffffffu, m[0], 8 * c + 4);
      const float lr0 = __shfl_sync(0xffffffffu, l[0], 8 * c), lr1 = __shfl_sync(0xffffffffu, l[0], 8 * c + 4);
      float mr[2] = {mr0, mr1}, lr[2] = {lr0, lr1};
      const int q4 = lane >> 2;
      constexpr int dB = kFp8 ? 1 : 8;
      auto dA = [&](int tm) { return kFp8 ? 16 * q4 + 2 * tm : 16 * tm + q4; };
      if (p.wph > 1) {
        const int rec = D + 2;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int row = 2 * c + i;
          if (row < R) {
            float* dstm = merge + (static_cast<size_t>(warp) * R + row) * rec;
#pragma unroll
            for (int tm = 0; tm < NO; ++tm) {
              dstm[dA(tm)] = o[tm][i];
              dstm[dA(tm) + dB] = o[tm][2 + i];
            }
          }
        }
        if (c == 0 && r0 < R) {
          float* dstm = merge + (static_cast<size_t>(warp) * R + r0) * rec;
          dstm[D] = m[0];
          dstm[D + 1] = l[0];
        }
        pkv::named_barrier_sync(1, nthreads_c);
        if (phase == 0) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int row = 2 * c + i;
            if (row >= R) continue;
            float mm = mr[i];
            for (int ph = 1; ph < p.wph; ++ph)
              mm = fmaxf(mm, merge[(static_cast<size_t>(ph * p.hkv + g) * R + row) * rec + D]);
            const float w0 = mm == -INFINITY ? 0.f : exp2f(mr[i] - mm);
            float ll = lr[i] * w0;
#pragma unroll
            for (int tm = 0; tm < NO; ++tm) {
              o[tm][i] *= w0;
              o[tm][2 + i] *= w0;
            }
            for (int ph = 1; ph < p.wph; ++ph) {
              const float* src = merge + (static_cast<size_t>(ph * p.hkv + g) * R + row) * rec;
              const float w = src[D] == -INFINITY ? 0.f : exp2f(src[D] - mm);
              ll += w * src[D + 1];
#pragma unroll
              for (int tm = 0; tm < NO; ++tm) {
                o[tm][i] += w * src[dA(tm)];
                o[tm][2 + i] += w * src[dA(tm) + dB];
              }
            }
            mr[i] = mm;
            lr[i] = ll;
          }
        }
        pkv::named_barrier_sync(1, nthreads_c);
      }
      // write the result (whole sequence) or this part's state; for an FP8
      // cache V's scale comes off here (P's 2^7 cancels against l)
      if (phase == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int row = 2 * c + i;
          if (row >= R) continue;
          const int head = (row / G) * p.hq + g * G + row % G;
          const float vs = kFp8 ? p.v_scale : 1.f;
          if (seg.nparts == 1) {
            const float ws = vs / lr[i];
            T* orow = static_cast<T*>(p.out) + (static_cast<size_t>(seg.b) * rows_per_seq + head) * D;
            if constexpr (kFp8) {
              // this lane's 16 outputs are contiguous: head_dim 16 q4 .. 16 q4 + 15
              uint32_t w[8];
#pragma unroll
              for (int tm = 0; tm < 8; ++tm) w[tm] = pkv::pack_bf16x2(o[tm][i] * ws, o[tm][2 + i] * ws);
              uint4* dst = reinterpret_cast<uint4*>(orow + 16 * q4);
              dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
              dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
#pragma unroll
              for (int tm = 0; tm < NO; ++tm) {
                orow[dA(tm)] = static_cast<T>(o[tm][i] * ws);
                orow[dA(tm) + dB] = static_cast<T>(o[tm][2 + i] * ws);
              }
            }
          } else {
            float* po = p.part_o + (static_cast<size_t>(seg.slot) * rows_per_seq + head) * D;
            if constexpr (kFp8) {
              float4* dst = reinterpret_cast<float4*>(po + 16 * q4);
#pragma unroll
              for (int u = 0; u < 4; ++u)
                dst[u] = make_float4(o[2 * u][i] * vs, o[2 * u][2 + i] * vs, o[2 * u + 1][i] * vs,
                                     o[2 * u + 1][2 + i] * vs);
            } else {
#pragma unroll
              for (int tm = 0; tm < NO; ++tm) {
                po[dA(tm)] = o[tm][i];
                po[dA(tm) + dB] = o[tm][2 + i];
              }
            }
            if (q4 == 0)
              *reinterpret_cast<float2*>(p.part_ml + (static_cast<size_t>(seg.slot) * rows_per_seq + head) * 2) =
                  make_float2(mr[i], lr[i]);
          }
        }
      }
    } else {
      // merge the warps that share KV head g (token phases)
      if (p.wph > 1) {
        const int rec = D + 2;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int rho = r0 + 8 * hh;
          if (rho < R) {
            float* dstm = merge + (static_cast<size_t>(warp) * R + rho) * rec;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              *reinterpret_cast<float2*>(dstm + j * 8 + 2 * c) = make_float2(o[j][2 * hh], o[j][2 * hh + 1]);
            if (c == 0) {
              dstm[D] = m[hh];
              dstm[D + 1] = l[hh];
            }
          }
        }
        pkv::named_barrier_sync(1, nthreads_c);
        if (phase == 0) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int rho = r0 + 8 * hh;
            if (rho >= R) continue;
            float mm = m[hh];
            for (int ph = 1; ph < p.wph; ++ph)
              mm = fmaxf(mm, merge[(static_cast<size_t>(ph * p.hkv + g) * R + rho) * rec + D]);
            const float w0 = mm == -INFINITY ? 0.f : exp2f(m[hh] - mm);
            float ll = l[hh] * w0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              o[j][2 * hh] *= w0;
              o[j][2 * hh + 1] *= w0;
            }
            for (int ph = 1; ph < p.wph; ++ph) {
              const float* src = merge + (static_cast<size_t>(ph * p.hkv + g) * R + rho) * rec;
              const float w = src[D] == -INFINITY ? 0.f : exp2f(src[D] - mm);
              ll += w * src[D + 1];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float2 v = *reinterpret_cast<const float2*>(src + j * 8 + 2 * c);
                o[j][2 * hh] += w * v.x;
                o[j][2 * hh + 1] += w * v.y;
              }
            }
            m[hh] = mm;
            l[hh] = ll;
          }
        }
        pkv::named_barrier_sync(1, nthreads_c);
      }

      // write the result (whole sequence) or this part's state
      if (phase == 0) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int rho = r0 + 8 * hh;
          if (rho >= R) continue;
          const int head = (rho / G) * p.hq + g * G + rho % G;
          if (seg.nparts == 1) {
            const float inv = 1.f / l[hh];
            uint32_t* orow = reinterpret_cast<uint32_t*>(static_cast<T*>(p.out) +
                                                         (static_cast<size_t>(seg.b) * rows_per_seq + head) * D);
#pragma unroll
            for (int j = 0; j < 16; ++j) orow[j * 4 + c] = pkv::pack_bf16x2(o[j][2 * hh] * inv, o[j][2 * hh + 1] * inv);
          } else {
            float* po = p.part_o + (static_cast<size_t>(seg.slot) * rows_per_seq + head) * D;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              *reinterpret_cast<float2*>(po + j * 8 + 2 * c) = make_float2(o[j][2 * hh], o[j][2 * hh + 1]);
          }
          if (seg.nparts > 1) {
            if (c == 0)
              *reinterpret_cast<float2*>(p.part_ml + (static_cast<size_t>(seg.slot) * rows_per_seq + head) * 2) =
                  make_float2(m[hh], l[hh]);
          }
        }
      }
    }
    if (seg.nparts > 1) combine_if_last<T, D>(p, seg, rows_per_seq, sh_flag, nthreads_c);
    return true;
  });
}

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
  // tickets: one per sequence, then one per slot (the merge groups)
  const size_t counters = align256((static_cast<size_t>(batch) + slots) * sizeof(int32_t));
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

