// Shared part of the paged decode / verify kernels: launch parameters, the
// split of the batch's context over the grid, and the log-sum-exp merge of
// split parts.  The kernels themselves are in decode_simt.cuh (CUDA cores)
// and decode_mma.cuh (tensor cores); decode_launch.cuh holds the host side.
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
  const long long grid = gridDim.x;
  if (p.batch <= nthreads) {
    // one pass when the batch fits the block: each thread loads one length,
    // one block-wide scan gives the total and the prefix that holds `start`
    const long long n = tid < p.batch ? round_up(context_len(p, tid), A) : 0;
    long long incl = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, off);
      if (tid % 32 >= off) incl += y;
    }
    if (tid % 32 == 31) sh[tid / 32] = incl;
    if (tid == 0) sh[32] = -1;
    __syncthreads();
    long long warp_prefix = 0;
    long long total = 0;
    for (int w = 0; w < nthreads / 32; ++w) {
      if (w < tid / 32) warp_prefix += sh[w];
      total += sh[w];
    }
    long long per = round_up((total + grid - 1) / grid, A);
    if (per < kMinTokensPerCta) per = round_up(kMinTokensPerCta, A);
    plan.per = per;
    plan.start = per * blockIdx.x;
    plan.end = plan.start + per < total ? plan.start + per : total;
    const long long excl = warp_prefix + incl - n;
    if (n > 0 && excl <= plan.start && plan.start < excl + n) {
      sh[32] = tid;
      sh[33] = excl;
    }
    __syncthreads();
    plan.b_first = plan.start < plan.end ? static_cast<int>(sh[32]) : -1;
    plan.cu_first = plan.b_first >= 0 ? sh[33] : 0;
    __syncthreads();
    return;
  }
  long long local = 0;
  for (int b = tid; b < p.batch; b += nthreads) local += round_up(context_len(p, b), A);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) local += __shfl_xor_sync(0xffffffffu, local, off);
  if (tid % 32 == 0) sh[tid / 32] = local;
  __syncthreads();
  long long total = 0;
  for (int w = 0; w < nthreads / 32; ++w) total += sh[w];
  __syncthreads();
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
// takes two rows at a time (so a 16-row sequence keeps all eight consumer
// warps busy), each lane owning D / 32 columns, and folds the parts in order
// in one pass: the running maximum m, the sum l and the weighted row are
// rescaled whenever a part raises m (every lane keeps the same m and l).
// Parts are loaded kJ at a time, every load of a batch issued before the
// first is used, so a batch costs one round trip to L2.
template <typename T, int D>
__device__ __forceinline__ void merge_parts(const Params& p, const Segment& seg, int rows_per_seq, int first,
                                            int step, int count, bool final, int nthreads_c) {
  constexpr int RW = 2;  // rows a warp merges together
  constexpr int PER = D / 32;
  constexpr int kJ = 4;
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
    float mm[RW], ll[RW], acc[RW][PER];
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      mm[r] = -INFINITY;
      ll[r] = 0.f;
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[r][e] = 0.f;
    }
    for (int j0 = 0; j0 < count; j0 += kJ) {
      float v[kJ][RW][PER];
      float2 ml[kJ][RW];
#pragma unroll
      for (int jj = 0; jj < kJ; ++jj)
#pragma unroll
        for (int r = 0; r < RW; ++r) {
          ml[jj][r] = make_float2(-INFINITY, 0.f);
#pragma unroll
          for (int e = 0; e < PER; ++e) v[jj][r][e] = 0.f;
          if (j0 + jj >= count || row0 + r >= rows_per_seq) continue;
          const size_t j = j0 + jj;
          ml[jj][r] = __ldcg(reinterpret_cast<const float2*>(ml_base + j * ml_stride + (row0 + r) * 2));
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
          const float mn = fmaxf(mm[r], ml[jj][r].x);
          // absent parts and rows, and parts that saw no key of this row (a
          // verify row whose part holds only keys past its position), carry
          // m = -inf: they add nothing, and a row none of whose parts saw a
          // key keeps m = -inf, l = 0 and a zero row
          if (mn == -INFINITY) continue;
          const float a = exp2f(mm[r] - mn);
          const float w = exp2f(ml[jj][r].x - mn);
          ll[r] = fmaf(ll[r], a, ml[jj][r].y * w);
#pragma unroll
          for (int e = 0; e < PER; ++e) acc[r][e] = fmaf(acc[r][e], a, w * v[jj][r][e]);
          mm[r] = mn;
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

}  // namespace
