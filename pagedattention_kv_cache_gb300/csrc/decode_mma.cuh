// paged_decode_mma_kernel: the tensor-core decode / verify kernel (bf16 and
// FP8 caches, head_dim 128).  The CTA plan, split and merge it uses are in
// decode_plan.cuh.
#pragma once

#include "decode_plan.cuh"

namespace {

// ------------------------------------------------------------------ tensor-core variant
//
// Past R = 2 rows per KV head (grouped-query heads x verify tokens) the
// CUDA-core loop of decode_simt.cuh runs out of registers and issue slots
// before HBM is saturated; with the layouts below this kernel is also the
// faster one at R = 1 and 2, so it runs every bf16 or FP8 cache with
// head_dim 128.  It keeps the same CTA plan, split and merge, but each
// consumer warp computes its 16-token chunks of a stage with mma.sync
// m16n8k16 (fp32 accumulate): S = Q K^T with the R rows in the M dimension
// (rows >= R are zero), online softmax on the accumulator fragments (O
// rescaled only when a row maximum grows by more than 2^8), and P V with P
// taken straight from the S fragments (as O^T = V^T P^T when R <= 8).  The
// eight keys an ldmatrix reads must sit in eight different bank groups; two
// stage layouts give that:
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
//  * O^T += V^T P^T (an FP8 cache always has R <= 8): P is f16 times 2^7 (the
//    lazy rescale lets P reach 2^8, and 2^15 is f16's top binade); l sums the
//    same rounded weights, so the factor cancels.  V^T's A fragment pairs two
//    keys of one head_dim index, which ldmatrix.trans cannot form from bytes:
//    each lane reads 16 consecutive codes of four key rows and byte-permutes
//    key pairs together.  m-tile t, row m then stands for head_dim index
//    16 m + 2t (m < 8) or 16 (m - 8) + 2t + 1, and a lane's accumulators cover
//    16 consecutive outputs of each of its two rows.
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
  {
    // the producer reads its block-table entries right after the plan: warm
    // L2 with the tables (when they are small) while the plan reads the lengths
    const size_t lines = (static_cast<size_t>(p.batch) * p.max_blocks * 4 + 127) / 128;
    if (lines <= 512) {
      const char* tb = reinterpret_cast<const char*>(p.block_tables);
      for (size_t i = threadIdx.x; i < lines; i += blockDim.x)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(tb + i * 128) : "memory");
    }
  }
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

}  // namespace
