// paged_decode_kernel: the CUDA-core decode / verify kernel (fp32 caches and
// head_dim 64).  The CTA plan, split and merge it uses are in decode_plan.cuh.
#pragma once

#include "decode_plan.cuh"

namespace {

// G query heads per KV head, QL query tokens per sequence.  A consumer warp
// holds R = G * QL rows: row rho is query token rho / G, head g * G + rho % G.
// T is the q / out element type, TC the cache's (T: an FP8 cache runs on the
// tensor-core kernel of decode_mma.cuh).
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

}  // namespace
