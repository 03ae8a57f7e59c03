// paged_varlen_prefill_attn: packed variable-length (chunked) prefill
// attention, reading history through block tables.
//
// What is computed ("3.6 ModelRunner, CUDA Graph, and benchmarks", section 2,
// prepare_prefill): sequence i owns query rows cu_seqlens_q[i] ..
// cu_seqlens_q[i+1]-1 and nk = cu_seqlens_k[i+1] - cu_seqlens_k[i] keys, of
// which the first c = nk - nq are history (prefix-cache hit or earlier
// chunks).  Query row r sits at absolute position c + r; causal attention lets
// it see keys 0..c + r.  With block tables the keys are gathered from the
// paged cache (after the new rows were stored); without, from the packed k/v
// rows of the sequence.
//
// How: a CTA owns one (sequence, KV head, query tile).  The G query heads
// sharing the KV head are packed into the tile's rows (row = token * G +
// head), so every K/V tile gathered through the block table serves all of
// them.  Q K^T and P V run on tensor cores (mma.sync m16n8k16, bf16 in,
// fp32 accumulate) with an online softmax in registers; K/V tiles are
// double-buffered in XOR-swizzled shared memory with cp.async.
#include "prefill_args.cuh"

namespace {

constexpr int kD = 128;
constexpr int kBM = 128;  // rows (token, head) per CTA
constexpr int kBN = 64;   // keys per tile
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowBytes = kD * 2;
constexpr int kChunks = kRowBytes / 16;  // 16

struct Params {
  __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const __nv_bfloat16* k_cache;
  const __nv_bfloat16* v_cache;
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* block_tables;
  unsigned int* err;
  int total_q;
  int total_k;
  int max_seqlen_q;
  int max_blocks;
  int batch;
  int hq;
  int hkv;
  int block_size;
  int num_blocks;
  float scale_log2;
  int causal;
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * kRowBytes + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 source bytes = zero fill
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Issue the cp.async copies of one 64-key tile of K and V for KV head g.
__device__ __forceinline__ void load_kv_tile(const Params& p, int seq, int g, int key0, int nk, int k_row0,
                                             uint32_t ks, uint32_t vs) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int i = 0; i < (kBN * kChunks) / kThreads; ++i) {
    const int idx = tid + i * kThreads;
    const int row = idx / kChunks;
    const int chunk = idx % kChunks;
    const int key = key0 + row;
    const __nv_bfloat16* ksrc = p.k_cache;
    const __nv_bfloat16* vsrc = p.v_cache;
    bool valid = key < nk;
    size_t off = 0;
    if (valid) {
      if (p.block_tables) {
        const int blk = key / p.block_size;
        const int phys = __ldg(p.block_tables + static_cast<size_t>(seq) * p.max_blocks + blk);
        if (phys < 0 || phys >= p.num_blocks) {
          if (chunk == 0) pkv::raise_error(p.err, PKV_DERR_BLOCK_RANGE);
          valid = false;
        } else {
          off = ((static_cast<size_t>(phys) * p.block_size + (key - blk * p.block_size)) * p.hkv + g) * kD;
        }
      } else {
        ksrc = p.k;
        vsrc = p.v;
        off = (static_cast<size_t>(k_row0 + key) * p.hkv + g) * kD;
      }
    }
    cp_async16(ks + swz(row, chunk), valid ? ksrc + off + chunk * 8 : p.q, valid);
    cp_async16(vs + swz(row, chunk), valid ? vsrc + off + chunk * 8 : p.q, valid);
  }
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const Params p) {
  pkv::pdl_enter();
  constexpr int TQ = kBM / G;  // query tokens per tile
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t sq = pkv::smem_u32(smem);
  const uint32_t sk0 = sq + kBM * kRowBytes;
  const uint32_t sv0 = sk0 + 2 * kBN * kRowBytes;

  const int seq = blockIdx.y;
  const int g = blockIdx.z;
  const int q_begin = __ldg(p.cu_q + seq);
  const int nq = __ldg(p.cu_q + seq + 1) - q_begin;
  const int k_begin = __ldg(p.cu_k + seq);
  const int nk = __ldg(p.cu_k + seq + 1) - k_begin;
  const int tok0 = blockIdx.x * TQ;
  // the same range rule as the tcgen05 kernel: rows inside q / out and the packed
  // k / v, and at most max_seqlen_q rows (the grid's size); otherwise skipped
  if (q_begin < 0 || nq < 0 || nk < nq || static_cast<long long>(q_begin) + nq > p.total_q || nq > p.max_seqlen_q ||
      (p.block_tables ? static_cast<long long>(nk) > static_cast<long long>(p.max_blocks) * p.block_size
                      : (k_begin < 0 || static_cast<long long>(k_begin) + nk > p.total_k))) {
    if (threadIdx.x == 0) pkv::raise_error(p.err, PKV_DERR_LEN_RANGE);
    return;
  }
  if (tok0 >= nq) return;
  const int cached = nk - nq;
  const int tok_last = min(nq, tok0 + TQ) - 1;
  const int keys_needed = p.causal ? cached + tok_last + 1 : nk;
  const int num_tiles = (keys_needed + kBN - 1) / kBN;

  const int tid = threadIdx.x;
  const int warp = tid / 32;
  const int lane = tid % 32;

  // Q tile: row m = token * G + head
#pragma unroll
  for (int i = 0; i < (kBM * kChunks) / kThreads; ++i) {
    const int idx = tid + i * kThreads;
    const int row = idx / kChunks;
    const int chunk = idx % kChunks;
    const int tok = tok0 + row / G;
    const bool valid = tok < nq;
    const __nv_bfloat16* src =
        p.q + (static_cast<size_t>(q_begin + (valid ? tok : 0)) * p.hq + g * G + row % G) * kD + chunk * 8;
    cp_async16(sq + swz(row, chunk), src, valid);
  }
  if (num_tiles > 0) load_kv_tile(p, seq, g, 0, nk, k_begin, sk0, sv0);
  cp_commit();

  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[j][e] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  uint32_t qf[8][4];

  const int r_lo = warp * 16 + lane / 4;  // this thread's two rows in the tile
  const int pos_lo = cached + tok0 + r_lo / G;
  const int pos_hi = cached + tok0 + (r_lo + 8) / G;

  for (int kt = 0; kt < num_tiles; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < num_tiles) {
      load_kv_tile(p, seq, g, (kt + 1) * kBN, nk, k_begin, sk0 + (buf ^ 1) * kBN * kRowBytes,
                   sv0 + (buf ^ 1) * kBN * kRowBytes);
      cp_commit();
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    if (kt == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int mi = lane / 8;
        const int row = warp * 16 + (mi & 1) * 8 + lane % 8;
        ldsm_x4(sq + swz(row, kk * 2 + (mi >> 1)), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    const uint32_t ks = sk0 + buf * kBN * kRowBytes;
    const uint32_t vs = sv0 + buf * kBN * kRowBytes;

    // S = Q K^T for 16 rows x 64 keys
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[j][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {
        const int mi = lane / 8;
        const int key_row = jp * 16 + (mi >> 1) * 8 + lane % 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(ks + swz(key_row, kk * 2 + (mi & 1)), b0, b1, b2, b3);
        mma_bf16(s[2 * jp], qf[kk], b0, b1);
        mma_bf16(s[2 * jp + 1], qf[kk], b2, b3);
      }
    }

    // mask + online softmax (exp2 domain)
    const int key0 = kt * kBN;
    const bool need_mask = p.causal ? (key0 + kBN - 1 > cached + tok0) : (key0 + kBN > nk);
    float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = s[j][e] * p.scale_log2;
        if (need_mask) {
          const int key = key0 + j * 8 + (lane % 4) * 2 + (e & 1);
          const int lim = p.causal ? (e < 2 ? pos_lo : pos_hi) : nk - 1;
          if (key > lim || key >= nk) x = -INFINITY;
        }
        s[j][e] = x;
        mt[e >> 1] = fmaxf(mt[e >> 1], x);
      }
    }
    float corr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], 1));
      mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], 2));
      const float mnew = fmaxf(m_run[h], mt[h]);
      corr[h] = mnew == -INFINITY ? 1.f : exp2f(m_run[h] - mnew);
      m_run[h] = mnew;
    }
    float rs[2] = {0.f, 0.f};
    uint32_t pf[4][4];
    // P enters the P.V product as bf16; the row sums add the same rounded
    // values, so numerator and denominator weigh every key identically.
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const float mr = m_run[e >> 1];
        const float p0 = mr == -INFINITY ? 0.f : exp2f(s[j][e] - mr);
        const float p1 = mr == -INFINITY ? 0.f : exp2f(s[j][e + 1] - mr);
        const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
        rs[e >> 1] += __low2float(pb) + __high2float(pb);
        pf[j / 2][(j & 1) * 2 + (e >> 1)] = *reinterpret_cast<const uint32_t*>(&pb);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) l_run[h] = l_run[h] * corr[h] + rs[h];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      o[j][0] *= corr[0];
      o[j][1] *= corr[0];
      o[j][2] *= corr[1];
      o[j][3] *= corr[1];
    }
    // A fragments of P for k-step kk (keys 16kk..16kk+15): {n-tile 2kk rows lo, rows hi, n-tile 2kk+1 lo, hi}
    // pf[kk] holds {2kk:c01, 2kk:c23, 2kk+1:c01, 2kk+1:c23} -> reorder to a0..a3
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint32_t a[4] = {pf[kk][0], pf[kk][1], pf[kk][2], pf[kk][3]};
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        const int mi = lane / 8;
        const int key_row = kk * 16 + (mi & 1) * 8 + lane % 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vs + swz(key_row, dp * 2 + (mi >> 1)), b0, b1, b2, b3);
        mma_bf16(o[2 * dp], a, b0, b1);
        mma_bf16(o[2 * dp + 1], a, b2, b3);
      }
    }
    __syncthreads();
  }

  // each lane summed only its own columns: reduce the row sums over the quad
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }

  // normalise and store the rows this thread owns
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = r_lo + h * 8;
    const int tok = tok0 + row / G;
    if (tok >= nq) continue;
    const float inv = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f;
    __nv_bfloat16* dst = p.out + (static_cast<size_t>(q_begin + tok) * p.hq + g * G + row % G) * kD;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int col = j * 8 + (lane % 4) * 2;
      *reinterpret_cast<uint32_t*>(dst + col) = pack_bf16(o[j][2 * h] * inv, o[j][2 * h + 1] * inv);
    }
  }
}

template <int G>
int launch(const Params& p, int max_seqlen_q, cudaStream_t stream) {
  constexpr int TQ = kBM / G;
  const size_t smem = static_cast<size_t>(kBM + 4 * kBN) * kRowBytes;
  auto kernel = prefill_kernel<G>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return PKV_ECUDA;
  dim3 grid((max_seqlen_q + TQ - 1) / TQ, p.batch, p.hkv);
  if (grid.x == 0) return PKV_OK;
  return pkv::launch_pdl(kernel, grid, dim3(kThreads), smem, stream, p) == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

}  // namespace

extern "C" int pkv_paged_varlen_prefill_attn(void* out, const void* q, const void* k, const void* v,
                                             const void* k_cache, const void* v_cache,
                                             const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                             int32_t max_seqlen_q, int32_t max_seqlen_k,
                                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                                             int32_t batch, int32_t total_q, int32_t total_k, int32_t num_q_heads,
                                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                             int32_t num_blocks, float scale, int32_t causal, void* workspace,
                                             size_t workspace_bytes, pkv_dtype dtype, pkv_stream_t stream) {
  if (batch < 0 || total_q < 0 || total_k < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_seqlen_q < 0 || max_seqlen_k < 0)
    return PKV_EINVAL;
  if (num_q_heads % num_kv_heads != 0) return PKV_EINVAL;
  if (dtype != PKV_BF16 || (head_dim != kD && head_dim != 64)) return PKV_EUNSUPPORTED;
  const int group = num_q_heads / num_kv_heads;
  if (group != 1 && group != 2 && group != 4 && group != 8) return PKV_EUNSUPPORTED;
  if (causal != 0 && causal != 1) return PKV_EINVAL;
  if (batch == 0 || max_seqlen_q == 0 || total_q == 0) return PKV_OK;
  if (!out || !q || !cu_seqlens_q || !cu_seqlens_k) return PKV_EINVAL;
  if (block_tables) {
    if (!k_cache || !v_cache || block_size <= 0 || num_blocks < 0 || max_blocks_per_seq < 0) return PKV_EINVAL;
    if (static_cast<long long>(max_blocks_per_seq) * block_size > INT32_MAX ||
        static_cast<long long>(num_blocks) * block_size > INT32_MAX)
      return PKV_EINVAL;
    if (!pkv::aligned16(k_cache) || !pkv::aligned16(v_cache)) return PKV_EALIGN;
  } else {
    if (!k || !v || total_k == 0) return PKV_EINVAL;
    if (!pkv::aligned16(k) || !pkv::aligned16(v)) return PKV_EALIGN;
  }
  if (!pkv::aligned16(out) || !pkv::aligned16(q)) return PKV_EALIGN;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255)) return PKV_EALIGN;
  int st = PKV_OK;
  unsigned int* err = pkv::device_error_word(&st);
  if (st != PKV_OK) return st;

  pkv::PrefillArgs a{};
  a.out = out;
  a.q = q;
  a.k = k;
  a.v = v;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.block_tables = block_tables;
  a.err = err;
  a.total_q = total_q;
  a.total_k = block_tables ? 0 : total_k;
  a.max_seqlen_q = max_seqlen_q;
  a.max_blocks = max_blocks_per_seq;
  a.batch = batch;
  a.hq = num_q_heads;
  a.hkv = num_kv_heads;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.causal = causal;
  a.group = group;
  a.head_dim = head_dim;
  a.workspace = workspace;
  a.workspace_bytes = workspace ? workspace_bytes : 0;
  if (pkv::prefill_tc_supported(a)) return pkv::prefill_tc_launch(a, stream);
  if (head_dim != kD) return PKV_EUNSUPPORTED;  // the mma.sync kernel below is head_dim 128 only

  Params p{};
  p.out = static_cast<__nv_bfloat16*>(out);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  p.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.block_tables = block_tables;
  p.err = err;
  p.total_q = total_q;
  p.total_k = total_k;
  p.max_seqlen_q = max_seqlen_q;
  p.max_blocks = max_blocks_per_seq;
  p.batch = batch;
  p.hq = num_q_heads;
  p.hkv = num_kv_heads;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = causal;
  switch (group) {
    case 1: return launch<1>(p, max_seqlen_q, stream);
    case 2: return launch<2>(p, max_seqlen_q, stream);
    case 4: return launch<4>(p, max_seqlen_q, stream);
    default: return launch<8>(p, max_seqlen_q, stream);
  }
}

extern "C" size_t pkv_paged_varlen_prefill_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                                          int32_t head_dim, int32_t max_seqlen_q) {
  if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0) return 0;
  return pkv::prefill_tc_workspace_bytes(batch, num_kv_heads, num_q_heads / num_kv_heads, head_dim, max_seqlen_q);
}
