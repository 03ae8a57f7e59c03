// paged_varlen_prefill_attn on the 5th-generation tensor cores (tcgen05).
//
// What is computed is the same as the mma.sync kernel in prefill.cu
// ("3.6 ModelRunner, CUDA Graph, and benchmarks", section 2, prepare_prefill):
// query row r of sequence i sits at absolute position c + r (c = nk - nq
// history tokens) and, causally, attends keys 0..c + r, read through the
// block table (or from the packed k/v rows when there is no history).
//
// How: one CTA per SM owns a pair of query tiles of one (sequence, KV head):
// tile A and the tile after it, B.  A tile's 128 rows are (token, query head
// of the KV group) pairs, token-major, so one TMA box of q covers them and
// every K/V tile serves all G heads of both query tiles.
//   warp 0     TMA producer (one thread): Q of both tiles once, then K and V
//              tiles of 128 keys into 2-stage rings (128-byte swizzled, one
//              box per 64-wide d slab; paged tiles are gathered block piece by
//              block piece).  Then the whole warp zeroes the V rows past the
//              last key in the last tile before the MMA thread may use it.
//   warp 1     MMA issuer: the whole warp runs the loop, one elected lane
//              issues each group of MMAs from one asm block, so the issuing
//              work stays warp-uniform and short (the warp shares its SMSP with
//              four busy softmax warps).  Per key tile j the tensor pipe runs
//                 P_A(j) V(j),  Q_A K(j+1)^T,  P_B(j) V(j),  Q_B K(j+1)^T
//              (each a group of eight M=128, N=128 MMAs), so each tile's
//              softmax has the other tile's two groups to hide behind.  S and
//              O of both tiles sit in TMEM (4 x 128 columns); P is written
//              over S in bf16 and read from TMEM as the A operand of P V.
//   warps 2-9  softmax of tile A, two threads per TMEM lane (= query row),
//              one per half of the key tile: scale, mask, row max (the two
//              warps on the same 32 rows exchange theirs through shared memory
//              at a 64-thread named barrier), exp2, bf16 P; O is
//              rescaled in TMEM only when the row max grows by more than 2^8;
//              final normalisation and store (each half 64 of the 128 columns).
//   warps 10-17  the same for tile B.
// Why this shape (measured on GB300): one issuing thread needs about 45
// cycles per tcgen05.mma whatever its N, and each barrier wait between MMA
// groups idles the pipe for ~100 cycles; four groups of N = 128 per key tile
// keep it busy ~83 % of the time even so, where 32- or 64-key tiles per
// query tile reached a fifth to a half.  The pair shares every K/V tile,
// halving the load bytes per flop.
// Every wait is bounded; on a timeout the CTA records an error, skips the
// remaining waits and still frees its TMEM.
#include <algorithm>

#include "prefill_args.cuh"
#include "tcgen05.cuh"

namespace {

using namespace pkv;

constexpr int kBM = 128;   // rows per query tile
constexpr int kBN = 128;   // keys per tile
constexpr int kStages = 2; // K ring and V ring depth
constexpr int kSoftmaxWarps = 8;  // per query tile: two threads per row, one per half of the key tile
constexpr int kThreads = 32 * (2 + 2 * kSoftmaxWarps);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S_A at 0, S_B at 128
constexpr uint32_t kColO = 256;  // O_A at 256, O_B at 384
constexpr uint32_t kSlabQ = kBM * 128;
constexpr uint32_t kSlabKV = kBN * 128;
constexpr uint32_t kRedBytes = 2 * 2 * 2 * kBM * 4;  // row maxima / sums exchanged by the halves: [tile parity][query tile][half][row]

// Sizes for head dimension D (64 or 128): a row of D bf16 is D / 64 slabs of
// 128 bytes (one 128-byte swizzle atom each), and each slab of a tile is a
// TMA box of its own.
template <int D>
struct Geo {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static constexpr int kSlabs = D / 64;
  static constexpr uint32_t kTileQ = kSlabs * kSlabQ;
  static constexpr uint32_t kTileKV = kSlabs * kSlabKV;
  static constexpr uint32_t kRedOffset = 2 * kTileQ + 2 * kStages * kTileKV;
  static constexpr uint32_t kBarOffset = kRedOffset + kRedBytes;
  static constexpr uint32_t kSmemBytes = kBarOffset + 256 + 1024;  // barriers + 1 KB for alignment
  // one CTA per SM even when two would fit (each holds all 512 TMEM columns)
  static constexpr uint32_t kLaunchSmem = kSmemBytes > 120 * 1024 ? kSmemBytes : 120 * 1024;
  static constexpr size_t kRecordBytes = static_cast<size_t>(kBM) * D * 4 + static_cast<size_t>(kBM) * 8;
};
static_assert(Geo<128>::kSmemBytes <= 227 * 1024, "shared memory plan exceeds an SM");
constexpr float kRescaleLog2 = 8.0f;

// Key-range split of long work items, used only when the pairs do not fill
// the GPU (small batches with long histories) and a workspace is given.  With
// P parts chosen on the host, a pair with more than kSplitMinTiles key tiles
// runs as up to P CTAs over consecutive ranges of its key tiles.  For each of
// its two query tiles, every part but the last to finish publishes its
// unnormalised O and its row maxima and sums (one record per part); the last
// merges the records and its own TMEM result by the log-sum-exp rule, in part
// order, and stores the output.
constexpr int kSplitMinTiles = 8;
constexpr int kMaxParts = 8;
constexpr uint64_t kSplitWaitNs = 1000000000ull;  // bound on the last part's wait for the records

// Per query tile X (A = 0, B = 1): S_FULL + X completes when S_X holds the
// scores of the next key tile (and so every P_X V issued before it has
// completed too), P_FULL + X when its softmax warps have written P over it.
// O_FINAL + X completes once, after the last P_X V: tile X's epilogue waits on
// it (A's can start while B still runs).  K and V stages are released
// separately, a K stage once both Q K^T products have read it, a V stage once
// both P V products have.  V_TAIL: the last V tile, once its rows past the
// last key are zeroed (only when that tile is partial).
enum Bar {
  Q_FULL = 0,
  K_FULL = 1,
  V_FULL = K_FULL + kStages,
  K_EMPTY = V_FULL + kStages,
  V_EMPTY = K_EMPTY + kStages,
  S_FULL = V_EMPTY + kStages,
  P_FULL = S_FULL + 2,
  O_FINAL = P_FULL + 2,  // per query tile
  V_TAIL = O_FINAL + 2,
  NUM_BARS
};
static_assert(NUM_BARS * 8 + 16 <= 256, "barrier area too small");

struct TcParams {
  __nv_bfloat16* out;
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* block_tables;
  unsigned int* err;
  int total_q;
  int total_k;
  int max_seqlen_q;
  int max_blocks;
  int hq;
  int hkv;
  int block_size;
  int num_blocks;
  float scale_log2;
  int causal;
  int paged;
  int piece_rows;  // rows per K/V TMA box (paged: min(block_size, kBN))
  int q_tiles;     // query tiles per sequence, rounded up to a whole number of pairs
  int parts_max;   // P: the most parts a long pair runs as (1: no split)
  int* tickets;    // [sequences x KV heads x q_tiles]: finish order of a split tile's parts, reset by the last
  int* ready;      // [same]: records published so far, reset by the last
  unsigned char* records;  // [same][P][record bytes]: O rows (D fp32 each), then m[kBM], l[kBM]
};

}  // namespace

namespace pkv {

// Parts a long pair may run as when the pairs alone leave SMs idle: as many
// as fit in one wave of one CTA per SM (at most kMaxParts), so the split
// never adds a second, mostly empty wave; 1 when the pairs fill the GPU.
int prefill_tc_parts(int batch, int num_kv_heads, int group, int max_seqlen_q, int sms) {
  const long long tq = kBM / group;
  const long long pairs = static_cast<long long>(batch) * num_kv_heads * ((max_seqlen_q + 2 * tq - 1) / (2 * tq));
  if (pairs <= 0 || 2 * pairs > sms) return 1;
  return static_cast<int>(std::min<long long>(kMaxParts, sms / pairs));
}

// Bytes of each of the two int arrays (tickets, ready counts) at the start of
// the prefill workspace: a half of the fixed counter area (split launches have
// at most one item per SM, far below its 8,192 counters), more only past it.
size_t prefill_tc_flag_bytes(long long items) {
  return std::max(kWorkspaceCounterBytes / 2, static_cast<size_t>((items * 4 + 255) / 256 * 256));
}

// Workspace of the tcgen05 prefill: tickets and ready counts (the counter
// area), then P records per (sequence, KV head, query tile); 0 when the
// current device's SMs are filled without splitting.
size_t prefill_tc_workspace_bytes(int batch, int num_kv_heads, int group, int head_dim, int max_seqlen_q) {
  if (batch <= 0 || num_kv_heads <= 0 || max_seqlen_q <= 0) return 0;
  if (head_dim != 64 && head_dim != 128) return 0;
  if (group != 1 && group != 2 && group != 4 && group != 8) return 0;
  DeviceInfo info;
  if (device_info(&info) != PKV_OK) return 0;
  const int parts = prefill_tc_parts(batch, num_kv_heads, group, max_seqlen_q, info.sms);
  if (parts == 1) return 0;
  const long long tq = kBM / group;
  const long long items = static_cast<long long>(batch) * num_kv_heads * 2 * ((max_seqlen_q + 2 * tq - 1) / (2 * tq));
  const size_t flags = prefill_tc_flag_bytes(items);
  const size_t record = head_dim == 64 ? Geo<64>::kRecordBytes : Geo<128>::kRecordBytes;
  return 2 * flags + static_cast<size_t>(items) * parts * record;
}

}  // namespace pkv

namespace {

struct Waiter {
  volatile int* abort_flag;
  unsigned int* err;
  __device__ __forceinline__ void operator()(uint64_t* bar, uint32_t parity) const {
    // one try_wait first: no shared-memory read of the abort flag on the fast path
    if (mbar_try_wait(bar, parity)) return;
    slow(bar, parity);
  }
  // For phases that have usually completed already (loads issued long
  // before): a test_wait returns at once.
  __device__ __forceinline__ void ready(uint64_t* bar, uint32_t parity) const {
    if (mbar_test_wait(bar, parity)) return;
    if (mbar_try_wait(bar, parity)) return;
    slow(bar, parity);
  }
  __device__ __noinline__ void slow(uint64_t* bar, uint32_t parity) const {
    if (*abort_flag) return;
    if (!mbar_wait(bar, parity)) {
      *abort_flag = 1;
      raise_error(err, PKV_DERR_WAIT_TIMEOUT);
    }
  }
};

// exp2(scale * s - m) for two scores (fma on the f32x2 pair, ex2.approx per
// element), rounded to bf16 and packed low = first; the two rounded values are
// added to the row-sum lanes acc (widened exactly: fma by 1 in fp32).
__device__ __forceinline__ uint32_t exp2_pair_bf16(uint32_t s0, uint32_t s1, float scale, float neg_m,
                                                   uint64_t& acc) {
  uint32_t out;
  asm("{\n\t.reg .b64 x, c, m;\n\t.reg .f32 a, b, sa, sb;\n\t.reg .b16 pa, pb, one;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 c, {%4, %4};\n\t"
      "mov.b64 m, {%5, %5};\n\t"
      "fma.rn.f32x2 x, x, c, m;\n\t"
      "mov.b64 {a, b}, x;\n\t"
      "ex2.approx.ftz.f32 a, a;\n\t"
      "ex2.approx.ftz.f32 b, b;\n\t"
      "cvt.rn.bf16x2.f32 %0, b, a;\n\t"
      "mov.b32 {pa, pb}, %0;\n\t"
      "mov.b16 one, 0x3f80;\n\t"
      "mov.b64 {sa, sb}, %1;\n\t"
      "fma.rn.f32.bf16 sa, pa, one, sa;\n\t"
      "fma.rn.f32.bf16 sb, pb, one, sb;\n\t"
      "mov.b64 %1, {sa, sb};\n\t}"
      : "=r"(out), "+l"(acc)
      : "r"(s0), "r"(s1), "f"(scale), "f"(neg_m));
  return out;
}

// Maximum of three floats in one instruction.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <int G, int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  pdl_enter();
  constexpr int TQ = kBM / G;
  constexpr int kD = D;
  constexpr int kSlabs = Geo<D>::kSlabs;
  constexpr uint32_t kTileQ = Geo<D>::kTileQ;
  constexpr uint32_t kTileKV = Geo<D>::kTileKV;
  constexpr size_t kRecordBytes = Geo<D>::kRecordBytes;
  // blocks launch in linear order: x runs over (sequence, KV head), y over
  // query-tile pairs from the last (most keys under the causal mask) to the
  // first, and, with a workspace, over the key-range parts of each pair
  const int seq = blockIdx.x / p.hkv;
  const int g = blockIdx.x % p.hkv;
  const int pairs = p.q_tiles / 2;
  const int pt = pairs - 1 - static_cast<int>(blockIdx.y) / p.parts_max;
  const int part = static_cast<int>(blockIdx.y) % p.parts_max;
  const int q_begin = __ldg(p.cu_q + seq);
  const int nq = __ldg(p.cu_q + seq + 1) - q_begin;
  const int k_begin = __ldg(p.cu_k + seq);
  const int nk = __ldg(p.cu_k + seq + 1) - k_begin;
  // cu_seqlens must describe rows inside q / out (and the packed k / v), and no
  // sequence may have more rows than max_seqlen_q, which sized the grid: such a
  // sequence is skipped whole and raises the range bit
  if (q_begin < 0 || nq < 0 || nk < nq || static_cast<long long>(q_begin) + nq > p.total_q || nq > p.max_seqlen_q ||
      (p.paged ? static_cast<long long>(nk) > static_cast<long long>(p.max_blocks) * p.block_size
               : (k_begin < 0 || static_cast<long long>(k_begin) + nk > p.total_k))) {
    if (threadIdx.x == 0) raise_error(p.err, PKV_DERR_LEN_RANGE);
    return;
  }
  const int tok0 = pt * 2 * TQ;  // first token of tile A; tile B starts TQ later
  if (tok0 >= nq) return;
  const int cached = nk - nq;
  // key tiles each query tile needs (0: the tile has no rows)
  int n_need[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const int t0 = tok0 + x * TQ;
    const int keys = t0 >= nq ? 0 : (p.causal ? cached + min(nq, t0 + TQ) : nk);
    n_need[x] = (keys + kBN - 1) / kBN;
  }
  const int n_all = max(n_need[0], n_need[1]);
  // this CTA's key tiles: j0 .. j0 + n_tiles - 1 (all of them, or one of up to P
  // consecutive ranges); tile X takes the first n_x of them
  const int parts = n_all > kSplitMinTiles ? min(p.parts_max, (n_all + kSplitMinTiles - 1) / kSplitMinTiles) : 1;
  if (part >= parts) return;
  const int j0 = part * n_all / parts;
  const int n_tiles = (part + 1) * n_all / parts - j0;
  const int n_a = max(0, min(n_tiles, n_need[0] - j0));
  const int n_b = max(0, min(n_tiles, n_need[1] - j0));
  // the last tile holds keys past nk: its V rows there are zeroed first
  const bool v_tail = (j0 + n_tiles) * kBN > nk;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  unsigned char* sq = smem;  // Q_A, then Q_B
  unsigned char* sk = sq + 2 * kTileQ;
  unsigned char* sv = sk + kStages * kTileKV;
  float* red = reinterpret_cast<float*>(smem + Geo<D>::kRedOffset);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Geo<D>::kBarOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_ticket = abort_flag + 1;  // split tiles' tickets, one per query tile

  const int tid = threadIdx.x;
  const int warp = tid / 32;
  const int lane = tid % 32;
  const int32_t* table = p.block_tables + static_cast<size_t>(seq) * p.max_blocks;

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(&bars[Q_FULL], 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[K_FULL + s], 1);
      mbar_init(&bars[V_FULL + s], 1);
      mbar_init(&bars[K_EMPTY + s], 1);
      mbar_init(&bars[V_EMPTY + s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars[S_FULL + x], 1);
      mbar_init(&bars[P_FULL + x], kSoftmaxWarps);  // one arrival per softmax warp
    }
    mbar_init(&bars[O_FINAL], 1);
    mbar_init(&bars[O_FINAL + 1], 1);
    mbar_init(&bars[V_TAIL], 1);
    fence_mbar_init();
  }
  const Waiter wait{abort_flag, p.err};
  // Loads tile j's K (is_v = false) or V into stage j % kStages, after the
  // stage's previous occupant (tile j - kStages) was released.
  auto load_tile = [&](int j, bool is_v) {
    const int st = j % kStages;
    const int use = j / kStages;
    uint64_t* full = &bars[(is_v ? V_FULL : K_FULL) + st];
    if (use > 0) wait(&bars[(is_v ? V_EMPTY : K_EMPTY) + st], (use - 1) & 1);
    unsigned char* dst = (is_v ? sv : sk) + st * kTileKV;
    const CUtensorMap* map = is_v ? &tm_v : &tm_k;
    const int key0 = (j0 + j) * kBN;
    if (p.paged) {
      const uint32_t piece_bytes = p.piece_rows * 128u;
      for (int r = 0; r < kBN; r += p.piece_rows) {
        const int key = key0 + r;
        if (key >= nk) break;
        const int blk = key / p.block_size;
        const int phys = __ldg(table + blk);
        if (phys < 0 || phys >= p.num_blocks) {
          raise_error(p.err, PKV_DERR_BLOCK_RANGE);
          continue;
        }
        const int row = phys * p.block_size + (key - blk * p.block_size);
        mbar_expect_tx(full, kSlabs * piece_bytes);
        tc::tma_load_3d(dst + r * 128, map, 0, g, row, full);
        if constexpr (kSlabs == 2) tc::tma_load_3d(dst + kSlabKV + r * 128, map, 64, g, row, full);
      }
    } else {
      const int row = k_begin + key0;
      mbar_expect_tx(full, kTileKV);
      tc::tma_load_3d(dst, map, 0, g, row, full);
      if constexpr (kSlabs == 2) tc::tma_load_3d(dst + kSlabKV, map, 64, g, row, full);
    }
    mbar_arrive(full);
  };
  // the producer thread issues Q and the first K/V tiles (stages still free)
  // before the CTA-wide sync, so their latency overlaps the TMEM allocation
  const int n_early = min(n_tiles, kStages);
  if (tid == 0) {
    tc::prefetch_tensormap(&tm_q);
    tc::prefetch_tensormap(&tm_k);
    tc::prefetch_tensormap(&tm_v);
    const int nx = n_b > 0 ? 2 : 1;
    mbar_expect_tx(&bars[Q_FULL], nx * kTileQ);
    for (int x = 0; x < nx; ++x) {
      tc::tma_load_3d(sq + x * kTileQ, &tm_q, 0, g * G, q_begin + tok0 + x * TQ, &bars[Q_FULL]);
      if constexpr (kSlabs == 2)
        tc::tma_load_3d(sq + x * kTileQ + kSlabQ, &tm_q, 64, g * G, q_begin + tok0 + x * TQ, &bars[Q_FULL]);
    }
    mbar_arrive(&bars[Q_FULL]);
    for (int j = 0; j < n_early; ++j) {
      load_tile(j, false);
      load_tile(j, true);
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // broadcast from lane 0 so the compiler treats the TMEM base as warp-uniform
  const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      if (parts > 1) {
        // a split part streams a key range no other CTA reads: request it into
        // L2 first, so that the ring's loads, which start only as stages free
        // up, find it there
        for (int j = n_early; j < n_tiles; ++j) {
          const int key0 = (j0 + j) * kBN;
          for (int r = 0; r < kBN; r += p.piece_rows) {
            const int key = key0 + r;
            if (key >= nk) break;
            int row = k_begin + key;
            if (p.paged) {
              const int blk = key / p.block_size;
              const int phys = __ldg(table + blk);
              if (phys < 0 || phys >= p.num_blocks) continue;  // raised by the load
              row = phys * p.block_size + (key - blk * p.block_size);
            }
            tc::tma_prefetch_3d(&tm_k, 0, g, row);
            if constexpr (kSlabs == 2) tc::tma_prefetch_3d(&tm_k, 64, g, row);
            tc::tma_prefetch_3d(&tm_v, 0, g, row);
            if constexpr (kSlabs == 2) tc::tma_prefetch_3d(&tm_v, 64, g, row);
          }
        }
      }
      // K(j) once the K stage is free (both Q K^T of tile j - 2 read it), V(j)
      // once the V stage is
      for (int j = n_early; j < n_tiles; ++j) {
        load_tile(j, false);
        load_tile(j, true);
      }
    }
    __syncwarp();  // every load issued before the warp turns to the last tile
    if (v_tail) {
      // In the last tile the V rows past nk hold whatever their block had there
      // (or were not loaded): zero them so 0 * stale never reaches O.  Every
      // load has been issued, so the stage's barrier is at the last tile's
      // phase or just past it, and a parity wait for that phase is exact.
      const int j = n_tiles - 1;
      const int st = j % kStages;
      wait(&bars[V_FULL + st], (j / kStages) & 1);
      unsigned char* vt = sv + st * kTileKV;
      const int first = nk - (j0 + j) * kBN;
      for (int idx = lane; idx < (kBN - first) * kSlabs * 8; idx += 32) {
        const int rr = first + idx / (kSlabs * 8);
        const int ch = idx % (kSlabs * 8);
        *reinterpret_cast<uint4*>(vt + (ch >> 3) * kSlabKV + rr * 128 + (ch & 7) * 16) = make_uint4(0, 0, 0, 0);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[V_TAIL]);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (its descriptor arithmetic stays warp-uniform);
    // one elected lane issues the MMAs and commits.
    {
      const bool leader = tc::elect_one();
      constexpr uint32_t idesc_qk = tc::idesc_bf16(kBM, kBN, 0, 0);
      constexpr uint32_t idesc_pv = tc::idesc_bf16(kBM, kD, 0, 1);
      // descriptors of the first Q, K and V slabs; later ones differ only in the
      // start-address field (address >> 4), so they are reached by adding offset >> 4
      const uint64_t q_desc = tc::smem_desc(smem_u32(sq), 16, 1024);
      const uint64_t k_desc = tc::smem_desc(smem_u32(sk), 16, 1024);
      const uint64_t v_desc = tc::smem_desc(smem_u32(sv), kSlabKV, 1024);
      const int n_x[2] = {n_a, n_b};
      // S_X = Q_X K(j)^T (S_X held P_X(j - 1), read by P_X(j - 1) V issued
      // before: the tensor pipe runs one thread's MMAs in order)
      auto issue_qk = [&](int x, int j) {
        const int st = j % kStages;
        // the chain's first step: tile X's Q slab 0 and stage st's K slab 0
        const uint64_t a0 = q_desc + ((x * kTileQ) >> 4);
        const uint64_t b0 = k_desc + ((st * kTileKV) >> 4);
        if (leader) {
          if constexpr (kD == 128)
            tc::mma_ss_k128(tmem + kColS + x * kBN, a0, b0, idesc_qk);
          else
            tc::mma_ss_k64(tmem + kColS + x * kBN, a0, b0, idesc_qk);
        }
        if (leader) tc::commit(&bars[S_FULL + x]);
      };
      // O_X += P_X(j) V(j)
      auto issue_pv = [&](int x, int j) {
        const int st = j % kStages;
        wait.ready(&bars[P_FULL + x], j & 1);
        tc::fence_after_sync();
        if (leader)
          tc::mma_ts_k128(tmem + kColO + x * kD, tmem + kColS + x * kBN, v_desc + ((st * kTileKV) >> 4), idesc_pv,
                          j > 0 ? 1u : 0u);
      };
      wait(&bars[Q_FULL], 0);
      if (n_tiles > 0) {
        wait.ready(&bars[K_FULL], 0);
        tc::fence_after_sync();
        for (int x = 0; x < 2; ++x)
          if (n_x[x] > 0) issue_qk(x, 0);
        if (leader) tc::commit(&bars[K_EMPTY]);
      }
      for (int x = 0; x < 2; ++x)
        if (leader && (n_x[x] == 0)) tc::commit(&bars[O_FINAL + x]);  // a tile with no key tile here: nothing to wait for
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j % kStages;
        if (v_tail && j == n_tiles - 1)
          wait(&bars[V_TAIL], 0);
        else
          wait.ready(&bars[V_FULL + st], (j / kStages) & 1);
        const bool next = j + 1 < n_tiles;
        bool k_next = false;  // K(j + 1) seen loaded
        for (int x = 0; x < 2; ++x) {
          if (j < n_x[x]) {
            issue_pv(x, j);
            if (leader && (j == n_x[x] - 1)) tc::commit(&bars[O_FINAL + x]);
            // the step's last P V (tile B's, or A's when B has no tile j) releases V(j)
            if (leader && (x == 1 || j >= n_x[1])) tc::commit(&bars[V_EMPTY + st]);
          }
          if (j + 1 < n_x[x]) {
            if (!k_next) {
              wait.ready(&bars[K_FULL + (j + 1) % kStages], ((j + 1) / kStages) & 1);
              tc::fence_after_sync();
              k_next = true;
            }
            issue_qk(x, j + 1);
          }
        }
        if (leader && next) tc::commit(&bars[K_EMPTY + (j + 1) % kStages]);
      }
      // no MMA may be in flight when TMEM is freed: tile B's last product (or
      // A's, when B has none here) is the last MMA issued
      wait(&bars[O_FINAL + (n_b > 0 ? 1 : 0)], 0);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue of tile X, one half of the keys
    const int x = (warp - 2) / kSoftmaxWarps;
    const int half = ((warp - 2) % kSoftmaxWarps) / 4;
    const int n_x = x == 0 ? n_a : n_b;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int gt = half * kBM + row;  // 0..255 within the tile's softmax threads
    const int tok_first = tok0 + x * TQ;  // first token of this query tile
    const int tok = tok_first + row / G;
    const int pos = cached + tok;  // absolute position of this query row
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t s_addr = lane_addr + kColS + x * kBN;
    const uint32_t o_addr = lane_addr + kColO + x * kD + half * (kD / 2);  // this half's D / 2 output columns
    const int lim = p.causal ? min(pos, nk - 1) : nk - 1;
    const int bar_id = 1 + x;                 // the tile's 8 softmax warps
    const int pair_id = 3 + x * 4 + quad;     // the tile's two warps (one per half) on these 32 rows
    constexpr int kGroup = 32 * kSoftmaxWarps;
    auto red_at = [&](int parity, int h) { return red + ((parity * 2 + x) * 2 + h) * kBM + row; };
    float m_run = -INFINITY;
    float l_run = 0.f;  // this half's keys only
    uint32_t r[64];

    for (int j = 0; j < n_x; ++j) {
      const int key0 = (j0 + j) * kBN + half * 64;  // first key of this half
      wait(&bars[S_FULL + x], j & 1);
      tc::fence_after_sync();
      // this half's 64 scores, held in registers: the other half writes its P
      // over them once both halves have exchanged their maxima
      tc::tmem_ld32(s_addr + half * 64, r);
      tc::tmem_ld32(s_addr + half * 64 + 32, r + 32);
      tc::tmem_wait_ld();
      if (key0 + 63 > (p.causal ? cached + tok_first : nk - 1)) {
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (key0 + e > lim) r[e] = __float_as_uint(-INFINITY);
      }
      // raw-score maximum of this half (the scale, > 0, is applied after), as
      // four chains of three-input maxima; then the row's, through shared memory
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int e = 0; e < 64; e += 8) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          mx[u] = max3(mx[u], __uint_as_float(r[e + 2 * u]), __uint_as_float(r[e + 2 * u + 1]));
      }
      *red_at(j & 1, half) = max3(fmaxf(mx[0], mx[1]), mx[2], mx[3]);
      named_barrier_sync(pair_id, 64);
      const float mt = fmaxf(*red_at(j & 1, 0), *red_at(j & 1, 1));
      const float m_new = fmaxf(m_run, mt * p.scale_log2);
      const bool grow = m_new > m_run + kRescaleLog2 || (m_run == -INFINITY && m_new != -INFINITY);
      const bool rescale = __any_sync(0xffffffffu, grow);  // the same in both halves' warps
      float factor = 1.f;
      if (rescale) {
        factor = (m_run == -INFINITY || m_new <= m_run) ? 1.f : exp2f(m_run - m_new);
        m_run = fmaxf(m_run, m_new);
      }
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      // P = exp2(scale * s - m) rounded to bf16, packed two per column: keys
      // half*64 .. half*64 + 63 are P columns half*32 .. half*32 + 31 of S.  The
      // row sum adds the same rounded values (two accumulators of two lanes,
      // so the adds do not form one long chain)
      uint64_t l_pair[2] = {0, 0};
#pragma unroll
      for (int e = 0; e < 32; ++e) r[e] = exp2_pair_bf16(r[2 * e], r[2 * e + 1], p.scale_log2, -m_use, l_pair[e % 2]);
      tc::tmem_st32(s_addr + half * 32, r);
      float l_tile = 0.f;
#pragma unroll
      for (int u = 0; u < 2; ++u)
        l_tile += __uint_as_float(static_cast<uint32_t>(l_pair[u])) +
                  __uint_as_float(static_cast<uint32_t>(l_pair[u] >> 32));
      l_run = l_run * factor + l_tile;
      if (rescale && j > 0) {
        // O_X holds the products up to tile j-1, complete: the S_X(j) commit
        // waited on above came after them; bring this half's columns to the new
        // maximum before P_X(j) V is issued
        uint32_t o[32];
#pragma unroll
        for (int c = 0; c < kD / 64; ++c) {
          tc::tmem_ld32(o_addr + c * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
          tc::tmem_st32(o_addr + c * 32, o);
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[P_FULL + x]);
    }

    wait(&bars[O_FINAL + x], 0);
    tc::fence_after_sync();
    // the row sum over both halves (the exchange buffers are free: every tile's
    // maxima were read before the last P_FULL)
    *red_at(0, half) = l_run;
    named_barrier_sync(pair_id, 64);
    l_run = *red_at(0, 0) + *red_at(0, 1);
    // this thread's 64 outputs, 32 at a time: TMEM O (zero when the tile saw no key in this part)
    auto load_o = [&](int c, uint32_t* o) {
      if (n_x > 0) {
        tc::tmem_ld32(o_addr + c * 32, o);
        tc::tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
    };
    if (parts == 1) {
      // normalised bf16 rows staged in this tile's Q buffer (free: every MMA has
      // completed), 16-byte chunk c of row r at chunk position c ^ (r mod the
      // chunks per row) so the eight rows of a quarter-warp hit distinct banks;
      // then copied out 512 contiguous bytes (when G > 1) per warp instruction
      constexpr int kChunks = kD / 8;  // 16-byte chunks per row
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      unsigned char* stage = sq + x * kTileQ;
#pragma unroll
      for (int c = 0; c < kD / 64; ++c) {
        uint32_t o[32];
        load_o(c, o);
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          float f[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) f[u] = __uint_as_float(o[e + u]) * inv;
          const int chunk = half * (kChunks / 2) + (c * 32 + e) / 8;
          *reinterpret_cast<uint4*>(stage + row * (kD * 2) + ((chunk ^ (row & (kChunks - 1))) << 4)) =
              Chunk<__nv_bfloat16>::pack(f);
        }
      }
      named_barrier_sync(bar_id, kGroup);
#pragma unroll 4
      for (int k = 0; k < kBM * kChunks / kGroup; ++k) {
        const int rr = k * (kGroup / kChunks) + gt / kChunks;
        const int chunk = gt % kChunks;
        const int tk = tok_first + rr / G;
        if (tk < nq) {
          const uint4 v =
              *reinterpret_cast<const uint4*>(stage + rr * (kD * 2) + ((chunk ^ (rr & (kChunks - 1))) << 4));
          __nv_bfloat16* o_row = p.out + (static_cast<size_t>(q_begin + tk) * p.hq + g * G + rr % G) * kD;
          reinterpret_cast<uint4*>(o_row)[chunk] = v;
        }
      }
    } else if (tok_first < nq) {
      // Split tile: every part but the last to finish publishes O (unnormalised),
      // m and l of each row; the last waits for those records and merges.  Each
      // half handles its D / 2 columns.
      const bool row_valid = tok < nq;
      __nv_bfloat16* dst = p.out + (static_cast<size_t>(q_begin + (row_valid ? tok : 0)) * p.hq + g * G + row % G) * kD +
                           half * (kD / 2);
      const int qt = 2 * pt + x;
      const long long item = (static_cast<long long>(seq) * p.hkv + g) * p.q_tiles + qt;
      const int leader = 64 + x * kGroup;  // first thread of this tile's softmax warps
      auto record = [&](int q) {
        return reinterpret_cast<float*>(p.records + (static_cast<size_t>(item) * p.parts_max + q) * kRecordBytes);
      };
      named_barrier_sync(bar_id, kGroup);
      if (threadIdx.x == leader) s_ticket[x] = atomicAdd(p.tickets + item, 1);
      named_barrier_sync(bar_id, kGroup);
      if (s_ticket[x] < parts - 1) {
        float* rec = record(part);
#pragma unroll
        for (int c = 0; c < kD / 64; ++c) {
          uint32_t o[32];
          load_o(c, o);
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            reinterpret_cast<uint4*>(rec + row * kD + half * (kD / 2) + c * 32 + e)[0] =
                make_uint4(o[e], o[e + 1], o[e + 2], o[e + 3]);
        }
        if (half == 0) {
          rec[kBM * kD + row] = m_run;
          rec[kBM * kD + kBM + row] = l_run;
        }
        __threadfence();
        named_barrier_sync(bar_id, kGroup);
        if (threadIdx.x == leader) atomicAdd(p.ready + item, 1);
      } else {
        if (threadIdx.x == leader) {
          // the other parts hold their tickets, so they are resident and publish
          // soon; the wait is still bounded
          const uint64_t t0 = globaltimer_ns();
          int ok = 0;
          while (true) {
            int v;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p.ready + item) : "memory");
            if (v == parts - 1) {
              ok = 1;
              break;
            }
            if (globaltimer_ns() - t0 > kSplitWaitNs) break;
            __nanosleep(100);
          }
          if (!ok) raise_error(p.err, PKV_DERR_WAIT_TIMEOUT);
          s_ticket[x] = ok ? 1 : -1;
        }
        named_barrier_sync(bar_id, kGroup);
        __threadfence();
        if (s_ticket[x] == 1) {
          // log-sum-exp merge over the parts that saw a key of this row, in part
          // order, so the result does not depend on the order they finished in
          float mq[kMaxParts], lq[kMaxParts];
          float mm = -INFINITY;
#pragma unroll
          for (int q = 0; q < kMaxParts; ++q) {
            mq[q] = -INFINITY;
            lq[q] = 0.f;
            if (q < parts) {
              mq[q] = q == part ? m_run : __ldcg(record(q) + kBM * kD + row);
              lq[q] = q == part ? l_run : __ldcg(record(q) + kBM * kD + kBM + row);
              if (lq[q] > 0.f) mm = fmaxf(mm, mq[q]);
            }
          }
          float total = 0.f;
#pragma unroll
          for (int q = 0; q < kMaxParts; ++q) {
            mq[q] = lq[q] > 0.f ? exp2f(mq[q] - mm) : 0.f;  // now the part's weight
            total += mq[q] * lq[q];
          }
          const float inv = total > 0.f ? 1.f / total : 0.f;
#pragma unroll
          for (int c = 0; c < kD / 64; ++c) {
            uint32_t o[32];
            load_o(c, o);
            if (row_valid) {
#pragma unroll
              for (int e = 0; e < 32; e += 8) {
                float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int q = 0; q < kMaxParts; ++q) {
                  if (q >= parts) break;
                  if (mq[q] == 0.f) continue;  // saw no key of this row: weight 0, record not read
                  float v8[8];
                  if (q == part) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) v8[u] = __uint_as_float(o[e + u]);
                  } else {
                    const float* src = record(q) + row * kD + half * (kD / 2) + c * 32 + e;
                    const float4 r0 = __ldcg(reinterpret_cast<const float4*>(src));
                    const float4 r1 = __ldcg(reinterpret_cast<const float4*>(src + 4));
                    v8[0] = r0.x, v8[1] = r0.y, v8[2] = r0.z, v8[3] = r0.w;
                    v8[4] = r1.x, v8[5] = r1.y, v8[6] = r1.z, v8[7] = r1.w;
                  }
#pragma unroll
                  for (int u = 0; u < 8; ++u) f[u] += mq[q] * v8[u];
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) f[u] *= inv;
                reinterpret_cast<uint4*>(dst + c * 32 + e)[0] = Chunk<__nv_bfloat16>::pack(f);
              }
            }
          }
        }
        named_barrier_sync(bar_id, kGroup);
        if (threadIdx.x == leader) {  // leave the tile's slots ready for the next call
          p.tickets[item] = 0;
          p.ready[item] = 0;
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int G, int D>
int launch(const PrefillArgs& a, cudaStream_t stream) {
  constexpr int TQ = kBM / G;
  constexpr int kD = D;
  alignas(64) CUtensorMap tm_q, tm_k, tm_v;
  if (encode_bf16_3d(&tm_q, a.q, kD, a.hq, a.total_q, 64, G, TQ) != PKV_OK) return PKV_ECUDA;
  const bool paged = a.block_tables != nullptr;
  const int piece = paged ? (a.block_size < kBN ? a.block_size : kBN) : kBN;
  const void* kb = paged ? a.k_cache : a.k;
  const void* vb = paged ? a.v_cache : a.v;
  const uint64_t rows = paged ? static_cast<uint64_t>(a.num_blocks) * a.block_size : a.total_k;
  if (encode_bf16_3d(&tm_k, kb, kD, a.hkv, rows, 64, 1, piece) != PKV_OK) return PKV_ECUDA;
  if (encode_bf16_3d(&tm_v, vb, kD, a.hkv, rows, 64, 1, piece) != PKV_OK) return PKV_ECUDA;
  TcParams p{};
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.block_tables = a.block_tables;
  p.err = a.err;
  p.total_q = a.total_q;
  p.total_k = a.total_k;
  p.max_seqlen_q = a.max_seqlen_q;
  p.max_blocks = a.max_blocks;
  p.hq = a.hq;
  p.hkv = a.hkv;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.causal = a.causal;
  p.paged = paged ? 1 : 0;
  p.piece_rows = piece;
  const int pairs = (a.max_seqlen_q + 2 * TQ - 1) / (2 * TQ);
  p.q_tiles = 2 * pairs;
  p.parts_max = 1;
  DeviceInfo info;
  if (device_info(&info) != PKV_OK) return PKV_ECUDA;
  const size_t ws_need = prefill_tc_workspace_bytes(a.batch, a.hkv, G, D, a.max_seqlen_q);
  if (a.workspace && ws_need > 0 && a.workspace_bytes >= ws_need) {
    const long long items = static_cast<long long>(a.batch) * a.hkv * p.q_tiles;
    const size_t flags = prefill_tc_flag_bytes(items);
    unsigned char* ws = static_cast<unsigned char*>(a.workspace);
    p.parts_max = prefill_tc_parts(a.batch, a.hkv, G, a.max_seqlen_q, info.sms);
    p.tickets = reinterpret_cast<int*>(ws);
    p.ready = reinterpret_cast<int*>(ws + flags);
    p.records = ws + 2 * flags;
  }
  auto kernel = prefill_tc_kernel<G, D>;
  constexpr uint32_t kSmemBytes = Geo<D>::kLaunchSmem;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes)) !=
      cudaSuccess)
    return PKV_ECUDA;
  dim3 grid(a.batch * a.hkv, pairs * p.parts_max);
  return launch_pdl(kernel, grid, dim3(kThreads), kSmemBytes, stream, tm_q, tm_k, tm_v, p) == cudaSuccess ? PKV_OK
                                                                                                  : PKV_ECUDA;
}

}  // namespace

namespace pkv {

bool prefill_tc_supported(const PrefillArgs& a) {
  if (a.group != 1 && a.group != 2 && a.group != 4 && a.group != 8) return false;
  if (a.head_dim != 64 && a.head_dim != 128) return false;
  if (a.total_q <= 0) return false;
  if (a.block_tables) {
    const int bs = a.block_size;
    const bool whole_tiles = bs % kBN == 0;
    const bool pieces = bs >= 8 && kBN % bs == 0;
    if (!(whole_tiles || pieces)) return false;
    if (static_cast<long long>(a.num_blocks) * bs <= 0) return false;
  } else if (a.total_k <= 0) {
    return false;
  }
  return true;
}

template <int D>
int launch_d(const PrefillArgs& a, cudaStream_t stream) {
  switch (a.group) {
    case 1: return launch<1, D>(a, stream);
    case 2: return launch<2, D>(a, stream);
    case 4: return launch<4, D>(a, stream);
    default: return launch<8, D>(a, stream);
  }
}

int prefill_tc_launch(const PrefillArgs& a, cudaStream_t stream) {
  return a.head_dim == 64 ? launch_d<64>(a, stream) : launch_d<128>(a, stream);
}

}  // namespace pkv
