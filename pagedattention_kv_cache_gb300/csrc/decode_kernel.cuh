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
// and decode_mma.cuh (the two kernels), decode_launch.cuh (host side).
#pragma once

#include "decode_launch.cuh"
