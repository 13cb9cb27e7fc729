// The routing decisions of tokens by one warp, for N_r = 32*Q experts (Q = 2, 4, 8)
// and K_r <= 8: lane l holds experts l + 32j, j < Q, so expert block j (experts
// 32j .. 32j+31) is the j-th value of every lane and each reduction over a block is one
// warp-wide redux.
//
// DeepSeek-V3 Technical Report reading guide (xyznot.com), Method §2: an expert is
// selected iff s_{i,t} + b_i is among the K_r largest keys, and its gate is its raw
// s_{i,t} normalised over the selected set.  pwwt.cn notes §1.3: with the group limit
// only the M groups with the largest sums of their K_r/M best keys are eligible; here a
// group is Q/G whole 32-expert blocks and K_r/M <= 2.  Keys are fp32(s + b), ties go to
// the lower expert (and group) index: the decisions are those of route_oct.cuh.  Each
// lane sorts its Q keys once, so a Top-K_r round needs two warp reductions over the
// lanes' leading keys and a shift of the winning lane's list.
#pragma once

#include <math_constants.h>

#include "common.cuh"
#include "route_select.cuh"

namespace moe {

// Order-preserving code of an fp32 key: a larger key gets a larger code, -0 is taken
// as +0 (so equal keys get equal codes), and code 0 lies below every key.
__device__ __forceinline__ uint32_t key_code(float k) {
  const uint32_t b = __float_as_uint(k == 0.f ? 0.f : k);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float code_key(uint32_t c) {
  return __uint_as_float((c & 0x80000000u) ? (c & 0x7fffffffu) : ~c);
}

// Sorts Q = 2, 4 or 8 values in descending order with a fixed comparator network.
template <int Q>
__device__ __forceinline__ void sort_desc(uint64_t (&k)[Q]) {
  auto cx = [&](int a, int b) {   // k[a] >= k[b] afterwards
    const uint64_t x = k[a], y = k[b];
    const bool sw = y > x;
    k[a] = sw ? y : x;
    k[b] = sw ? x : y;
  };
  if constexpr (Q == 2) {
    cx(0, 1);
  } else if constexpr (Q == 4) {
    cx(0, 1); cx(2, 3); cx(0, 2); cx(1, 3); cx(1, 2);
  } else {
    static_assert(Q == 8, "Q is 2, 4 or 8");
    // Batcher's odd-even merge sort of eight values: 19 comparators
    cx(0, 1); cx(2, 3); cx(4, 5); cx(6, 7);
    cx(0, 2); cx(1, 3); cx(4, 6); cx(5, 7);
    cx(1, 2); cx(5, 6);
    cx(0, 4); cx(1, 5); cx(2, 6); cx(3, 7);
    cx(2, 4); cx(3, 5);
    cx(1, 2); cx(3, 4); cx(5, 6);
  }
}

// Group limit, Top-K_r and gates of NT tokens at once (independent chains, so the warp
// interleaves their reductions) from the warp's s (lane l: experts l + 32j) and b, with
// G groups of Q/G blocks (G = 1: no group limit); for a token with valid[n], lane
// r < K_r writes its r-th selected expert and gate.  Called by all 32 lanes of the warp.
template <int Q, int G, int NT>
__device__ __forceinline__ void warp_decide(const float (&s)[NT][Q], const float (&b)[Q], const int (&t)[NT],
                                            const bool (&valid)[NT], const RouteOut& p) {
  static_assert(Q % G == 0, "a group is whole 32-expert blocks");
  const int lane = threadIdx.x & 31;
  uint32_t u[NT][Q];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int j = 0; j < Q; ++j) u[n][j] = key_code(__fadd_rn(s[n][j], b[j]));

  if constexpr (G > 1) {
    constexpr int BPG = Q / G;            // blocks per group
    const int kg = p.K_r / p.M;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      // each block's two best codes (the second equals the first when the best is tied)
      uint32_t m1[Q], m2[Q];
#pragma unroll
      for (int j = 0; j < Q; ++j) m1[j] = __reduce_max_sync(0xffffffffu, u[n][j]);
#pragma unroll
      for (int j = 0; j < Q; ++j) {
        const unsigned eq = __ballot_sync(0xffffffffu, u[n][j] == m1[j]);
        const uint32_t rest = __reduce_max_sync(0xffffffffu, u[n][j] == m1[j] ? 0u : u[n][j]);
        m2[j] = __popc(eq) >= 2 ? m1[j] : rest;
      }
      // group scores: the best key (K_r/M = 1) or the fp32 sum of the best two in
      // descending order (K_r/M = 2); every lane holds all G of them
      float gs[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        uint32_t t1 = 0, t2 = 0;
#pragma unroll
        for (int j = g * BPG; j < (g + 1) * BPG; ++j) {
          const uint32_t lo = min(t1, m1[j]);
          t1 = max(t1, m1[j]);
          t2 = max(max(t2, m2[j]), lo);
        }
        gs[g] = kg == 1 ? code_key(t1) : __fadd_rn(code_key(t1), code_key(t2));
      }
      // lane g < G ranks group g (higher score first, ties to the lower index); the M
      // best are kept
      float mine = gs[0];
#pragma unroll
      for (int g = 1; g < G; ++g) mine = lane == g ? gs[g] : mine;
      int rank = 0;
#pragma unroll
      for (int h = 0; h < G; ++h) rank += (gs[h] > mine || (gs[h] == mine && h < lane)) ? 1 : 0;
      const unsigned gkeep = __ballot_sync(0xffffffffu, lane < G && rank < p.M);
#pragma unroll
      for (int j = 0; j < Q; ++j)
        if (!((gkeep >> (j / BPG)) & 1u)) u[n][j] = 0u;
    }
  }

  // Each lane orders its Q keys once, as 64-bit values (code, then Q-1-j: a higher
  // code first, and of equal codes the lower expert index, since lane l holds experts
  // l + 32j); a round then looks only at each lane's head.
  uint64_t k[NT][Q];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int j = 0; j < Q; ++j) k[n][j] = ((uint64_t)u[n][j] << 32) | (uint32_t)(Q - 1 - j);
#pragma unroll
  for (int n = 0; n < NT; ++n) sort_desc<Q>(k[n]);

  // K_r rounds: the warp's best head code (redux max), of equal ones the lowest expert
  // index (redux min); the lane that held it drops its head
  int my_idx[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) my_idx[n] = 0;
  for (int r = 0; r < p.K_r; ++r) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const uint32_t head = (uint32_t)(k[n][0] >> 32);
      const uint32_t m = __reduce_max_sync(0xffffffffu, head);
      const uint32_t e = (uint32_t)lane + 32u * (uint32_t)(Q - 1 - (int)(uint32_t)k[n][0]);
      const uint32_t cand = (head == m && m != 0u) ? e : 0xffffffffu;
      const uint32_t w = __reduce_min_sync(0xffffffffu, cand);
      const bool won = cand == w;
#pragma unroll
      for (int j = 0; j + 1 < Q; ++j) k[n][j] = won ? k[n][j + 1] : k[n][j];
      k[n][Q - 1] = won ? 0ull : k[n][Q - 1];
      if (lane == r) my_idx[n] = (int)w;
    }
  }
  // gates: lane r < K_r fetches the raw s of its expert; the normaliser adds them in
  // round order
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int w = my_idx[n];
    float my_s = 0.f;
#pragma unroll
    for (int j = 0; j < Q; ++j) {
      const float v = __shfl_sync(0xffffffffu, s[n][j], w & 31);
      my_s = (w >> 5) == j ? v : my_s;
    }
    float total = 0.f;
    for (int r = 0; r < p.K_r; ++r) total = __fadd_rn(total, __shfl_sync(0xffffffffu, my_s, r));
    if (valid[n] && lane < p.K_r) {
      p.topk_idx[(size_t)t[n] * p.K_r + lane] = w;
      p.topk_gate[(size_t)t[n] * p.K_r + lane] = __fdiv_rn(my_s, total);
    }
  }
}

}  // namespace moe
