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
// the lower expert (and group) index: the decisions are those of route_oct.cuh.
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

  // K_r rounds: the warp's best remaining code, ties to the lower expert index
  unsigned taken[NT];
  int my_idx[NT];
  float my_s[NT], total[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) { taken[n] = 0; my_idx[n] = 0; my_s[n] = 0.f; total[n] = 0.f; }
  for (int r = 0; r < p.K_r; ++r) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      uint32_t best = 0u;
      int bj = 0;
      float bs = 0.f;
#pragma unroll
      for (int j = 0; j < Q; ++j) {
        const uint32_t c = ((taken[n] >> j) & 1u) ? 0u : u[n][j];
        if (c > best) { best = c; bj = j; bs = s[n][j]; }
      }
      const uint32_t m = __reduce_max_sync(0xffffffffu, best);
      const uint32_t cand = (best == m && m != 0u) ? (uint32_t)(lane + 32 * bj) : 0xffffffffu;
      const uint32_t w = __reduce_min_sync(0xffffffffu, cand);
      if (cand == w) taken[n] |= 1u << bj;   // the lane that holds expert w
      const float sw = __shfl_sync(0xffffffffu, bs, (int)(w & 31u));
      total[n] = __fadd_rn(total[n], sw);
      if (lane == r) { my_idx[n] = (int)w; my_s[n] = sw; }
    }
  }
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    if (valid[n] && lane < p.K_r) {
      p.topk_idx[(size_t)t[n] * p.K_r + lane] = my_idx[n];
      p.topk_gate[(size_t)t[n] * p.K_r + lane] = __fdiv_rn(my_s[n], total[n]);
    }
  }
}

}  // namespace moe
