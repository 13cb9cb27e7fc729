// Warp-cooperative routing decision for one token: biased Top-K_r with the optional
// group limit, gates from the raw affinities, and the per-token normalised
// affinities used by the sequence-wise statistic.
//
// DeepSeek-V3 Technical Report reading guide (xyznot.com), Method §2: an expert is
// selected iff s_{i,t} + b_i is among the K_r largest keys, and its gate is its raw
// s_{i,t} normalised over the selected set.  pwwt.cn notes §1.3: with the group
// limit only the M groups with the largest sums of their K_r/M best keys are
// eligible.
#pragma once

#include <math_constants.h>

#include "common.cuh"

namespace moe {

constexpr int kMaxExperts = 256;
constexpr int kMaxSlots = kMaxExperts / 32;

struct RouteOut {
  int T, N_r, K_r, G, M;
  int32_t* topk_idx;   // [T, K_r]
  float* topk_gate;    // [T, K_r]
  float* s_out;        // [T, N_r] or null
  float* sprime;       // [T, N_r] or null: s_{i,t} / sum_j s_{j,t}
};

// s_row: the token's N_r fp32 affinities (shared memory); b_sm: biases (shared).
// All 32 lanes of the warp must call it with the same token.
__device__ __forceinline__ void route_token(const float* s_row, const float* b_sm, int t,
                                            const RouteOut& p) {
  const int lane = threadIdx.x & 31;
  const int N_r = p.N_r;
  float sv[kMaxSlots], key[kMaxSlots];
#pragma unroll
  for (int j = 0; j < kMaxSlots; ++j) {
    const int i = j * 32 + lane;
    const bool ok = i < N_r;
    sv[j] = ok ? s_row[i] : 0.f;
    key[j] = ok ? __fadd_rn(sv[j], b_sm[i]) : -CUDART_INF_F;   // one fp32 rounding
  }
  const size_t rowbase = (size_t)t * N_r;
  if (p.s_out) {
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j) {
      const int i = j * 32 + lane;
      if (i < N_r) p.s_out[rowbase + i] = sv[j];
    }
  }
  if (p.sprime) {
    float part = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j) part = __fadd_rn(part, sv[j]);
    const float rs = warp_sum(part);   // butterfly: every lane holds the same sum
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j) {
      const int i = j * 32 + lane;
      if (i < N_r) p.sprime[rowbase + i] = __fdiv_rn(sv[j], rs);
    }
  }

  if (p.G > 1) {
    const int per = N_r / p.G, kg = p.K_r / p.M;
    float my_gscore = -CUDART_INF_F;   // lane g ends with group g's score
    for (int g = 0; g < p.G; ++g) {
      float tmp[kMaxSlots];
#pragma unroll
      for (int j = 0; j < kMaxSlots; ++j) {
        const int i = j * 32 + lane;
        tmp[j] = (i < N_r && i / per == g) ? key[j] : -CUDART_INF_F;
      }
      float acc = 0.f;
      for (int r = 0; r < kg; ++r) {
        KeyIdxVal best{-CUDART_INF_F, 0x7fffffff, 0.f};
#pragma unroll
        for (int j = 0; j < kMaxSlots; ++j) {
          const int i = j * 32 + lane;
          if (better(tmp[j], i, best.key, best.idx)) best = KeyIdxVal{tmp[j], i, 0.f};
        }
        best = warp_argmax(best);
        acc = __fadd_rn(acc, best.key);   // descending key order
#pragma unroll
        for (int j = 0; j < kMaxSlots; ++j)
          if (j * 32 + lane == best.idx) tmp[j] = -CUDART_INF_F;
      }
      if (lane == g) my_gscore = acc;
    }
    unsigned keep = 0;
    float gs = my_gscore;
    for (int r = 0; r < p.M; ++r) {
      KeyIdxVal best = warp_argmax(KeyIdxVal{gs, lane, 0.f});
      keep |= 1u << best.idx;
      if (lane == best.idx) gs = -CUDART_INF_F;
    }
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j) {
      const int i = j * 32 + lane;
      if (i < N_r && !((keep >> (i / per)) & 1u)) key[j] = -CUDART_INF_F;
    }
  }

  float total = 0.f, my_s = 0.f;
  int my_idx = 0;
  for (int k = 0; k < p.K_r; ++k) {
    KeyIdxVal best{-CUDART_INF_F, 0x7fffffff, 0.f};
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j) {
      const int i = j * 32 + lane;
      if (i < N_r && better(key[j], i, best.key, best.idx)) best = KeyIdxVal{key[j], i, sv[j]};
    }
    best = warp_argmax(best);
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j)
      if (j * 32 + lane == best.idx) key[j] = -CUDART_INF_F;
    total = __fadd_rn(total, best.val);
    if (lane == k) { my_idx = best.idx; my_s = best.val; }
  }
  if (lane < p.K_r) {
    p.topk_idx[(size_t)t * p.K_r + lane] = my_idx;
    p.topk_gate[(size_t)t * p.K_r + lane] = __fdiv_rn(my_s, total);
  }
}

__device__ __forceinline__ float sigmoid_f32(float z) {
  return __fdiv_rn(1.f, __fadd_rn(1.f, expf(-z)));
}

}  // namespace moe
