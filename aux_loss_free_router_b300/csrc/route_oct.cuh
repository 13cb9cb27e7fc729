// The routing decision of one token held by eight threads, for N_r = 32*Q experts
// (Q = 2, 4, 8) and K_r <= 8: thread `part` of the token holds experts
// 32q + 4*part .. 32q + 4*part + 3 of every 32-expert block q.
//
// DeepSeek-V3 Technical Report reading guide (xyznot.com), Method §2: an expert is
// selected iff s_{i,t} + b_i is among the K_r largest keys, and its gate is its raw
// s_{i,t} normalised over the selected set.  pwwt.cn notes §1.3: with the group limit
// only the M groups with the largest sums of their K_r/M best keys are eligible; here a
// group is Q/G whole 32-expert blocks and K_r/M <= 2.  Keys are fp32(s + b), ties go to
// the lower expert (and group) index.
#pragma once

#include <math_constants.h>

#include "common.cuh"
#include "route_select.cuh"

namespace moe {

// Top-8 list of (key, index, s) triples in descending key order, ties to the lower
// index (better()); empty slots hold -inf.
struct Top8 {
  float k[8], s[8];
  int i[8];
};

__device__ __forceinline__ void top8_clear(Top8& L) {
#pragma unroll
  for (int j = 0; j < 8; ++j) { L.k[j] = -CUDART_INF_F; L.i[j] = 0x7fffffff; L.s[j] = 0.f; }
}

// Insert (key, idx, sv) if it beats the last entry.
__device__ __forceinline__ void top8_insert(Top8& L, float key, int idx, float sv) {
  if (!better(key, idx, L.k[7], L.i[7])) return;
  bool c[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) c[j] = better(key, idx, L.k[j], L.i[j]);
#pragma unroll
  for (int j = 7; j >= 1; --j) {
    if (c[j - 1]) { L.k[j] = L.k[j - 1]; L.i[j] = L.i[j - 1]; L.s[j] = L.s[j - 1]; }
    else if (c[j]) { L.k[j] = key; L.i[j] = idx; L.s[j] = sv; }
  }
  if (c[0]) { L.k[0] = key; L.i[0] = idx; L.s[0] = sv; }
}

__device__ __forceinline__ void top8_cswap(Top8& L, int a, int b) {   // L[a] before L[b]
  if (better(L.k[b], L.i[b], L.k[a], L.i[a])) {
    const float tk = L.k[a], ts = L.s[a];
    const int ti = L.i[a];
    L.k[a] = L.k[b]; L.i[a] = L.i[b]; L.s[a] = L.s[b];
    L.k[b] = tk; L.i[b] = ti; L.s[b] = ts;
  }
}

// Top 8 of this lane's list and that of lane ^ xr: taking, slot by slot, the better of
// the list and the partner's reversed list keeps the eight best as a bitonic sequence,
// which three half-cleaner stages sort.  Both lanes end with the same list.
__device__ __forceinline__ void top8_merge(Top8& L, int xr) {
  float pk[8], ps[8];
  int pi[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    pk[j] = __shfl_xor_sync(0xffffffffu, L.k[j], xr);
    pi[j] = __shfl_xor_sync(0xffffffffu, L.i[j], xr);
    ps[j] = __shfl_xor_sync(0xffffffffu, L.s[j], xr);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (better(pk[7 - j], pi[7 - j], L.k[j], L.i[j])) {
      L.k[j] = pk[7 - j]; L.i[j] = pi[7 - j]; L.s[j] = ps[7 - j];
    }
#pragma unroll
  for (int d = 4; d >= 1; d >>= 1)
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if ((j & d) == 0) top8_cswap(L, j, j + d);
}

// Whether router_select_oct_kernel takes the shape: 64, 128 or 256 experts, K_r <= 8,
// and with the group limit groups of whole 32-expert blocks keeping K_r/M <= 2 keys.
__host__ __device__ inline bool oct_select_ok(int N_r, int K_r, int G, int M) {
  if (N_r != 64 && N_r != 128 && N_r != 256) return false;
  if (K_r > 8) return false;
  if (G == 1) return true;
  return (N_r / 32) % G == 0 && K_r / M <= 2;
}

// Group limit, Top-K_r and gates of token t from its eight threads' (s, b) values;
// thread `part` < K_r writes the part-th selected expert and its gate.  All 32 lanes of
// the warp call it (the shuffles span the token's eight lanes).
template <int Q>
__device__ __forceinline__ void oct_decide(const float (&sv)[Q][4], const float (&bv)[Q][4],
                                           int part, int t, bool valid, const RouteOut& p) {
  // group limit: bit q of `keep` marks an eligible 32-expert block (G divides Q and both
  // are powers of two)
  unsigned keep = (1u << Q) - 1u;
  if (p.G > 1) {
    const int G = p.G, kg = p.K_r / p.M;
    const int gsh = __ffs(Q / G) - 1;   // blocks per group = Q/G, a power of two: shift, not divide
    float b1[Q], b2[Q];                 // each block's two best keys over the token
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      float t1 = -CUDART_INF_F, t2 = -CUDART_INF_F;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float k = __fadd_rn(sv[q][j], bv[q][j]);
        const float lo = fminf(t1, k);
        t1 = fmaxf(t1, k);
        t2 = fmaxf(t2, lo);
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        const float a1 = __shfl_xor_sync(0xffffffffu, t1, o);
        const float a2 = __shfl_xor_sync(0xffffffffu, t2, o);
        const float lo = fminf(t1, a1);
        t1 = fmaxf(t1, a1);
        t2 = fmaxf(fmaxf(t2, a2), lo);
      }
      b1[q] = t1;
      b2[q] = t2;
    }
    // group g = blocks [g*bq, (g+1)*bq): fold the blocks' pairs, score = best (kg = 1)
    // or fp32 sum of the best two in descending order (kg = 2)
    float gs[Q];
#pragma unroll
    for (int g = 0; g < Q; ++g) {
      gs[g] = -CUDART_INF_F;
      if (g < G) {
        float t1 = -CUDART_INF_F, t2 = -CUDART_INF_F;
#pragma unroll
        for (int q = 0; q < Q; ++q) {
          if ((q >> gsh) == g) {
            const float lo = fminf(t1, b1[q]);
            t1 = fmaxf(t1, b1[q]);
            t2 = fmaxf(fmaxf(t2, b2[q]), lo);
          }
        }
        gs[g] = kg == 1 ? t1 : __fadd_rn(t1, t2);
      }
    }
    unsigned gkeep = 0;
    for (int m = 0; m < p.M; ++m) {      // M best groups, ties to the lower index
      float best = -CUDART_INF_F;
      int bg = -1;
#pragma unroll
      for (int g = 0; g < Q; ++g)
        if (g < G && !((gkeep >> g) & 1u) && (bg < 0 || gs[g] > best)) { best = gs[g]; bg = g; }
      gkeep |= 1u << bg;
    }
    keep = 0;
#pragma unroll
    for (int q = 0; q < Q; ++q)
      if ((gkeep >> (q >> gsh)) & 1u) keep |= 1u << q;
  }

  Top8 L;
  top8_clear(L);
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    if ((keep >> q) & 1u) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        top8_insert(L, __fadd_rn(sv[q][j], bv[q][j]), 32 * q + 4 * part + j, sv[q][j]);
    }
  }
  top8_merge(L, 1);
  top8_merge(L, 2);
  top8_merge(L, 4);
  float total = 0.f, my_s = 0.f;
  int my_i = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < p.K_r) total = __fadd_rn(total, L.s[j]);
    if (j == part) { my_s = L.s[j]; my_i = L.i[j]; }
  }
  if (valid && part < p.K_r) {
    p.topk_idx[(size_t)t * p.K_r + part] = my_i;
    p.topk_gate[(size_t)t * p.K_r + part] = __fdiv_rn(my_s, total);
  }
}

}  // namespace moe
