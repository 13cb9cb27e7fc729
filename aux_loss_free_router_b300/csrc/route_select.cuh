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

// Tokens per P-sum window: the selection kernels sum s_{i,t} / sum_j s_{j,t} over the
// tokens of each window that belong to one sequence.
constexpr int kPWindow = 32;

struct RouteOut {
  int T, N_r, K_r, G, M;
  int32_t* topk_idx;   // [T, K_r]
  float* topk_gate;    // [T, K_r]
  float* s_out;        // [T, N_r] or null
  // [T, N_r] or null.  For every run of tokens [t, t') that lies in one kPWindow-token
  // window and one sequence, row t receives sum_{t <= x < t'} s_{i,x} / sum_j s_{j,x};
  // other rows are not written.
  float* pwin;
  const int32_t* seq_offsets;   // [n_seq + 1], used when pwin is set
  int n_seq;
};

// Index of the sequence holding token t: the largest j with seq_offsets[j] <= t.
__device__ __forceinline__ int seq_of(int t, const int32_t* __restrict__ off, int n_seq) {
  int lo = 0, hi = n_seq;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(off + mid) <= t) lo = mid; else hi = mid;
  }
  return lo;
}

// Window sums of one expert column: v(r) gives s'_{i, t0+r} for the window's ntok
// tokens, seqid[r] their sequences; each run of one sequence is written to the row of
// its first token.
template <typename F>
__device__ __forceinline__ void window_runs(F v, const int* seqid, int ntok, int t0, int N_r,
                                            int i, float* __restrict__ pwin) {
  float acc = 0.f;
  int start = 0;
  for (int r = 0; r < ntok; ++r) {
    acc = __fadd_rn(acc, v(r));
    if (r == ntok - 1 || seqid[r + 1] != seqid[r]) {
      pwin[(size_t)(t0 + start) * N_r + i] = acc;
      acc = 0.f;
      start = r + 1;
    }
  }
}

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

constexpr int kFastK = 8;    // per-thread selection keeps the 8 largest keys
constexpr int kFastG = 16;   // and handles up to 16 groups of whole 32-column chunks

// One thread takes the whole decision for its token.  c1/c2 hold the two largest keys
// of every 32-column chunk; with the group limit a group is per/32 whole chunks and
// keeps its K_r/M <= 2 best keys.  Candidates are visited in ascending expert index
// and only a strictly larger key displaces a list entry, so equal keys keep the lower
// index first, as the definition requires.
__device__ __forceinline__ void select_row(const float* s_row, const float* b,
                                           const float (&c1)[kMaxSlots],
                                           const float (&c2)[kMaxSlots], int t,
                                           const RouteOut& p) {
  if (t >= p.T) return;
  const int N_r = p.N_r;
  unsigned keep = 0xffffffffu;
  int per = N_r, n_keep = 1;
  if (p.G > 1) {
    per = N_r / p.G;
    const int cpg = per / 32, kg = p.K_r / p.M;
    float gs[kFastG];
#pragma unroll
    for (int g = 0; g < kFastG; ++g) {
      float t1 = -CUDART_INF_F, t2 = -CUDART_INF_F;
#pragma unroll
      for (int c = 0; c < kMaxSlots; ++c) {
        if (c / cpg == g && c < N_r / 32) {   // chunk c belongs to group g
          const float lo = fminf(t1, c1[c]);
          t1 = fmaxf(t1, c1[c]);
          t2 = fmaxf(lo, fmaxf(t2, c2[c]));
        }
      }
      gs[g] = kg == 1 ? t1 : __fadd_rn(t1, t2);   // fp32, descending order
    }
    keep = 0;
    for (int m = 0; m < p.M; ++m) {
      float best = -CUDART_INF_F;
      int bg = 0;
#pragma unroll
      for (int g = kFastG - 1; g >= 0; --g)   // descending scan: ties settle on the lower g
        if (g < p.G && !((keep >> g) & 1u) && gs[g] >= best) { best = gs[g]; bg = g; }
      keep |= 1u << bg;
    }
    n_keep = p.M;
  }
  float lk[kFastK];
  int li[kFastK];
#pragma unroll
  for (int j = 0; j < kFastK; ++j) { lk[j] = -CUDART_INF_F; li[j] = 0; }
  for (int m = 0; m < n_keep; ++m) {
    const int g = p.G > 1 ? (int)__fns(keep, 0, m + 1) : 0;   // m-th kept group, ascending
    const int c0 = g * per;
    for (int j0 = 0; j0 < per; ++j0) {
      const int i = c0 + j0;
      const float v = __fadd_rn(s_row[i], b[i]);
      if (v > lk[kFastK - 1]) {
        bool cj[kFastK];
#pragma unroll
        for (int j = 0; j < kFastK; ++j) cj[j] = v > lk[j];
#pragma unroll
        for (int j = kFastK - 1; j >= 1; --j) {
          const float nk = cj[j - 1] ? lk[j - 1] : (cj[j] ? v : lk[j]);
          const int ni = cj[j - 1] ? li[j - 1] : (cj[j] ? i : li[j]);
          lk[j] = nk;
          li[j] = ni;
        }
        if (cj[0]) { lk[0] = v; li[0] = i; }
      }
    }
  }
  float total = 0.f, sel[kFastK];
#pragma unroll
  for (int j = 0; j < kFastK; ++j) {
    sel[j] = j < p.K_r ? s_row[li[j]] : 0.f;
    if (j < p.K_r) total = __fadd_rn(total, sel[j]);
  }
#pragma unroll
  for (int j = 0; j < kFastK; ++j) {
    if (j < p.K_r) {
      p.topk_idx[(size_t)t * p.K_r + j] = li[j];
      p.topk_gate[(size_t)t * p.K_r + j] = __fdiv_rn(sel[j], total);
    }
  }
}

// Whether select_row() handles the shape: K_r <= 8, and either no group limit or
// groups made of whole 32-expert chunks (at most 16 groups) keeping <= 2 keys each.
inline bool fast_select_ok(int N_r, int K_r, int G, int M) {
  if (K_r > kFastK || N_r % 32 != 0) return false;
  if (G == 1) return true;
  const int per = N_r / G;
  return per % 32 == 0 && G <= kFastG && K_r / M <= 2;
}

// 1 / (1 + e^-z) from the fast exponential and the fast reciprocal (absolute error
// about 1e-7, well inside the affinity tolerances).
__device__ __forceinline__ float sigmoid_f32(float z) {
  return __fdividef(1.f, __fadd_rn(1.f, __expf(-z)));
}

}  // namespace moe
