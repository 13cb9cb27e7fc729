// Expert FFNs in fp32 on CUDA cores (used for fp32 layers, where tensor-core TF32
// would miss the fp32 tolerance).  Same row space and segment schedule as the
// tensor-core path: a block walks tiles (segment, n-tile, m-tile) computed on the
// device from expert_offset, so no host synchronisation is needed.
#include <algorithm>

#include "common.cuh"
#include "ffn_sched.cuh"
#include "launch.h"

namespace moe {

namespace {

constexpr int BM = 64, BN = 64, BK = 32;
constexpr int kLd = BM * BK / 256;   // elements of each operand a thread loads per K step

__device__ __forceinline__ float silu_f32(float z) { return __fdiv_rn(z, __fadd_rn(1.f, expf(-z))); }

// MODE 0: h = silu(x Wg^T) * (x Wu^T) over K = d, N = I.
// MODE 1: y = h Wd^T over K = I, N = d.
template <int MODE>
__global__ void __launch_bounds__(256) ffn_simt_kernel(FfnShape s, const float* __restrict__ a_routed,
                                                       const float* __restrict__ a_shared,
                                                       const int32_t* __restrict__ expert_offset,
                                                       const float* __restrict__ w0,
                                                       const float* __restrict__ w1,
                                                       const float* __restrict__ ws0,
                                                       const float* __restrict__ ws1,
                                                       float* __restrict__ out, int32_t* err) {
  __shared__ SegTable tab;
  __shared__ float As[BK][BM + 1];   // +1: the transposing stores hit 32 banks
  __shared__ float B0[BK][BN + 1];
  __shared__ float B1[BK][BN + 1];
  pdl_release();
  pdl_wait();
  const int K = MODE == 0 ? s.d : s.I;
  const int N = MODE == 0 ? s.I : s.d;
  const int n_tiles_n = (N + BN - 1) / BN;
  build_seg_table(tab, expert_offset, s.T, s.K_r, s.N_r, s.N_s, BM, n_tiles_n, false, err);
  __syncthreads();
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int tile = blockIdx.x; tile < tab.total; tile += gridDim.x) {
    const TileCoord tc = decode_tile(tab, tile, n_tiles_n);
    const bool shared = tc.seg >= s.N_r;
    const int e = shared ? tc.seg - s.N_r : tc.seg;
    // Input rows: routed -> x_perm / h rows; shared (MODE 0) -> u rows; shared (MODE 1) ->
    // h rows of that shared expert.
    const float* A;
    if (MODE == 0) A = shared ? a_shared : a_routed + (size_t)tc.row0 * K;
    else A = a_routed + (size_t)tc.out_row0 * K;
    const float* W0 = (shared ? ws0 : w0) + (size_t)e * N * K;
    const float* W1 = MODE == 0 ? (shared ? ws1 : w1) + (size_t)e * N * K : nullptr;
    const int m0 = tc.m * BM, n0 = tc.n * BN;
    float acc0[4][4], acc1[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc0[i][j] = acc1[i][j] = 0.f;
    // the next K step's operands are loaded into registers while this one computes
    float ra[kLd], rb0[kLd], rb1[kLd];
    auto load_step = [&](int k0) {
#pragma unroll
      for (int q = 0; q < kLd; ++q) {
        const int x = threadIdx.x + 256 * q;
        const int r = x / BK, c = x % BK, gk = k0 + c;
        ra[q] = (m0 + r < tc.rows && gk < K) ? A[(size_t)(m0 + r) * K + gk] : 0.f;
        const bool ok = n0 + r < N && gk < K;
        rb0[q] = ok ? W0[(size_t)(n0 + r) * K + gk] : 0.f;
        if (MODE == 0) rb1[q] = ok ? W1[(size_t)(n0 + r) * K + gk] : 0.f;
      }
    };
    load_step(0);
    for (int k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
      for (int q = 0; q < kLd; ++q) {
        const int x = threadIdx.x + 256 * q;
        const int r = x / BK, c = x % BK;
        As[c][r] = ra[q];
        B0[c][r] = rb0[q];
        if (MODE == 0) B1[c][r] = rb1[q];
      }
      __syncthreads();
      if (k0 + BK < K) load_step(k0 + BK);
#pragma unroll
      for (int c = 0; c < BK; ++c) {
        float av[4], bv0[4], bv1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = As[c][ty + 16 * i];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          bv0[j] = B0[c][tx + 16 * j];
          if (MODE == 0) bv1[j] = B1[c][tx + 16 * j];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc0[i][j] = fmaf(av[i], bv0[j], acc0[i][j]);
            if (MODE == 0) acc1[i][j] = fmaf(av[i], bv1[j], acc1[i][j]);
          }
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = m0 + ty + 16 * i;
      if (r >= tc.rows) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = n0 + tx + 16 * j;
        if (n >= N) continue;
        const float v = MODE == 0 ? silu_f32(acc0[i][j]) * acc1[i][j] : acc0[i][j];
        out[(size_t)(tc.out_row0 + r) * N + n] = v;
      }
    }
  }
}

int grid_for(const FfnShape& s, int N) {
  const long long routed = (long long)s.T * s.K_r;
  const long long m_tiles = routed / BM + s.N_r + (long long)s.N_s * ((s.T + BM - 1) / BM);
  const long long tiles = m_tiles * ((N + BN - 1) / BN);
  const long long cap = 8LL * device_sm_count();
  return (int)std::max(1LL, std::min(tiles, cap));
}

}  // namespace

cudaError_t launch_ffn_up_simt(const FfnShape& s, const float* x_perm, const float* u,
                               const int32_t* expert_offset, const moe_expert_weights* w,
                               float* h, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  const cudaError_t err = launch_pdl(ffn_simt_kernel<0>, dim3(grid_for(s, s.I)), dim3(256), 0, st, 0, s,
                                     x_perm, u, expert_offset, (const float*)w->gate,
                                     (const float*)w->up, (const float*)w->s_gate,
                                     (const float*)w->s_up, h, dev_error_ptr());
  return err != cudaSuccess ? err : cudaGetLastError();
}

cudaError_t launch_ffn_down_simt(const FfnShape& s, const float* h,
                                 const int32_t* expert_offset, const moe_expert_weights* w,
                                 float* y, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  const cudaError_t err = launch_pdl(ffn_simt_kernel<1>, dim3(grid_for(s, s.d)), dim3(256), 0, st, 0, s, h,
                                     (const float*)nullptr, expert_offset, (const float*)w->down,
                                     (const float*)nullptr, (const float*)w->s_down,
                                     (const float*)nullptr, y, dev_error_ptr());
  return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace moe
