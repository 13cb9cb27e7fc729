// Router for fp32 (and any shape): affinity GEMM on CUDA cores, sigmoid, then the
// warp-level biased Top-K of route_select.cuh.  Also the deterministic per-sequence
// reduction of the normalised affinities.
#include "launch.h"
#include "route_select.cuh"

namespace moe {

namespace {

constexpr int kTok = 32;   // tokens per block
constexpr int kKc = 32;    // reduction chunk

template <typename TIn>
__global__ void __launch_bounds__(256) router_simt_kernel(const TIn* __restrict__ u,
                                                          const TIn* __restrict__ e,
                                                          const float* __restrict__ b,
                                                          int d, RouteOut p) {
  extern __shared__ float sm[];
  const int N_r = p.N_r;
  float* s_tile = sm;                          // [kTok][N_r]
  float* u_tile = s_tile + kTok * N_r;         // [kTok][kKc+1]
  float* e_tile = u_tile + kTok * (kKc + 1);   // [N_r][kKc+1]
  float* b_sm = e_tile + N_r * (kKc + 1);      // [N_r]

  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * kTok;
  const int ty = tid >> 3, tx = tid & 7;
  for (int i = tid; i < N_r; i += blockDim.x) b_sm[i] = b[i];

  float acc[kMaxExperts / 8];
#pragma unroll
  for (int j = 0; j < kMaxExperts / 8; ++j) acc[j] = 0.f;

  for (int k0 = 0; k0 < d; k0 += kKc) {
    for (int x = tid; x < kTok * kKc; x += blockDim.x) {
      const int r = x / kKc, c = x % kKc, t = t0 + r, k = k0 + c;
      u_tile[r * (kKc + 1) + c] = (t < p.T && k < d) ? to_f32(u[(size_t)t * d + k]) : 0.f;
    }
    for (int x = tid; x < N_r * kKc; x += blockDim.x) {
      const int r = x / kKc, c = x % kKc, k = k0 + c;
      e_tile[r * (kKc + 1) + c] = (k < d) ? to_f32(e[(size_t)r * d + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int c = 0; c < kKc; ++c) {
      const float uv = u_tile[ty * (kKc + 1) + c];
#pragma unroll
      for (int j = 0; j < kMaxExperts / 8; ++j) {
        const int i = tx + 8 * j;
        if (i < N_r) acc[j] = fmaf(uv, e_tile[i * (kKc + 1) + c], acc[j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < kMaxExperts / 8; ++j) {
    const int i = tx + 8 * j;
    if (i < N_r) s_tile[ty * N_r + i] = sigmoid_f32(acc[j]);
  }
  __syncthreads();
  const int warp = tid >> 5;
  for (int r = warp; r < kTok; r += blockDim.x / 32) {
    const int t = t0 + r;
    if (t < p.T) route_token(s_tile + r * N_r, b_sm, t, p);
  }
}

// partial[(j*Z + z)*N_r + i] = sum over slab z of sequence j of sprime[t, i] (fp64).
__global__ void __launch_bounds__(256) seq_psum_partial_kernel(const float* __restrict__ sprime,
                                                               const int32_t* __restrict__ seq_offsets,
                                                               int N_r, int Z,
                                                               double* __restrict__ partial) {
  __shared__ double red[8][32];
  const int j = blockIdx.x, z = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int i = blockIdx.y * 32 + lane;
  const int a = seq_offsets[j], bnd = seq_offsets[j + 1];
  const int len = bnd - a;
  const int L = (len + Z - 1) / Z;
  const int t_begin = a + z * L;
  const int t_end = min(t_begin + L, bnd);
  double acc = 0.0;
  if (i < N_r)
    for (int t = t_begin + warp; t < t_end; t += 8) acc += (double)sprime[(size_t)t * N_r + i];
  red[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && i < N_r) {
    double s = 0.0;
    for (int w = 0; w < 8; ++w) s += red[w][lane];
    partial[((size_t)j * Z + z) * N_r + i] = s;
  }
}

__global__ void seq_psum_final_kernel(const double* __restrict__ partial, int n_seq, int N_r,
                                      int Z, float* __restrict__ out) {
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= n_seq * N_r) return;
  const int j = x / N_r, i = x % N_r;
  double s = 0.0;
  for (int z = 0; z < Z; ++z) s += partial[((size_t)j * Z + z) * N_r + i];
  out[x] = (float)s;
}

}  // namespace

size_t router_simt_smem(int N_r) {
  return sizeof(float) * ((size_t)kTok * N_r + kTok * (kKc + 1) + (size_t)N_r * (kKc + 1) + N_r);
}

cudaError_t launch_router_simt(const void* u, const void* e, moe_dtype dt, const float* b,
                               int d, const RouteOut& p, cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  const size_t smem = router_simt_smem(p.N_r);
  const dim3 grid((p.T + kTok - 1) / kTok);
  if (dt == MOE_F32) {
    auto k = router_simt_kernel<float>;
    cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    k<<<grid, 256, smem, st>>>((const float*)u, (const float*)e, b, d, p);
  } else {
    auto k = router_simt_kernel<__nv_bfloat16>;
    cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    k<<<grid, 256, smem, st>>>((const __nv_bfloat16*)u, (const __nv_bfloat16*)e, b, d, p);
  }
  return cudaGetLastError();
}

cudaError_t launch_seq_psum(const float* sprime, const int32_t* seq_offsets, int n_seq,
                            int N_r, double* partial, float* out, cudaStream_t st) {
  if (n_seq == 0) return cudaSuccess;
  const dim3 grid(n_seq, (N_r + 31) / 32, kSeqSlabs);
  seq_psum_partial_kernel<<<grid, 256, 0, st>>>(sprime, seq_offsets, N_r, kSeqSlabs, partial);
  const int n = n_seq * N_r;
  seq_psum_final_kernel<<<(n + 255) / 256, 256, 0, st>>>(partial, n_seq, N_r, kSeqSlabs, out);
  return cudaGetLastError();
}

}  // namespace moe
