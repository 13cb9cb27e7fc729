// Router pieces on CUDA cores: the affinity GEMM for fp32 layers, the routing
// decision kernel shared by every layer dtype (sigmoid, bias, group limit, Top-K_r,
// gates; DeepSeek-V3 Technical Report reading guide, Method §2), and the
// deterministic per-sequence reduction of the normalised affinities.
#include "launch.h"
#include "route_select.cuh"

namespace moe {

namespace {

constexpr int kTok = 32;   // tokens per block
constexpr int kKc = 32;    // reduction chunk

// z = u e^T on CUDA cores (fp32 layers, or shapes the tensor-core GEMM does not
// take): 32 tokens x N_r centroids per block, fp32 FMA over 32-wide chunks of d.
template <typename TIn>
__global__ void __launch_bounds__(256) router_gemm_simt_kernel(const TIn* __restrict__ u,
                                                               const TIn* __restrict__ e,
                                                               int T, int d, int N_r,
                                                               float* __restrict__ z) {
  extern __shared__ float sm[];
  float* u_tile = sm;                          // [kTok][kKc+1]
  float* e_tile = u_tile + kTok * (kKc + 1);   // [N_r][kKc+1]
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * kTok;
  const int ty = tid >> 3, tx = tid & 7;
  float acc[kMaxExperts / 8];
#pragma unroll
  for (int j = 0; j < kMaxExperts / 8; ++j) acc[j] = 0.f;
  for (int k0 = 0; k0 < d; k0 += kKc) {
    for (int x = tid; x < kTok * kKc; x += blockDim.x) {
      const int r = x / kKc, c = x % kKc, t = t0 + r, k = k0 + c;
      u_tile[r * (kKc + 1) + c] = (t < T && k < d) ? to_f32(u[(size_t)t * d + k]) : 0.f;
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
  const int t = t0 + ty;
  if (t < T) {
#pragma unroll
    for (int j = 0; j < kMaxExperts / 8; ++j) {
      const int i = tx + 8 * j;
      if (i < N_r) z[(size_t)t * N_r + i] = acc[j];
    }
  }
}

// The routing decision for 32 tokens per block (one warp): z = the fixed-order fp32 sum
// of the S split-K partials, s = sigmoid(z) into shared memory, then either one thread
// per token (select_row, the common shapes) or one warp per token (route_token), and
// coalesced writes of s and s / sum(s).
__global__ void __launch_bounds__(32) router_select_kernel(const float* __restrict__ z_part,
                                                           int S, const float* __restrict__ b,
                                                           RouteOut p, int fast) {
  __shared__ float s_tile[kTok * (kMaxExperts + 1)];
  __shared__ float b_sm[kMaxExperts];
  __shared__ float rs_sm[kTok];
  const int lane = threadIdx.x, N_r = p.N_r, T = p.T, stride = N_r + 1;
  const int t0 = blockIdx.x * kTok;
  for (int i = lane; i < N_r; i += 32) b_sm[i] = b[i];
  for (int r = 0; r < kTok; ++r) {
    const int t = t0 + r;
    if (t >= T) break;
    for (int i = lane; i < N_r; i += 32) {
      float z = z_part[(size_t)t * N_r + i];
      for (int sp = 1; sp < S; ++sp) z = __fadd_rn(z, z_part[((size_t)sp * T + t) * N_r + i]);
      s_tile[r * stride + i] = sigmoid_f32(z);
    }
  }
  __syncwarp();
  if (!fast) {
    for (int r = 0; r < kTok; ++r) {
      const int t = t0 + r;
      if (t < T) route_token(s_tile + r * stride, b_sm, t, p);
    }
    return;
  }
  const int t = t0 + lane;
  float rowsum = 0.f;
  if (t < T) {
    const float* row = s_tile + lane * stride;
    float c1[kMaxSlots], c2[kMaxSlots];
#pragma unroll
    for (int c = 0; c < kMaxSlots; ++c) {
      c1[c] = c2[c] = -CUDART_INF_F;
      if (c < N_r / 32) {
#pragma unroll 8
        for (int j = 0; j < 32; ++j) {
          const int i = c * 32 + j;
          const float sv = row[i];
          rowsum = __fadd_rn(rowsum, sv);
          const float k = __fadd_rn(sv, b_sm[i]);
          c2[c] = fmaxf(c2[c], fminf(c1[c], k));
          c1[c] = fmaxf(c1[c], k);
        }
      }
    }
    select_row(row, b_sm, c1, c2, t, p);
  }
  rs_sm[lane] = rowsum;
  __syncwarp();
  if (p.s_out || p.sprime) {
    for (int r = 0; r < kTok; ++r) {
      const int tr = t0 + r;
      if (tr >= T) break;
      const float rs = rs_sm[r];
      for (int i = lane; i < N_r; i += 32) {
        const float sv = s_tile[r * stride + i];
        if (p.s_out) p.s_out[(size_t)tr * N_r + i] = sv;
        if (p.sprime) p.sprime[(size_t)tr * N_r + i] = __fdiv_rn(sv, rs);
      }
    }
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

cudaError_t launch_router_gemm_simt(const void* u, const void* e, moe_dtype dt, int T, int d,
                                    int N_r, float* z, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const size_t smem = sizeof(float) * ((size_t)kTok * (kKc + 1) + (size_t)N_r * (kKc + 1));
  const dim3 grid((T + kTok - 1) / kTok);
  if (dt == MOE_F32) {
    router_gemm_simt_kernel<float><<<grid, 256, smem, st>>>((const float*)u, (const float*)e, T,
                                                            d, N_r, z);
  } else {
    router_gemm_simt_kernel<__nv_bfloat16><<<grid, 256, smem, st>>>(
        (const __nv_bfloat16*)u, (const __nv_bfloat16*)e, T, d, N_r, z);
  }
  return cudaGetLastError();
}

cudaError_t launch_router_select(const float* z_part, int S, const float* b, const RouteOut& p,
                                 cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  const int fast = fast_select_ok(p.N_r, p.K_r, p.G, p.M) ? 1 : 0;
  router_select_kernel<<<(p.T + kTok - 1) / kTok, 32, 0, st>>>(z_part, S, b, p, fast);
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
