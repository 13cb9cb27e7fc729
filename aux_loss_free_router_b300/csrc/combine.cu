// Combine: h'_t = u_t + sum_s FFN_s(u_t) + sum_k g_{t,k} FFN_{idx_k}(u_t)
// (DeepSeek-V3 Technical Report reading guide, Method §2, equation for h'_t;
// pwwt.cn notes §四: the gate-weighted sum of the experts' outputs back at the token).
//
// One warp per token and column chunk; each lane owns 16-byte column vectors, so every
// row read is a fully coalesced 512-byte warp access.  Small batches (decode) split each
// row into column chunks over gridDim.y so that enough warps have loads in flight.  The
// fp32 accumulation order of every element is fixed: u, shared experts ascending,
// routed slots k ascending (deterministic, and independent of the chunking).  A routed
// row index outside [0, T*K_r) (inv_row = -1 marks an entry dispatch skipped) is read as
// row 0 with gate 0, so it adds nothing, and MOE_ERR_INVALID_ARG is recorded in the
// device error word.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

// Below this many token warps a row is split into column chunks.
constexpr int kTargetWarps = 2048;

template <typename TIn> struct Vec;
template <> struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void load(const float* p, float (&v)[4]) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  }
};
template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __bfloat1622float2(h[q]);
      v[2 * q] = f.x; v[2 * q + 1] = f.y;
    }
  }
};

template <typename TOut, int N> __device__ void store_vec(TOut* p, const float (&v)[N]);
template <> __device__ void store_vec<float, 4>(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
template <> __device__ void store_vec<float, 8>(float* p, const float (&v)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
template <> __device__ void store_vec<__nv_bfloat16, 8>(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 x;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&x);
#pragma unroll
  for (int q = 0; q < 4; ++q) h[q] = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
  *reinterpret_cast<uint4*>(p) = x;
}
template <> __device__ void store_vec<__nv_bfloat16, 4>(__nv_bfloat16* p, const float (&v)[4]) {
  uint2 x;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&x);
  h[0] = __floats2bfloat162_rn(v[0], v[1]);
  h[1] = __floats2bfloat162_rn(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) = x;
}

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(256) combine_kernel(const TIn* __restrict__ u,
                                                      const TIn* __restrict__ y,
                                                      const float* __restrict__ gate,
                                                      const int32_t* __restrict__ inv_row,
                                                      int T, int d, int K_r, int N_s,
                                                      int pass_per_chunk,
                                                      TOut* __restrict__ out, int32_t* err) {
  constexpr int V = Vec<TIn>::N;
  pdl_release();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;
  const int c_begin = blockIdx.y * pass_per_chunk * 64 * V;
  const int c_end = min(d, c_begin + pass_per_chunk * 64 * V);
  const size_t routed_rows = (size_t)T * K_r;
  float my_g = lane < K_r ? gate[(size_t)t * K_r + lane] : 0.f;
  int my_r = lane < K_r ? inv_row[(size_t)t * K_r + lane] : 0;
  if ((size_t)(unsigned)my_r >= routed_rows) {     // also catches negative rows: the slot
    if (blockIdx.y == 0) record_error(err, MOE_ERR_INVALID_ARG);   // adds exactly 0 * y[0]
    my_r = 0;
    my_g = 0.f;
  }
  // two 16-byte column vectors per lane per pass: twice the loads in flight
  for (int c0 = c_begin; c0 < c_end; c0 += 64 * V) {
    const int ca = c0 + lane * V, cb = ca + 32 * V;
    const bool oka = ca < c_end, okb = cb < c_end;
    float acc[2][V], tmp[2][V];
#pragma unroll
    for (int q = 0; q < V; ++q) acc[0][q] = acc[1][q] = 0.f;
    if (oka) Vec<TIn>::load(u + (size_t)t * d + ca, acc[0]);
    if (okb) Vec<TIn>::load(u + (size_t)t * d + cb, acc[1]);
    for (int s = 0; s < N_s; ++s) {
      const TIn* row = y + (routed_rows + (size_t)s * T + t) * d;
      if (oka) Vec<TIn>::load(row + ca, tmp[0]);
      if (okb) Vec<TIn>::load(row + cb, tmp[1]);
#pragma unroll
      for (int q = 0; q < V; ++q) {
        acc[0][q] = __fadd_rn(acc[0][q], tmp[0][q]);
        acc[1][q] = __fadd_rn(acc[1][q], tmp[1][q]);
      }
    }
#pragma unroll 4
    for (int k = 0; k < K_r; ++k) {
      const float g = __shfl_sync(0xffffffffu, my_g, k);
      const int r = __shfl_sync(0xffffffffu, my_r, k);
      const TIn* row = y + (size_t)r * d;
      if (oka) Vec<TIn>::load(row + ca, tmp[0]);
      if (okb) Vec<TIn>::load(row + cb, tmp[1]);
#pragma unroll
      for (int q = 0; q < V; ++q) {
        acc[0][q] = fmaf(g, tmp[0][q], acc[0][q]);
        acc[1][q] = fmaf(g, tmp[1][q], acc[1][q]);
      }
    }
    if (oka) store_vec<TOut, V>(out + (size_t)t * d + ca, acc[0]);
    if (okb) store_vec<TOut, V>(out + (size_t)t * d + cb, acc[1]);
  }
}

template <typename TIn, typename TOut>
cudaError_t run(const void* u, const void* y, const float* gate, const int32_t* inv_row, int T,
                int d, int K_r, int N_s, void* out, cudaStream_t st) {
  constexpr int kCols = 64 * Vec<TIn>::N;              // columns of one pass of a warp
  const int passes = (d + kCols - 1) / kCols;
  const int chunks = std::min(passes, std::max(1, kTargetWarps / T));
  const int ppc = (passes + chunks - 1) / chunks;
  const dim3 grid((T + 7) / 8, (passes + ppc - 1) / ppc);
  const cudaError_t err = launch_pdl(combine_kernel<TIn, TOut>, grid, dim3(256), 0, st, 0, (const TIn*)u,
                                     (const TIn*)y, gate, inv_row, T, d, K_r, N_s, ppc, (TOut*)out,
                                     dev_error_ptr());
  return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const void* u, const void* y, moe_dtype dt, const float* gate,
                           const int32_t* inv_row, int T, int d, int K_r, int N_s,
                           void* out, moe_dtype out_dt, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (dt == MOE_F32)
    return out_dt == MOE_F32 ? run<float, float>(u, y, gate, inv_row, T, d, K_r, N_s, out, st)
                             : run<float, __nv_bfloat16>(u, y, gate, inv_row, T, d, K_r, N_s, out, st);
  return out_dt == MOE_F32
             ? run<__nv_bfloat16, float>(u, y, gate, inv_row, T, d, K_r, N_s, out, st)
             : run<__nv_bfloat16, __nv_bfloat16>(u, y, gate, inv_row, T, d, K_r, N_s, out, st);
}

}  // namespace moe
