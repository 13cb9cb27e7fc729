// E4M3 quantisation with fp32 block scales: activations per 1x128 tile, weights per
// 128x128 block (DeepSeek-V3 Technical Report reading guide, Key ideas, FP8
// bullet; pwwt.cn notes §三).  scale = amax / 448 (IEEE fp32 division), 1 for an
// all-zero block; code = E4M3(x / scale), round to nearest even, saturating.
#include <cuda_fp8.h>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

__device__ __forceinline__ float block_scale(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
}

__device__ __forceinline__ uint8_t to_e4m3(float x, float scale, float inv) {
  return (uint8_t)__nv_cvt_float_to_fp8(div_by_scale(x, scale, inv), __NV_SATFINITE, __NV_E4M3);
}

// One warp per (row, 128-column tile); each lane owns 4 consecutive values.
template <typename TIn>
__global__ void __launch_bounds__(256) quant_1x128_kernel(const TIn* __restrict__ x,
                                                          long long rows, long long cols,
                                                          uint8_t* __restrict__ q,
                                                          float* __restrict__ scale) {
  pdl_release();
  pdl_wait();
  const long long tiles_per_row = cols / 128;
  const long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= rows * tiles_per_row) return;
  const long long r = w / tiles_per_row, tc = w % tiles_per_row;
  const TIn* src = x + r * cols + tc * 128 + lane * 4;
  float v[4];
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[k] = to_f32(src[k]);
    amax = fmaxf(amax, fabsf(v[k]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sc = block_scale(amax);
  const float inv = __frcp_rn(sc);
  uint32_t packed = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) packed |= (uint32_t)to_e4m3(v[k], sc, inv) << (8 * k);
  *reinterpret_cast<uint32_t*>(q + r * cols + tc * 128 + lane * 4) = packed;
  if (lane == 0) scale[w] = sc;
}

// One block per 128x128 block.
template <typename TIn>
__global__ void __launch_bounds__(256) quant_128x128_kernel(const TIn* __restrict__ x,
                                                            long long cols,
                                                            uint8_t* __restrict__ q,
                                                            float* __restrict__ scale) {
  __shared__ float red[8];
  pdl_release();
  pdl_wait();
  const long long br = blockIdx.y, bc = blockIdx.x;
  const TIn* base = x + br * 128 * cols + bc * 128;
  float amax = 0.f;
  for (int e = threadIdx.x; e < 128 * 128; e += blockDim.x) {
    const int r = e >> 7, c = e & 127;
    amax = fmaxf(amax, fabsf(to_f32(base[(long long)r * cols + c])));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  float m = 0.f;
  for (int k = 0; k < (int)(blockDim.x >> 5); ++k) m = fmaxf(m, red[k]);
  const float sc = block_scale(m);
  const float inv = __frcp_rn(sc);
  uint8_t* qb = q + br * 128 * cols + bc * 128;
  for (int e = threadIdx.x; e < 128 * 128; e += blockDim.x) {
    const int r = e >> 7, c = e & 127;
    qb[(long long)r * cols + c] = to_e4m3(to_f32(base[(long long)r * cols + c]), sc, inv);
  }
  if (threadIdx.x == 0) scale[br * gridDim.x + bc] = sc;
}

}  // namespace

cudaError_t launch_quantize_e4m3(const void* x, moe_dtype x_dt, int64_t rows, int64_t cols,
                                 int block_rows, uint8_t* q, float* scale, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  cudaError_t err;
  if (block_rows == 1) {
    const long long warps = rows * (cols / 128);
    const dim3 blocks((unsigned)((warps + 7) / 8));
    if (x_dt == MOE_F32)
      err = launch_pdl(quant_1x128_kernel<float>, blocks, dim3(256), 0, st, 0, (const float*)x,
                       (long long)rows, (long long)cols, q, scale);
    else
      err = launch_pdl(quant_1x128_kernel<__nv_bfloat16>, blocks, dim3(256), 0, st, 0,
                       (const __nv_bfloat16*)x, (long long)rows, (long long)cols, q, scale);
  } else {
    const dim3 grid((unsigned)(cols / 128), (unsigned)(rows / 128));
    if (x_dt == MOE_F32)
      err = launch_pdl(quant_128x128_kernel<float>, grid, dim3(256), 0, st, 0, (const float*)x,
                       (long long)cols, q, scale);
    else
      err = launch_pdl(quant_128x128_kernel<__nv_bfloat16>, grid, dim3(256), 0, st, 0,
                       (const __nv_bfloat16*)x, (long long)cols, q, scale);
  }
  return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace moe
