// Shared device helpers: error word, bounded waits, warp reductions, dtype loads.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Kernels that can time out receive the device address of the library's error word
// (MOE_OK or MOE_ERR_TIMEOUT) and raise it with this.
__device__ __forceinline__ void record_error(int32_t* err, int32_t code) {
  if (err) atomicMax(err, code);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Every spin in this library gives up after this long, records MOE_ERR_TIMEOUT and
// lets the kernel return.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// (key, index) is better than (key', index') when key > key', or equal keys and a
// lower index.  A total order on finite keys, so every lane of a butterfly reduction
// ends with the same winner.
__device__ __forceinline__ bool better(float k, int i, float k2, int i2) {
  return k > k2 || (k == k2 && i < i2);
}

struct KeyIdxVal {
  float key;
  int idx;
  float val;
};

__device__ __forceinline__ KeyIdxVal warp_argmax(KeyIdxVal a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float k2 = __shfl_xor_sync(0xffffffffu, a.key, o);
    int i2 = __shfl_xor_sync(0xffffffffu, a.idx, o);
    float v2 = __shfl_xor_sync(0xffffffffu, a.val, o);
    if (better(k2, i2, a.key, a.idx)) { a.key = k2; a.idx = i2; a.val = v2; }
  }
  return a;
}

inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// x / scale for E4M3 quantisation from inv = RN(1 / scale), taken once per tile: q =
// RN(x inv), the remainder r = x - q scale exact by fma, then RN(q + r inv) (Markstein's
// correction step).  It is meant only for a quotient that is then rounded to E4M3: over
// 4e9 operand pairs of the quantisers' shape (|x| <= amax, scale = amax / 448, amax from
// 2^-63 to 2^64) the E4M3 codes of this quotient and of the IEEE one (__fdiv_rn) were
// identical (the fp32 quotients themselves can differ where x/scale is far below the
// smallest E4M3 step), and the quantiser tests compare the codes with the oracle's fp32
// division.
__device__ __forceinline__ float div_by_scale(float x, float scale, float inv) {
  const float q = __fmul_rn(x, inv);
  const float r = __fmaf_rn(-q, scale, x);
  return __fmaf_rn(r, inv, q);
}

// Programmatic dependent launch.  The forward kernels are launched with launch_pdl, so
// the GPU may schedule a kernel while the one before it in the stream still runs.  Each
// such kernel calls pdl_wait() before its first access to global memory that another
// kernel writes, and before allocating tensor memory: the wait returns once the previous
// kernel has completed and its writes are visible (a kernel launched without the
// attribute, or after a non-kernel node, returns at once).  pdl_release() lets the next
// kernel in the stream be scheduled; it is issued first thing, and the next kernel's
// blocks then wait in their own pdl_wait().
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kernel` with the programmatic-serialization attribute (and a cluster shape when
// cluster_x > 1; kernels with compiled-in cluster dimensions pass 0).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       unsigned cluster_x, Args... args) {
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace moe
