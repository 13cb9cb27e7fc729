// Pieces shared by the two grouped expert GEMMs (tc_gate_up.cu, tc_down.cu): the
// per-launch tile counters, the CTA-pair launch, and the epilogue helpers.
#pragma once

#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "ffn_sched.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace moe {
namespace ffn_tc {

constexpr int BK = 64;           // K per step: one 128-byte swizzle row of bf16
constexpr int SMALL_ROWS = 32;   // token box of an MMA with <= 64 tokens (<= 32 rows per CTA)
constexpr int THREADS = 192;     // producer warp, MMA warp, four epilogue warps
constexpr int TQ = 4;            // tile-index ring between the roles of a CTA pair

struct TcArgs {
  FfnShape s;
  const int32_t* expert_offset;
  __nv_bfloat16* out;
  int32_t* err;
  int* tile_ctr;     // [claimed, done], zero at launch; pairs claim tiles in order
  // gate/up only, optional: the pre-activations a = x W_gate^T and c = x W_up^T in bf16,
  // in the same row space and layout as h (kept for the backward pass)
  __nv_bfloat16* save_a = nullptr;
  __nv_bfloat16* save_c = nullptr;
  // gate/up reading the routed token rows straight from u: u [T, d] and perm_token
  // [T*K_r] (the token of each row of the routed row space)
  const __nv_bfloat16* u = nullptr;
  const int32_t* perm = nullptr;
};

// silu(g) * u = g * u / (1 + e^-g), with the fast reciprocal division (the result is
// rounded to bf16).
__device__ __forceinline__ float swiglu(float g, float u) {
  return __fdividef(g * u, 1.f + __expf(-g));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 16 tokens x 32 features of one warp (lane = feature, v[j] = token j) to token rows:
// through the warp's scratch, then 16-byte pieces of 8 features.
__device__ __forceinline__ void store_transposed(__nv_bfloat16* scr, const float (&v)[16], int lane,
                                                 __nv_bfloat16* out, size_t row0, int j0, int n_tok,
                                                 int f0, int N) {
#pragma unroll
  for (int j = 0; j < 16; ++j) scr[j * 32 + lane] = __float2bfloat16_rn(v[j]);
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int item = i * 32 + lane;      // 16 tokens x 4 pieces of 8 features
    const int tok = item >> 2, piece = item & 3;
    const int f = f0 + piece * 8;
    if (j0 + tok < n_tok && f < N) {
      const uint4 val = *reinterpret_cast<const uint4*>(scr + tok * 32 + piece * 8);
      *reinterpret_cast<uint4*>(out + (row0 + j0 + tok) * N + f) = val;
    }
  }
  __syncwarp();
}

// One of the library's per-launch tile counters on the current device (defined in
// tc_down.cu): slots are taken round-robin from a built-in array of 64, so that up to
// 64 launches in flight at once count separately.
int* tile_counter(cudaError_t* err);

// Called once by every CTA of a launch, after its producer's last claim: the last CTA
// to get here puts the slot back to zero for the next launch that takes it (in stream
// order that launch reads the counter only after this one has completed).
__device__ __forceinline__ void release_tile_counter(int* ctr) {
  __threadfence();
  if (atomicAdd(ctr + 1, 1) == (int)(gridDim.x * gridDim.y * gridDim.z) - 1) {
    __threadfence();
    atomicExch(ctr, 0);
    atomicExch(ctr + 1, 0);
  }
}

// Launch `kernel` as persistent CTA pairs (clusters of two): as many pairs as fit on
// the device at once (cached per device in `fit_cache`), at most `tiles_ub`, with the
// programmatic-serialization attribute.
template <typename Kernel>
cudaError_t launch_pairs(Kernel kernel, int* fit_cache, std::mutex& mu, size_t smem,
                         long long tiles_ub, const CUtensorMap* m, TcArgs a, cudaStream_t st,
                         int threads = THREADS) {
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (device_sm_count() / 2));
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int fit;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (fit_cache[dev] == 0) {
      int n = 0;
      if ((err = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg)) != cudaSuccess) return err;
      fit_cache[dev] = n;
    }
    fit = fit_cache[dev];
  }
  if (fit < 1) return cudaErrorInvalidConfiguration;
  cfg.gridDim = dim3(2 * (int)std::min<long long>(fit, std::max<long long>(1, tiles_ub)));
  a.tile_ctr = tile_counter(&err);
  if (a.tile_ctr == nullptr) return err;
  err = launch_pdl(kernel, cfg.gridDim, cfg.blockDim, smem, st, 2, m[0], m[1], m[2], m[3], m[4], m[5], m[6],
                   m[7], a);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace ffn_tc
}  // namespace moe
