// Affinity GEMM z = u e^T for bf16 layers on the sm_103a tensor cores
// (DeepSeek-V3 Technical Report reading guide, Method §2: s_{i,t} = Sigmoid(u_t^T e_i);
// this kernel forms u_t^T e_i, router_select_kernel the rest).
//
// CTA (m, s) computes the fp32 partial product of 128 tokens with all N_r centroids
// over the s-th slice of the d dimension (split-K, so that a few thousand tokens still
// fill the SMs): warp 0 streams u [128 x 64] and e [N_r x 64] tiles by TMA into a
// 4-stage ring, warp 1 issues M=128, N=N_r MMAs into TMEM, warps 2..5 write the
// accumulator rows to z_part[s] (one token row per thread).
#include <algorithm>

#include "launch.h"
#include "route_select.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moe {

namespace {

constexpr int BM = 128, BK = 64, STAGES = 4, THREADS = 192;
constexpr int A_BYTES = BM * BK * 2;

struct RCtrl {
  uint64_t full[STAGES], empty[STAGES], tfull, fin;
  uint32_t tmem_base;
  int abort_flag;
};

__global__ void __launch_bounds__(THREADS, 1)
    router_gemm_tc_kernel(const __grid_constant__ CUtensorMap mU,
                          const __grid_constant__ CUtensorMap mE, int d, int n_pad,
                          uint32_t tmem_cols, int T, int N_r, int kb_per_split,
                          float* __restrict__ z_part, int32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_off = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_off & 1023u)) & 1023u);
  const int sbytes = A_BYTES + n_pad * BK * 2;
  RCtrl& C = *reinterpret_cast<RCtrl*>(base + STAGES * sbytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * BM;
  const int nk = (d + BK - 1) / BK;
  const int kb0 = blockIdx.y * kb_per_split;
  const int nkb = min(nk, kb0 + kb_per_split) - kb0;   // >= 1 by construction

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      tc::mbar_init(&C.full[i], 1);
      tc::mbar_init(&C.empty[i], 1);
    }
    tc::mbar_init(&C.tfull, 1);
    tc::mbar_init(&C.fin, 1);
    C.abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&C.tmem_base, tmem_cols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = C.tmem_base;
  volatile int* abort_flag = &C.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      for (; it < nkb; ++it) {
        const int st = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!tc::mbar_wait(&C.empty[st], ph ^ 1, abort_flag, err)) break;
        uint8_t* sa = base + st * sbytes;
        tc::mbar_arrive_expect_tx(&C.full[st], (uint32_t)sbytes);
        tc::tma_load_2d(sa, &mU, &C.full[st], (kb0 + it) * BK, t0);
        tc::tma_load_2d(sa + A_BYTES, &mE, &C.full[st], (kb0 + it) * BK, 0);
      }
      if (*abort_flag)
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          tc::mbar_drain(&C.full[j % STAGES], (j / STAGES) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(BM, n_pad);
      bool ok = true;
      for (int it = 0; it < nkb; ++it) {
        const int st = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!tc::mbar_wait(&C.full[st], ph, abort_flag, err)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t a0 = tc::smem_u32(base + st * sbytes);
        const uint64_t ad = tc::sdesc_sw128(a0), bd = tc::sdesc_sw128(a0 + A_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc::mma_bf16(tmem_base, ad + 2 * kk, bd + 2 * kk, idesc, (it | kk) != 0);
        tc::mma_commit(&C.empty[st]);
      }
      if (ok) tc::mma_commit(&C.tfull);
      tc::mma_commit(&C.fin);
      tc::mbar_drain(&C.fin, 0);
    }
  } else {
    const int q = warp & 3;   // TMEM lane quarter of this warp
    const bool got = tc::mbar_wait(&C.tfull, 0, abort_flag, err);
    if (__all_sync(0xffffffffu, got)) {
      tc::fence_after_sync();
      const int t = t0 + q * 32 + lane;
      float* zrow = z_part + ((size_t)blockIdx.y * T + t) * N_r;
      for (int c = 0; c < n_pad / 32; ++c) {
        uint32_t z[32];
        tc::tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + c * 32, z);
        tc::tmem_ld_wait();
        if (t < T) {
          float4* dst = reinterpret_cast<float4*>(zrow + c * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(z[4 * v]), __uint_as_float(z[4 * v + 1]),
                                 __uint_as_float(z[4 * v + 2]), __uint_as_float(z[4 * v + 3]));
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, tmem_cols);
  }
}

}  // namespace

int router_tc_splits(int T, int d) {
  const int nk = (d + BK - 1) / BK;
  const int m_tiles = std::max(1, (T + BM - 1) / BM);
  const int S = std::min({std::max(1, nk / 2), std::max(1, device_sm_count() / m_tiles), 16});
  const int per = (nk + S - 1) / S;
  return (nk + per - 1) / per;   // every split gets at least one k-block
}

cudaError_t launch_router_gemm_tc(const void* u, const void* e, int T, int d, int N_r,
                                  float* z_part, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int n_pad = (N_r + 31) / 32 * 32;
  uint32_t cols = 32;
  while (cols < (uint32_t)n_pad) cols <<= 1;
  CUtensorMap mU, mE;
  const uint64_t rb = (uint64_t)d * 2;
  if (!make_tmap_2d(&mU, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, u, d, T, rb, BK, BM) ||
      !make_tmap_2d(&mE, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, e, d, N_r, rb, BK, n_pad))
    return cudaErrorInvalidValue;
  const size_t smem = (size_t)STAGES * (A_BYTES + n_pad * BK * 2) + sizeof(RCtrl) + 1024;
  cudaError_t err = cudaFuncSetAttribute(router_gemm_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int nk = (d + BK - 1) / BK;
  const int S = router_tc_splits(T, d);
  const int per = (nk + S - 1) / S;
  const dim3 grid((T + BM - 1) / BM, S);
  router_gemm_tc_kernel<<<grid, THREADS, smem, st>>>(mU, mE, d, n_pad, cols, T, N_r, per, z_part,
                                                     dev_error_ptr());
  return cudaGetLastError();
}

}  // namespace moe
