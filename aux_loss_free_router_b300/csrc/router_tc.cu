// Affinity GEMM z = u e^T for bf16 layers on the sm_103a tensor cores
// (DeepSeek-V3 Technical Report reading guide, Method §2: s_{i,t} = Sigmoid(u_t^T e_i);
// this kernel forms u_t^T e_i, router_select_kernel the rest).
//
// Split-K CTA-pair GEMM; see router_gemm_tc_kernel.
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

// A CTA pair (cluster of two) computes the fp32 partial product of 256 tokens with all
// N_r centroids over the s-th slice of d (split-K, so that a few thousand tokens still
// fill the SMs), as M=256 pair MMAs: each CTA loads its 128 token rows and half of the
// centroid rows per K step (16 + N_r/4 KB), and its TMEM receives its 128 tokens' rows.
// Warp 0 streams the tiles by TMA into a 4-stage ring (completion counted on the even
// CTA's barrier), one thread of the even CTA issues the MMAs, warps 2..5 of both CTAs
// write the accumulator rows to z_part[s] (one token row per thread).
__global__ void __launch_bounds__(THREADS, 1)
    router_gemm_tc_kernel(const __grid_constant__ CUtensorMap mU,
                          const __grid_constant__ CUtensorMap mE, int d, int n_r,
                          uint32_t tmem_cols, int T, int kb_per_split,
                          float* __restrict__ z_part, int32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  pdl_release();
  pdl_wait();
  const uint32_t raw_off = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_off & 1023u)) & 1023u);
  const int half = n_r / 2;                       // centroid rows per CTA
  const int sbytes = A_BYTES + half * BK * 2;
  RCtrl& C = *reinterpret_cast<RCtrl*>(base + STAGES * sbytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_rank();
  const bool leader = rank == 0;
  const int t0 = (blockIdx.x >> 1) * (2 * BM) + (int)rank * BM;   // this CTA's tokens
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
    tc::tmem_alloc_pair(&C.tmem_base, tmem_cols);
    tc::tmem_relinquish_pair();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  tc::cluster_sync();   // both CTAs' barriers exist before any remote copy
  const uint32_t tmem_base = C.tmem_base;
  volatile int* abort_flag = &C.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      for (int it = 0; it < nkb; ++it) {
        const int st = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!tc::mbar_wait(&C.empty[st], ph ^ 1, abort_flag, err)) break;
        const uint32_t bar = tc::cluster_addr(&C.full[st], 0);
        if (leader) tc::mbar_arrive_expect_tx(&C.full[st], (uint32_t)(2 * sbytes));
        uint8_t* sa = base + st * sbytes;
        tc::tma_load_2d_pair(sa, &mU, bar, (kb0 + it) * BK, t0);
        tc::tma_load_2d_pair(sa + A_BYTES, &mE, bar, (kb0 + it) * BK, (int)rank * half);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      const uint32_t idesc = tc::idesc_bf16(2 * BM, n_r);
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
          tc::mma_bf16_pair(tmem_base, ad + 2 * kk, bd + 2 * kk, idesc, (it | kk) != 0);
        tc::mma_commit_pair(&C.empty[st]);
      }
      if (ok) tc::mma_commit_pair(&C.tfull);
      tc::mma_commit_pair(&C.fin);
    }
  } else {
    const int q = warp & 3;   // TMEM lane quarter of this warp
    const bool got = tc::mbar_wait(&C.tfull, 0, abort_flag, err);
    if (__all_sync(0xffffffffu, got)) {
      tc::fence_after_sync();
      const int t = t0 + q * 32 + lane;
      float* zrow = z_part + ((size_t)blockIdx.y * T + t) * n_r;
      for (int c = 0; c < n_r / 32; ++c) {
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
  if (*abort_flag && warp == 0 && lane == 0) {
    // copies this CTA issued report to the even CTA's barriers: give them time to land
    const uint64_t w0 = global_ns();
    while (global_ns() - w0 < 10000000ull) {
    }
  }
  if (warp == 1 && lane == 0) tc::mbar_drain(&C.fin, 0);
  __syncthreads();
  tc::cluster_sync();   // neither CTA leaves while its peer may still touch it
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem_base, tmem_cols);
  }
}

int pair_count(int T) { return std::max(1, (T + 2 * BM - 1) / (2 * BM)); }

}  // namespace

int router_tc_splits(int T, int d) {
  const int nk = (d + BK - 1) / BK;
  const int S = std::min({std::max(1, nk / 2), std::max(1, (device_sm_count() / 2) / pair_count(T)), 16});
  const int per = (nk + S - 1) / S;
  return (nk + per - 1) / per;   // every split gets at least one k-block
}

cudaError_t launch_router_gemm_tc(const void* u, const void* e, int T, int d, int N_r,
                                  float* z_part, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  // N_r is a multiple of 32 here: half of it (a CTA's centroid rows) is a multiple of 16
  uint32_t cols = 32;
  while (cols < (uint32_t)N_r) cols <<= 1;
  CUtensorMap mU, mE;
  const uint64_t rb = (uint64_t)d * 2;
  if (!make_tmap_2d(&mU, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, u, d, T, rb, BK, BM) ||
      !make_tmap_2d(&mE, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, e, d, N_r, rb, BK, N_r / 2))
    return cudaErrorInvalidValue;
  const size_t smem = (size_t)STAGES * (A_BYTES + (N_r / 2) * BK * 2) + sizeof(RCtrl) + 1024;
  cudaError_t err = cudaFuncSetAttribute(router_gemm_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int nk = (d + BK - 1) / BK;
  const int S = router_tc_splits(T, d);
  const int per = (nk + S - 1) / S;
  err = launch_pdl(router_gemm_tc_kernel, dim3(2 * pair_count(T), S), dim3(THREADS), smem, st, 2, mU, mE,
                   d, N_r, cols, T, per, z_part, dev_error_ptr());
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace moe
