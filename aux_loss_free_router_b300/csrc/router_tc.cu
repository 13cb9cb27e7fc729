// Router for bf16 layers: the T x d x N_r affinity GEMM on the sm_103a tensor cores,
// fused with sigmoid, the bias add, the group-limited biased Top-K_r and the gate
// normalisation (DeepSeek-V3 Technical Report reading guide, Method §2: s, g' and g).
//
// One CTA per 128-token tile.  warp 0 streams u [128 x 64] and e [N_r x 64] tiles by
// TMA into a 4-stage ring; warp 1 issues M=128, N=N_r MMAs into TMEM (fp32);
// warps 2..5 turn the accumulator rows into s = sigmoid(z) in shared memory (reusing
// the ring); then all six warps take the routing decision of one token each at a
// time with route_token().
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
  float b[kMaxExperts];
};

inline int stage_bytes(int n_pad) { return A_BYTES + n_pad * BK * 2; }

__global__ void __launch_bounds__(THREADS, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap mU, const __grid_constant__ CUtensorMap mE,
                     const float* __restrict__ b, int d, int n_pad, uint32_t tmem_cols, RouteOut p,
                     int32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_off = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_off & 1023u)) & 1023u);
  const int sbytes = A_BYTES + n_pad * BK * 2;
  RCtrl& C = *reinterpret_cast<RCtrl*>(base + STAGES * sbytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * BM;
  const int nk = (d + BK - 1) / BK;
  const int N_r = p.N_r;

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
  for (int i = threadIdx.x; i < N_r; i += blockDim.x) C.b[i] = b[i];
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
      for (; it < nk; ++it) {
        const int st = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!tc::mbar_wait(&C.empty[st], ph ^ 1, abort_flag, err)) break;
        uint8_t* sa = base + st * sbytes;
        tc::mbar_arrive_expect_tx(&C.full[st], (uint32_t)sbytes);
        tc::tma_load_2d(sa, &mU, &C.full[st], it * BK, t0);
        tc::tma_load_2d(sa + A_BYTES, &mE, &C.full[st], it * BK, 0);
      }
      if (*abort_flag)
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          tc::mbar_drain(&C.full[j % STAGES], (j / STAGES) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(BM, n_pad);
      bool ok = true;
      for (int it = 0; it < nk; ++it) {
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
    // accumulator rows -> s = sigmoid(z) in shared memory, row stride N_r + 1 floats
    const int q = warp & 3;
    const bool got = tc::mbar_wait(&C.tfull, 0, abort_flag, err);
    if (__all_sync(0xffffffffu, got)) {
      tc::fence_after_sync();
      float* s_tile = reinterpret_cast<float*>(base);
      const int r = q * 32 + lane;
      for (int c = 0; c < n_pad / 32; ++c) {
        uint32_t z[32];
        tc::tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + c * 32, z);
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int i = c * 32 + j;
          if (i < N_r) s_tile[r * (N_r + 1) + i] = sigmoid_f32(__uint_as_float(z[j]));
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
  if (*abort_flag) return;
  const float* s_tile = reinterpret_cast<const float*>(base);
  for (int r = warp; r < BM; r += THREADS / 32) {
    const int t = t0 + r;
    if (t < p.T) route_token(s_tile + r * (N_r + 1), C.b, t, p);
  }
}

}  // namespace

cudaError_t launch_router_tc(const void* u, const void* e, const float* b, int d,
                             const RouteOut& p, cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  const int n_pad = (p.N_r + 31) / 32 * 32;
  uint32_t cols = 32;
  while (cols < (uint32_t)n_pad) cols <<= 1;
  CUtensorMap mU, mE;
  const uint64_t rb = (uint64_t)d * 2;
  if (!make_tmap_2d(&mU, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, u, d, p.T, rb, BK, BM) ||
      !make_tmap_2d(&mE, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, e, d, p.N_r, rb, BK, n_pad))
    return cudaErrorInvalidValue;
  const size_t ring = (size_t)STAGES * stage_bytes(n_pad);
  const size_t s_tile = (size_t)BM * (p.N_r + 1) * sizeof(float);
  const size_t smem = std::max(ring, s_tile) + sizeof(RCtrl) + 1024;
  cudaError_t err = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  const int grid = (p.T + BM - 1) / BM;
  router_tc_kernel<<<grid, THREADS, smem, st>>>(mU, mE, b, d, n_pad, cols, p, dev_error_ptr());
  return cudaGetLastError();
}

}  // namespace moe
