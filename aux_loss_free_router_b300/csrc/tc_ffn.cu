// Grouped SwiGLU expert GEMMs on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One persistent CTA per SM walks the tiles of the segment schedule
// (ffn_sched.cuh).  Warp roles:
//   warp 0      TMA producer: A tile [128 rows x 64 K] and B tile [256 rows x 64 K]
//               per stage, 128-byte swizzled, into a 4-stage shared-memory ring.
//   warp 1      allocates 512 TMEM columns and issues the MMAs (one thread):
//               M=128, N=256, K=16 per instruction into one of two 256-column fp32
//               accumulators, so the epilogue of tile i overlaps the MMAs of i+1.
//   warps 2..5  epilogue: TMEM -> registers -> bf16 -> global.
//
// gate/up (MODE 0): the B tile stacks 128 rows of W_gate over the same 128 rows of
//   W_up, so one N=256 MMA produces both halves; the epilogue forms
//   silu(gate) * up for a [128 x 128] tile of h.
// down (MODE 1): B is 256 rows of W_down; the epilogue writes a [128 x 256] tile
//   of y.
// Rows of an A tile past the end of its segment belong to the next segment (or are
// zero-filled past the tensor end); they are computed and not stored.
#include <algorithm>

#include "common.cuh"
#include "ffn_sched.cuh"
#include "launch.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moe {

namespace {

constexpr int BM = 128, BK = 64, BN = 256, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int THREADS = 192;

struct Ctrl {
  uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], fin;
  uint32_t tmem_base;
  int abort_flag;
  SegTable tab;
};

constexpr size_t kSmemBytes = (size_t)STAGES * STAGE_BYTES + sizeof(Ctrl) + 1024;

struct TcArgs {
  FfnShape s;
  const int32_t* expert_offset;
  __nv_bfloat16* out;
  int32_t* err;
};

__device__ __forceinline__ float silu(float z) { return z / (1.f + __expf(-z)); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const float (&v)[32], int valid) {
  if (valid >= 32) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      d4[q] = make_uint4(pack_bf16(v[8 * q + 0], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                         pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < valid) dst[j] = __float2bfloat16_rn(v[j]);
  }
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    tc_ffn_kernel(const __grid_constant__ CUtensorMap mA_r, const __grid_constant__ CUtensorMap mA_s,
                  const __grid_constant__ CUtensorMap mB0_r, const __grid_constant__ CUtensorMap mB1_r,
                  const __grid_constant__ CUtensorMap mB0_s, const __grid_constant__ CUtensorMap mB1_s,
                  TcArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_off = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_off & 1023u)) & 1023u);
  Ctrl& C = *reinterpret_cast<Ctrl*>(base + STAGES * STAGE_BYTES);

  const FfnShape s = args.s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = MODE == 0 ? s.d : s.I;
  const int N = MODE == 0 ? s.I : s.d;
  constexpr int BNO = MODE == 0 ? BN / 2 : BN;   // output columns per tile
  const int n_tiles_n = (N + BNO - 1) / BNO;
  const int nk = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      tc::mbar_init(&C.full[i], 1);
      tc::mbar_init(&C.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&C.tfull[i], 1);
      tc::mbar_init(&C.tempty[i], 128);
    }
    tc::mbar_init(&C.fin, 1);
    C.abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&mA_r);
    tc::tma_prefetch_desc(&mB0_r);
  }
  if (warp == 1) {
    tc::tmem_alloc(&C.tmem_base, TMEM_COLS);
    tc::tmem_relinquish();
  }
  build_seg_table(C.tab, args.expert_offset, s.T, s.K_r, s.N_r, s.N_s, BM, n_tiles_n);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = C.tmem_base;
  const int total = C.tab.total;
  volatile int* abort_flag = &C.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer --
      int it = 0;
      for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
        const TileCoord tcd = decode_tile(C.tab, tile, n_tiles_n);
        const bool shared = tcd.seg >= s.N_r;
        const int e = shared ? tcd.seg - s.N_r : tcd.seg;
        const CUtensorMap* mA = (MODE == 0 && shared) ? &mA_s : &mA_r;
        const int a_row = (MODE == 0 ? (shared ? 0 : tcd.row0) : tcd.out_row0) + tcd.m * BM;
        const CUtensorMap* mB0 = shared ? &mB0_s : &mB0_r;
        const CUtensorMap* mB1 = shared ? &mB1_s : &mB1_r;
        const int b_row = e * N + tcd.n * BNO;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!tc::mbar_wait(&C.empty[st], ph ^ 1, abort_flag, args.err)) { ok = false; break; }
          uint8_t* sa = base + st * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          tc::mbar_arrive_expect_tx(&C.full[st], STAGE_BYTES);
          tc::tma_load_2d(sa, mA, &C.full[st], kb * BK, a_row);
          if (MODE == 0) {
            tc::tma_load_2d(sb, mB0, &C.full[st], kb * BK, b_row);
            tc::tma_load_2d(sb + B_BYTES / 2, mB1, &C.full[st], kb * BK, b_row);
          } else {
            tc::tma_load_2d(sb, mB0, &C.full[st], kb * BK, b_row);
          }
        }
        if (!ok) break;
      }
      if (*abort_flag) {
        // let the copies already issued land before the CTA exits
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          tc::mbar_drain(&C.full[j % STAGES], (j / STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer --
      constexpr uint32_t idesc = tc::idesc_bf16(BM, BN);
      int it = 0, tcount = 0;
      for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x, ++tcount) {
        const int acc = tcount & 1;
        const uint32_t aph = (tcount >> 1) & 1;
        if (!tc::mbar_wait(&C.tempty[acc], aph ^ 1, abort_flag, args.err)) break;
        tc::fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!tc::mbar_wait(&C.full[st], ph, abort_flag, args.err)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t a0 = tc::smem_u32(base + st * STAGE_BYTES);
          const uint64_t ad = tc::sdesc_sw128(a0), bd = tc::sdesc_sw128(a0 + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_bf16(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
          tc::mma_commit(&C.empty[st]);
        }
        if (!ok) break;
        tc::mma_commit(&C.tfull[acc]);
      }
      // every MMA issued by this thread has finished once `fin` flips
      tc::mma_commit(&C.fin);
      tc::mbar_drain(&C.fin, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int q = warp & 3;   // TMEM lane quarter this warp can access
    int tcount = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++tcount) {
      // warp-uniform decisions: the TMEM loads below are warp-collective
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const TileCoord tcd = decode_tile(C.tab, tile, n_tiles_n);
      const int acc = tcount & 1;
      const uint32_t aph = (tcount >> 1) & 1;
      const bool got = tc::mbar_wait(&C.tfull[acc], aph, abort_flag, args.err);
      if (!__all_sync(0xffffffffu, got)) break;
      tc::fence_after_sync();
      const int row_local = tcd.m * BM + q * 32 + lane;
      const bool row_ok = row_local < tcd.rows;
      __nv_bfloat16* out_row = args.out + (size_t)(tcd.out_row0 + row_local) * N;
      const uint32_t t_base = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      if (MODE == 0) {
#pragma unroll 1
        for (int c = 0; c < BNO / 32; ++c) {
          uint32_t g[32], u[32];
          tc::tmem_ld32(t_base + c * 32, g);
          tc::tmem_ld32(t_base + BNO + c * 32, u);
          tc::tmem_ld_wait();
          const int col0 = tcd.n * BNO + c * 32;
          if (row_ok && col0 < N) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = silu(__uint_as_float(g[j])) * __uint_as_float(u[j]);
            store_row32(out_row + col0, v, N - col0);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BNO / 32; ++c) {
          uint32_t y[32];
          tc::tmem_ld32(t_base + c * 32, y);
          tc::tmem_ld_wait();
          const int col0 = tcd.n * BNO + c * 32;
          if (row_ok && col0 < N) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(y[j]);
            store_row32(out_row + col0, v, N - col0);
          }
        }
      }
      tc::fence_before_sync();
      tc::mbar_arrive(&C.tempty[acc]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int MODE>
cudaError_t launch(const FfnShape& s, const CUtensorMap* maps, const int32_t* off, void* out,
                   cudaStream_t st) {
  const int N = MODE == 0 ? s.I : s.d;
  const int bno = MODE == 0 ? BN / 2 : BN;
  const long long m_ub = (long long)s.T * s.K_r / BM + s.N_r + (long long)s.N_s * ((s.T + BM - 1) / BM);
  const long long tiles_ub = m_ub * ((N + bno - 1) / bno);
  const int grid = (int)std::min<long long>(device_sm_count(), std::max<long long>(1, tiles_ub));
  auto k = tc_ffn_kernel<MODE>;
  cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  TcArgs a{s, off, static_cast<__nv_bfloat16*>(out), dev_error_ptr()};
  k<<<grid, THREADS, kSmemBytes, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], a);
  return cudaGetLastError();
}

constexpr CUtensorMapDataType kBF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;

}  // namespace

cudaError_t launch_ffn_up_tc(const FfnShape& s, const void* x_perm, const void* u,
                             const int32_t* expert_offset, const moe_expert_weights* w, void* h,
                             cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  CUtensorMap m[6];
  const uint64_t rb = (uint64_t)s.d * 2;
  const uint64_t routed = (uint64_t)s.T * s.K_r;
  bool ok = make_tmap_2d(&m[0], kBF16, x_perm, s.d, routed, rb, BK, BM) &&
            make_tmap_2d(&m[1], kBF16, u, s.d, s.T, rb, BK, BM) &&
            make_tmap_2d(&m[2], kBF16, w->gate, s.d, (uint64_t)s.N_r * s.I, rb, BK, BN / 2) &&
            make_tmap_2d(&m[3], kBF16, w->up, s.d, (uint64_t)s.N_r * s.I, rb, BK, BN / 2);
  if (ok && s.N_s > 0) {
    ok = make_tmap_2d(&m[4], kBF16, w->s_gate, s.d, (uint64_t)s.N_s * s.I, rb, BK, BN / 2) &&
         make_tmap_2d(&m[5], kBF16, w->s_up, s.d, (uint64_t)s.N_s * s.I, rb, BK, BN / 2);
  } else {
    m[4] = m[2];
    m[5] = m[3];
  }
  if (!ok) return cudaErrorInvalidValue;
  return launch<0>(s, m, expert_offset, h, st);
}

cudaError_t launch_ffn_down_tc(const FfnShape& s, const void* h, const int32_t* expert_offset,
                               const moe_expert_weights* w, void* y, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  CUtensorMap m[6];
  const uint64_t rb = (uint64_t)s.I * 2;
  const uint64_t rows = (uint64_t)s.T * s.K_r + (uint64_t)s.N_s * s.T;
  bool ok = make_tmap_2d(&m[0], kBF16, h, s.I, rows, rb, BK, BM) &&
            make_tmap_2d(&m[2], kBF16, w->down, s.I, (uint64_t)s.N_r * s.d, rb, BK, BN);
  if (ok && s.N_s > 0)
    ok = make_tmap_2d(&m[4], kBF16, w->s_down, s.I, (uint64_t)s.N_s * s.d, rb, BK, BN);
  else
    m[4] = m[2];
  if (!ok) return cudaErrorInvalidValue;
  m[1] = m[0];
  m[3] = m[2];
  m[5] = m[4];
  return launch<1>(s, m, expert_offset, y, st);
}

}  // namespace moe
