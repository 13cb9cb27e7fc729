// Grouped SwiGLU expert GEMMs in FP8 (E4M3) on the sm_103a tensor cores, with fp32
// block scales: tokens and the SwiGLU output per 1x128 tile, weights per 128x128
// block (DeepSeek-V3 Technical Report reading guide, Key ideas, FP8 bullet;
// pwwt.cn notes §三).
//
// The scales change every 128 elements of K, so each 128-wide K chunk is multiplied
// on the tensor cores on its own (four kind::f8f6f4 MMAs of K=32 into a TMEM
// buffer) and the epilogue warps promote it into fp32 registers with that chunk's
// scales: acc += P * (scale_x[row, chunk] * scale_w[block, chunk]).  Two TMEM
// buffers alternate, so the MMAs of chunk c+1 run while chunk c is promoted: the
// tensor-core form of the pages' promotion to CUDA cores every 128 elements.
//
// One persistent CTA per SM walks the segment schedule (ffn_sched.cuh).  Warp roles:
//   warp 0      TMA producer: A [128 rows x 128 B] and B [256 rows x 128 B] per
//               stage, 128-byte swizzled, 4-stage ring.
//   warp 1      allocates 512 TMEM columns, issues the MMAs (one thread).
//   warps 2..17 epilogue: four warps per TMEM lane quarter, each holding 64 fp32
//               accumulators of its row (one quarter of the tile's columns), so
//               four warps per scheduler hide the TMEM-load latency.
//
// gate/up (MODE 0): B = 128 rows of W_gate over the same 128 rows of W_up; the
//   epilogue forms h = silu(gate) * up for 128 columns of a row, quantises that 1x128
//   tile to E4M3 (the four quarters exchange their amax through shared memory) and
//   writes the codes and the scale.
// down (MODE 1): B = 256 rows of W_down (two 128-row scale blocks); y is bf16.
#include <cuda_fp8.h>

#include <algorithm>

#include "common.cuh"
#include "ffn_sched.cuh"
#include "launch.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moe {

namespace {

constexpr int BM = 128, BK = 128, BN = 256, STAGES = 4;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int EPI_WARPS = 16;
constexpr int kLoadGroup = 8;   // TMEM columns loaded per wait in the promotion
constexpr int THREADS = 64 + EPI_WARPS * 32;

struct Ctrl {
  uint64_t full[STAGES], empty[STAGES], pfull[2], pempty[2], xbar[2], fin;
  uint32_t tmem_base;
  int abort_flag;
  float amax[2][4][BM];   // [tile parity][column quarter][row]
  SegTable tab;
};

constexpr size_t kSmemBytes = (size_t)STAGES * STAGE_BYTES + sizeof(Ctrl) + 1024;

struct Fp8Args {
  FfnShape s;
  const int32_t* expert_offset;
  const float* a_scale_r;    // scales of the routed A rows (x_perm / h), [rows, K/128]
  const float* a_scale_s;    // MODE 0: scales of u for the shared experts, [T, d/128]
  const float* b0_scale_r;   // gate (MODE 0) or down (MODE 1) block scales, routed
  const float* b1_scale_r;   // up block scales, routed (MODE 0)
  const float* b0_scale_s;   // the same for the shared experts
  const float* b1_scale_s;
  void* out;                 // MODE 0: h codes [R, I]; MODE 1: y bf16 [R, d]
  float* out_scale;          // MODE 0: h scales [R, I/128]
  int32_t* err;
  // MODE 0, optional: the fp32 pre-activations a = x W_gate^T and c = x W_up^T rounded
  // to bf16, [R, I] in h's row space (kept for the backward pass)
  __nv_bfloat16* save_a = nullptr;
  __nv_bfloat16* save_c = nullptr;
};

__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.f + __expf(-z)); }

__device__ __forceinline__ uint32_t e4m3_code(float x, float scale, float inv) {
  return (uint32_t)__nv_cvt_float_to_fp8(div_by_scale(x, scale, inv), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    tc_ffn_fp8_kernel(const __grid_constant__ CUtensorMap mA_r,
                      const __grid_constant__ CUtensorMap mA_s,
                      const __grid_constant__ CUtensorMap mB0_r,
                      const __grid_constant__ CUtensorMap mB1_r,
                      const __grid_constant__ CUtensorMap mB0_s,
                      const __grid_constant__ CUtensorMap mB1_s, Fp8Args args) {
  extern __shared__ uint8_t smem_raw[];
  pdl_release();
  pdl_wait();
  const uint32_t raw_off = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_off & 1023u)) & 1023u);
  Ctrl& C = *reinterpret_cast<Ctrl*>(base + STAGES * STAGE_BYTES);

  const FfnShape s = args.s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = MODE == 0 ? s.d : s.I;
  const int N = MODE == 0 ? s.I : s.d;
  constexpr int BNO = MODE == 0 ? BN / 2 : BN;   // output columns per tile
  const int n_tiles_n = (N + BNO - 1) / BNO;
  const int nk = K / BK;                          // K is a multiple of 128

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      tc::mbar_init(&C.full[i], 1);
      tc::mbar_init(&C.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&C.pfull[i], 1);
      tc::mbar_init(&C.pempty[i], EPI_WARPS * 32);
      tc::mbar_init(&C.xbar[i], EPI_WARPS * 32);
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
  build_seg_table(C.tab, args.expert_offset, s.T, s.K_r, s.N_r, s.N_s, BM, n_tiles_n, false,
                  args.err);
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
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          tc::mbar_drain(&C.full[j % STAGES], (j / STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer --
      constexpr uint32_t idesc = tc::idesc_e4m3(BM, BN);
      int it = 0, c = 0;   // stage counter, K-chunk counter (TMEM buffer = c & 1)
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total && !*abort_flag; tile += gridDim.x) {
        for (int kb = 0; kb < nk; ++kb, ++it, ++c) {
          const int buf = c & 1;
          if (!tc::mbar_wait(&C.pempty[buf], ((c >> 1) & 1) ^ 1, abort_flag, args.err)) {
            ok = false;
            break;
          }
          const int st = it % STAGES;
          if (!tc::mbar_wait(&C.full[st], (it / STAGES) & 1, abort_flag, args.err)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a0 = tc::smem_u32(base + st * STAGE_BYTES);
          const uint64_t ad = tc::sdesc_sw128(a0), bd = tc::sdesc_sw128(a0 + A_BYTES);
          const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk)
            tc::mma_e4m3(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, kk != 0);
          tc::mma_commit(&C.empty[st]);
          tc::mma_commit(&C.pfull[buf]);
        }
      }
      tc::mma_commit(&C.fin);
      tc::mbar_drain(&C.fin, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int q = warp & 3;              // TMEM lane quarter this warp can access
    const int cq = (warp - 2) >> 2;      // column quarter of the tile
    const int row_in_tile = q * 32 + lane;
    const int nkc_out = N / 128;         // scale columns of the output (MODE 0)
    const int nblk = N / 128;            // 128-row weight blocks per expert along N
    int c = 0, tcount = 0;
    bool alive = true;
    for (int tile = blockIdx.x; alive && tile < total; tile += gridDim.x, ++tcount) {
      // Only what the chunk loop needs stays live across it (the register budget is
      // 96 per thread): the scale offsets, -1 where this thread has no valid row or
      // block.  The tile's coordinates are decoded again for the output.
      int a_off, b_off;
      bool shared;
      {
        const TileCoord tcd = decode_tile(C.tab, tile, n_tiles_n);
        shared = tcd.seg >= s.N_r;
        const int e = shared ? tcd.seg - s.N_r : tcd.seg;
        const int row_local = tcd.m * BM + row_in_tile;
        const int a_row = (MODE == 0 && shared) ? row_local
                          : (MODE == 0 ? tcd.row0 : tcd.out_row0) + row_local;
        a_off = row_local < tcd.rows ? a_row * nk : -1;
        const int blk0 = MODE == 0 ? tcd.n : tcd.n * 2 + (cq >> 1);
        b_off = blk0 < nblk ? (e * nblk + blk0) * nk : -1;
      }
      const float* a_sc = (MODE == 0 && shared) ? args.a_scale_s : args.a_scale_r;
      const float* b0 = shared ? args.b0_scale_s : args.b0_scale_r;
      const float* b1 = shared ? args.b1_scale_s : args.b1_scale_r;   // same block layout

      float acc[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0.f;

      // scales of chunk kb+1 are fetched while chunk kb is promoted
      float sa_n = a_off >= 0 ? __ldg(a_sc + a_off) : 0.f;
      float sb0_n = b_off >= 0 ? __ldg(b0 + b_off) : 0.f;
      float sb1_n = (MODE == 0 && b_off >= 0) ? __ldg(b1 + b_off) : 0.f;
#pragma unroll 1
      for (int kb = 0; kb < nk; ++kb, ++c) {
        const float sa = sa_n, sb0 = sb0_n, sb1 = sb1_n;
        if (kb + 1 < nk) {
          sa_n = a_off >= 0 ? __ldg(a_sc + a_off + kb + 1) : 0.f;
          sb0_n = b_off >= 0 ? __ldg(b0 + b_off + kb + 1) : 0.f;
          if (MODE == 0) sb1_n = b_off >= 0 ? __ldg(b1 + b_off + kb + 1) : 0.f;
        }
        const int buf = c & 1;
        const bool got = tc::mbar_wait(&C.pfull[buf], (c >> 1) & 1, abort_flag, args.err);
        if (!__all_sync(0xffffffffu, got)) { alive = false; break; }
        tc::fence_after_sync();
        const uint32_t t_base = tmem_base + (uint32_t)(buf * BN) + ((uint32_t)(q * 32) << 16);
        // this thread's 64 columns: MODE 0 gate cq*32.. and up 128+cq*32.., MODE 1
        // cq*64..; loaded kLoadGroup at a time per wait
#pragma unroll
        for (int g0 = 0; g0 < 64; g0 += kLoadGroup) {
          uint32_t pv[kLoadGroup];
#pragma unroll
          for (int x = 0; x < kLoadGroup; x += 8) {
            const int c = g0 + x;
            const int col = MODE == 0 ? (c < 32 ? cq * 32 + c : BN / 2 + cq * 32 + (c - 32))
                                      : cq * 64 + c;
            tc::tmem_ld8(t_base + col, *reinterpret_cast<uint32_t(*)[8]>(&pv[x]));
          }
          tc::tmem_ld_wait();
          // the group's 8 columns share one scale (the gate / up boundary is at 32)
          const float sc = sa * (MODE == 0 && g0 >= 32 ? sb1 : sb0);
#pragma unroll
          for (int j = 0; j < kLoadGroup; j += 2)
            tc::fma2(acc[g0 + j], acc[g0 + j + 1], __uint_as_float(pv[j]), __uint_as_float(pv[j + 1]), sc);
        }
        tc::fence_before_sync();
        tc::mbar_arrive(&C.pempty[buf]);
      }
      if (!alive) break;

      const TileCoord tcd = decode_tile(C.tab, tile, n_tiles_n);
      const int row_local = tcd.m * BM + row_in_tile;
      const bool row_ok = row_local < tcd.rows;
      const size_t out_row = (size_t)tcd.out_row0 + row_local;
      if (MODE == 0) {
        if (args.save_a && row_ok) {
          const size_t o = out_row * N + tcd.n * 128 + cq * 32;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            reinterpret_cast<uint4*>(args.save_a + o)[v] =
                make_uint4(pack_bf16(acc[8 * v], acc[8 * v + 1]), pack_bf16(acc[8 * v + 2], acc[8 * v + 3]),
                           pack_bf16(acc[8 * v + 4], acc[8 * v + 5]), pack_bf16(acc[8 * v + 6], acc[8 * v + 7]));
            reinterpret_cast<uint4*>(args.save_c + o)[v] =
                make_uint4(pack_bf16(acc[32 + 8 * v], acc[33 + 8 * v]), pack_bf16(acc[34 + 8 * v], acc[35 + 8 * v]),
                           pack_bf16(acc[36 + 8 * v], acc[37 + 8 * v]), pack_bf16(acc[38 + 8 * v], acc[39 + 8 * v]));
          }
        }
        // h for this thread's 32 columns, then the 1x128 tile scale from all four quarters
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          acc[j] = silu(acc[j]) * acc[32 + j];
          amax = fmaxf(amax, fabsf(acc[j]));
        }
        const int tb = tcount & 1;
        C.amax[tb][cq][row_in_tile] = amax;
        tc::mbar_arrive(&C.xbar[tb]);   // release: the amax store is visible after the wait
        const bool xg = tc::mbar_wait(&C.xbar[tb], (tcount >> 1) & 1, abort_flag, args.err);
        if (!__all_sync(0xffffffffu, xg)) break;
        float tile_amax = 0.f;
#pragma unroll
        for (int x = 0; x < 4; ++x) tile_amax = fmaxf(tile_amax, C.amax[tb][x][row_in_tile]);
        const float scale = tile_amax > 0.f ? __fdiv_rn(tile_amax, 448.f) : 1.f;
        const float inv = __frcp_rn(scale);
        if (row_ok) {
          uint8_t* hq = static_cast<uint8_t*>(args.out) + out_row * N + tcd.n * 128 + cq * 32;
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const int j = v * 16 + x * 4;
              w[x] = e4m3_code(acc[j], scale, inv) | (e4m3_code(acc[j + 1], scale, inv) << 8) |
                     (e4m3_code(acc[j + 2], scale, inv) << 16) | (e4m3_code(acc[j + 3], scale, inv) << 24);
            }
            reinterpret_cast<uint4*>(hq)[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          if (cq == 0) args.out_scale[out_row * nkc_out + tcd.n] = scale;
        }
      } else {
        const int col0 = tcd.n * BN + cq * 64;
        if (row_ok && col0 < N) {
          __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(args.out) + out_row * N + col0;
#pragma unroll
          for (int v = 0; v < 8; ++v)
            reinterpret_cast<uint4*>(yrow)[v] =
                make_uint4(pack_bf16(acc[8 * v + 0], acc[8 * v + 1]), pack_bf16(acc[8 * v + 2], acc[8 * v + 3]),
                           pack_bf16(acc[8 * v + 4], acc[8 * v + 5]), pack_bf16(acc[8 * v + 6], acc[8 * v + 7]));
        }
      }
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
cudaError_t launch(const FfnShape& s, const CUtensorMap* maps, const Fp8Args& a, cudaStream_t st) {
  const int N = MODE == 0 ? s.I : s.d;
  const int bno = MODE == 0 ? BN / 2 : BN;
  const long long m_ub = (long long)s.T * s.K_r / BM + s.N_r + (long long)s.N_s * ((s.T + BM - 1) / BM);
  const long long tiles_ub = m_ub * ((N + bno - 1) / bno);
  const int grid = (int)std::min<long long>(device_sm_count(), std::max<long long>(1, tiles_ub));
  auto k = tc_ffn_fp8_kernel<MODE>;
  cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  err = launch_pdl(k, dim3(grid), dim3(THREADS), kSmemBytes, st, 0, maps[0], maps[1], maps[2], maps[3],
                   maps[4], maps[5], a);
  return err != cudaSuccess ? err : cudaGetLastError();
}

constexpr CUtensorMapDataType kU8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;

}  // namespace

cudaError_t launch_ffn_up_fp8(const FfnShape& s, const void* x_perm, const float* x_perm_scale,
                              const void* u, const float* u_scale, const int32_t* expert_offset,
                              const moe_expert_weights* w, void* h, float* h_scale,
                              cudaStream_t st, void* save_a, void* save_c) {
  if (s.T == 0) return cudaSuccess;
  CUtensorMap m[6];
  const uint64_t rb = (uint64_t)s.d;
  const uint64_t routed = (uint64_t)s.T * s.K_r;
  bool ok = make_tmap_2d(&m[0], kU8, x_perm, s.d, routed, rb, BK, BM) &&
            make_tmap_2d(&m[1], kU8, u, s.d, s.T, rb, BK, BM) &&
            make_tmap_2d(&m[2], kU8, w->gate, s.d, (uint64_t)s.N_r * s.I, rb, BK, BN / 2) &&
            make_tmap_2d(&m[3], kU8, w->up, s.d, (uint64_t)s.N_r * s.I, rb, BK, BN / 2);
  if (ok && s.N_s > 0) {
    ok = make_tmap_2d(&m[4], kU8, w->s_gate, s.d, (uint64_t)s.N_s * s.I, rb, BK, BN / 2) &&
         make_tmap_2d(&m[5], kU8, w->s_up, s.d, (uint64_t)s.N_s * s.I, rb, BK, BN / 2);
  } else {
    m[4] = m[2];
    m[5] = m[3];
  }
  if (!ok) return cudaErrorInvalidValue;
  Fp8Args a{s, expert_offset, x_perm_scale, u_scale, w->gate_scale, w->up_scale,
            s.N_s > 0 ? w->s_gate_scale : w->gate_scale, s.N_s > 0 ? w->s_up_scale : w->up_scale,
            h, h_scale, dev_error_ptr(), static_cast<__nv_bfloat16*>(save_a),
            static_cast<__nv_bfloat16*>(save_c)};
  return launch<0>(s, m, a, st);
}

cudaError_t launch_ffn_down_fp8(const FfnShape& s, const void* h, const float* h_scale,
                                const int32_t* expert_offset, const moe_expert_weights* w,
                                void* y, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  CUtensorMap m[6];
  const uint64_t rb = (uint64_t)s.I;
  const uint64_t rows = (uint64_t)s.T * s.K_r + (uint64_t)s.N_s * s.T;
  bool ok = make_tmap_2d(&m[0], kU8, h, s.I, rows, rb, BK, BM) &&
            make_tmap_2d(&m[2], kU8, w->down, s.I, (uint64_t)s.N_r * s.d, rb, BK, BN);
  if (ok && s.N_s > 0)
    ok = make_tmap_2d(&m[4], kU8, w->s_down, s.I, (uint64_t)s.N_s * s.d, rb, BK, BN);
  else
    m[4] = m[2];
  if (!ok) return cudaErrorInvalidValue;
  m[1] = m[0];
  m[3] = m[2];
  m[5] = m[4];
  Fp8Args a{s, expert_offset, h_scale, nullptr, w->down_scale, nullptr,
            s.N_s > 0 ? w->s_down_scale : w->down_scale, nullptr, y, nullptr, dev_error_ptr()};
  return launch<1>(s, m, a, st);
}

}  // namespace moe
