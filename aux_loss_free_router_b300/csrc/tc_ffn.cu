// Grouped SwiGLU expert GEMMs on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Weights on the M side, tokens on the N side: each MMA computes a [128 features x
// n tokens] block of the transposed output, D^T = W X^T.  The MMA's N (tokens) goes
// down to 16 in steps of 16, so the last tile of an expert's segment is sized to the
// tokens it has (at most 15 padding tokens), where a token-major M tile would pad up
// to 127 rows: on the DeepSeek-V3 layer that is about a fifth of the routed work.
//
// One persistent CTA per SM walks the tiles of the segment schedule (ffn_sched.cuh):
// segment-major, then feature tile, then token tile, so CTAs running at the same time
// share an expert's weight tile through L2.  Warp roles:
//   warp 0      TMA producer into a 4-stage shared-memory ring (48 KB per stage).
//   warp 1      allocates 512 TMEM columns and issues the MMAs (one thread) into one
//               of two 256-column fp32 accumulators, so the epilogue of tile i
//               overlaps the MMAs of tile i+1.
//   warps 2..5  epilogue: TMEM lane = feature, column = token; each warp transposes
//               32 features x 16 tokens through its own shared-memory scratch and
//               writes 16-byte pieces of token rows.
//
// gate/up (MODE 0): a stage holds W_gate and W_up [128 features x 64 K] and X [128
//   tokens x 64 K]; two MMAs per K step give gate (columns 0..127) and up (128..255)
//   of the same features; the epilogue writes h = silu(gate) * up.
// down (MODE 1): a stage holds W_down [128 features x 64 K] and H [256 tokens x 64 K];
//   the epilogue writes y.
// Tokens past the end of a tile's segment are loaded (or zero-filled past the tensor
// end) but sit beyond the MMA's N or are not stored; features past the end of the
// output width are computed from the next expert's rows (or zeros) and not stored.
#include <algorithm>

#include "common.cuh"
#include "ffn_sched.cuh"
#include "launch.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moe {

namespace {

constexpr int BF = 128, BK = 64, STAGES = 4;
constexpr int W_BYTES = BF * BK * 2;          // one weight tile
constexpr int STAGE_BYTES = 3 * W_BYTES;      // MODE 0: Wg, Wu, X[128]; MODE 1: Wd, H[256]
constexpr int TMEM_COLS = 512, ACC_COLS = 256;
constexpr int THREADS = 192;
constexpr int SCRATCH = 16 * 32 * 2;          // per epilogue warp: 16 tokens x 32 features bf16

template <int MODE> struct Tiles {
  static constexpr int BT = MODE == 0 ? 128 : 256;   // tokens per tile (MMA N at most)
};

struct Ctrl {
  uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], fin;
  uint32_t tmem_base;
  int abort_flag;
  SegTable tab;
};

constexpr size_t kSmemBytes = (size_t)STAGES * STAGE_BYTES + 4 * SCRATCH + sizeof(Ctrl) + 1024;

struct TcArgs {
  FfnShape s;
  const int32_t* expert_offset;
  __nv_bfloat16* out;
  int32_t* err;
};

__device__ __forceinline__ float silu(float z) { return z / (1.f + __expf(-z)); }

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    tc_ffn_kernel(const __grid_constant__ CUtensorMap mX_r, const __grid_constant__ CUtensorMap mX_s,
                  const __grid_constant__ CUtensorMap mW0_r, const __grid_constant__ CUtensorMap mW1_r,
                  const __grid_constant__ CUtensorMap mW0_s, const __grid_constant__ CUtensorMap mW1_s,
                  TcArgs args) {
  constexpr int BT = Tiles<MODE>::BT;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_off = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_off & 1023u)) & 1023u);
  uint8_t* scratch = base + STAGES * STAGE_BYTES;
  Ctrl& C = *reinterpret_cast<Ctrl*>(scratch + 4 * SCRATCH);

  const FfnShape s = args.s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = MODE == 0 ? s.d : s.I;
  const int N = MODE == 0 ? s.I : s.d;            // output width (features)
  const int n_ft = (N + BF - 1) / BF;             // feature tiles per expert
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
    tc::tma_prefetch_desc(&mX_r);
    tc::tma_prefetch_desc(&mW0_r);
  }
  if (warp == 1) {
    tc::tmem_alloc(&C.tmem_base, TMEM_COLS);
    tc::tmem_relinquish();
  }
  build_seg_table(C.tab, args.expert_offset, s.T, s.K_r, s.N_r, s.N_s, BT, n_ft);
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
        const TileCoord tcd = decode_tile(C.tab, tile, n_ft);
        const bool shared = tcd.seg >= s.N_r;
        const int e = shared ? tcd.seg - s.N_r : tcd.seg;
        const CUtensorMap* mX = (MODE == 0 && shared) ? &mX_s : &mX_r;
        const int x_row = (MODE == 0 ? (shared ? 0 : tcd.row0) : tcd.out_row0) + tcd.m * BT;
        const CUtensorMap* mW0 = shared ? &mW0_s : &mW0_r;
        const CUtensorMap* mW1 = shared ? &mW1_s : &mW1_r;
        const int w_row = e * N + tcd.n * BF;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!tc::mbar_wait(&C.empty[st], ph ^ 1, abort_flag, args.err)) { ok = false; break; }
          uint8_t* sw = base + st * STAGE_BYTES;
          tc::mbar_arrive_expect_tx(&C.full[st], STAGE_BYTES);
          tc::tma_load_2d(sw, mW0, &C.full[st], kb * BK, w_row);
          if (MODE == 0) {
            tc::tma_load_2d(sw + W_BYTES, mW1, &C.full[st], kb * BK, w_row);
            tc::tma_load_2d(sw + 2 * W_BYTES, mX, &C.full[st], kb * BK, x_row);
          } else {
            tc::tma_load_2d(sw + W_BYTES, mX, &C.full[st], kb * BK, x_row);
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
      int it = 0, tcount = 0;
      for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x, ++tcount) {
        const TileCoord tcd = decode_tile(C.tab, tile, n_ft);
        const int n_tok = min(BT, tcd.rows - tcd.m * BT);
        const uint32_t idesc = tc::idesc_bf16(BF, (n_tok + 15) & ~15);
        const int acc = tcount & 1;
        const uint32_t aph = (tcount >> 1) & 1;
        if (!tc::mbar_wait(&C.tempty[acc], aph ^ 1, abort_flag, args.err)) break;
        tc::fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * ACC_COLS);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!tc::mbar_wait(&C.full[st], ph, abort_flag, args.err)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t s0 = tc::smem_u32(base + st * STAGE_BYTES);
          const uint64_t w0 = tc::sdesc_sw128(s0);
          if (MODE == 0) {
            const uint64_t w1 = tc::sdesc_sw128(s0 + W_BYTES), x = tc::sdesc_sw128(s0 + 2 * W_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              tc::mma_bf16(d_tmem, w0 + 2 * kk, x + 2 * kk, idesc, (kb | kk) != 0);        // gate
              tc::mma_bf16(d_tmem + BT, w1 + 2 * kk, x + 2 * kk, idesc, (kb | kk) != 0);   // up
            }
          } else {
            const uint64_t x = tc::sdesc_sw128(s0 + W_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              tc::mma_bf16(d_tmem, w0 + 2 * kk, x + 2 * kk, idesc, (kb | kk) != 0);
          }
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
    const int q = warp & 3;   // TMEM lane quarter this warp can access: features q*32..
    __nv_bfloat16* scr = reinterpret_cast<__nv_bfloat16*>(scratch + q * SCRATCH);  // [16][32]
    int tcount = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++tcount) {
      // warp-uniform decisions: the TMEM loads below are warp-collective
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const TileCoord tcd = decode_tile(C.tab, tile, n_ft);
      const int n_tok = min(BT, tcd.rows - tcd.m * BT);
      const int acc = tcount & 1;
      const uint32_t aph = (tcount >> 1) & 1;
      const bool got = tc::mbar_wait(&C.tfull[acc], aph, abort_flag, args.err);
      if (!__all_sync(0xffffffffu, got)) break;
      tc::fence_after_sync();
      const uint32_t t_base = tmem_base + (uint32_t)(acc * ACC_COLS) + ((uint32_t)(q * 32) << 16);
      const int f0 = tcd.n * BF + q * 32;                 // first feature of this warp
      const size_t row0 = (size_t)tcd.out_row0 + (size_t)tcd.m * BT;
#pragma unroll 1
      for (int j0 = 0; j0 < n_tok; j0 += 16) {
        uint32_t a[16];
        float v[16];
        if (MODE == 0) {
          uint32_t b[16];
          tc::tmem_ld16(t_base + j0, a);
          tc::tmem_ld16(t_base + BT + j0, b);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = silu(__uint_as_float(a[j])) * __uint_as_float(b[j]);
        } else {
          tc::tmem_ld16(t_base + j0, a);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(a[j]);
        }
        // transpose: lane = feature -> 16-byte pieces of 8 features of one token
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
            *reinterpret_cast<uint4*>(args.out + (row0 + j0 + tok) * N + f) = val;
          }
        }
        __syncwarp();
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
  constexpr int BT = Tiles<MODE>::BT;
  const int N = MODE == 0 ? s.I : s.d;
  const long long t_ub = (long long)s.T * s.K_r / BT + s.N_r + (long long)s.N_s * ((s.T + BT - 1) / BT);
  const long long tiles_ub = t_ub * ((N + BF - 1) / BF);
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
  constexpr int BT = Tiles<0>::BT;
  CUtensorMap m[6];
  const uint64_t rb = (uint64_t)s.d * 2;
  const uint64_t routed = (uint64_t)s.T * s.K_r;
  bool ok = make_tmap_2d(&m[0], kBF16, x_perm, s.d, routed, rb, BK, BT) &&
            make_tmap_2d(&m[1], kBF16, u, s.d, s.T, rb, BK, BT) &&
            make_tmap_2d(&m[2], kBF16, w->gate, s.d, (uint64_t)s.N_r * s.I, rb, BK, BF) &&
            make_tmap_2d(&m[3], kBF16, w->up, s.d, (uint64_t)s.N_r * s.I, rb, BK, BF);
  if (ok && s.N_s > 0) {
    ok = make_tmap_2d(&m[4], kBF16, w->s_gate, s.d, (uint64_t)s.N_s * s.I, rb, BK, BF) &&
         make_tmap_2d(&m[5], kBF16, w->s_up, s.d, (uint64_t)s.N_s * s.I, rb, BK, BF);
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
  constexpr int BT = Tiles<1>::BT;
  CUtensorMap m[6];
  const uint64_t rb = (uint64_t)s.I * 2;
  const uint64_t rows = (uint64_t)s.T * s.K_r + (uint64_t)s.N_s * s.T;
  bool ok = make_tmap_2d(&m[0], kBF16, h, s.I, rows, rb, BK, BT) &&
            make_tmap_2d(&m[2], kBF16, w->down, s.I, (uint64_t)s.N_r * s.d, rb, BK, BF);
  if (ok && s.N_s > 0)
    ok = make_tmap_2d(&m[4], kBF16, w->s_down, s.I, (uint64_t)s.N_s * s.d, rb, BK, BF);
  else
    m[4] = m[2];
  if (!ok) return cudaErrorInvalidValue;
  m[1] = m[0];
  m[3] = m[2];
  m[5] = m[4];
  return launch<1>(s, m, expert_offset, y, st);
}

}  // namespace moe
