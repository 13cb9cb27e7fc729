// The FP8 backward pass's own kernels: the three GEMMs of every expert linear layer
// run in E4M3 - Fprop (recomputed), Dgrad and Wgrad - with fp32 block scales and fp32
// promotion every 128 elements of the contraction, and Wgrad reads the activations the
// forward kept in E4M3 (pwwt.cn notes §三; DeepSeek-V3 Technical Report reading guide,
// Key ideas, FP8 bullet).  An activation tile lies along the contraction of the GEMM
// that reads it: 1x128 (one token, 128 features) for Fprop and Dgrad, 128x1 (one
// feature, 128 tokens of an expert's segment) for Wgrad, whose contraction runs over
// the tokens; weights keep their 128x128 blocks, which are blocks of W^T too.
//
// The Dgrad GEMMs are the forward's FP8 down-projection kernel run on transposed E4M3
// weights (fp8_transpose_kernel); this file holds the rest:
//   fp8_swiglu_bwd_kernel   dA = dH c silu'(a), dC = dH silu(a); their 1x128 E4M3 tiles
//                           for Dgrad and bf16 copies for Wgrad;
//   fp8_colquant_kernel     Wgrad operands: 128x1 E4M3 tiles over each segment's tokens,
//                           written transposed (tokens contiguous: K-major for the MMA);
//   fp8_wgrad_kernel        per expert, dW = sum over its 128-token blocks of
//                           diag(sa) (A B^T) diag(sb) on the tensor cores
//                           (tcgen05 kind::f8f6f4), promoted in fp32 registers.
#include <cuda_fp8.h>

#include <algorithm>

#include "common.cuh"
#include "ffn_sched.cuh"
#include "launch.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moe {

namespace {

__device__ __forceinline__ uint32_t e4m3_code(float x, float scale, float inv) {
  return (uint32_t)__nv_cvt_float_to_fp8(div_by_scale(x, scale, inv), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float e4m3_value(uint32_t code) {
  __nv_fp8_e4m3 v;
  v.__x = (__nv_fp8_storage_t)code;
  return float(v);
}

// scale = amax / 448 in fp32, 1 for an all-zero tile
__device__ __forceinline__ float tile_scale(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
}

// ------------------------------------------------------------ weight transpose ----
// One CTA per 64 x 64 byte tile of one expert's [R, C] matrix.
__global__ void __launch_bounds__(256) fp8_transpose_kernel(const uint8_t* __restrict__ src,
                                                            const float* __restrict__ src_s, int R,
                                                            int C, uint8_t* __restrict__ dst,
                                                            float* __restrict__ dst_s, int ldd, int col0) {
  __shared__ uint8_t tile[64][64 + 16];
  const int e = blockIdx.z, r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
  const int t = threadIdx.x, row = t >> 2, chunk = (t & 3) * 16;
  const uint8_t* s = src + (size_t)e * R * C;
  *reinterpret_cast<uint4*>(&tile[row][chunk]) =
      *reinterpret_cast<const uint4*>(s + (size_t)(r0 + row) * C + c0 + chunk);
  __syncthreads();
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    w[k] = (uint32_t)tile[chunk + 4 * k][row] | ((uint32_t)tile[chunk + 4 * k + 1][row] << 8) |
           ((uint32_t)tile[chunk + 4 * k + 2][row] << 16) | ((uint32_t)tile[chunk + 4 * k + 3][row] << 24);
  uint8_t* d = dst + (size_t)e * C * ldd;
  *reinterpret_cast<uint4*>(d + (size_t)(c0 + row) * ldd + col0 + r0 + chunk) = make_uint4(w[0], w[1], w[2], w[3]);
  if (t == 0 && (r0 & 127) == 0 && (c0 & 127) == 0) {   // one scale per 128 x 128 block
    const int br = r0 >> 7, bc = c0 >> 7;
    dst_s[(size_t)e * (C / 128) * (ldd / 128) + (size_t)bc * (ldd / 128) + (col0 >> 7) + br] =
        src_s[(size_t)e * (R / 128) * (C / 128) + (size_t)br * (C / 128) + bc];
  }
}

// ------------------------------------------------------------ SwiGLU backward ----
// One warp per (row, 128-column tile of I); lane l takes columns 4l .. 4l+3.
__global__ void __launch_bounds__(256) fp8_swiglu_bwd_kernel(
    const __nv_bfloat16* __restrict__ dH, const __nv_bfloat16* __restrict__ a,
    const __nv_bfloat16* __restrict__ c, long long rows, int I, uint8_t* __restrict__ ac_q,
    float* __restrict__ ac_s, __nv_bfloat16* __restrict__ dA, __nv_bfloat16* __restrict__ dC) {
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int tiles = I / 128;
  if (w >= rows * tiles) return;
  const long long r = w / tiles;
  const int t = (int)(w % tiles);
  const size_t o = (size_t)r * I + t * 128 + lane * 4;
  float vh[4], va[4], vc[4], ga[4], gc[4];
  {
    const uint2 h2 = *reinterpret_cast<const uint2*>(dH + o);
    const uint2 a2 = *reinterpret_cast<const uint2*>(a + o);
    const uint2 c2 = *reinterpret_cast<const uint2*>(c + o);
    const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&h2);
    const __nv_bfloat162* ap = reinterpret_cast<const __nv_bfloat162*>(&a2);
    const __nv_bfloat162* cp = reinterpret_cast<const __nv_bfloat162*>(&c2);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      vh[2 * k] = __low2float(hp[k]); vh[2 * k + 1] = __high2float(hp[k]);
      va[2 * k] = __low2float(ap[k]); va[2 * k + 1] = __high2float(ap[k]);
      vc[2 * k] = __low2float(cp[k]); vc[2 * k + 1] = __high2float(cp[k]);
    }
  }
  float amax_a = 0.f, amax_c = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float sg = __fdividef(1.f, 1.f + __expf(-va[k]));
    const float silu = va[k] * sg;
    const float dsilu = sg * (1.f + va[k] * (1.f - sg));
    ga[k] = vh[k] * vc[k] * dsilu;
    gc[k] = vh[k] * silu;
    amax_a = fmaxf(amax_a, fabsf(ga[k]));
    amax_c = fmaxf(amax_c, fabsf(gc[k]));
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) {
    amax_a = fmaxf(amax_a, __shfl_xor_sync(0xffffffffu, amax_a, s));
    amax_c = fmaxf(amax_c, __shfl_xor_sync(0xffffffffu, amax_c, s));
  }
  const float sa = tile_scale(amax_a), sc = tile_scale(amax_c);
  const float ia = __frcp_rn(sa), ic = __frcp_rn(sc);
  uint32_t qa = 0, qc = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    qa |= e4m3_code(ga[k], sa, ia) << (8 * k);
    qc |= e4m3_code(gc[k], sc, ic) << (8 * k);
  }
  uint8_t* qrow = ac_q + (size_t)r * 2 * I;
  *reinterpret_cast<uint32_t*>(qrow + t * 128 + lane * 4) = qa;
  *reinterpret_cast<uint32_t*>(qrow + I + t * 128 + lane * 4) = qc;
  if (lane == 0) {
    ac_s[(size_t)r * (2 * tiles) + t] = sa;
    ac_s[(size_t)r * (2 * tiles) + tiles + t] = sc;
  }
  __nv_bfloat162 pa[2] = {__floats2bfloat162_rn(ga[0], ga[1]), __floats2bfloat162_rn(ga[2], ga[3])};
  __nv_bfloat162 pc[2] = {__floats2bfloat162_rn(gc[0], gc[1]), __floats2bfloat162_rn(gc[2], gc[3])};
  *reinterpret_cast<uint2*>(dA + o) = *reinterpret_cast<uint2*>(pa);
  *reinterpret_cast<uint2*>(dC + o) = *reinterpret_cast<uint2*>(pc);
}

// ------------------------------------------------------ padded segment blocks ----
// blk[i] = 128-token blocks before segment i (segment i < N_r: rows off[i]..off[i+1],
// shared segments T rows); blk[nseg] = all.  One warp; a routed segment outside
// [0, T*K_r] counts as empty and records MOE_ERR_INVALID_ARG.
__device__ __forceinline__ void segment_blocks(int* blk, int* seg_rows, const int32_t* __restrict__ off,
                                               int T, int K_r, int N_r, int N_s, int32_t* err) {
  const int lane = threadIdx.x & 31, nseg = N_r + N_s;
  const int span = (nseg + 31) / 32;
  int local = 0;
  for (int q = 0; q < span; ++q) {
    const int i = lane * span + q;
    if (i < nseg) {
      int rows = T;
      if (i < N_r) {
        const int r0 = off[i];
        rows = off[i + 1] - r0;
        if (r0 < 0 || rows < 0 || (long long)r0 + rows > (long long)T * K_r) {
          if (blockIdx.x == 0 && blockIdx.y == 0) record_error(err, MOE_ERR_INVALID_ARG);
          rows = 0;
        }
      }
      seg_rows[i] = rows;
      local += (rows + 127) >> 7;
    }
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - local;
  for (int q = 0; q < span; ++q) {
    const int i = lane * span + q;
    if (i < nseg) {
      blk[i] = run;
      run += (seg_rows[i] + 127) >> 7;
    }
  }
  if (lane == 31) blk[nseg] = incl;
}

// ------------------------------------------------- Wgrad operand quantisation ----
// Work items (128-token block, 64 columns), taken by a grid of CTAs that each build the
// block table once and then walk items blockIdx.x, blockIdx.x + gridDim.x, ...
constexpr int CQ_COLS = 64;

__global__ void __launch_bounds__(256) fp8_colquant_kernel(ColQuantSrc src, const int32_t* __restrict__ off,
                                                           int T, int K_r, int N_r, int N_s, int C,
                                                           uint8_t* __restrict__ q, float* __restrict__ scale,
                                                           long long Rp, int32_t* err) {
  __shared__ int blk[kMaxSegs + 1];
  __shared__ int seg_rows[kMaxSegs];
  __shared__ float tile[128][CQ_COLS + 1];
  __shared__ float red[4][CQ_COLS];
  const int nseg = N_r + N_s;
  if (threadIdx.x < 32) segment_blocks(blk, seg_rows, off, T, K_r, N_r, N_s, err);
  __syncthreads();
  const int ncc = C / CQ_COLS;
  const long long items = (long long)blk[nseg] * ncc;
  for (long long item = blockIdx.x; item < items; item += gridDim.x) {
    const int b = (int)(item / ncc);
    const int c0 = (int)(item - (long long)b * ncc) * CQ_COLS;
    int lo = 0, hi = nseg;                       // the segment: last i with blk[i] <= b
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (blk[mid] <= b) lo = mid; else hi = mid;
    }
    const int seg = lo;
    const int r0 = (b - blk[seg]) * 128;
    const int n_valid = min(128, seg_rows[seg] - r0);
    const bool sh = seg >= N_r;
    const long long src_row0 = sh ? (long long)(seg - N_r) * src.shared_stride + r0 : (long long)off[seg] + r0;
    const void* base = sh ? src.shared : src.routed;
    const float* bscale = sh ? src.shared_scale : src.routed_scale;
    {
      const int row = threadIdx.x >> 1, half = threadIdx.x & 1;    // 32 columns each
      float v[32];
      if (row < n_valid) {
        const long long gr = src_row0 + row;
        if (bscale == nullptr) {
          const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) +
                                                          (size_t)gr * C + c0 + half * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 x = p[k];
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              v[8 * k + 2 * j] = __low2float(h[j]);
              v[8 * k + 2 * j + 1] = __high2float(h[j]);
            }
          }
        } else {
          const float s = bscale[(size_t)gr * (C / 128) + (c0 >> 7)];
          const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(base) + (size_t)gr * C +
                                                          c0 + half * 32);
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const uint4 x = p[k];
            const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int j = 0; j < 16; ++j) v[16 * k + j] = e4m3_value((wv[j >> 2] >> (8 * (j & 3))) & 0xffu) * s;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) tile[row][half * 32 + j] = v[j];
    }
    __syncthreads();
    const int col = threadIdx.x & (CQ_COLS - 1), part = threadIdx.x >> 6;   // 32 rows each
    float amax = 0.f;
#pragma unroll 8
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(tile[part * 32 + j][col]));
    red[part][col] = amax;
    __syncthreads();
    const float s = tile_scale(fmaxf(fmaxf(red[0][col], red[1][col]), fmaxf(red[2][col], red[3][col])));
    const float inv = __frcp_rn(s);
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      w[k] = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) w[k] |= e4m3_code(tile[part * 32 + 4 * k + j][col], s, inv) << (8 * j);
    }
    uint4* dst = reinterpret_cast<uint4*>(q + (size_t)(c0 + col) * Rp + (size_t)b * 128 + part * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    if (part == 0) scale[(size_t)b * C + c0 + col] = s;
    __syncthreads();                             // tile and red are free for the next item
  }
}

// ------------------------------------------------------------------- Wgrad GEMM ----
// One persistent CTA per SM walks the tiles (expert, 128 rows of M, 256 columns of N),
// expert-major.  Warp roles, as in the forward's FP8 kernel:
//   warp 0      TMA producer: A [128 rows x 128 tokens] and B [256 rows x 128 tokens]
//               per stage (E4M3, 128-byte swizzled), 4-stage ring;
//   warp 1      allocates 512 TMEM columns; one thread issues, per 128-token block, four
//               kind::f8f6f4 MMAs of K = 32 into one of two 256-column TMEM buffers;
//   warps 2..17 promote each block into fp32 registers: acc += P * (sa[row] * sb[col]),
//               four warps per TMEM lane quarter, 64 columns each, and store the tile.
//               Output: 32 x 32 fp32 boxes written to per-warp scratch, stored by TMA.
//               A block's 256 column scales sit in a shared-memory double buffer: the
//               epilogue loads the next block's while it promotes this one (an mbarrier
//               per buffer says all 512 epilogue threads have stored theirs).
constexpr int WG_BM = 128, WG_BK = 128, WG_BN = 256, WG_STAGES = 3;
constexpr int WG_A = WG_BM * WG_BK, WG_B = WG_BN * WG_BK, WG_STAGE = WG_A + WG_B;
constexpr int WG_EPI_WARPS = 16, WG_THREADS = 64 + WG_EPI_WARPS * 32;
constexpr int WG_SCR = 32 * 32 * 4;   // per epilogue warp: a 32 x 32 fp32 store box

struct WgCtrl {
  uint64_t full[WG_STAGES], empty[WG_STAGES], pfull[2], pempty[2], sfill[2], fin;
  uint32_t tmem_base;
  int abort_flag;
  float sbuf[2][WG_BN];   // column scales of a 128-token block, by block parity
  int blk[kMaxSegs + 1];
  int seg_rows[kMaxSegs];
};

constexpr size_t kWgSmem = (size_t)WG_STAGES * WG_STAGE + (size_t)WG_EPI_WARPS * WG_SCR + sizeof(WgCtrl) + 1024;
static_assert(kWgSmem <= 227 * 1024, "shared memory per CTA");

struct WgArgs {
  const float* sa;           // [Rp/128, M]
  const float* sb;           // [Rp/128, N]
  int M, N, T, K_r, N_r, N_s;
  const int32_t* expert_offset;
  float* out;                // [N_r][M, N]
  float* out_s;              // [N_s][M, N]
  int32_t* err;
};

__global__ void __launch_bounds__(WG_THREADS, 1)
    fp8_wgrad_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB,
                     const __grid_constant__ CUtensorMap mO, const __grid_constant__ CUtensorMap mOs, WgArgs g) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_off = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_off & 1023u)) & 1023u);
  float* scr_all = reinterpret_cast<float*>(base + WG_STAGES * WG_STAGE);
  WgCtrl& C = *reinterpret_cast<WgCtrl*>(base + WG_STAGES * WG_STAGE + WG_EPI_WARPS * WG_SCR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nseg = g.N_r + g.N_s;
  const int mt = g.M / WG_BM, nt = (g.N + WG_BN - 1) / WG_BN;
  const int total = nseg * mt * nt;

  if (threadIdx.x == 0) {
    for (int i = 0; i < WG_STAGES; ++i) {
      tc::mbar_init(&C.full[i], 1);
      tc::mbar_init(&C.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&C.pfull[i], 1);
      tc::mbar_init(&C.pempty[i], WG_EPI_WARPS * 32);
      tc::mbar_init(&C.sfill[i], WG_EPI_WARPS * 32);   // every epilogue thread, per use
    }
    tc::mbar_init(&C.fin, 1);
    C.abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&mA);
    tc::tma_prefetch_desc(&mB);
  }
  if (warp == 1) {
    tc::tmem_alloc(&C.tmem_base, 512);
    tc::tmem_relinquish();
  }
  if (warp == 2) segment_blocks(C.blk, C.seg_rows, g.expert_offset, g.T, g.K_r, g.N_r, g.N_s, g.err);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = C.tmem_base;
  volatile int* abort_flag = &C.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer --
      int it = 0;
      for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
        const int seg = tile / (mt * nt), rem = tile - seg * (mt * nt);
        const int m = rem / nt, n = rem - m * nt;
        bool ok = true;
        for (int kb = C.blk[seg]; kb < C.blk[seg + 1]; ++kb, ++it) {
          const int st = it % WG_STAGES;
          if (!tc::mbar_wait(&C.empty[st], ((it / WG_STAGES) & 1) ^ 1, abort_flag, g.err)) { ok = false; break; }
          uint8_t* sa = base + st * WG_STAGE;
          tc::mbar_arrive_expect_tx(&C.full[st], WG_STAGE);
          tc::tma_load_2d(sa, &mA, &C.full[st], kb * WG_BK, m * WG_BM);
          tc::tma_load_2d(sa + WG_A, &mB, &C.full[st], kb * WG_BK, n * WG_BN);
        }
        if (!ok) break;
      }
      if (*abort_flag) {
        for (int j = (it > WG_STAGES ? it - WG_STAGES : 0); j < it; ++j)
          tc::mbar_drain(&C.full[j % WG_STAGES], (j / WG_STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer --
      constexpr uint32_t idesc = tc::idesc_e4m3(WG_BM, WG_BN);
      int it = 0, c = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total && !*abort_flag; tile += gridDim.x) {
        const int seg = tile / (mt * nt);
        for (int kb = C.blk[seg]; kb < C.blk[seg + 1]; ++kb, ++it, ++c) {
          const int buf = c & 1;
          if (!tc::mbar_wait(&C.pempty[buf], ((c >> 1) & 1) ^ 1, abort_flag, g.err)) { ok = false; break; }
          const int st = it % WG_STAGES;
          if (!tc::mbar_wait(&C.full[st], (it / WG_STAGES) & 1, abort_flag, g.err)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t a0 = tc::smem_u32(base + st * WG_STAGE);
          const uint64_t ad = tc::sdesc_sw128(a0), bd = tc::sdesc_sw128(a0 + WG_A);
          const uint32_t d_tmem = tmem_base + (uint32_t)(buf * WG_BN);
#pragma unroll
          for (int kk = 0; kk < WG_BK / 32; ++kk) tc::mma_e4m3(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, kk != 0);
          tc::mma_commit(&C.empty[st]);
          tc::mma_commit(&C.pfull[buf]);
        }
      }
      tc::mma_commit(&C.fin);
      tc::mbar_drain(&C.fin, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int q = warp & 3;               // TMEM lane quarter
    const int cq = (warp - 2) >> 2;       // column quarter: 64 columns
    const int et = threadIdx.x - 64;      // 0 .. 511
    // the (tile, block) after (tile, kb) in this CTA's walk, or tile = -1
    auto next_chunk = [&](int tile, int kb, int& nt_tile, int& nkb) {
      const int seg = tile / (mt * nt);
      if (kb + 1 < C.blk[seg + 1]) { nt_tile = tile; nkb = kb + 1; return; }
      for (int t2 = tile + (int)gridDim.x; t2 < total; t2 += (int)gridDim.x) {
        const int s2 = t2 / (mt * nt);
        if (C.blk[s2 + 1] > C.blk[s2]) { nt_tile = t2; nkb = C.blk[s2]; return; }
      }
      nt_tile = -1;
      nkb = 0;
    };
    // the scale of column et (< 256) of (tile, block kb), 0 past N
    auto col_scale = [&](int tile, int kb) -> float {
      const int rem = tile - (tile / (mt * nt)) * (mt * nt);
      const int col = (rem % nt) * WG_BN + et;
      return (et < WG_BN && col < g.N) ? __ldg(g.sb + (size_t)kb * g.N + col) : 0.f;
    };
    int c = 0;
    bool alive = true;
    bool staged = false;                  // sbuf[c & 1] already holds this block's scales
    for (int tile = blockIdx.x; alive && tile < total; tile += gridDim.x) {
      const int seg = tile / (mt * nt), rem = tile - seg * (mt * nt);
      const int m = rem / nt, n = rem - m * nt;
      const int row = m * WG_BM + q * 32 + lane;            // < M: M is a multiple of 128
      const int col0 = n * WG_BN + cq * 64;
      const bool cols_ok = col0 < g.N;                        // N is a multiple of 64
      float acc[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0.f;
#pragma unroll 1
      for (int kb = C.blk[seg]; kb < C.blk[seg + 1]; ++kb, ++c) {
        const int buf = c & 1;
        if (!staged) {
          if (et < WG_BN) C.sbuf[buf][et] = col_scale(tile, kb);
          tc::mbar_arrive(&C.sfill[buf]);   // release: the store is visible after the wait
        }
        const bool filled = tc::mbar_wait(&C.sfill[buf], (c >> 1) & 1, abort_flag, g.err);
        if (!__all_sync(0xffffffffu, filled)) { alive = false; break; }
        int t2, kb2;
        next_chunk(tile, kb, t2, kb2);
        const float pf = t2 >= 0 ? col_scale(t2, kb2) : 0.f;   // in flight during the promotion
        const float sa = __ldg(g.sa + (size_t)kb * g.M + row);
        const bool got = tc::mbar_wait(&C.pfull[buf], (c >> 1) & 1, abort_flag, g.err);
        if (!__all_sync(0xffffffffu, got)) { alive = false; break; }
        tc::fence_after_sync();
        const uint32_t t_base = tmem_base + (uint32_t)(buf * WG_BN) + ((uint32_t)(q * 32) << 16) + cq * 64;
        const float* sbs = C.sbuf[buf] + cq * 64;
#pragma unroll
        for (int g0 = 0; g0 < 64; g0 += 8) {
          uint32_t pv[8];
          tc::tmem_ld8(t_base + g0, pv);
          const float4 s0 = *reinterpret_cast<const float4*>(sbs + g0);
          const float4 s1 = *reinterpret_cast<const float4*>(sbs + g0 + 4);
          tc::tmem_ld_wait();
          const float sb[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
          for (int j = 0; j < 8; j += 2)
            tc::fma2_scaled(acc[g0 + j], acc[g0 + j + 1], __uint_as_float(pv[j]), __uint_as_float(pv[j + 1]), sa,
                            sb[j], sb[j + 1]);
        }
        tc::fence_before_sync();
        tc::mbar_arrive(&C.pempty[buf]);
        // the next block's scales into the other buffer: every thread finished reading
        // it (block c - 1) before arriving on this block's sfill, which this thread
        // has waited for
        if (t2 >= 0) {
          if (et < WG_BN) C.sbuf[buf ^ 1][et] = pf;
          tc::mbar_arrive(&C.sfill[buf ^ 1]);
        }
        staged = t2 >= 0;
      }
      if (!alive) break;
      if (cols_ok) {
        // 32 rows x 64 columns as two 32 x 32 boxes: written to the warp's scratch with
        // the 128-byte swizzle, stored by TMA (mO routed experts, mOs shared ones)
        const CUtensorMap* om = seg < g.N_r ? &mO : &mOs;
        const int z = seg < g.N_r ? seg : seg - g.N_r;
        uint8_t* scr = reinterpret_cast<uint8_t*>(scr_all) + (warp - 2) * WG_SCR;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (lane == 0) tc::bulk_wait_read();   // the previous box has left the scratch
          __syncwarp();
          uint8_t* rowp = scr + lane * 128;
#pragma unroll
          for (int v = 0; v < 8; ++v)
            *reinterpret_cast<float4*>(rowp + ((v ^ (lane & 7)) << 4)) =
                make_float4(acc[32 * h + 4 * v], acc[32 * h + 4 * v + 1], acc[32 * h + 4 * v + 2], acc[32 * h + 4 * v + 3]);
          tc::fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
            tc::tma_store_3d(om, scr, col0 + 32 * h, row - lane, z);
            tc::bulk_commit();
          }
        }
      }
    }
  }

  if (warp >= 2 && lane == 0) tc::bulk_wait_all();   // this warp's output stores are done
  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // a wait that ran out may have left TMA copies in flight: give them time to land
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 10000000ull) {
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, 512);
  }
}

constexpr CUtensorMapDataType kU8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;

}  // namespace

cudaError_t launch_fp8_transpose(const uint8_t* src, const float* src_s, int E, int R, int C,
                                 uint8_t* dst, float* dst_s, int ldd, int col0, cudaStream_t st) {
  if (E == 0) return cudaSuccess;
  fp8_transpose_kernel<<<dim3(C / 64, R / 64, E), 256, 0, st>>>(src, src_s, R, C, dst, dst_s, ldd, col0);
  return cudaGetLastError();
}

cudaError_t launch_fp8_swiglu_bwd(const void* dH, const void* a, const void* c, long long rows, int I,
                                  uint8_t* ac_q, float* ac_s, void* dA, void* dC, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const long long warps = rows * (I / 128);
  fp8_swiglu_bwd_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(
      (const __nv_bfloat16*)dH, (const __nv_bfloat16*)a, (const __nv_bfloat16*)c, rows, I, ac_q, ac_s,
      (__nv_bfloat16*)dA, (__nv_bfloat16*)dC);
  return cudaGetLastError();
}

cudaError_t launch_fp8_colquant(const ColQuantSrc& src, const int32_t* expert_offset, int T, int K_r,
                                int N_r, int N_s, int C, uint8_t* q, float* scale, long long Rp,
                                cudaStream_t st) {
  const long long items_ub = (Rp / 128) * (C / CQ_COLS);
  if (items_ub == 0) return cudaSuccess;
  const int grid = (int)std::min<long long>(items_ub, 8LL * device_sm_count());   // about 6 resident per SM
  fp8_colquant_kernel<<<grid, 256, 0, st>>>(src, expert_offset, T, K_r, N_r, N_s, C, q, scale, Rp,
                                            dev_error_ptr());
  return cudaGetLastError();
}

cudaError_t launch_fp8_wgrad(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                             int M, int N, long long Rp, const int32_t* expert_offset, int T, int K_r,
                             int N_r, int N_s, float* out, float* out_s, cudaStream_t st) {
  CUtensorMap mA, mB, mO, mOs;
  const CUtensorMapDataType kF32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  if (!make_tmap_2d(&mA, kU8, qa, (uint64_t)Rp, (uint64_t)M, (uint64_t)Rp, WG_BK, WG_BM) ||
      !make_tmap_2d(&mB, kU8, qb, (uint64_t)Rp, (uint64_t)N, (uint64_t)Rp, WG_BK, WG_BN) ||
      !make_tmap_3d(&mO, kF32, out, N, M, N_r, (uint64_t)N * 4, (uint64_t)M * N * 4, 32, 32))
    return cudaErrorInvalidValue;
  if (N_s > 0) {
    if (!make_tmap_3d(&mOs, kF32, out_s, N, M, N_s, (uint64_t)N * 4, (uint64_t)M * N * 4, 32, 32))
      return cudaErrorInvalidValue;
  } else {
    mOs = mO;   // never used
  }
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    err = cudaFuncSetAttribute(fp8_wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWgSmem);
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  const long long tiles = (long long)(N_r + N_s) * (M / WG_BM) * ((N + WG_BN - 1) / WG_BN);
  const int grid = (int)std::max<long long>(1, std::min<long long>(device_sm_count(), tiles));
  WgArgs g{sa, sb, M, N, T, K_r, N_r, N_s, expert_offset, out, out_s, dev_error_ptr()};
  fp8_wgrad_kernel<<<grid, WG_THREADS, kWgSmem, st>>>(mA, mB, mO, mOs, g);
  return cudaGetLastError();
}

}  // namespace moe
