// Grouped gate/up GEMM with the SwiGLU epilogue, on the sm_103a tensor cores: tcgen05
// pair MMAs over TMEM, fed by TMA.  h = silu(x W_gate^T) * (x W_up^T) over the expert
// segments of the FFN row space (DeepSeek-V3 Technical Report reading guide, Method §2:
// the experts' FFN terms of h'_t; SwiGLU is the reading taken for the unnamed FFN).
//
// Weights on the M side, tokens on the N side: each MMA computes a block of the
// transposed output, D^T = W X^T.  The MMA's N (tokens) goes down to 16 in steps of
// 16, so the last tile of an expert's segment is sized to the tokens it has (at most
// 15 padding tokens), where a token-major M tile would pad up to 127 rows.
//
// Two CTAs on two SMs form a pair (a cluster of two) and issue M=256 MMAs together
// (cta_group::2): each CTA holds 128 of the 256 weight rows (64 W_gate rows over the
// same features' 64 W_up rows) and half of the token rows of a K step, and receives its
// 128 rows of the accumulator in its own TMEM.  Per SM a K step of 64 moves 32 KB
// (16 KB of weights, 16 KB of tokens) for 128 x 256 x 64 MACs.
//
// Tiles hold at most 256 tokens, so the two 256-column TMEM accumulators alternate and
// the SwiGLU epilogue of tile i (two special-function operations per element) overlaps
// the MMAs of tile i+1.  A wider tile would have to take both accumulators and stall the
// next tile's MMAs behind its epilogue.
//
// Persistent pairs (as many as fit) take the tiles of the segment schedule
// (ffn_sched.cuh: segment-major, then token tile of up to 256, then feature tile of 128)
// in order from a per-launch device counter, so the pairs running at one time always
// work on neighbouring tiles and share their token and weight tiles through L2.  Warp
// roles in each CTA:
//   warp 0      TMA producer: this CTA's weight and token rows into a 6-stage ring
//               (32 KB per stage; for batches of at most 128 tokens, tiles of up to 128
//               tokens and 8 stages of 24 KB); completion is counted on the even CTA's
//               barrier.
//   warp 1      allocates 512 TMEM columns (with the peer); in the even CTA one thread
//               issues the pair MMAs into one of two 256-column accumulators.
//   warps 2..5  epilogue: TMEM lanes 0..63 hold gate and lanes 64..127 up of the same
//               64 features; per 16 tokens the four warps stage their raw values in
//               shared memory and each thread forms 8 features of h for one token and
//               writes them as 16 bytes.
// Tokens past the end of a tile's segment are loaded (or zero-filled past the tensor
// end) but sit beyond the MMA's N or are not stored; features past I are computed from
// the next expert's rows (or zeros) and not stored.
//
// GATHER variant (moe_expert_gate_up_gather): a routed tile's token rows come straight
// from u at the rows perm_token gives, copied by the 128 lanes of warps 0 and 6..8 with
// cp.async into the same swizzled layout; each CTA counts its lanes' copies of a stage
// on a gfull barrier, the even CTA's MMA thread waits on its own, and the odd CTA's idle
// MMA warp relays its CTA's to the even CTA's full barrier.  A generic-to-async proxy
// fence precedes the MMAs' reads.  h is bit-identical to the x_perm path's; the kernel
// ran about 2.5 times longer (a stage's round trip through the copies, the barriers and
// the relay is longer than the six-stage ring covers), so the layer keeps x_perm by
// default.
#include "tc_ffn_common.cuh"
#include "tmap.h"

namespace moe {

namespace {

using namespace ffn_tc;

constexpr int STAGES = 6, BT = 256;
// gathering from u: warp 0 and warps 6..8 copy the routed token rows (128 lanes)
constexpr int GWARPS = 4, GTHREADS = THREADS + 32 * (GWARPS - 1);
constexpr int A_BYTES = 128 * BK * 2;           // this CTA's 128 weight rows
constexpr int B_BYTES = (BT / 2) * BK * 2;      // this CTA's half of the token rows
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 32 KB
// Small batches (at most 128 tokens): tiles of up to 128 tokens and stages of 16 KB of
// weights and an 8 KB token box (up to 64 rows a CTA), 8 of them in the same space, so
// that 8 K steps of weights are in flight instead of 6.
constexpr int S_BT = 128, S_XROWS = 64, S_STAGES = 8;
constexpr int S_STAGE_BYTES = A_BYTES + S_XROWS * BK * 2;   // 24 KB
static_assert(S_STAGES * S_STAGE_BYTES <= STAGES * STAGE_BYTES, "small-batch ring in the same space");
constexpr int TMEM_COLS = 512, ACC_COLS = 256;
constexpr int XCH = 2 * 16 * 128 * 4;           // raw values [2 buffers][16 tokens][128 rows]

struct Ctrl {
  uint64_t full[S_STAGES], empty[S_STAGES], tfull[2], tempty[2], xfull[2], xempty[2], fin;
  uint64_t gfull[S_STAGES];   // token rows gathered from u: the gather lanes' copies done
  uint64_t tq_full[TQ], tq_empty[TQ];
  int tq[TQ];
  uint32_t tmem_base;
  int abort_flag;
  SegTable tab;
};

constexpr size_t kSmemBytes = (size_t)STAGES * STAGE_BYTES + XCH + sizeof(Ctrl) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

template <bool GATHER, bool SMALL>
__global__ void __launch_bounds__(GATHER ? GTHREADS : THREADS, 1)
    tc_gate_up_kernel(const __grid_constant__ CUtensorMap mX_r, const __grid_constant__ CUtensorMap mX_s,
                  const __grid_constant__ CUtensorMap mW0_r, const __grid_constant__ CUtensorMap mW1_r,
                  const __grid_constant__ CUtensorMap mW0_s, const __grid_constant__ CUtensorMap mW1_s,
                  const __grid_constant__ CUtensorMap mXs_r, const __grid_constant__ CUtensorMap mXs_s,
                  TcArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_off = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_off & 1023u)) & 1023u);
  float* xch = reinterpret_cast<float*>(base + STAGES * STAGE_BYTES);
  Ctrl& C = *reinterpret_cast<Ctrl*>(base + STAGES * STAGE_BYTES + XCH);

  constexpr int NST = SMALL ? S_STAGES : STAGES;         // stages of the ring
  constexpr int SB = SMALL ? S_STAGE_BYTES : STAGE_BYTES;  // bytes of a stage
  const FfnShape s = args.s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_rank();
  const bool leader = rank == 0;
  const int K = s.d;
  const int N = s.I;                              // output width
  const int n_ft = (N + 128 - 1) / 128;         // feature tiles per expert
  const int nk = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      tc::mbar_init(&C.full[i], GATHER ? 2 : 1);   // gathering: and the odd CTA's relay
      tc::mbar_init(&C.empty[i], 1);
      tc::mbar_init(&C.gfull[i], 32 * GWARPS);      // the gather lanes
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&C.tfull[i], 1);
      tc::mbar_init(&C.tempty[i], 8);      // one arrival per epilogue warp of both CTAs
      tc::mbar_init(&C.xfull[i], 128);
      tc::mbar_init(&C.xempty[i], 128);
    }
    for (int i = 0; i < TQ; ++i) {
      tc::mbar_init(&C.tq_full[i], 1);
      // readers of a tile index: the even CTA's MMA thread, the four epilogue warps of
      // each CTA and the odd CTA's producer (and, gathering, the odd CTA's relay and the
      // three more gather warps of each CTA)
      tc::mbar_init(&C.tq_empty[i], GATHER ? 11 + 2 * (GWARPS - 1) : 10);
    }
    tc::mbar_init(&C.fin, 1);
    C.abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&mX_r);
    tc::tma_prefetch_desc(&mW0_r);
  }
  pdl_release();
  pdl_wait();   // before the tile counter, expert_offset and tensor memory are touched
  if (warp == 1) {
    tc::tmem_alloc_pair(&C.tmem_base, TMEM_COLS);
    tc::tmem_relinquish_pair();
  }
  build_seg_table(C.tab, args.expert_offset, s.T, s.K_r, s.N_r, s.N_s, SMALL ? S_BT : BT, n_ft, true,
                  args.err);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  tc::cluster_sync();   // both CTAs' barriers exist before any remote arrive or copy
  const uint32_t tmem_base = C.tmem_base;
  const int total = C.tab.total;
  volatile int* abort_flag = &C.abort_flag;

  // Tiles are claimed in order from a device counter by the even CTA's producer, so
  // pairs that start together work on neighbouring tiles (which share token and weight
  // tiles through L2) however long their earlier tiles took.  The claimed index goes
  // to every role of both CTAs through the TQ-slot ring tq; -1 ends the run.
  auto next_tile = [&](int k) -> int {          // a reader's k-th tile index
    const int slot = k % TQ;
    const bool got = tc::mbar_wait(&C.tq_full[slot], (k / TQ) & 1, abort_flag, args.err);
    const int t = got ? *reinterpret_cast<volatile int*>(&C.tq[slot]) : -1;
    return t;
  };
  auto release_tile = [&](int k) {              // done reading slot k % TQ (value in hand)
    tc::mbar_arrive_cluster_relaxed(tc::cluster_addr(&C.tq_empty[k % TQ], 0));
  };
  auto claim_tile = [&](int k) -> int {         // even CTA's producer: publish tile k
    const int slot = k % TQ;
    if (!tc::mbar_wait(&C.tq_empty[slot], ((k / TQ) & 1) ^ 1, abort_flag, args.err)) return -2;
    int t = atomicAdd(args.tile_ctr, 1);
    if (t >= total) t = -1;
    C.tq[slot] = t;
    tc::st_cluster_s32(tc::cluster_addr(&C.tq[slot], 1), t);
    tc::mbar_arrive(&C.tq_full[slot]);
    tc::mbar_arrive_cluster(tc::cluster_addr(&C.tq_full[slot], 1));
    return t;
  };

  if (GATHER && (warp == 0 || warp >= 6)) {
    // -------------------------------------------- producer, rows gathered from u --
    // Warp 0's lane 0 claims tiles (even CTA) and issues the weights' TMA copies (and,
    // for a shared expert's tile, the token rows' copy: those rows are consecutive rows
    // of u).  For a routed tile the 128 lanes of warps 0 and 6..8 copy 16-byte pieces of
    // this CTA's token rows of the K step from u, at the rows perm gives, into the
    // 128-byte-swizzled layout the MMA reads: gather lane g takes piece g & 7 of rows
    // (g >> 3) + 16i.  Each lane's copies of a stage are counted on the stage's gfull
    // barrier.
    constexpr unsigned FULLM = 0xffffffffu;
    const bool claimer = warp == 0 && leader;
    const int gl = (warp == 0 ? 0 : warp - 5) * 32 + lane;
    int it = 0;
    int tile = 0;
    if (lane == 0) tile = claimer ? claim_tile(0) : next_tile(0);
    tile = __shfl_sync(FULLM, tile, 0);
    const int chunk = gl & 7;
    for (int k = 0; tile >= 0; ++k) {
      if (__shfl_sync(FULLM, *abort_flag, 0)) break;
      int next = -1;
      if (lane == 0) {
        if (claimer) next = claim_tile(k + 1);            // one tile ahead of the loads
        else release_tile(k);
      }
      next = __shfl_sync(FULLM, next, 0);
      if (claimer && next == -2) break;
      const TileCoord tcd = decode_tile(C.tab, tile, n_ft);
      const bool shared = tcd.seg >= s.N_r;
      const int e = shared ? tcd.seg - s.N_r : tcd.seg;
      const int n_tok = tcd.n_tok;
      const int half = ((n_tok + 15) & ~15) >> 1;     // token rows per CTA
      const bool small = half <= SMALL_ROWS;
      const CUtensorMap* mX = small ? &mXs_s : &mX_s;
      const uint32_t stage_tx =
          (uint32_t)A_BYTES + (shared ? (uint32_t)((small ? SMALL_ROWS : BT / 2) * BK * 2) : 0u);
      const int x_row = tcd.tok0 + (int)rank * half;   // the CTA's first row within the segment
      const CUtensorMap* mW0 = shared ? &mW0_s : &mW0_r;
      const CUtensorMap* mW1 = shared ? &mW1_s : &mW1_r;
      const int w_row = e * N + tcd.n * 128 + (int)rank * (128 / 2);
      // this lane's rows: the token (-1: zero-filled, past the tile's tokens; -2: not
      // copied, past the CTA's half of the MMA)
      int tokr[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rho = (gl >> 3) + 16 * i;
        int t = -2;
        if (!shared && rho < half) {
          t = -1;
          if ((int)rank * half + rho < n_tok) {
            t = __ldg(args.perm + tcd.row0 + x_row + rho);
            if (t < 0 || t >= s.T) {                    // not a token: report, copy zeros
              record_error(args.err, MOE_ERR_INVALID_ARG);
              t = -1;
            }
          }
        }
        tokr[i] = t;
      }
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int st = it % NST;
        const uint32_t ph = (it / NST) & 1;
        const bool got = tc::mbar_wait(&C.empty[st], ph ^ 1, abort_flag, args.err);
        if (!__all_sync(FULLM, got)) { ok = false; break; }
        uint8_t* sa = base + st * SB;
        if (warp == 0 && lane == 0) {
          const uint32_t bar = tc::cluster_addr(&C.full[st], 0);   // the even CTA's barrier
          if (leader) tc::mbar_arrive_expect_tx(&C.full[st], 2 * stage_tx);
          tc::tma_load_2d_pair(sa, mW0, bar, kb * BK, w_row);                 // 64 gate rows
          tc::tma_load_2d_pair(sa + A_BYTES / 2, mW1, bar, kb * BK, w_row);   // 64 up rows
          if (shared) tc::tma_load_2d_pair(sa + A_BYTES, mX, bar, kb * BK, x_row);
        }
        if (!shared) {
          const uint32_t sb = tc::smem_u32(sa + A_BYTES);
          const int col = kb * BK + chunk * 8;           // d is a multiple of 8
          const bool in_row = col < s.d;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rho = (gl >> 3) + 16 * i;
            if (tokr[i] >= -1) {
              const bool copy = tokr[i] >= 0 && in_row;
              const __nv_bfloat16* src = copy ? args.u + (size_t)tokr[i] * s.d + col : args.u;
              tc::cp_async16(sb + (uint32_t)(rho * 128 + ((chunk ^ (rho & 7)) << 4)), src, copy ? 16u : 0u);
            }
          }
        }
        tc::cp_async_mbar_arrive(&C.gfull[st]);
      }
      if (!ok) break;
      if (!claimer) next = lane == 0 ? next_tile(k + 1) : 0;
      tile = __shfl_sync(FULLM, next, 0);
    }
    tc::cp_async_wait_all();
  } else if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer --
      int it = 0;
      int tile = leader ? claim_tile(0) : next_tile(0);
      for (int k = 0; tile >= 0 && !*abort_flag; ++k) {
        int next = -1;
        if (leader) {
          next = claim_tile(k + 1);                     // one tile ahead of the loads
          if (next == -2) break;
        } else {
          release_tile(k);
        }
        const TileCoord tcd = decode_tile(C.tab, tile, n_ft);
        const bool shared = tcd.seg >= s.N_r;
        const int e = shared ? tcd.seg - s.N_r : tcd.seg;
        const int n_tok = tcd.n_tok;
        const int half = ((n_tok + 15) & ~15) >> 1;     // token rows per CTA
        // a tile of <= 64 tokens loads 32-row token boxes (decode-sized batches)
        const bool small = half <= SMALL_ROWS;
        const CUtensorMap* mX = shared ? (small ? &mXs_s : &mX_s) : (small ? &mXs_r : &mX_r);
        const uint32_t stage_tx =
            (uint32_t)(A_BYTES + (small ? SMALL_ROWS : (SMALL ? S_XROWS : BT / 2)) * BK * 2);
        const int x_row = (shared ? 0 : tcd.row0) + tcd.tok0 + (int)rank * half;
        const CUtensorMap* mW0 = shared ? &mW0_s : &mW0_r;
        const CUtensorMap* mW1 = shared ? &mW1_s : &mW1_r;
        const int w_row = e * N + tcd.n * 128 + (int)rank * (128 / 2);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % NST;
          const uint32_t ph = (it / NST) & 1;
          if (!tc::mbar_wait(&C.empty[st], ph ^ 1, abort_flag, args.err)) { ok = false; break; }
          const uint32_t bar = tc::cluster_addr(&C.full[st], 0);   // the even CTA's barrier
          if (leader) tc::mbar_arrive_expect_tx(&C.full[st], 2 * stage_tx);
          uint8_t* sa = base + st * SB;
          tc::tma_load_2d_pair(sa, mW0, bar, kb * BK, w_row);                   // 64 gate rows
          tc::tma_load_2d_pair(sa + A_BYTES / 2, mW1, bar, kb * BK, w_row);     // 64 up rows
          tc::tma_load_2d_pair(sa + A_BYTES, mX, bar, kb * BK, x_row);
        }
        if (!ok) break;
        tile = leader ? next : next_tile(k + 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer --
      int it = 0, tcount = 0;
      for (;; ++tcount) {
        const int tile = next_tile(tcount);
        if (tile < 0 || *abort_flag) break;
        release_tile(tcount);
        const TileCoord tcd = decode_tile(C.tab, tile, n_ft);
        const int n_tok = tcd.n_tok;
        const uint32_t idesc = tc::idesc_bf16(256, (n_tok + 15) & ~15);
        const int acc = tcount & 1;
        const uint32_t aph = (tcount >> 1) & 1;
        if (!tc::mbar_wait(&C.tempty[acc], aph ^ 1, abort_flag, args.err)) break;
        tc::fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * ACC_COLS);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % NST;
          const uint32_t ph = (it / NST) & 1;
          if (!tc::mbar_wait(&C.full[st], ph, abort_flag, args.err)) { ok = false; break; }
          if constexpr (GATHER) {
            // this CTA's gathered rows have landed (the odd CTA's: its relay's arrival on
            // full); the generic-proxy copies are ordered before the MMA's reads
            if (!tc::mbar_wait(&C.gfull[st], ph, abort_flag, args.err)) { ok = false; break; }
            tc::fence_proxy_async_shared();
          }
          tc::fence_after_sync();
          const uint32_t s0 = tc::smem_u32(base + st * SB);
          const uint64_t a = tc::sdesc_sw128(s0), b = tc::sdesc_sw128(s0 + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_bf16_pair(d_tmem, a + 2 * kk, b + 2 * kk, idesc, (kb | kk) != 0);
          tc::mma_commit_pair(&C.empty[st]);
        }
        if (!ok) break;
        tc::mma_commit_pair(&C.tfull[acc]);
      }
      // every pair MMA has finished once `fin` flips (in both CTAs)
      tc::mma_commit_pair(&C.fin);
    } else if (GATHER && lane == 0) {
      // ------------------------------------------- relay (odd CTA, gathering) --
      // Once this CTA's gather lanes' copies of a stage have landed, order them before
      // the pair MMA's reads and arrive on the even CTA's full barrier of the stage.
      int it = 0;
      bool ok = true;
      for (int tcount = 0; ok; ++tcount) {
        const int tile = next_tile(tcount);
        if (tile < 0 || *abort_flag) break;
        release_tile(tcount);
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % NST;
          if (!tc::mbar_wait(&C.gfull[st], (it / NST) & 1, abort_flag, args.err)) { ok = false; break; }
          tc::fence_proxy_async_shared();
          tc::mbar_arrive_cluster(tc::cluster_addr(&C.full[st], 0));
        }
      }
    }
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------ epilogue --
    const int q = warp & 3;   // TMEM lane quarter this warp can access
    const uint32_t tempty0 = tc::cluster_addr(&C.tempty[0], 0);
    const uint32_t tempty1 = tc::cluster_addr(&C.tempty[1], 0);
    int tcount = 0, cc = 0;
    for (;; ++tcount) {
      // warp-uniform decisions: the TMEM loads below are warp-collective
      const int tile = __shfl_sync(0xffffffffu, next_tile(tcount), 0);
      if (tile < 0 || __shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      __syncwarp();
      if (lane == 0) release_tile(tcount);
      const TileCoord tcd = decode_tile(C.tab, tile, n_ft);
      const int n_tok = tcd.n_tok;
      const int acc = tcount & 1;
      const uint32_t aph = (tcount >> 1) & 1;
      const bool got = tc::mbar_wait(&C.tfull[acc], aph, abort_flag, args.err);
      if (!__all_sync(0xffffffffu, got)) break;
      tc::fence_after_sync();
      const uint32_t t_base = tmem_base + (uint32_t)(acc * ACC_COLS) + ((uint32_t)(q * 32) << 16);
      const size_t row0 = (size_t)tcd.out_row0 + (size_t)tcd.tok0;
      bool alive = true;
      {
        // lanes 0..63: gate rows, 64..127: up rows of the same 64 features.  Per 16
        // tokens all four warps put their raw values in shared memory, then each
        // thread forms 8 features of h for one token and writes them as 16 bytes.
        const int t = q * 32 + lane;                 // this thread's piece: token t/8,
        const int tok = t >> 3, piece = t & 7;       // features 8*piece .. 8*piece+7
        const int f = tcd.n * 128 + (int)rank * 64 + piece * 8;
#pragma unroll 1
        for (int j0 = 0; j0 < n_tok; j0 += 16, ++cc) {
          const int xb = cc & 1;
          const uint32_t xph = (cc >> 1) & 1;
          float* S = xch + xb * (16 * 128);                   // [16 tokens][128 rows]
          uint32_t a[16];
          tc::tmem_ld16(t_base + j0, a);
          tc::tmem_ld_wait();
          bool ok = tc::mbar_wait(&C.xempty[xb], xph ^ 1, abort_flag, args.err);
          if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
#pragma unroll
          for (int j = 0; j < 16; ++j) S[j * 128 + q * 32 + lane] = __uint_as_float(a[j]);
          tc::mbar_arrive(&C.xfull[xb]);   // release: the stores are visible after the wait
          ok = tc::mbar_wait(&C.xfull[xb], xph, abort_flag, args.err);
          if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
          const float4* g4 = reinterpret_cast<const float4*>(S + tok * 128 + piece * 8);
          const float4* u4 = reinterpret_cast<const float4*>(S + tok * 128 + 64 + piece * 8);
          const float4 g0 = g4[0], g1 = g4[1], u0 = u4[0], u1 = u4[1];
          tc::mbar_arrive(&C.xempty[xb]);
          if (j0 + tok < n_tok && f < N) {
            const uint4 hv = make_uint4(pack_bf16(swiglu(g0.x, u0.x), swiglu(g0.y, u0.y)),
                                        pack_bf16(swiglu(g0.z, u0.z), swiglu(g0.w, u0.w)),
                                        pack_bf16(swiglu(g1.x, u1.x), swiglu(g1.y, u1.y)),
                                        pack_bf16(swiglu(g1.z, u1.z), swiglu(g1.w, u1.w)));
            *reinterpret_cast<uint4*>(args.out + (row0 + j0 + tok) * N + f) = hv;
            if (args.save_a) {
              const size_t o = (row0 + j0 + tok) * N + f;
              *reinterpret_cast<uint4*>(args.save_a + o) =
                  make_uint4(pack_bf16(g0.x, g0.y), pack_bf16(g0.z, g0.w), pack_bf16(g1.x, g1.y),
                             pack_bf16(g1.z, g1.w));
              *reinterpret_cast<uint4*>(args.save_c + o) =
                  make_uint4(pack_bf16(u0.x, u0.y), pack_bf16(u0.z, u0.w), pack_bf16(u1.x, u1.y),
                             pack_bf16(u1.z, u1.w));
            }
          }
        }
      }
      if (!alive) break;
      tc::fence_before_sync();
      __syncwarp();
      // the accumulator's columns are in registers: the MMA may overwrite them
      if (lane == 0) tc::mbar_arrive_cluster_relaxed(acc ? tempty1 : tempty0);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // copies this CTA issued report to the even CTA's barriers: give them time to land
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 10000000ull) {
    }
  }
  if (warp == 1 && lane == 0) tc::mbar_drain(&C.fin, 0);
  __syncthreads();
  tc::cluster_sync();   // neither CTA leaves while its peer may still touch it
  if (threadIdx.x == 0) release_tile_counter(args.tile_ctr);   // the producer's claims are done
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}


constexpr CUtensorMapDataType kBF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;

}  // namespace

cudaError_t launch_ffn_up_tc(const FfnShape& s, const void* x_perm, const void* u,
                             const int32_t* expert_offset, const moe_expert_weights* w, void* h,
                             cudaStream_t st, void* save_a, void* save_c) {
  if (s.T == 0) return cudaSuccess;
  CUtensorMap m[8];
  const uint64_t rb = (uint64_t)s.d * 2;
  const uint64_t routed = (uint64_t)s.T * s.K_r;
  // tokens: 128-row boxes (a CTA's half of a 256-token tile) and 32-row boxes (tiles of
  // <= 64 tokens); weights: 64-row boxes
  // small batches: a CTA's token box is at most 64 rows (tiles of <= 128 tokens)
  const bool small_batch = s.T <= S_BT;
  const uint32_t xbox = small_batch ? S_XROWS : BT / 2;
  bool ok = make_tmap_2d(&m[0], kBF16, x_perm, s.d, routed, rb, BK, xbox) &&
            make_tmap_2d(&m[1], kBF16, u, s.d, s.T, rb, BK, xbox) &&
            make_tmap_2d(&m[6], kBF16, x_perm, s.d, routed, rb, BK, SMALL_ROWS) &&
            make_tmap_2d(&m[7], kBF16, u, s.d, s.T, rb, BK, SMALL_ROWS) &&
            make_tmap_2d(&m[2], kBF16, w->gate, s.d, (uint64_t)s.N_r * s.I, rb, BK, 64) &&
            make_tmap_2d(&m[3], kBF16, w->up, s.d, (uint64_t)s.N_r * s.I, rb, BK, 64);
  if (ok && s.N_s > 0) {
    ok = make_tmap_2d(&m[4], kBF16, w->s_gate, s.d, (uint64_t)s.N_s * s.I, rb, BK, 64) &&
         make_tmap_2d(&m[5], kBF16, w->s_up, s.d, (uint64_t)s.N_s * s.I, rb, BK, 64);
  } else {
    m[4] = m[2];
    m[5] = m[3];
  }
  if (!ok) return cudaErrorInvalidValue;
  const int bt = small_batch ? S_BT : BT;
  const long long t_ub = (long long)s.T * s.K_r / bt + s.N_r + (long long)s.N_s * ((s.T + bt - 1) / bt);
  static std::mutex mu;
  static int fit[64] = {}, fit_small[64] = {};
  TcArgs a{s, expert_offset, static_cast<__nv_bfloat16*>(h), dev_error_ptr(), nullptr,
           static_cast<__nv_bfloat16*>(save_a), static_cast<__nv_bfloat16*>(save_c)};
  if (small_batch)
    return launch_pairs(tc_gate_up_kernel<false, true>, fit_small, mu, kSmemBytes,
                        t_ub * ((s.I + 127) / 128), m, a, st);
  return launch_pairs(tc_gate_up_kernel<false, false>, fit, mu, kSmemBytes, t_ub * ((s.I + 127) / 128), m, a, st);
}

cudaError_t launch_ffn_up_tc_gather(const FfnShape& s, const void* u, const int32_t* perm_token,
                                    const int32_t* expert_offset, const moe_expert_weights* w, void* h,
                                    cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  CUtensorMap m[8];
  const uint64_t rb = (uint64_t)s.d * 2;
  // tokens of the shared experts: 128-row and 32-row boxes of u (the routed rows are
  // gathered by the kernel's lanes); weights: 64-row boxes
  bool ok = make_tmap_2d(&m[1], kBF16, u, s.d, s.T, rb, BK, BT / 2) &&
            make_tmap_2d(&m[7], kBF16, u, s.d, s.T, rb, BK, SMALL_ROWS) &&
            make_tmap_2d(&m[2], kBF16, w->gate, s.d, (uint64_t)s.N_r * s.I, rb, BK, 64) &&
            make_tmap_2d(&m[3], kBF16, w->up, s.d, (uint64_t)s.N_r * s.I, rb, BK, 64);
  if (ok && s.N_s > 0) {
    ok = make_tmap_2d(&m[4], kBF16, w->s_gate, s.d, (uint64_t)s.N_s * s.I, rb, BK, 64) &&
         make_tmap_2d(&m[5], kBF16, w->s_up, s.d, (uint64_t)s.N_s * s.I, rb, BK, 64);
  } else {
    m[4] = m[2];
    m[5] = m[3];
  }
  if (!ok) return cudaErrorInvalidValue;
  m[0] = m[1];
  m[6] = m[7];
  const long long t_ub = (long long)s.T * s.K_r / BT + s.N_r + (long long)s.N_s * ((s.T + BT - 1) / BT);
  static std::mutex mu;
  static int fit[64] = {};
  TcArgs a{s, expert_offset, static_cast<__nv_bfloat16*>(h), dev_error_ptr(), nullptr};
  a.u = static_cast<const __nv_bfloat16*>(u);
  a.perm = perm_token;
  return launch_pairs(tc_gate_up_kernel<true, false>, fit, mu, kSmemBytes, t_ub * ((s.I + 127) / 128), m, a, st,
                      GTHREADS);
}

}  // namespace moe
