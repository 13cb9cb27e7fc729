// Grouped down-projection GEMM on the sm_103a tensor cores: tcgen05 pair MMAs over
// TMEM, fed by TMA.  y = h W_down^T over the expert segments of the FFN row space
// (DeepSeek-V3 Technical Report reading guide, Method §2: the experts' FFN terms of
// h'_t).
//
// Weights on the M side, tokens on the N side: each MMA computes a block of the
// transposed output, D^T = W H^T.  The MMA's N (tokens) goes down to 16 in steps of 16,
// so a tile is sized to the tokens it has (at most 15 padding tokens).
//
// Two CTAs on two SMs form a pair (a cluster of two) and issue M=256 MMAs together
// (cta_group::2): each CTA holds 128 of the 256 W_down rows and half of the token rows
// of a K step, and receives its 128 rows of the accumulator in its own TMEM.  A pair
// tile holds up to 512 tokens of one expert segment as two MMAs of N <= 256 that share
// each weight stage, so an expert with up to 512 tokens streams its weight slab once,
// and per K step of 64 an SM loads 16 KB of weights for up to 256 token rows.  Such a
// tile takes both 256-column TMEM slots, so the next tile's MMAs wait for its
// epilogue; the epilogue here only converts and stores, so that wait is short.
//
// Operands sit in a ring of 16 KB chunks (one 128-row x 64-K operand each): a K step
// takes three chunks (weights, tokens 0..255, tokens 256..511) for a tile of more than
// 256 tokens and two otherwise, so both kinds of tile keep the whole ring in flight.
// Each chunk has an "empty" barrier (the MMAs that read it have finished); the first
// chunk of a K step has the "full" barrier its TMA loads complete on.  Batches of at
// most 128 tokens use the same space as a plain ring of 8 stages (16 KB of weights and an
// 8 KB token box each) with tiles of up to 128 tokens.
//
// Persistent pairs (as many as fit) take the tiles of the segment schedule
// (ffn_sched.cuh: segment-major, then token tile of up to 512, then feature tile of 256)
// in order from a per-launch device counter, so the pairs running at one time always
// work on neighbouring tiles and share their token and weight tiles through L2.  Warp
// roles in each CTA:
//   warp 0      TMA producer: this CTA's weight and token rows into the chunk ring;
//               completion is counted on the even CTA's barrier.
//   warp 1      allocates 512 TMEM columns (with the peer): two 256-column slots.  In
//               the even CTA one thread issues the pair MMAs.  A tile of at most 256
//               tokens takes one slot (the slots alternate, so its epilogue overlaps the
//               next tile's MMAs); a larger tile takes both, tokens 0..255 in the slot
//               due next.
//   warps 2..5  epilogue: TMEM lane = W_down row, column = token; each warp transposes
//               32 features x 16 tokens through its own shared-memory scratch and
//               writes 16-byte pieces of token rows.
// Tokens past the end of a tile's segment are loaded (or zero-filled past the tensor
// end) but sit beyond the MMA's N or are not stored; features past d are computed from
// the next expert's rows (or zeros) and not stored.
#include "tc_ffn_common.cuh"
#include "tmap.h"

namespace moe {

namespace ffn_tc {

// Tile counters: one slot per launch, taken round-robin from kTileCounters, so that
// launches in flight at the same time (up to kTileCounters of them) count separately.
// A slot is two ints (tiles claimed, CTAs done); the last CTA of a launch zeroes both,
// so a slot is zero whenever no launch holds it.
constexpr int kTileCounters = 64;
__device__ int g_tile_ctr[2 * kTileCounters];

int* tile_counter(cudaError_t* err) {
  static std::mutex mu;
  static int* base[64] = {};
  static unsigned next_slot = 0;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) { *err = cudaErrorInvalidDevice; return nullptr; }
  std::lock_guard<std::mutex> lock(mu);
  if (base[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_tile_ctr);
    if (*err != cudaSuccess) return nullptr;
    base[dev] = static_cast<int*>(p);
  }
  return base[dev] + 2 * (next_slot++ % kTileCounters);
}

}  // namespace ffn_tc

namespace {

using namespace ffn_tc;

constexpr int HALF = 256;                       // tokens of one MMA (N <= 256)
constexpr int BT = 2 * HALF;                    // tokens of a pair tile at most
constexpr int CHUNK = 128 * BK * 2;             // one operand of a K step: 16 KB
constexpr int NCHUNK = 13;                      // operand ring: 208 KB
constexpr int TMEM_COLS = 512, SLOT_COLS = 256;
constexpr int SCRATCH = 16 * 32 * 2;            // per epilogue warp: 16 tokens x 32 rows bf16
// Small batches (at most 128 tokens, so no expert segment holds more): tiles of up to 128
// tokens, one MMA each, through a ring of stages of 16 KB of weights and an 8 KB token box
// (up to 64 rows a CTA), so that 8 K steps of weights are in flight where the chunk ring
// holds 6 (a K step there gives a whole 16 KB chunk to a box of at most 4 KB).
constexpr int S_BT = 128, S_XROWS = 64, S_STAGES = 8;
constexpr int S_STAGE = CHUNK + S_XROWS * BK * 2;

struct Ctrl {
  uint64_t full[NCHUNK], empty[NCHUNK], tfull[2], tempty[2], fin;
  uint64_t tq_full[TQ], tq_empty[TQ];
  int tq[TQ];
  uint32_t tmem_base;
  int abort_flag;
  SegTable tab;
};

constexpr size_t kSmemBytes = (size_t)NCHUNK * CHUNK + 4 * SCRATCH + sizeof(Ctrl) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
static_assert(NCHUNK <= 32, "chunk parities are kept in one 32-bit word");
static_assert(S_STAGES * S_STAGE <= NCHUNK * CHUNK && S_STAGES <= NCHUNK,
              "the small-batch ring uses the chunk ring's space and barriers");

// The MMA halves of a tile of n_tok tokens: N of each (multiples of 16; n1 = 0 when
// one MMA covers the tile).
struct TileGeo {
  int n0, n1;
  __device__ __forceinline__ explicit TileGeo(int n_tok) {
    const int n_pad = (n_tok + 15) & ~15;
    n0 = min(n_pad, HALF);
    n1 = n_pad - n0;
  }
  __device__ __forceinline__ bool wide() const { return n1 > 0; }
  __device__ __forceinline__ int chunks() const { return n1 > 0 ? 3 : 2; }
};

// Token rows one CTA loads for an MMA of N tokens, and the box that covers them.
__device__ __forceinline__ int box_rows(int n) { return (n >> 1) <= SMALL_ROWS ? SMALL_ROWS : 128; }

// TMEM slots of a tile: a tile of <= 256 tokens takes slot `toggle` and flips it; a
// wider one takes `toggle` for tokens 0..255 and the other slot for the rest.  The MMA
// issuer and the epilogue walk the same tile sequence, so they agree on the slots.
struct Slots {
  int toggle = 0;
  uint32_t uses = 0;   // bit s: parity of the tiles that used slot s so far
  __device__ __forceinline__ void take(bool wide, int& s0, int& s1) {
    s0 = toggle;
    s1 = toggle ^ 1;
    if (!wide) toggle ^= 1;
  }
  __device__ __forceinline__ uint32_t parity(int s) const { return (uses >> s) & 1u; }
  __device__ __forceinline__ void used(int s) { uses ^= 1u << s; }
};

__device__ __forceinline__ int ring_next(int c, int by) {
  c += by;
  return c >= NCHUNK ? c - NCHUNK : c;
}

template <bool SMALL>
__global__ void __launch_bounds__(THREADS, 1)
    tc_down_kernel(const __grid_constant__ CUtensorMap mX_r, const __grid_constant__ CUtensorMap mX_s,
                  const __grid_constant__ CUtensorMap mW0_r, const __grid_constant__ CUtensorMap mW1_r,
                  const __grid_constant__ CUtensorMap mW0_s, const __grid_constant__ CUtensorMap mW1_s,
                  const __grid_constant__ CUtensorMap mXs_r, const __grid_constant__ CUtensorMap mXs_s,
                  TcArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_off = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_off & 1023u)) & 1023u);
  uint8_t* scratch = base + NCHUNK * CHUNK;
  Ctrl& C = *reinterpret_cast<Ctrl*>(scratch + 4 * SCRATCH);

  const FfnShape s = args.s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_rank();
  const bool leader = rank == 0;
  const int K = s.I;
  const int N = s.d;                              // output width
  const int n_ft = (N + 256 - 1) / 256;         // feature tiles per expert
  const int nk = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NCHUNK; ++i) {
      tc::mbar_init(&C.full[i], 1);
      tc::mbar_init(&C.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&C.tfull[i], 1);
      tc::mbar_init(&C.tempty[i], 8);      // one arrival per epilogue warp of both CTAs
    }
    for (int i = 0; i < TQ; ++i) {
      tc::mbar_init(&C.tq_full[i], 1);
      // readers of a tile index: the even CTA's MMA thread, the four epilogue warps of
      // each CTA and the odd CTA's producer
      tc::mbar_init(&C.tq_empty[i], 10);
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

  if (warp == 0 && SMALL) {
    if (lane == 0) {
      // ---------------------------------------------- producer, small batches --
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
        const int half = ((tcd.n_tok + 15) & ~15) >> 1;   // token rows a CTA: <= 64
        const bool sm = half <= SMALL_ROWS;
        const CUtensorMap* mXb = sm ? &mXs_r : &mX_r;     // 32-row or 64-row boxes
        const uint32_t stage_tx = (uint32_t)(CHUNK + (sm ? SMALL_ROWS : S_XROWS) * BK * 2);
        const int x_row = tcd.out_row0 + tcd.tok0 + (int)rank * half;
        const CUtensorMap* mW0 = shared ? &mW0_s : &mW0_r;
        const int w_row = e * N + tcd.n * 256 + (int)rank * (256 / 2);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % S_STAGES;
          const uint32_t ph = (it / S_STAGES) & 1;
          if (!tc::mbar_wait(&C.empty[st], ph ^ 1, abort_flag, args.err)) { ok = false; break; }
          const uint32_t bar = tc::cluster_addr(&C.full[st], 0);   // the even CTA's barrier
          if (leader) tc::mbar_arrive_expect_tx(&C.full[st], 2 * stage_tx);
          uint8_t* sa = base + st * S_STAGE;
          tc::tma_load_2d_pair(sa, mW0, bar, kb * BK, w_row);            // 128 down rows
          tc::tma_load_2d_pair(sa + CHUNK, mXb, bar, kb * BK, x_row);
        }
        if (!ok) break;
        tile = leader ? next : next_tile(k + 1);
      }
    }
  } else if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer --
      int ptr = 0;
      uint32_t chunk_uses = 0;                          // bit c: parity of chunk c's uses
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
        const TileGeo g(tcd.n_tok);
        const bool shared = tcd.seg >= s.N_r;
        const int e = shared ? tcd.seg - s.N_r : tcd.seg;
        const bool sm0 = box_rows(g.n0) == SMALL_ROWS, sm1 = box_rows(g.n1) == SMALL_ROWS;
        const CUtensorMap* mXb = &mX_r;                                    // 128-row boxes
        const CUtensorMap* mXsm = &mXs_r;                                  // 32-row boxes
        const uint32_t stage_tx = (uint32_t)(CHUNK + box_rows(g.n0) * BK * 2 +
                                             (g.wide() ? box_rows(g.n1) * BK * 2 : 0));
        const int x_base = tcd.out_row0 + tcd.tok0;                       // h rows
        const int x_row0 = x_base + (int)rank * (g.n0 >> 1);
        const int x_row1 = x_base + HALF + (int)rank * (g.n1 >> 1);
        const CUtensorMap* mW0 = shared ? &mW0_s : &mW0_r;
        const int w_row = e * N + tcd.n * 256 + (int)rank * (256 / 2);
        const int nch = g.chunks();
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          int c[3];
          for (int j = 0; j < nch; ++j) {
            c[j] = ring_next(ptr, j);
            if (!tc::mbar_wait(&C.empty[c[j]], ((chunk_uses >> c[j]) & 1u) ^ 1u, abort_flag,
                               args.err)) {
              ok = false;
              break;
            }
          }
          if (!ok) break;
          const uint32_t bar = tc::cluster_addr(&C.full[c[0]], 0);   // the even CTA's barrier
          if (leader) tc::mbar_arrive_expect_tx(&C.full[c[0]], 2 * stage_tx);
          uint8_t* A = base + c[0] * CHUNK;
          tc::tma_load_2d_pair(A, mW0, bar, kb * BK, w_row);                 // 128 down rows
          tc::tma_load_2d_pair(base + c[1] * CHUNK, sm0 ? mXsm : mXb, bar, kb * BK, x_row0);
          if (g.wide())
            tc::tma_load_2d_pair(base + c[2] * CHUNK, sm1 ? mXsm : mXb, bar, kb * BK, x_row1);
          for (int j = 0; j < nch; ++j) chunk_uses ^= 1u << c[j];
          ptr = ring_next(ptr, nch);
        }
        if (!ok) break;
        tile = leader ? next : next_tile(k + 1);
      }
    }
  } else if (warp == 1 && SMALL) {
    if (lane == 0 && leader) {
      // -------------------------------------------- MMA issuer, small batches --
      int it = 0;
      Slots sl;
      for (int tcount = 0;; ++tcount) {
        const int tile = next_tile(tcount);
        if (tile < 0 || *abort_flag) break;
        release_tile(tcount);
        const TileCoord tcd = decode_tile(C.tab, tile, n_ft);
        int s0, s1;
        sl.take(false, s0, s1);
        if (!tc::mbar_wait(&C.tempty[s0], sl.parity(s0) ^ 1u, abort_flag, args.err)) break;
        tc::fence_after_sync();
        const uint32_t d0 = tmem_base + (uint32_t)(s0 * SLOT_COLS);
        const uint32_t idesc0 = tc::idesc_bf16(256, (tcd.n_tok + 15) & ~15);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % S_STAGES;
          if (!tc::mbar_wait(&C.full[st], (it / S_STAGES) & 1, abort_flag, args.err)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint64_t a = tc::sdesc_sw128(tc::smem_u32(base + st * S_STAGE));
          const uint64_t b0 = tc::sdesc_sw128(tc::smem_u32(base + st * S_STAGE + CHUNK));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_bf16_pair(d0, a + 2 * kk, b0 + 2 * kk, idesc0, (kb | kk) != 0);
          tc::mma_commit_pair(&C.empty[st]);
        }
        if (!ok) break;
        tc::mma_commit_pair(&C.tfull[s0]);
        sl.used(s0);
      }
      // every pair MMA has finished once `fin` flips (in both CTAs)
      tc::mma_commit_pair(&C.fin);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer --
      int ptr = 0;
      uint32_t starts = 0;                // bit c: parity of the K steps that began at chunk c
      Slots sl;
      for (int tcount = 0;; ++tcount) {
        const int tile = next_tile(tcount);
        if (tile < 0 || *abort_flag) break;
        release_tile(tcount);
        const TileCoord tcd = decode_tile(C.tab, tile, n_ft);
        const TileGeo g(tcd.n_tok);
        int s0, s1;
        sl.take(g.wide(), s0, s1);
        if (!tc::mbar_wait(&C.tempty[s0], sl.parity(s0) ^ 1u, abort_flag, args.err)) break;
        tc::fence_after_sync();
        const uint32_t d0 = tmem_base + (uint32_t)(s0 * SLOT_COLS);
        const uint32_t d1 = tmem_base + (uint32_t)(s1 * SLOT_COLS);
        const uint32_t idesc0 = tc::idesc_bf16(256, g.n0);
        const uint32_t idesc1 = tc::idesc_bf16(256, g.wide() ? g.n1 : 16);
        const int nch = g.chunks();
        bool ok = true, have_s1 = !g.wide();
        for (int kb = 0; kb < nk; ++kb) {
          const int c0 = ptr, c1 = ring_next(ptr, 1), c2 = ring_next(ptr, 2);
          if (!tc::mbar_wait(&C.full[c0], (starts >> c0) & 1u, abort_flag, args.err)) {
            ok = false;
            break;
          }
          starts ^= 1u << c0;
          tc::fence_after_sync();
          const uint64_t a = tc::sdesc_sw128(tc::smem_u32(base + c0 * CHUNK));
          const uint64_t b0 = tc::sdesc_sw128(tc::smem_u32(base + c1 * CHUNK));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_bf16_pair(d0, a + 2 * kk, b0 + 2 * kk, idesc0, (kb | kk) != 0);
          if (g.wide()) {
            if (!have_s1) {   // tokens 256.. go to the other slot once its epilogue is done
              if (!tc::mbar_wait(&C.tempty[s1], sl.parity(s1) ^ 1u, abort_flag, args.err)) {
                ok = false;
                break;
              }
              tc::fence_after_sync();
              have_s1 = true;
            }
            const uint64_t b1 = tc::sdesc_sw128(tc::smem_u32(base + c2 * CHUNK));
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              tc::mma_bf16_pair(d1, a + 2 * kk, b1 + 2 * kk, idesc1, (kb | kk) != 0);
          }
          tc::mma_commit_pair(&C.empty[c0]);
          tc::mma_commit_pair(&C.empty[c1]);
          if (g.wide()) tc::mma_commit_pair(&C.empty[c2]);
          ptr = ring_next(ptr, nch);
        }
        if (!ok) break;
        tc::mma_commit_pair(&C.tfull[s0]);
        sl.used(s0);
        if (g.wide()) {
          tc::mma_commit_pair(&C.tfull[s1]);
          sl.used(s1);
        }
      }
      // every pair MMA has finished once `fin` flips (in both CTAs)
      tc::mma_commit_pair(&C.fin);
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int q = warp & 3;   // TMEM lane quarter this warp can access
    __nv_bfloat16* scr = reinterpret_cast<__nv_bfloat16*>(scratch + q * SCRATCH);
    Slots sl;
    bool alive = true;
    for (int tcount = 0; alive; ++tcount) {
      // warp-uniform decisions: the TMEM loads below are warp-collective
      const int tile = __shfl_sync(0xffffffffu, next_tile(tcount), 0);
      if (tile < 0 || __shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      __syncwarp();
      if (lane == 0) release_tile(tcount);
      const TileCoord tcd = decode_tile(C.tab, tile, n_ft);
      const int n_tok = tcd.n_tok;
      const TileGeo g(n_tok);
      int s0, s1;
      sl.take(g.wide(), s0, s1);
      const size_t row0 = (size_t)tcd.out_row0 + (size_t)tcd.tok0;
      for (int h = 0; h < (g.wide() ? 2 : 1); ++h) {
        const int slot = h ? s1 : s0;
        const bool got = tc::mbar_wait(&C.tfull[slot], sl.parity(slot), abort_flag, args.err);
        if (!__all_sync(0xffffffffu, got)) { alive = false; break; }
        tc::fence_after_sync();
        const uint32_t t_base =
            tmem_base + (uint32_t)(slot * SLOT_COLS) + ((uint32_t)(q * 32) << 16);
        const int tok_begin = h * HALF;
        const int n_here = min(n_tok - tok_begin, HALF);
        {
          const int f0 = tcd.n * 256 + (int)rank * 128 + q * 32;
#pragma unroll 1
          for (int j0 = 0; j0 < n_here; j0 += 16) {
            uint32_t a[16];
            float v[16];
            tc::tmem_ld16(t_base + j0, a);
            tc::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(a[j]);
            store_transposed(scr, v, lane, args.out, row0 + tok_begin, j0, n_here, f0, N);
          }
        }
        // the slot's columns are in registers: the MMA may overwrite them
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_cluster_relaxed(tc::cluster_addr(&C.tempty[slot], 0));
        sl.used(slot);
      }
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

cudaError_t launch_ffn_down_tc(const FfnShape& s, const void* h, const int32_t* expert_offset,
                               const moe_expert_weights* w, void* y, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  CUtensorMap m[8];
  const uint64_t rb = (uint64_t)s.I * 2;
  const uint64_t rows = (uint64_t)s.T * s.K_r + (uint64_t)s.N_s * s.T;
  // h: 128-row boxes (a CTA's half of a 256-token MMA) and 32-row boxes (MMAs of <= 64
  // tokens); W_down: 128-row boxes
  // small batches: the token box of a CTA is at most 64 rows (tiles of <= 128 tokens)
  const bool small = s.T <= S_BT;
  bool ok = make_tmap_2d(&m[0], kBF16, h, s.I, rows, rb, BK, small ? S_XROWS : HALF / 2) &&
            make_tmap_2d(&m[6], kBF16, h, s.I, rows, rb, BK, SMALL_ROWS) &&
            make_tmap_2d(&m[2], kBF16, w->down, s.I, (uint64_t)s.N_r * s.d, rb, BK, 128);
  if (ok && s.N_s > 0)
    ok = make_tmap_2d(&m[4], kBF16, w->s_down, s.I, (uint64_t)s.N_s * s.d, rb, BK, 128);
  else
    m[4] = m[2];
  if (!ok) return cudaErrorInvalidValue;
  m[1] = m[0];
  m[3] = m[2];
  m[5] = m[4];
  m[7] = m[6];
  const int bt = small ? S_BT : BT;
  const long long t_ub = (long long)s.T * s.K_r / bt + s.N_r + (long long)s.N_s * ((s.T + bt - 1) / bt);
  static std::mutex mu;
  static int fit[64] = {}, fit_small[64] = {};
  TcArgs a{s, expert_offset, static_cast<__nv_bfloat16*>(y), dev_error_ptr(), nullptr};
  if (small)
    return launch_pairs(tc_down_kernel<true>, fit_small, mu, kSmemBytes, t_ub * ((s.d + 255) / 256), m, a, st);
  return launch_pairs(tc_down_kernel<false>, fit, mu, kSmemBytes, t_ub * ((s.d + 255) / 256), m, a, st);
}

}  // namespace moe
