// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA, for the bf16 kind.
//
// "DeepSeek-V3 Technical Report", DeepSeekMoE paragraph: each routed expert
// is an FFN applied to the tokens routed to it, and the shared experts to
// every token.  Each FFN is SwiGLU: h = silu(u W1^T) * (u W3^T), y = h W2^T.
//
// Two launches per layer, one persistent kernel each:
//   gate/up: [a | b] = A W13^T per 128 x 256 tile, h = silu(a) * b in the
//            epilogue (the tile's 256 MMA columns are 128 gate rows and the
//            128 matching up rows of W13, so a tile yields 128 h columns);
//   down:    y = h W2^T per 128 x 256 tile.
// The work list covers every (group, M tile, N tile) of the routed experts
// (segment sizes read from `offsets` in device memory) followed by the
// shared class (all T rows, intermediate N_s * I).  The CTAs run in
// clusters of two, and a cluster's unit of work is a pair of tiles that
// share one operand, loaded once from L2 and multicast into both CTAs:
//   - two M tiles of one group with the same weight (B) tile: each CTA
//     loads its own A rows and half of the B tile for both;
//   - the odd last M tile of a group with two of its N tiles: each CTA
//     loads half of the A rows for both and its own B tile;
//   - an odd last (M, N) tile, paired with an empty tile past the segment.
// Each CTA still holds whole A and B tiles and runs its own 128 x 256 MMAs;
// what the pair saves is L2 reads (a stage reads 48 KiB from L2 per CTA,
// 32 KiB when B is shared), not what each SM takes in (48 KiB a stage
// either way); experts_pair.cu's pair MMAs lower that.  Cluster c takes
// units c, c + clusters, ...; inside a group the M pair varies fastest, so
// the clusters running at the same time share each weight tile through L2.
// (The gathering gate/up GEMM keeps one tile per CTA: its A rows come from
// gather warps, not TMA.)
//
// Roles (224 threads, one CTA per SM):
//   warps 0, 6  TMA producers (even / odd stages): A and B tiles into a
//               4-stage shared-memory ring, one TMA load each per stage
//   warp 1      allocates TMEM; one thread issues tcgen05.mma (M=128, N=256,
//               K=16) into one of two 256-column fp32 accumulators
//   warps 2..5  epilogue: tcgen05.ld the accumulator (warp w reads TMEM
//               lanes 32*(w%4) .. +31), SwiGLU or copy, bf16 stores with
//               the segment's tail rows masked
// Every wait is bounded (see mbar_wait); a wait that gives up sets the
// error word and a block-wide abort flag so that all roles leave, drain
// their own copies in flight and free TMEM.
#include <algorithm>
#include <map>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace bf16gemm {

constexpr int BM = 128, BN = 256, BK = 64;  // BK * 2 bytes = one 128-byte swizzle row
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;         // 16 KiB
constexpr int B_BYTES = BN * BK * 2;         // 32 KiB
constexpr int THREADS = 224;
constexpr int PRODUCER2 = 6;                 // warp of the second producer
constexpr int GATHER_WARP0 = 7;              // gathering gate/up: warps 7..10, one per ring slot
constexpr int THREADS_GATHER = THREADS + STAGES * 32;
constexpr int MAX_GROUPS = 1025;             // 1024 routed experts + the shared class
constexpr uint32_t TMEM_COLS = 512;          // two 256-column accumulators
constexpr uint32_t IDESC = idesc_f32acc(1, 1, BM, BN);
constexpr uint16_t kPairMask = 0x3;          // both CTAs of a cluster

enum { GATEUP = 0, DOWN = 1 };
// Operand a pair unit's two tiles share.
enum { SHARE_B = 0, SHARE_A = 1 };

struct ClassDesc {
  __nv_bfloat16* out;  // output rows of the class
  int ld_out;          // output row stride, elements
  int n_out;           // output columns (h columns for gate/up, d for down)
  int k_dim;           // reduction length
  __nv_bfloat16* ab;   // gate/up, optional: [a | b] of every expert kept for the backward
  int ld_ab;           // its row stride (2I per expert of the class)
  const float* gate;   // down, optional: every output row is multiplied by gate[row]
};

struct Params {
  CUtensorMap a_map[2];   // [0] routed rows, [1] shared rows: 128-row box
  CUtensorMap b_map[2];   // [0] routed weights, [1] shared weights: whole B tile
  CUtensorMap a_half[2];  // the same A with a 64-row box (units sharing A)
  CUtensorMap b_half[2];  // the same B with a half-tile box (units sharing B)
  CUtensorMap b_mix[2];   // gate/up: 64 W1 rows then the matching 64 W3 rows (pair half tiles)
  ClassDesc cls[2];
  const int32_t* offsets;
  int n_rows;  // T * K: permuted rows, the bound of every segment
  int E;
  int T;
  int has_shared;
  int inter;  // I: intermediate size of one expert
  int d;
  // gathering gate/up only: routed A rows are x[token_of_row[r]]
  const int32_t* token_of_row;
  const __nv_bfloat16* x_rows;  // [T, d]
};

struct Smem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
  int n_groups;
  int gstart[MAX_GROUPS + 1];  // first tile of every group
  int mtiles[MAX_GROUPS];      // M tiles of every group
  int off[MAX_GROUPS];         // first row of every routed group (copy of offsets[0..E])
  int gather_tok[STAGES][BM];  // gathering gate/up: x row of each tile row, per ring slot
};

constexpr size_t kRingBytes = static_cast<size_t>(STAGES) * (A_BYTES + B_BYTES);
constexpr size_t kSmemBytes = 1024 + kRingBytes + sizeof(Smem);
static_assert(kSmemBytes <= 232448, "above the 227 KiB of shared memory a block may use");

struct Tile {
  int share;    // pair units: SHARE_B or SHARE_A
  int cls;      // 0 routed, 1 shared
  int group;    // routed expert index (cls 0)
  int row0;     // first row of the group in its class's row space
  int rows;     // valid rows of the group
  int mt, nt;   // tile coordinates inside the group
};

template <int MODE>
__device__ __forceinline__ int out_tile_cols() { return MODE == GATEUP ? BN / 2 : BN; }

template <int MODE>
__device__ __forceinline__ int n_tiles_of(const Params& p, int cls) {
  return ceil_div(p.cls[cls].n_out, out_tile_cols<MODE>());
}

// Pair units of a group of mt M tiles and nt N tiles: M pairs sharing a B
// tile, then, for an odd last M tile, N pairs sharing its A rows (an odd
// last N tile pairs with an empty tile).
__device__ __forceinline__ int pair_units(int mt, int nt) {
  return (mt / 2) * nt + (mt & 1) * ((nt + 1) / 2);
}

// Warp-cooperative build of the work table from the segment offsets:
// first work item (tile, or pair unit) of every group.
template <int MODE, bool PAIR>
__device__ void build_tile_table(const Params& p, Smem& s) {
  const int lane = threadIdx.x % 32;
  const int G = p.E + (p.has_shared ? 1 : 0);
  const int per = ceil_div(G, 32);
  const int g0 = lane * per, g1 = min(G, g0 + per);
  int sum = 0;
  for (int g = g0; g < g1; ++g) {
    int rows, cls;
    if (g < p.E) {
      int o0;
      rows = checked_segment(p.offsets, g, p.n_rows, o0);
      cls = 0;
      s.off[g] = o0;
    } else {
      rows = p.T;
      cls = 1;
    }
    const int mt = ceil_div(max(rows, 0), BM);
    s.mtiles[g] = mt;
    const int nt = n_tiles_of<MODE>(p, cls);
    sum += PAIR ? pair_units(mt, nt) : mt * nt;
  }
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  int run = incl - sum;
  for (int g = g0; g < g1; ++g) {
    s.gstart[g] = run;
    const int nt = n_tiles_of<MODE>(p, g < p.E ? 0 : 1);
    run += PAIR ? pair_units(s.mtiles[g], nt) : s.mtiles[g] * nt;
  }
  if (lane == 31) {
    s.gstart[G] = incl;
    s.n_groups = G;
    s.off[p.E] = p.offsets[p.E];
  }
}

// This CTA's tile of work item t (rank: the CTA's rank in its cluster).
template <int MODE, bool PAIR>
__device__ __forceinline__ Tile decode_tile(const Params& p, const Smem& s, int t, int rank) {
  int lo = 0, hi = s.n_groups;  // gstart[lo] <= t < gstart[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.gstart[mid] <= t) lo = mid; else hi = mid;
  }
  Tile tl;
  tl.cls = lo < p.E ? 0 : 1;
  tl.group = lo;
  const int local = t - s.gstart[lo];
  const int mt_count = s.mtiles[lo];
  tl.share = SHARE_B;
  if (!PAIR) {
    tl.mt = local % mt_count;
    tl.nt = local / mt_count;
  } else {
    const int nt_count = n_tiles_of<MODE>(p, tl.cls);
    const int pm = mt_count / 2;
    if (local < pm * nt_count) {
      tl.nt = local / pm;
      tl.mt = 2 * (local % pm) + rank;
    } else {
      const int l2 = local - pm * nt_count;
      tl.mt = mt_count - 1;
      if (2 * l2 + 1 < nt_count) {
        tl.share = SHARE_A;
        tl.nt = 2 * l2 + rank;
      } else {
        tl.nt = nt_count - 1;
        tl.mt += rank;  // the partner of an odd last tile: no rows, nothing stored
      }
    }
  }
  if (tl.cls == 0) { tl.row0 = s.off[lo]; tl.rows = s.off[lo + 1] - tl.row0; }
  else { tl.row0 = 0; tl.rows = p.T; }
  return tl;
}

template <int MODE, bool GATHER>
__global__ void __launch_bounds__(GATHER ? THREADS_GATHER : THREADS, 1)
    experts_bf16_kernel(const __grid_constant__ Params p) {
  constexpr bool PAIR = !GATHER;  // launched in clusters of two
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Smem& s = *reinterpret_cast<Smem*>(ring + kRingBytes);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  volatile int* abort_flag = &s.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      tma_prefetch_desc(&p.a_map[i]);
      tma_prefetch_desc(&p.b_map[i]);
      if (PAIR) { tma_prefetch_desc(&p.a_half[i]); tma_prefetch_desc(&p.b_half[i]); }
    }
    // a stage is full once the producer's TMA bytes have landed (in a pair,
    // also the partner's multicast half) and, when gathering, the slot's
    // gather warp has arrived; it is empty again once the MMAs of this CTA
    // and, in a pair, of the partner (whose copy of the slot the multicast
    // also writes) have read it
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&s.full[i], GATHER ? 2 : 1);
      mbar_init(&s.empty[i], PAIR ? 2 : 1);
    }
    for (int i = 0; i < 2; ++i) { mbar_init(&s.tfull[i], 1); mbar_init(&s.tempty[i], 4); }
    mbar_init(&s.done, 1);
    s.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  if (warp == 2) build_tile_table<MODE, PAIR>(p, s);
  __syncthreads();
  // both CTAs' barriers are initialised before either multicasts into the other
  if (PAIR) cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_base;
  const int total = s.gstart[s.n_groups];
  // work items: a cluster's pair units, or this CTA's tiles
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const int w_first = PAIR ? static_cast<int>(blockIdx.x) >> 1 : static_cast<int>(blockIdx.x);
  const int w_step = PAIR ? static_cast<int>(gridDim.x) >> 1 : static_cast<int>(gridDim.x);

  if (warp == 0 || warp == PRODUCER2) {
    // ----------------------------------------------------------- producers
    // Two threads fill the ring: warp 0 the even stages of the CTA's stage
    // sequence (ring slots 0 and 2), warp 6 the odd ones (slots 1 and 3).
    // A stage is two TMA loads: the A rows and the whole 256-row B tile.
    if (lane == 0) {
      const uint32_t par = warp == 0 ? 0u : 1u;
      const uint64_t pol_a = l2_policy_evict_last();
      const uint64_t pol_b = l2_policy_evict_normal();
      uint32_t g = 0;     // stages of the CTA so far
      uint32_t mine = 0;  // stages issued by this thread
      bool stop = false;
      for (int t = w_first; t < total && !stop && !*abort_flag; t += w_step) {
        const Tile tl = decode_tile<MODE, PAIR>(p, s, t, rank);
        const int nk = p.cls[tl.cls].k_dim / BK;
        const int a_row = tl.row0 + tl.mt * BM;
        const CUtensorMap* am = &p.a_map[tl.cls];
        const CUtensorMap* bm = &p.b_map[tl.cls];
        // B coordinates.  Gate/up: (k, i0, 0, matrix) in the [n][2][I][d]
        // view, i.e. 128 W1 rows and the matching 128 W3 rows.  Down:
        // (k inside the matrix, first row) in the [n * d, I] view; the shared
        // class walks K over its N_s matrices.
        int bmat = 0, bi = 0, bxk = 0, brow = 0;
        if (MODE == GATEUP) {
          const int n0 = tl.nt * (BN / 2);
          bmat = tl.cls == 0 ? tl.group : n0 / p.inter;
          bi = n0 % p.inter;
        } else {
          brow = (tl.cls == 0 ? tl.group : 0) * p.d + tl.nt * BN;
        }
        for (int kb = 0; kb < nk; ++kb, ++g) {
          if ((g & 1u) == par) {
            const int stage = static_cast<int>(par + 2 * (mine & 1u));
            const uint32_t sphase = (mine >> 1) & 1u;
            if (!mbar_wait(&s.empty[stage], sphase ^ 1u, abort_flag)) { stop = true; break; }
            uint8_t* sa = ring + stage * A_BYTES;
            uint8_t* sb = ring + STAGES * A_BYTES + stage * B_BYTES;
            // gathering: the routed A rows come from the slot's gather warp
            const bool a_by_tma = !GATHER || tl.cls != 0;
            mbar_arrive_expect_tx(&s.full[stage], (a_by_tma ? A_BYTES : 0) + B_BYTES);
            if (PAIR && tl.share == SHARE_B) {
              // own A rows; this CTA's half of the common B tile, for both
              // (gate/up: W1 rows from rank 0, the matching W3 rows from
              // rank 1; down: the first or the second 128 rows)
              tma_load_2d(sa, am, &s.full[stage], kb * BK, a_row, pol_a);
              uint8_t* sbh = sb + rank * (B_BYTES / 2);
              const CUtensorMap* bh = &p.b_half[tl.cls];
              if (MODE == GATEUP)
                tma_load_4d_mc(sbh, bh, &s.full[stage], kb * BK, bi, rank, bmat, kPairMask, pol_b);
              else
                tma_load_2d_mc(sbh, bh, &s.full[stage], bxk, brow + rank * (BN / 2), kPairMask, pol_b);
            } else if (PAIR) {
              // this CTA's half of the common A rows, for both; own B tile
              tma_load_2d_mc(sa + rank * (A_BYTES / 2), &p.a_half[tl.cls], &s.full[stage], kb * BK,
                             a_row + rank * (BM / 2), kPairMask, pol_a);
              if (MODE == GATEUP) tma_load_4d(sb, bm, &s.full[stage], kb * BK, bi, 0, bmat, pol_b);
              else tma_load_2d(sb, bm, &s.full[stage], bxk, brow, pol_b);
            } else {
              if (MODE == GATEUP) tma_load_4d(sb, bm, &s.full[stage], kb * BK, bi, 0, bmat, pol_b);
              else tma_load_2d(sb, bm, &s.full[stage], bxk, brow, pol_b);
              if (a_by_tma) tma_load_2d(sa, am, &s.full[stage], kb * BK, a_row, pol_a);
            }
            ++mine;
          }
          if (MODE == DOWN) {
            bxk += BK;
            if (bxk == p.inter) { bxk = 0; brow += p.d; }
          }
        }
      }
      // Drain: wait until this thread's last loads (one per slot) have landed.
      for (uint32_t i = 0; i < 2 && i < mine; ++i) {
        const uint32_t j = mine - 1 - i;
        mbar_wait_drain(&s.full[par + 2 * (j & 1u)], (j >> 1) & 1u);
      }
    }
  } else if (GATHER && warp >= GATHER_WARP0) {
    // ------------------------------------------------------- gather warps
    // Warp GATHER_WARP0 + j fills the A rows of ring slot j (stages
    // j, j + 4, ...) for routed tiles: row r of the tile is row
    // token_of_row[segment row] of x (kept per tile in a warp-private
    // shared table), copied in 16-byte pieces with cp.async, eight lanes
    // per 128-byte row, into the 128-byte-swizzled layout the MMA
    // descriptors read (the layout TMA writes).  Each lane waits for its own copies, makes
    // them visible to the async proxy, and lane 0 arrives on the slot's
    // full barrier.  Rows past the segment are not written (their MMA rows
    // are never stored).
    const int slot = warp - GATHER_WARP0;
    const uint64_t pol_x = l2_policy_evict_last();
    int* rowsrc = s.gather_tok[slot];  // x row of each tile row (-1: none)
    const int rsub = lane >> 3, c = lane & 7;  // 8 lanes cover one 128-byte row
    uint32_t g = 0;  // stages of the CTA so far
    bool stop = false;
    for (int t = w_first; t < total && !stop && !*abort_flag; t += w_step) {
      const Tile tl = decode_tile<MODE, PAIR>(p, s, t, rank);
      const int nk = p.cls[tl.cls].k_dim / BK;
      const bool routed = tl.cls == 0;
      if (routed) {
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = lane + 32 * j, m = tl.mt * BM + r;
          int tok = -1;
          if (m < tl.rows) {
            tok = p.token_of_row[tl.row0 + m];
            if (tok < 0 || tok >= p.T) { raise_error(kErrIndex); tok = -1; }
          }
          rowsrc[r] = tok;
        }
        __syncwarp();
      }
      for (int kb = 0; kb < nk; ++kb, ++g) {
        if (static_cast<int>(g & 3u) != slot) continue;
        if (!mbar_wait(&s.empty[slot], ((g >> 2) & 1u) ^ 1u, abort_flag)) { stop = true; break; }
        if (routed) {
          const uint32_t sa = smem_u32(ring + slot * A_BYTES);
          const __nv_bfloat16* xk = p.x_rows + kb * BK + c * 8;
#pragma unroll 8
          for (int j = 0; j < BM / 4; ++j) {
            const int r = 4 * j + rsub;
            const int tok = rowsrc[r];
            if (tok >= 0) cp_async_16(sa + sw128_offset(r, c), xk + static_cast<size_t>(tok) * p.d, pol_x);
          }
          cp_async_wait_all();
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.full[slot]);
      }
    }
    cp_async_wait_all();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int it = 0;
      bool any = false;
      for (int t = w_first; t < total && !*abort_flag; t += w_step, ++it) {
        const Tile tl = decode_tile<MODE, PAIR>(p, s, t, rank);
        const int nk = p.cls[tl.cls].k_dim / BK;
        const int acc = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
        if (!mbar_wait(&s.tempty[acc], use ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&s.full[stage], phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(ring + stage * A_BYTES);
          const uint32_t b0 = smem_u32(ring + STAGES * A_BYTES + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            mma_bf16_ss(d_tmem, sdesc_kmajor_sw128(a0 + k * 32), sdesc_kmajor_sw128(b0 + k * 32),
                        IDESC, (kb | k) != 0 ? 1u : 0u);
          }
          any = true;
          // the slot is free again once both CTAs of a pair have read it
          if (PAIR) mma_commit_mc(&s.empty[stage], kPairMask);
          else mma_commit(&s.empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&s.tfull[acc]);
      }
      // Drain: every MMA issued by this thread has completed after this.
      if (any) {
        mma_commit(&s.done);
        mbar_wait_drain(&s.done, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r_in_tile = q * 32 + lane;
    int it = 0;
    for (int t = w_first; t < total; t += w_step, ++it) {
      const Tile tl = decode_tile<MODE, PAIR>(p, s, t, rank);
      const ClassDesc& cd = p.cls[tl.cls];
      const int acc = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
      if (!mbar_wait(&s.tfull[acc], use, abort_flag)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + static_cast<uint32_t>(acc * BN) +
                             (static_cast<uint32_t>(q * 32) << 16);
      const int m = tl.mt * BM + r_in_tile;
      const bool valid = m < tl.rows;
      const int n_base = tl.nt * out_tile_cols<MODE>();
      __nv_bfloat16* orow = cd.out + static_cast<size_t>(tl.row0 + (valid ? m : 0)) * cd.ld_out + n_base;
      if (MODE == GATEUP) {
        // training forward: a and b of this row and these columns, kept for
        // the backward at [expert of the columns][a | b] (a 128-column tile
        // never straddles two shared experts: I % 128 == 0)
        __nv_bfloat16* abrow =
            cd.ab != nullptr && valid
                ? cd.ab + static_cast<size_t>(tl.row0 + m) * cd.ld_ab +
                      (n_base / p.inter) * 2 * p.inter + n_base % p.inter
                : nullptr;
#pragma unroll 1
        for (int c = 0; c < (BN / 2) / 16; ++c) {
          float a[16], b[16];
          tmem_ld16(taddr + c * 16, a);
          tmem_ld16(taddr + BN / 2 + c * 16, b);
          tmem_ld_wait();
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            pk[i] = pack_bf16x2(silu_f(a[2 * i]) * b[2 * i], silu_f(a[2 * i + 1]) * b[2 * i + 1]);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 16);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
          if (abrow != nullptr) {
            uint4* da = reinterpret_cast<uint4*>(abrow + c * 16);
            uint4* db = reinterpret_cast<uint4*>(abrow + p.inter + c * 16);
            da[0] = make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                               pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
            da[1] = make_uint4(pack_bf16x2(a[8], a[9]), pack_bf16x2(a[10], a[11]),
                               pack_bf16x2(a[12], a[13]), pack_bf16x2(a[14], a[15]));
            db[0] = make_uint4(pack_bf16x2(b[0], b[1]), pack_bf16x2(b[2], b[3]),
                               pack_bf16x2(b[4], b[5]), pack_bf16x2(b[6], b[7]));
            db[1] = make_uint4(pack_bf16x2(b[8], b[9]), pack_bf16x2(b[10], b[11]),
                               pack_bf16x2(b[12], b[13]), pack_bf16x2(b[14], b[15]));
          }
        }
      } else {
        // the routed rows' gate, folded in before the one rounding to bf16
        const float gm = cd.gate != nullptr && valid ? cd.gate[tl.row0 + m] : 1.f;
#pragma unroll 1
        for (int c = 0; c < BN / 16; ++c) {
          float v[16];
          tmem_ld16(taddr + c * 16, v);
          tmem_ld_wait();
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(v[2 * i] * gm, v[2 * i + 1] * gm);
          if (valid && n_base + c * 16 < cd.n_out) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 16);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.tempty[acc]);
    }
  }
  __syncthreads();
  // neither CTA of a pair leaves while the other may still multicast into
  // it or arrive on its barriers
  if (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace bf16gemm

// ------------------------------------------------------------------- host
// h (and, FP8, its scales), then the gate of every permuted row.
static size_t experts_h_bytes(const moe_cfg_t& c) {
  const size_t tk = static_cast<size_t>(c.T) * c.K;
  const size_t hr = tk * c.inter, hs = static_cast<size_t>(c.T) * c.n_shared * c.inter;
  if (c.dtype == MOE_DTYPE_FP32) return align_up((hr + hs) * 4, 256);
  if (c.dtype == MOE_DTYPE_BF16) return align_up((hr + hs) * 2, 256);
  // FP8: E4M3 codes plus one fp32 scale per 128 values
  return align_up(hr + hs, 256) + align_up((hr + hs) / 128 * 4, 256);
}

size_t experts_scratch_bytes(const moe_cfg_t& c) {
  return experts_h_bytes(c) + align_up(static_cast<size_t>(c.T) * c.K * 4, 256);
}

float* experts_gate_rows(const moe_cfg_t& c, void* ws) {
  return reinterpret_cast<float*>(static_cast<char*>(ws) + experts_h_bytes(c));
}

void experts_scratch_carve(const moe_cfg_t& c, void* ws, void** h, float** h_scales) {
  const size_t tk = static_cast<size_t>(c.T) * c.K;
  const size_t hr = tk * c.inter, hs = static_cast<size_t>(c.T) * c.n_shared * c.inter;
  *h = ws;
  *h_scales = nullptr;
  if (c.dtype == MOE_DTYPE_FP8_E4M3)
    *h_scales = reinterpret_cast<float*>(static_cast<char*>(ws) + align_up(hr + hs, 256));
}

// Clusters of two CTAs that can be resident at once (one CTA per SM), per
// (device, kernel).
int experts_pair_clusters(const void* func, const cudaLaunchConfig_t& cfg) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> known;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(mu);
  auto it = known.find({dev, func});
  if (it != known.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sm_count() / 2;
  }
  n = std::min(n, sm_count() / 2);
  known[{dev, func}] = n;
  return n;
}

template <int MODE, bool GATHER>
static cudaError_t launch_bf16_gemm(const bf16gemm::Params& prm, cudaStream_t st) {
  using namespace bf16gemm;
  const void* func = reinterpret_cast<const void*>(experts_bf16_kernel<MODE, GATHER>);
  cudaError_t e = ensure_smem_limit(func, static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  if (GATHER) {
    experts_bf16_kernel<MODE, GATHER><<<sm_count(), THREADS_GATHER, kSmemBytes, st>>>(prm);
    return cudaGetLastError();
  }
  // persistent clusters of two CTAs (pair units), as many as fit at once
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2);
  cfg.gridDim = dim3(2 * experts_pair_clusters(func, cfg));
  e = cudaLaunchKernelEx(&cfg, experts_bf16_kernel<MODE, GATHER>, prm);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// A-like operand (rows of `inner` bf16 elements, 128-byte swizzle) encoded
// twice: box of `rows` rows and of rows / 2 rows.
static CUresult encode_bf16_pair(CUtensorMap* full, CUtensorMap* half, const void* base,
                                 uint64_t inner, uint64_t outer, uint32_t rows) {
  using namespace bf16gemm;
  const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle SW = CU_TENSOR_MAP_SWIZZLE_128B;
  CUresult r = encode_tensor_map_2d(full, BF, const_cast<void*>(base), inner, outer, inner * 2, BK,
                                    rows, SW);
  if (r == CUDA_SUCCESS)
    r = encode_tensor_map_2d(half, BF, const_cast<void*>(base), inner, outer, inner * 2, BK,
                             rows / 2, SW);
  return r;
}

template <int MODE>
cudaError_t launch_bf16_pair_gemm(const bf16gemm::Params& prm, cudaStream_t st);  // experts_pair.cu

cudaError_t launch_experts_bf16(const ExpertsArgs& a, cudaStream_t st) {
  using namespace bf16gemm;
  const moe_cfg_t& c = *a.cfg;
  const int64_t tk = static_cast<int64_t>(c.T) * c.K;
  const int I = c.inter, Ns = c.n_shared;
  __nv_bfloat16* h_routed = static_cast<__nv_bfloat16*>(a.h);
  __nv_bfloat16* h_shared = h_routed + tk * I;
  const bool has_shared = Ns > 0;
  const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;

  // ---- gate/up: A = x_perm (or, gathering, x[token_of_row]) / x, B = W13
  const bool gather = a.token_of_row != nullptr;
  // Pair MMAs (experts_pair.cu) when the segments average at least 128
  // rows; with fewer the GEMMs only stream weights, and the multicast pairs
  // of this file keep more of B in flight per SM.  Measured on one B300:
  // V3 prefill (256 rows per expert) equal, T = 4096 x 6 of 64 experts
  // (384 rows) 2-3% faster with pair MMAs, V3 decode (4 rows) 3.7% slower.
  const bool pair_mma = !gather && tk >= static_cast<int64_t>(BM) * c.E;
  Params g{};
  g.offsets = a.offsets; g.n_rows = static_cast<int>(tk); g.E = c.E; g.T = c.T; g.has_shared = has_shared ? 1 : 0;
  g.inter = I; g.d = c.d;
  g.token_of_row = a.token_of_row;
  g.x_rows = static_cast<const __nv_bfloat16*>(a.x);
  // (gathering never reads the routed A map; it is encoded over x to stay valid)
  CUresult r = gather ? encode_bf16_pair(&g.a_map[0], &g.a_half[0], a.x, c.d, c.T, BM)
                      : encode_bf16_pair(&g.a_map[0], &g.a_half[0], a.x_perm, c.d, tk, BM);
  if (r == CUDA_SUCCESS) r = encode_gate_up_map(&g.b_map[0], BF, a.w13, c.E, I, c.d, 2, BK, 2);
  if (r == CUDA_SUCCESS) r = encode_gate_up_map(&g.b_half[0], BF, a.w13, c.E, I, c.d, 2, BK, 1);
  if (r == CUDA_SUCCESS) r = encode_gate_up_map(&g.b_mix[0], BF, a.w13, c.E, I, c.d, 2, BK, 2, 64);
  if (r == CUDA_SUCCESS && has_shared) {
    r = encode_bf16_pair(&g.a_map[1], &g.a_half[1], a.x, c.d, c.T, BM);
    if (r == CUDA_SUCCESS) r = encode_gate_up_map(&g.b_map[1], BF, a.ws13, Ns, I, c.d, 2, BK, 2);
    if (r == CUDA_SUCCESS) r = encode_gate_up_map(&g.b_half[1], BF, a.ws13, Ns, I, c.d, 2, BK, 1);
    if (r == CUDA_SUCCESS) r = encode_gate_up_map(&g.b_mix[1], BF, a.ws13, Ns, I, c.d, 2, BK, 2, 64);
  } else {
    g.a_map[1] = g.a_map[0];
    g.b_map[1] = g.b_map[0];
    g.a_half[1] = g.a_half[0];
    g.b_half[1] = g.b_half[0];
    g.b_mix[1] = g.b_mix[0];
  }
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  g.cls[0] = ClassDesc{h_routed, I, I, c.d, a.ab, 2 * I};
  g.cls[1] = ClassDesc{h_shared, Ns * I, Ns * I, c.d, a.ab_shared, Ns * 2 * I};
  cudaError_t e = gather     ? launch_bf16_gemm<GATEUP, true>(g, st)
                  : pair_mma ? launch_bf16_pair_gemm<GATEUP>(g, st)
                             : launch_bf16_gemm<GATEUP, false>(g, st);
  if (e != cudaSuccess) return e;

  // ---- down: A = h, B = W2
  Params dn = g;
  r = encode_bf16_pair(&dn.a_map[0], &dn.a_half[0], h_routed, I, tk, BM);
  if (r == CUDA_SUCCESS)
    r = encode_bf16_pair(&dn.b_map[0], &dn.b_half[0], a.w2, I, static_cast<uint64_t>(c.E) * c.d, BN);
  if (r == CUDA_SUCCESS && has_shared) {
    r = encode_bf16_pair(&dn.a_map[1], &dn.a_half[1], h_shared, static_cast<uint64_t>(Ns) * I, c.T,
                         BM);
    if (r == CUDA_SUCCESS)
      r = encode_bf16_pair(&dn.b_map[1], &dn.b_half[1], a.ws2, I, static_cast<uint64_t>(Ns) * c.d,
                           BN);
  } else {
    dn.a_map[1] = dn.a_map[0];
    dn.b_map[1] = dn.b_map[0];
    dn.a_half[1] = dn.a_half[0];
    dn.b_half[1] = dn.b_half[0];
  }
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  dn.cls[0] = ClassDesc{static_cast<__nv_bfloat16*>(a.y_perm), c.d, c.d, I, nullptr, 0,
                        a.gate_of_row};
  dn.cls[1] = ClassDesc{static_cast<__nv_bfloat16*>(a.y_shared), c.d, c.d, Ns * I};
  return pair_mma ? launch_bf16_pair_gemm<DOWN>(dn, st) : launch_bf16_gemm<DOWN, false>(dn, st);
}

}  // namespace moe
