// Grouped expert GEMMs in FP8 E4M3 with fine-grained scales, on the
// 5th-generation tensor cores (tcgen05 + TMEM) fed by TMA.
//
// "DeepSeek-V3 Technical Report":
//   - fine-grained quantisation paragraph / Appendix B.2: activations carry
//     one fp32 scale per 1 x 128 tile, weights one per 128 x 128 block;
//   - increased-precision accumulation paragraph: every N_C = 128 elements
//     of the reduction, the tensor-core partial sum is moved to fp32 CUDA
//     -core registers, where the scales are applied.
// Here the reduction is cut in 128-element K blocks (one pipeline stage).
// The tensor cores write each block's partial product, as two 128-column
// halves, into a ring of four 128-column TMEM partials; each column half is
// promoted by its own epilogue warpgroup, which reads the partial
// (tcgen05.ld), multiplies it by sa[row, kb] * sw[col block, kb], adds it
// to fp32 registers and hands it back.  The MMAs can run up to three
// half-blocks ahead of the promotion.
//
// Two launches per layer, one persistent kernel each:
//   gate/up: per 128 x 256 tile the 256 MMA columns are 128 rows of W1 and
//            the matching 128 rows of W3; the epilogue forms
//            h = silu(a) * b for 128 h columns and quantises h again in
//            1 x 128 tiles (codes + fp32 scales) for the down projection;
//   down:    y = h W2^T per 128 x 256 tile, bf16 output.
// The work list and its order are those of the bf16 kernel: every
// (group, M tile, N tile) of the routed experts, then the shared class;
// M varies fastest inside a group so concurrently running CTAs share each
// weight tile through L2.
//
// Roles (384 threads = 3 warpgroups, one CTA per SM):
//   warps 0, 3  TMA producers (even / odd K blocks): A and B tiles into a
//               4-stage ring (48 KB/stage), one TMA load each per stage
//   warp 1      allocates 512 TMEM columns; warps 1 and 2 issue
//               tcgen05.mma.kind::f8f6f4 (M=128, N=128, K=32), 4 per block
//               and column half, one thread each, for alternate K blocks
//   warps 4..11 promotion + epilogue.  Warp w reads TMEM lanes
//               32*(w%4)..+31 (its rows); warpgroup 1 owns column half 0,
//               warpgroup 2 half 1.  Gate/up: a half is 64 gate columns and
//               the 64 matching up columns (the B tile interleaves W1 and W3
//               in 64-row chunks), so SwiGLU needs no exchange;
//               the two halves of a row swap one amax through shared memory
//               for the 1 x 128 requantisation.  Down: a half is one
//               128-column weight block.
// Registers: launched at 168 per thread; warpgroup 0 gives its share down
// to 40 and the two epilogue warpgroups take 232 each (4*32*40 +
// 8*32*232 = 384*168), room for 128 fp32 accumulators, one batch of TMEM
// loads and the scales, which are loaded two K blocks ahead (no spills).
// Every wait is bounded; a wait that gives up sets the error word and the
// block-wide abort flag, so all roles leave, drain their own copies in
// flight and free TMEM.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace fp8gemm {

constexpr int BM = 128, BN = 256, BK = 128;  // BK bytes = one 128-byte swizzle row = one scale block
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;             // 16 KiB
constexpr int B_BYTES = BN * BK;             // 32 KiB
constexpr int EPI_WARPS = 8;
constexpr int EPI_WARP0 = 4;                 // first epilogue warp (warpgroup 1)
constexpr int THREADS = 128 + EPI_WARPS * 32;
constexpr uint32_t REGS_LOW = 40, REGS_HIGH = 232;  // after setmaxnreg
static_assert(4 * 32 * REGS_LOW + EPI_WARPS * 32 * REGS_HIGH <= THREADS * 168,
              "register split above the launch allocation");
constexpr int MAX_GROUPS = 1025;             // 1024 routed experts + the shared class
constexpr int PN = BN / 2;                   // columns of one TMEM partial (one column half)
constexpr uint32_t TMEM_COLS = 512;          // four 128-column partials
constexpr uint32_t IDESC = idesc_f32acc(0, 0, BM, PN);  // E4M3 x E4M3 -> fp32, N = 128

enum { GATEUP = 0, DOWN = 1 };

struct ClassDesc {
  void* out;              // gate/up: E4M3 h codes [rows, n_out]; down: bf16 y [rows, n_out]
  float* out_scales;      // gate/up: h scales [rows, n_out / 128]; down: unused
  const float* a_scales;  // [rows, k_dim / 128]
  const float* w_scales;  // block scales of the class's weight matrices
  int n_out;              // output columns (row stride of out)
  int k_dim;              // reduction length
  const float* gate;      // down, optional: every output row is multiplied by gate[row]
  __nv_bfloat16* ab;      // gate/up, optional: [a | b] rows [rows, 2I] kept for the backward
};

struct Params {
  CUtensorMap a_map[2];  // [0] routed rows, [1] shared rows
  CUtensorMap b_map[2];  // [0] routed weights, [1] shared weights
  ClassDesc cls[2];
  const int32_t* offsets;
  int n_rows;  // T * K: permuted rows, the bound of every segment
  int E;
  int T;
  int has_shared;
  int inter;  // I
  int d;
  int out32;  // both classes' outputs 32-byte aligned: 32-byte stores
};

struct Smem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t pfull[4];
  uint64_t pempty[4];
  uint64_t xch;
  uint64_t done[2];
  uint32_t tmem_base;
  int abort;
  int n_groups;
  float red[2][2][BM];         // [tile parity][column half][row]: |h| maxima
  int gstart[MAX_GROUPS + 1];  // first tile of every group
  int mtiles[MAX_GROUPS];      // M tiles of every group
  int off[MAX_GROUPS];         // first row of every routed group (copy of offsets[0..E])
};

constexpr size_t kRingBytes = static_cast<size_t>(STAGES) * (A_BYTES + B_BYTES);
constexpr size_t kSmemBytes = 1024 + kRingBytes + sizeof(Smem);
static_assert(kSmemBytes <= 232448, "above the 227 KiB of shared memory a block may use");

struct Tile {
  int cls;     // 0 routed, 1 shared
  int group;   // routed expert index (cls 0)
  int row0;    // first row of the group in its class's row space
  int rows;    // valid rows of the group
  int mt, nt;  // tile coordinates inside the group
};

template <int MODE>
__device__ __forceinline__ int out_tile_cols() { return MODE == GATEUP ? BN / 2 : BN; }

template <int MODE>
__device__ __forceinline__ int n_tiles_of(const Params& p, int cls) {
  return ceil_div(p.cls[cls].n_out, out_tile_cols<MODE>());
}

template <int MODE>
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
    sum += mt * n_tiles_of<MODE>(p, cls);
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
    const int cls = g < p.E ? 0 : 1;
    run += s.mtiles[g] * n_tiles_of<MODE>(p, cls);
  }
  if (lane == 31) {
    s.gstart[G] = incl;
    s.n_groups = G;
    s.off[p.E] = p.offsets[p.E];
  }
}

// Group of tile t, searching forward from group g (a CTA's tiles ascend, so
// each role keeps its last group as the hint).
__device__ __forceinline__ int group_from(const Smem& s, int t, int g) {
  while (s.gstart[g + 1] <= t) ++g;
  return g;
}

template <int MODE>
__device__ __forceinline__ Tile decode_tile(const Params& p, const Smem& s, int t, int& g) {
  g = group_from(s, t, g);
  const int lo = g;
  Tile tl;
  tl.cls = lo < p.E ? 0 : 1;
  tl.group = lo;
  const int local = t - s.gstart[lo];
  const int mt_count = s.mtiles[lo];
  tl.mt = local % mt_count;
  tl.nt = local / mt_count;
  if (tl.cls == 0) { tl.row0 = s.off[lo]; tl.rows = s.off[lo + 1] - tl.row0; }
  else { tl.row0 = 0; tl.rows = p.T; }
  return tl;
}

// Scales of the epilogue thread's row and columns, K block after K block.
// Activation: sa[row, kb] (a row past the segment reads the segment's first
// row: its sums are never stored).  Gate/up: the W1 block and the matching
// W3 block of the tile's 128 h columns (the W3 block row lies `up` floats
// after the W1 one).  Down: the thread's 128-column block of W2 (0 for a
// block past d); the shared class walks K over its N_s matrices, so the
// cursor steps to the next matrix every I/128 blocks.  Loads are issued two
// K blocks before use.
template <int MODE>
struct ScaleCursor {
  const float* a;   // activation scales of the row, next block to load
  const float* w;   // gate/up: W1 block of the next block; down: W2 block at kl = 0 of the current matrix
  int up;           // gate/up: floats from a W1 block to the matching W3 block
  int kl;           // down: next K block inside the current matrix
  int kbs;          // down: K blocks per matrix
  int mat_floats;   // down: scale floats per matrix
  bool col_ok;      // down: the column block lies inside d

  __device__ __forceinline__ void init(const Params& p, const Tile& tl, int hf, size_t grow) {
    const ClassDesc& cd = p.cls[tl.cls];
    const int I = p.inter;
    a = cd.a_scales + grow * (cd.k_dim / BK);
    kl = 0;
    if (MODE == GATEUP) {
      const int n0 = tl.nt * (BN / 2);
      const int mat = tl.cls == 0 ? tl.group : n0 / I;
      const int i0 = n0 % I;
      const int kd = p.d / BK, nbs = 2 * I / BK;
      w = cd.w_scales + (static_cast<size_t>(mat) * nbs + i0 / BK) * kd;
      up = (I / BK) * kd;
      col_ok = true;
    } else {
      const int nbs = p.d / BK;
      const int nb = tl.nt * 2 + hf;
      kbs = I / BK;
      mat_floats = nbs * kbs;
      col_ok = nb < nbs;
      const int mat = tl.cls == 0 ? tl.group : 0;
      w = cd.w_scales + (static_cast<size_t>(mat) * nbs + (col_ok ? nb : 0)) * kbs;
    }
  }

  // Loads the next K block's scales and advances.
  __device__ __forceinline__ void next(float& sa, float& s0, float& s1) {
    sa = __ldg(a);
    ++a;
    if (MODE == GATEUP) {
      s0 = __ldg(w);
      s1 = __ldg(w + up);
      ++w;
    } else {
      s0 = col_ok ? __ldg(w + kl) : 0.f;
      s1 = 0.f;
      if (++kl == kbs) { kl = 0; w += mat_floats; }
    }
  }
};

// Promotion of one K block for one column half: waits for the half's TMEM
// partial, adds partial * sa * sw to the fp32 accumulators and hands the
// partial back to its MMA issuer.  K block pc of the CTA lives in partial
// 2 * (pc % 2) + hf (issuer pc % 2, column half hf).  lane_addr: the warp's
// TMEM lanes at column 0.  Returns false if the wait gave up.
template <int MODE>
__device__ __forceinline__ bool promote_block(Smem& s, float (&acc)[128], uint32_t lane_addr,
                                              int hf, int lane, uint32_t pc, float sa, float s0,
                                              float s1, volatile int* abort_flag) {
  const int buf = 2 * static_cast<int>(pc & 1u) + hf;
  if (!mbar_wait(&s.pfull[buf], (pc >> 1) & 1u, abort_flag)) return false;
  tc_fence_after();
  const uint32_t taddr = lane_addr + static_cast<uint32_t>(buf * PN);
  // Two batches of 32 + 32 columns (what the register budget allows without
  // spilling): gate/up 32 gate columns with their 32 up columns, down 64
  // consecutive columns.  The partial goes back to the MMA issuer as soon
  // as the last batch is in registers (tcgen05.wait::ld returns once the
  // loads have completed), before that batch's FMAs.
  constexpr int NB = 2;  // batches
  constexpr int W = 128 / (2 * NB);           // columns per load
#pragma unroll
  for (int r = 0; r < NB; ++r) {
    float x0[W], x1[W];
    if (MODE == GATEUP) {
      tmem_ld_cols<W>(taddr + r * W, x0);        // gate columns
      tmem_ld_cols<W>(taddr + 64 + r * W, x1);   // matching up columns
    } else {
      tmem_ld_cols<W>(taddr + r * 2 * W, x0);
      tmem_ld_cols<W>(taddr + r * 2 * W + W, x1);
    }
    tmem_ld_wait();
    if (r == NB - 1) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.pempty[buf]);
    }
    if (MODE == GATEUP) {
      const float sg = sa * s0, su = sa * s1;
#pragma unroll
      for (int i = 0; i < W; i += 2) {
        ffma2_bcast(acc[r * W + i], acc[r * W + i + 1], x0[i], x0[i + 1], sg);
        ffma2_bcast(acc[64 + r * W + i], acc[64 + r * W + i + 1], x1[i], x1[i + 1], su);
      }
    } else {
      const float sc = sa * s0;
#pragma unroll
      for (int i = 0; i < W; i += 2) {
        ffma2_bcast(acc[r * 2 * W + i], acc[r * 2 * W + i + 1], x0[i], x0[i + 1], sc);
        ffma2_bcast(acc[r * 2 * W + W + i], acc[r * 2 * W + W + i + 1], x1[i], x1[i + 1], sc);
      }
    }
  }
  return true;
}

// KEEP_AB (gate/up of a training forward): also store a and b in bf16; a
// separate instantiation, since the stores cost the epilogue registers.
template <int MODE, bool KEEP_AB = false>
__global__ void __launch_bounds__(THREADS, 1) experts_fp8_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Smem& s = *reinterpret_cast<Smem*>(ring + kRingBytes);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  volatile int* abort_flag = &s.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) { tma_prefetch_desc(&p.a_map[i]); tma_prefetch_desc(&p.b_map[i]); }
    for (int i = 0; i < STAGES; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], 1); }
    for (int i = 0; i < 4; ++i) { mbar_init(&s.pfull[i], 1); mbar_init(&s.pempty[i], 4); }
    mbar_init(&s.xch, EPI_WARPS * 32);
    mbar_init(&s.done[0], 1);
    mbar_init(&s.done[1], 1);
    s.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  if (warp == 2) build_tile_table<MODE>(p, s);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_base;
  const int total = s.gstart[s.n_groups];

  if (warp < EPI_WARP0) {
    regs_dec<REGS_LOW>();
  if (warp == 0 || warp == 3) {
    // ----------------------------------------------------------- producers
    // Two threads fill the ring: warp 0 the even K blocks of the CTA's block
    // sequence (ring slots 0 and 2), warp 3 the odd ones (slots 1 and 3).
    // A stage is two TMA loads: the A rows and the whole 256-row B tile.
    if (lane == 0) {
      const uint32_t par = warp == 0 ? 0u : 1u;
      uint32_t g = 0;     // K blocks of the CTA so far
      uint32_t mine = 0;  // K blocks issued by this thread
      bool stop = false;
      int gh = 0;         // group of the last tile
      for (int t = blockIdx.x; t < total && !stop && !*abort_flag; t += gridDim.x) {
        const Tile tl = decode_tile<MODE>(p, s, t, gh);
        const int nk = p.cls[tl.cls].k_dim / BK;
        const int a_row = tl.row0 + tl.mt * BM;
        const CUtensorMap* am = &p.a_map[tl.cls];
        const CUtensorMap* bm = &p.b_map[tl.cls];
        // B coordinates.  Gate/up: (k, 0, 0, i0 / 64, matrix) in the
        // [n][I/64][2][64][d] view: 64 W1 rows, their 64 W3 rows, the next 64
        // W1 rows and their W3 rows, so each column half of the tile holds
        // matching gate and up rows.  Down:
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
            mbar_arrive_expect_tx(&s.full[stage], A_BYTES + B_BYTES);
            // (the L2 policies are created at each use: registers are scarce here)
            if (MODE == GATEUP)
              tma_load_5d(sb, bm, &s.full[stage], kb * BK, 0, 0, bi / 64, bmat, l2_policy_evict_normal());
            else
              tma_load_2d(sb, bm, &s.full[stage], bxk, brow, l2_policy_evict_normal());
            tma_load_2d(sa, am, &s.full[stage], kb * BK, a_row, l2_policy_evict_last());
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
  } else if (warp == 1 || warp == 2) {
    // ----------------------------------------------------------------- MMA
    // Two issuing threads: warp 1 takes the even K blocks of the CTA's
    // block sequence (TMEM partials 0 and 1, ring stages 0 and 2), warp 2
    // the odd ones (partials 2 and 3, stages 1 and 3).  Each K block and
    // column half is a separate accumulation into its own partial, so the
    // two threads need no mutual order.
    if (lane == 0) {
      const int par = warp - 1;
      uint32_t pc = 0;   // K blocks of the CTA so far
      uint32_t mine = 0; // K blocks of this issuer so far
      bool any = false, ok = true;
      const int shared0 = s.gstart[p.E];  // first tile of the shared class
      for (int t = blockIdx.x; t < total && ok && !*abort_flag; t += gridDim.x) {
        // only the tile's K length matters here: it depends on the class alone
        const int nk = p.cls[t >= shared0 ? 1 : 0].k_dim / BK;
        uint32_t kb0 = (pc & 1u) == static_cast<uint32_t>(par) ? 0u : 1u;
        for (uint32_t kb = kb0; kb < static_cast<uint32_t>(nk); kb += 2, ++mine) {
          const int stage = par + 2 * static_cast<int>(mine & 1u);
          const uint32_t sphase = (mine >> 1) & 1u;
          if (!mbar_wait(&s.full[stage], sphase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = sdesc_kmajor_sw128(smem_u32(ring + stage * A_BYTES));
          // the two column halves: B rows [0, 128) and [128, 128 + 128) of the
          // stage, each into its own partial 2 * par + h
          for (int h = 0; h < 2; ++h) {
            const int buf = 2 * par + h;
            if (!mbar_wait(&s.pempty[buf], (mine & 1u) ^ 1u, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint64_t bd = sdesc_kmajor_sw128(
                smem_u32(ring + STAGES * A_BYTES + stage * B_BYTES + h * (B_BYTES / 2)));
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * PN);
#pragma unroll
            for (int k = 0; k < BK / 32; ++k)  // +32 bytes along K = +2 in the address field
              mma_fp8_ss(d_tmem, ad + 2 * k, bd + 2 * k, IDESC, k != 0 ? 1u : 0u);
            any = true;
            mma_commit(&s.pfull[buf]);
          }
          if (!ok) break;
          mma_commit(&s.empty[stage]);
        }
        pc += static_cast<uint32_t>(nk);
      }
      if (any) {
        mma_commit(&s.done[par]);
        mbar_wait_drain(&s.done[par], 0);
      }
    }
  }
  } else {
    regs_inc<REGS_HIGH>();
    // ------------------------------------------------- promotion + epilogue
    // The TMEM base and the tile count are read from shared memory again
    // here, so that no value computed before the role split (where the
    // producer/MMA warpgroup's 40-register budget applies) is live in this
    // warpgroup's loops.
    const uint32_t tmem_base_e = *reinterpret_cast<volatile uint32_t*>(&s.tmem_base);
    const int total_e = reinterpret_cast<volatile int*>(s.gstart)[s.n_groups];
    const int q = warp & 3;                   // TMEM lane quarter of this warp
    const int hf = (warp - EPI_WARP0) >> 2;   // column half
    const uint32_t lane_addr = tmem_base_e + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t pc = 0;
    int gh = 0;  // group of the last tile
    for (int t = blockIdx.x; t < total_e; t += gridDim.x) {
      const int r_in_tile = q * 32 + lane;
      // Only the scale cursor and the K count stay live through the K loop;
      // the tile is decoded again for the store (register pressure).
      int nk;
      ScaleCursor<MODE> sc;
      {
        const Tile tl = decode_tile<MODE>(p, s, t, gh);
        nk = p.cls[tl.cls].k_dim / BK;
        const int m = tl.mt * BM + r_in_tile;
        sc.init(p, tl, hf, static_cast<size_t>(tl.row0) + (m < tl.rows ? m : 0));
      }
      float acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.f;
      // two-slot register ring of scales, loaded two K blocks ahead
      float sa0, w00, w10, sa1 = 0.f, w01 = 0.f, w11 = 0.f;
      sc.next(sa0, w00, w10);
      if (nk > 1) sc.next(sa1, w01, w11);
      bool ok = true;
      for (int kb = 0; kb < nk; kb += 2) {
        {
          const float a_ = sa0, b_ = w00, c_ = w10;
          if (kb + 2 < nk) sc.next(sa0, w00, w10);
          if (!promote_block<MODE>(s, acc, lane_addr, hf, lane, pc, a_, b_, c_, abort_flag)) {
            ok = false;
            break;
          }
          ++pc;
        }
        if (kb + 1 < nk) {
          const float a_ = sa1, b_ = w01, c_ = w11;
          if (kb + 3 < nk) sc.next(sa1, w01, w11);
          if (!promote_block<MODE>(s, acc, lane_addr, hf, lane, pc, a_, b_, c_, abort_flag)) {
            ok = false;
            break;
          }
          ++pc;
        }
      }
      if (!ok) break;

      const Tile tl = decode_tile<MODE>(p, s, t, gh);
      const ClassDesc& cd = p.cls[tl.cls];
      const int m = tl.mt * BM + r_in_tile;
      const bool valid = m < tl.rows;
      const size_t grow = static_cast<size_t>(tl.row0) + (valid ? m : 0);
      if (MODE == GATEUP) {
        // training forward: a and b of this row's 64 h columns, kept in bf16
        // for the backward at [a | b] (I columns each)
        if (KEEP_AB && cd.ab != nullptr && valid) {
          __nv_bfloat16* arow = cd.ab + grow * (2 * static_cast<size_t>(p.inter)) +
                                tl.nt * (BN / 2) + hf * 64;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            reinterpret_cast<uint4*>(arow)[c] =
                make_uint4(pack_bf16x2(acc[8 * c], acc[8 * c + 1]), pack_bf16x2(acc[8 * c + 2], acc[8 * c + 3]),
                           pack_bf16x2(acc[8 * c + 4], acc[8 * c + 5]), pack_bf16x2(acc[8 * c + 6], acc[8 * c + 7]));
            reinterpret_cast<uint4*>(arow + p.inter)[c] =
                make_uint4(pack_bf16x2(acc[64 + 8 * c], acc[64 + 8 * c + 1]),
                           pack_bf16x2(acc[64 + 8 * c + 2], acc[64 + 8 * c + 3]),
                           pack_bf16x2(acc[64 + 8 * c + 4], acc[64 + 8 * c + 5]),
                           pack_bf16x2(acc[64 + 8 * c + 6], acc[64 + 8 * c + 7]));
          }
        }
        // h = silu(a) * b, then one E4M3 scale per row and 128 h columns
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const float h = silu_fast(acc[i]) * acc[64 + i];
          acc[i] = h;
          amax = fmaxf(amax, fabsf(h));
        }
        const int it = (t - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x);
        const int xb = it & 1;
        s.red[xb][hf][r_in_tile] = amax;
        mbar_arrive(&s.xch);
        if (!mbar_wait(&s.xch, static_cast<uint32_t>(it) & 1u, abort_flag)) break;
        amax = fmaxf(amax, s.red[xb][hf ^ 1][r_in_tile]);
        const float scale = fp8_scale_of(amax);
        // codes of h / scale as h * fl32(1 / scale): one correctly rounded
        // reciprocal per row instead of 64 divisions (a code can differ from
        // that of the exact quotient only for a value within one fp32 ulp of
        // an E4M3 rounding midpoint)
        const float rs = __frcp_rn(scale);
        if (valid) {
          const int n0 = tl.nt * (BN / 2);
          uint8_t* orow = static_cast<uint8_t*>(cd.out) + grow * cd.n_out + n0 + hf * 64;
          uint32_t w[16];
#pragma unroll
          for (int v = 0; v < 16; ++v)
            w[v] = quant4_e4m3_mul(acc[v * 4 + 0], acc[v * 4 + 1], acc[v * 4 + 2], acc[v * 4 + 3], rs);
          if (p.out32) {
            st_global_32B(orow, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
            st_global_32B(orow + 32, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
          } else {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              reinterpret_cast<uint4*>(orow)[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
          }
          if (hf == 0) cd.out_scales[grow * (cd.n_out / BK) + n0 / BK] = scale;
        }
      } else {
        const int n_base = tl.nt * BN + hf * 128;
        if (valid) {
          // the routed rows' gate, folded in before the one rounding to bf16
          const float gm = cd.gate != nullptr ? cd.gate[grow] : 1.f;
          __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(cd.out) + grow * cd.n_out + n_base;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            if (n_base + c * 16 < cd.n_out) {
              uint32_t w[8];
#pragma unroll
              for (int i = 0; i < 8; ++i)
                w[i] = pack_bf16x2(acc[c * 16 + 2 * i] * gm, acc[c * 16 + 2 * i + 1] * gm);
              if (p.out32) {
                st_global_32B(orow + c * 16, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
              } else {
                uint4* dst = reinterpret_cast<uint4*>(orow + c * 16);
                dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
              }
            }
          }
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace fp8gemm

template <int MODE, bool KEEP_AB = false>
static cudaError_t launch_fp8_gemm(const fp8gemm::Params& prm, cudaStream_t st) {
  using namespace fp8gemm;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(experts_fp8_kernel<MODE, KEEP_AB>),
                                    static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  experts_fp8_kernel<MODE, KEEP_AB><<<sm_count(), THREADS, kSmemBytes, st>>>(prm);
  return cudaGetLastError();
}

cudaError_t launch_experts_fp8(const ExpertsArgs& a, cudaStream_t st) {
  using namespace fp8gemm;
  const moe_cfg_t& c = *a.cfg;
  const int64_t tk = static_cast<int64_t>(c.T) * c.K;
  const int I = c.inter, Ns = c.n_shared;
  uint8_t* h_routed = static_cast<uint8_t*>(a.h);
  uint8_t* h_shared = h_routed + tk * I;
  float* hs_routed = a.h_scales;
  float* hs_shared = a.h_scales + tk * (I / BK);
  const bool has_shared = Ns > 0;
  const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapSwizzle SW = CU_TENSOR_MAP_SWIZZLE_128B;

  // ---- gate/up: A = x_perm / x_q (E4M3), B = W13 (E4M3)
  Params g{};
  g.offsets = a.offsets; g.n_rows = static_cast<int>(tk); g.E = c.E; g.T = c.T; g.has_shared = has_shared ? 1 : 0;
  g.inter = I; g.d = c.d;
  CUresult r = encode_tensor_map_2d(&g.a_map[0], U8, const_cast<void*>(a.x_perm), c.d, tk,
                                    static_cast<uint64_t>(c.d), BK, BM, SW);
  if (r == CUDA_SUCCESS)
    r = encode_gate_up_map_interleaved(&g.b_map[0], U8, a.w13, c.E, I, c.d, 1, BK);
  if (r == CUDA_SUCCESS && has_shared) {
    r = encode_tensor_map_2d(&g.a_map[1], U8, const_cast<void*>(a.x), c.d, c.T,
                             static_cast<uint64_t>(c.d), BK, BM, SW);
    if (r == CUDA_SUCCESS)
      r = encode_gate_up_map_interleaved(&g.b_map[1], U8, a.ws13, Ns, I, c.d, 1, BK);
  } else {
    g.a_map[1] = g.a_map[0];
    g.b_map[1] = g.b_map[0];
  }
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const auto al32 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 31u) == 0; };
  g.out32 = al32(h_routed) && al32(h_shared) ? 1 : 0;
  g.cls[0] = ClassDesc{h_routed, hs_routed, a.x_perm_scales, a.w13_scales, I, c.d, nullptr, a.ab};
  g.cls[1] = ClassDesc{h_shared, hs_shared, has_shared ? a.x_scales : a.x_perm_scales,
                       has_shared ? a.ws13_scales : a.w13_scales, Ns * I, c.d, nullptr,
                       has_shared ? a.ab_shared : nullptr};
  cudaError_t e = a.ab != nullptr ? launch_fp8_gemm<GATEUP, true>(g, st) : launch_fp8_gemm<GATEUP>(g, st);
  if (e != cudaSuccess) return e;

  // ---- down: A = h codes, B = W2 (E4M3)
  Params dn = g;
  r = encode_tensor_map_2d(&dn.a_map[0], U8, h_routed, I, tk, static_cast<uint64_t>(I), BK, BM, SW);
  if (r == CUDA_SUCCESS)
    r = encode_tensor_map_2d(&dn.b_map[0], U8, const_cast<void*>(a.w2), I,
                             static_cast<uint64_t>(c.E) * c.d, static_cast<uint64_t>(I), BK,
                             BN, SW);
  if (r == CUDA_SUCCESS && has_shared) {
    r = encode_tensor_map_2d(&dn.a_map[1], U8, h_shared, static_cast<uint64_t>(Ns) * I, c.T,
                             static_cast<uint64_t>(Ns) * I, BK, BM, SW);
    if (r == CUDA_SUCCESS)
      r = encode_tensor_map_2d(&dn.b_map[1], U8, const_cast<void*>(a.ws2), I,
                               static_cast<uint64_t>(Ns) * c.d, static_cast<uint64_t>(I), BK,
                               BN, SW);
  } else {
    dn.a_map[1] = dn.a_map[0];
    dn.b_map[1] = dn.b_map[0];
  }
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  dn.out32 = al32(a.y_perm) && (!has_shared || al32(a.y_shared)) ? 1 : 0;
  dn.cls[0] = ClassDesc{a.y_perm, nullptr, hs_routed, a.w2_scales, c.d, I, a.gate_of_row};
  dn.cls[1] = ClassDesc{has_shared ? a.y_shared : a.y_perm, nullptr,
                        has_shared ? hs_shared : hs_routed,
                        has_shared ? a.ws2_scales : a.w2_scales, c.d, Ns > 0 ? Ns * I : I};
  return launch_fp8_gemm<DOWN>(dn, st);
}

}  // namespace moe
