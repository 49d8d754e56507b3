// Backward grouped GEMMs of the expert FFNs on the 5th-generation tensor
// cores (tcgen05 + TMEM), fed by TMA, for the bf16 kind.
//
// "DeepSeek-V3 Technical Report", mixed precision framework paragraph: a
// linear layer has three GEMMs, Fprop, Dgrad and Wgrad; DualPipe paragraph:
// the MLP backward splits into backward for input and backward for weights.
// With a = x W1^T, b = x W3^T, h = silu(a) b, y = h W2^T and dy given:
//   Dgrad (input):  dh = dy W2 (per expert),  da = dh b silu'(a),
//                   db = dh silu(a),           dx = [da | db] W13
//   Wgrad (weights): dW2 = dy^T h,             dW13 = [da | db]^T x
//
// The weights are stored [.., N rows, K cols] for the forward; the backward
// contracts over their other dimension.  Instead of transposing anything,
// those operands are read "MN-major": TMA copies 64-column x 64-row boxes
// (128-byte rows, 128-byte swizzle) and the MMA descriptors say that the
// N (or M) index is the contiguous one.  Likewise Wgrad reads both of its
// operands, activation rows of a segment, MN-major with the token rows as K.
//
// One persistent kernel per GEMM, three kinds:
//   DG_SWIGLU  dh tile = dy rows x W2 (A K-major, B MN-major); the epilogue
//              reads the [a | b] rows (kept by the training forward, or
//              recomputed), writes [da | db] over them and h = silu(a) b
//              (kept for dW2)
//   DG_PLAIN   dx tile = [da | db] rows x W13 (A K-major, B MN-major)
//   WG         dW tile = A^T B over the rows of one segment (both
//              MN-major); K is the segment length, so the last K block is
//              ragged: A's rows past the segment are zeroed in shared memory
//              before the MMAs read them
// The work list is every (group, M tile, N tile); groups are the E routed
// experts, then the shared experts.  Inside a group the M tile varies
// fastest for Dgrad (the CTAs running together share a weight tile through
// L2) and the N tile for Wgrad (they write whole row bands of the gradient).  Roles, barriers, bounded waits and the abort path are those of
// the forward grouped GEMM (experts_sm100.cu): warps 0 and 6 produce, warp 1
// issues MMAs into two 256-column fp32 accumulators, warps 2..5 drain them.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace bwdgemm {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KiB
constexpr int B_BYTES = BN * BK * 2;  // 32 KiB
constexpr int BOX_BYTES = 64 * BK * 2;  // one 64 x 64 MN-major box, 8 KiB
constexpr int THREADS = 224;
constexpr int PRODUCER2 = 6;
constexpr int MAX_GROUPS = 1025 + 64;  // routed experts + shared experts
constexpr uint32_t TMEM_COLS = 512;
static_assert(BN == 256, "the Wgrad epilogue drains an accumulator as four 64-column chunks");

enum Kind { DG_SWIGLU = 0, DG_PLAIN = 1, WG = 2 };

// Instruction descriptors: bit 15 marks A MN-major, bit 16 B MN-major.
constexpr uint32_t IDESC_DG = idesc_f32acc(1, 1, BM, BN) | (1u << 16);
constexpr uint32_t IDESC_WG = idesc_f32acc(1, 1, BM, BN) | (1u << 15) | (1u << 16);

struct ClassDesc {
  int k_dim;       // Dgrad: reduction length of every group of the class
  int b_row_step;  // Dgrad: B map rows between consecutive groups
  int a_col_step;  // Wgrad: A map column base of group j is j * a_col_step
  int b_col_step;  // Wgrad: B map column base of group j is j * b_col_step
  __nv_bfloat16* out;
  int ld_out;              // Dgrad: output row stride (elements)
  int out_col_step;        // Dgrad: output column base of group j
  size_t out_group_stride; // Wgrad: elements between the matrices of groups j, j + 1
  __nv_bfloat16* ab;       // DG_SWIGLU: [a | b] rows in, [da | db] out
  int ld_ab;
  int ab_col_step;
};

struct Params {
  CUtensorMap a_map[2];  // [0] routed class, [1] shared class
  CUtensorMap b_map[2];
  CUtensorMap out_map[2];  // Wgrad: the class's gradients [groups][m_dim][n_dim], box 1 x 32 x 64
  ClassDesc cls[2];
  const int32_t* offsets;
  int n_rows;  // T * K: permuted rows, the bound of every segment
  int E;
  int T;
  int n_sh;   // groups of the shared class
  int n_dim;  // output columns of a group (Dgrad: also the SwiGLU width I)
  int m_dim;  // Wgrad: output rows of a group
};

struct Smem {
  // Wgrad epilogue: per epilogue warp, 32 rows x 64 bf16 columns (128-byte
  // rows, 16-byte pieces XOR-swizzled by the row) on their way to a TMA store
  alignas(16) uint8_t stage_out[4][32 * 128];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
  int n_groups;
  int gstart[MAX_GROUPS + 1];
  int mtiles[MAX_GROUPS];
  int off[MAX_GROUPS];  // first row of every routed group (copy of offsets[0..E])
};

constexpr size_t kRingBytes = static_cast<size_t>(STAGES) * (A_BYTES + B_BYTES);
constexpr size_t kSmemBytes = 1024 + kRingBytes + sizeof(Smem);
static_assert(kSmemBytes <= 232448, "above the 227 KiB of shared memory a block may use");

struct Tile {
  int cls;    // 0 routed, 1 shared
  int j;      // group index inside its class
  int row0;   // Dgrad: first A row; Wgrad: first K row
  int rows;   // Dgrad: valid A rows; Wgrad: K length
  int mt, nt;
};

template <int KIND>
__device__ __forceinline__ int tiles_n(const Params& p) { return ceil_div(p.n_dim, BN); }

// Warp-cooperative tile table: Dgrad groups have ceil(rows / 128) M tiles,
// Wgrad groups ceil(m_dim / 128) whatever their K.
template <int KIND>
__device__ void build_tile_table(const Params& p, Smem& s) {
  const int lane = threadIdx.x % 32;
  const int G = p.E + p.n_sh;
  const int per = ceil_div(G, 32);
  const int g0 = lane * per, g1 = min(G, g0 + per);
  const int nt = tiles_n<KIND>(p);
  int sum = 0;
  for (int g = g0; g < g1; ++g) {
    int rows;
    if (g < p.E) {
      int o0;
      rows = checked_segment(p.offsets, g, p.n_rows, o0);
      s.off[g] = o0;
    } else {
      rows = p.T;
    }
    const int mt = KIND == WG ? ceil_div(p.m_dim, BM) : ceil_div(max(rows, 0), BM);
    s.mtiles[g] = mt;
    sum += mt * nt;
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
    run += s.mtiles[g] * nt;
  }
  if (lane == 31) {
    s.gstart[G] = incl;
    s.n_groups = G;
    s.off[p.E] = p.offsets[p.E];
  }
}

template <int KIND>
__device__ __forceinline__ Tile decode_tile(const Params& p, const Smem& s, int t) {
  int lo = 0, hi = s.n_groups;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.gstart[mid] <= t) lo = mid; else hi = mid;
  }
  Tile tl;
  tl.cls = lo < p.E ? 0 : 1;
  tl.j = tl.cls == 0 ? lo : lo - p.E;
  const int local = t - s.gstart[lo];
  if (KIND == WG) {
    // N tile fastest: the CTAs of a wave write whole row bands of the
    // gradient matrix (long contiguous runs in DRAM)
    const int nt_count = tiles_n<KIND>(p);
    tl.nt = local % nt_count;
    tl.mt = local / nt_count;
  } else {
    // M tile fastest: the CTAs of a wave share one weight tile through L2
    const int mt_count = s.mtiles[lo];
    tl.mt = local % mt_count;
    tl.nt = local / mt_count;
  }
  if (tl.cls == 0) { tl.row0 = s.off[lo]; tl.rows = max(s.off[lo + 1] - tl.row0, 0); }
  else { tl.row0 = 0; tl.rows = p.T; }
  return tl;
}

template <int KIND>
__device__ __forceinline__ int k_blocks(const Params& p, const Tile& tl) {
  return KIND == WG ? ceil_div(tl.rows, BK) : p.cls[tl.cls].k_dim / BK;
}

// Shared-memory descriptor of an MN-major operand stored as consecutive
// 64-column boxes of BK rows with the 128-byte swizzle: inside a box, K row
// r is the 128-byte line r (8-row atoms 1024 bytes apart); the next 64
// columns of M or N start BOX_BYTES further on.
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);         // start address
  d |= static_cast<uint64_t>(BOX_BYTES >> 4) << 16;            // leading byte offset: next 64 of M/N
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                 // stride byte offset: next 8 K rows
  d |= static_cast<uint64_t>(1) << 46;                         // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                         // 128-byte swizzle
  return d;
}

// silu and its derivative from one exponential.
__device__ __forceinline__ void silu_and_grad(float a, float& silu, float& dsilu) {
  const float sg = 1.0f / (1.0f + __expf(-a));
  silu = a * sg;
  dsilu = sg * fmaf(a, 1.0f - sg, 1.0f);
}

template <int KIND>
__global__ void __launch_bounds__(THREADS, 1) bwd_gemm_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Smem& s = *reinterpret_cast<Smem*>(ring + kRingBytes);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  volatile int* abort_flag = &s.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) { tma_prefetch_desc(&p.a_map[i]); tma_prefetch_desc(&p.b_map[i]); }
    for (int i = 0; i < STAGES; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], 1); }
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
  if (warp == 2) build_tile_table<KIND>(p, s);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_base;
  const int total = s.gstart[s.n_groups];

  if (warp == 0 || warp == PRODUCER2) {
    // ----------------------------------------------------------- producers
    // Warp 0 fills the even stages of the CTA's stage sequence, warp 6 the
    // odd ones.  Dgrad: A is one K-major box, B four MN-major boxes.
    // Wgrad: A two MN-major boxes, B four.
    if (lane == 0) {
      const uint32_t par = warp == 0 ? 0u : 1u;
      const uint64_t pol_a = l2_policy_evict_last();
      const uint64_t pol_b = l2_policy_evict_normal();
      uint32_t g = 0, mine = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < total && !stop && !*abort_flag; t += gridDim.x) {
        const Tile tl = decode_tile<KIND>(p, s, t);
        const ClassDesc& cd = p.cls[tl.cls];
        const int nk = k_blocks<KIND>(p, tl);
        const CUtensorMap* am = &p.a_map[tl.cls];
        const CUtensorMap* bm = &p.b_map[tl.cls];
        const int n0 = tl.nt * BN;
        for (int kb = 0; kb < nk; ++kb, ++g) {
          if ((g & 1u) != par) continue;
          const int stage = static_cast<int>(par + 2 * (mine & 1u));
          const uint32_t sphase = (mine >> 1) & 1u;
          if (!mbar_wait(&s.empty[stage], sphase ^ 1u, abort_flag)) { stop = true; break; }
          uint8_t* sa = ring + stage * A_BYTES;
          uint8_t* sb = ring + STAGES * A_BYTES + stage * B_BYTES;
          mbar_arrive_expect_tx(&s.full[stage], A_BYTES + B_BYTES);
          if (KIND == WG) {
            const int krow = tl.row0 + kb * BK;
            const int ac = tl.j * cd.a_col_step + tl.mt * BM;
            const int bc = tl.j * cd.b_col_step + n0;
#pragma unroll
            for (int c = 0; c < BM / 64; ++c)
              tma_load_2d(sa + c * BOX_BYTES, am, &s.full[stage], ac + 64 * c, krow, pol_a);
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_2d(sb + c * BOX_BYTES, bm, &s.full[stage], bc + 64 * c, krow, pol_b);
          } else {
            const int krow = tl.j * cd.b_row_step + kb * BK;
            tma_load_2d(sa, am, &s.full[stage], kb * BK, tl.row0 + tl.mt * BM, pol_a);
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_2d(sb + c * BOX_BYTES, bm, &s.full[stage], n0 + 64 * c, krow, pol_b);
          }
          ++mine;
        }
      }
      for (uint32_t i = 0; i < 2 && i < mine; ++i) {
        const uint32_t j = mine - 1 - i;
        mbar_wait_drain(&s.full[par + 2 * (j & 1u)], (j >> 1) & 1u);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    // Lane 0 issues.  For Wgrad the whole warp first zeroes the K rows of a
    // ragged last block that lie past the segment (in every box of A and
    // B: each K row is one 128-byte line of a box), then makes the writes
    // visible to the tensor cores.
    uint32_t stage = 0, phase = 0;
    int it = 0;
    bool any = false;
    for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x, ++it) {
      const Tile tl = decode_tile<KIND>(p, s, t);
      const int nk = k_blocks<KIND>(p, tl);
      const int acc = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
      // every lane waits; the warp leaves together if any lane gave up
      if (!__all_sync(0xffffffffu, mbar_wait(&s.tempty[acc], use ^ 1u, abort_flag))) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb) {
        if (!__all_sync(0xffffffffu, mbar_wait(&s.full[stage], phase, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint8_t* sa = ring + stage * A_BYTES;
        uint8_t* sb = ring + STAGES * A_BYTES + stage * B_BYTES;
        if (KIND == WG) {
          const int valid = min(tl.rows - kb * BK, BK);
          if (valid < BK) {
            // Zero A's K rows past the segment (16-byte chunks from line
            // `valid` to the end of both A boxes): their products with B
            // vanish whatever B holds there, as long as it is finite (B's
            // rows past a segment are rows of the next segment, written by
            // the library, or TMA's zero fill past the end of the tensor).
            const uint32_t from = static_cast<uint32_t>(valid) * 128u + lane * 16u;
#pragma unroll
            for (int box = 0; box < BM / 64; ++box)
              for (uint32_t o = from; o < static_cast<uint32_t>(BOX_BYTES); o += 512u)
                *reinterpret_cast<uint4*>(sa + box * BOX_BYTES + o) = make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
          }
          __syncwarp();
        }
        if (lane == 0) {
          const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = KIND == WG ? sdesc_mnmajor_sw128(a0 + k * 2048)
                                           : sdesc_kmajor_sw128(a0 + k * 32);
            mma_bf16_ss(d_tmem, ad, sdesc_mnmajor_sw128(b0 + k * 2048),
                        KIND == WG ? IDESC_WG : IDESC_DG, (kb | k) != 0 ? 1u : 0u);
          }
          mma_commit(&s.empty[stage]);
        }
        __syncwarp();
        any = true;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      // (a group without rows commits at once: its accumulator is not read)
      if (lane == 0) mma_commit(&s.tfull[acc]);
      __syncwarp();
    }
    if (lane == 0 && any) {
      mma_commit(&s.done);
      mbar_wait_drain(&s.done, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int r_in_tile = q * 32 + lane;
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const Tile tl = decode_tile<KIND>(p, s, t);
      const ClassDesc& cd = p.cls[tl.cls];
      const int acc = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
      if (!mbar_wait(&s.tfull[acc], use, abort_flag)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + static_cast<uint32_t>(acc * BN) +
                             (static_cast<uint32_t>(q * 32) << 16);
      const int n_base = tl.nt * BN;
      if (KIND == WG) {
        // The weight-gradient tile is written whole (64 KiB per tile, about
        // as much time as its MMAs take): per 64-column chunk each lane puts
        // its row into the warp's staging rows (the 128-byte swizzle), and
        // lane 0 hands the 32 x 64 chunk to a TMA store through the class's
        // 3-D map of the gradients.  The staging rows are reused once the
        // warp's previous store has read them; the TMEM loads of the next
        // chunk are in flight meanwhile.  m_dim is a multiple of 128, so
        // every row is inside the matrix.
        const bool empty = tl.rows == 0;
        uint8_t* stg = s.stage_out[q];
        auto put = [&](const float (&x0)[32], const float (&x1)[32], int c) {
          // the warp's previous store has read the staging rows
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float* x = j < 4 ? x0 + 8 * j : x1 + 8 * (j - 4);
            const uint4 w = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                                       pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) = w;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && n_base + c * 64 < p.n_dim) {  // (chunks past the matrix: no store)
            tma_store_3d(&p.out_map[tl.cls], stg, n_base + c * 64, tl.mt * BM + q * 32, tl.j);
            bulk_commit();
          }
        };
        float a0[32], a1[32], b0[32], b1[32];
        if (empty) {
#pragma unroll
          for (int i = 0; i < 32; ++i) a0[i] = a1[i] = 0.f;
#pragma unroll
          for (int c = 0; c < BN / 64; ++c) put(a0, a1, c);
        } else {
          // chunk c + 1's TMEM loads are in flight while chunk c is stored
          tmem_ld32(taddr, a0);
          tmem_ld32(taddr + 32, a1);
          tmem_ld_wait();
          tmem_ld32(taddr + 64, b0);
          tmem_ld32(taddr + 96, b1);
          put(a0, a1, 0);
          tmem_ld_wait();
          tmem_ld32(taddr + 128, a0);
          tmem_ld32(taddr + 160, a1);
          put(b0, b1, 1);
          tmem_ld_wait();
          tmem_ld32(taddr + 192, b0);
          tmem_ld32(taddr + 224, b1);
          put(a0, a1, 2);
          tmem_ld_wait();
          put(b0, b1, 3);
        }
      } else {
        const int m = tl.mt * BM + r_in_tile;
        const bool valid = m < tl.rows;
        const size_t row = static_cast<size_t>(tl.row0 + (valid ? m : 0));
        __nv_bfloat16* orow = cd.out + row * cd.ld_out + tl.j * cd.out_col_step + n_base;
#pragma unroll 1
        for (int c = 0; c < BN / 16; ++c) {
          float v[16];
          tmem_ld16(taddr + c * 16, v);
          tmem_ld_wait();
          if (!valid || n_base + c * 16 >= p.n_dim) continue;
          if (KIND == DG_SWIGLU) {
            // v = dh; [a | b] of the same row and columns (kept by the
            // training forward, or recomputed)
            __nv_bfloat16* arow = cd.ab + row * cd.ld_ab + tl.j * cd.ab_col_step + n_base + c * 16;
            __nv_bfloat16* brow = arow + p.n_dim;
            uint4 araw[2], braw[2];
            araw[0] = reinterpret_cast<const uint4*>(arow)[0];
            araw[1] = reinterpret_cast<const uint4*>(arow)[1];
            braw[0] = reinterpret_cast<const uint4*>(brow)[0];
            braw[1] = reinterpret_cast<const uint4*>(brow)[1];
            const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(araw);
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(braw);
            uint32_t da[8], db[8], hh[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float2 av = __bfloat1622float2(a2[i]);
              const float2 bv = __bfloat1622float2(b2[i]);
              float s0, g0, s1, g1;
              silu_and_grad(av.x, s0, g0);
              silu_and_grad(av.y, s1, g1);
              const float dh0 = v[2 * i], dh1 = v[2 * i + 1];
              da[i] = pack_bf16x2(dh0 * bv.x * g0, dh1 * bv.y * g1);
              db[i] = pack_bf16x2(dh0 * s0, dh1 * s1);
              hh[i] = pack_bf16x2(s0 * bv.x, s1 * bv.y);
            }
            uint4* ad = reinterpret_cast<uint4*>(arow);
            uint4* bd = reinterpret_cast<uint4*>(brow);
            uint4* hd = reinterpret_cast<uint4*>(orow + c * 16);
            ad[0] = make_uint4(da[0], da[1], da[2], da[3]);
            ad[1] = make_uint4(da[4], da[5], da[6], da[7]);
            bd[0] = make_uint4(db[0], db[1], db[2], db[3]);
            bd[1] = make_uint4(db[4], db[5], db[6], db[7]);
            hd[0] = make_uint4(hh[0], hh[1], hh[2], hh[3]);
            hd[1] = make_uint4(hh[4], hh[5], hh[6], hh[7]);
          } else {
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
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
    // the warp's last gradient stores have completed
    if (KIND == WG && lane == 0) bulk_wait_all();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace bwdgemm

// ------------------------------------------------------------------- host
template <int KIND>
static cudaError_t launch_bwd_gemm(const bwdgemm::Params& prm, cudaStream_t st) {
  using namespace bwdgemm;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(bwd_gemm_kernel<KIND>),
                                    static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  bwd_gemm_kernel<KIND><<<sm_count(), THREADS, kSmemBytes, st>>>(prm);
  return cudaGetLastError();
}

size_t experts_bwd_scratch_bytes(const moe_cfg_t& c) {
  const size_t tk = static_cast<size_t>(c.T) * c.K, T = c.T, I = c.inter, Ns = c.n_shared;
  // [a | b] (then [da | db]) and h, routed rows then shared rows, bf16
  return align_up((tk + T * Ns) * 3 * I * 2, 256);
}

ExpertsBwdScratch experts_bwd_scratch_carve(const moe_cfg_t& c, void* ws) {
  const size_t tk = static_cast<size_t>(c.T) * c.K, T = c.T, I = c.inter, Ns = c.n_shared;
  ExpertsBwdScratch r;
  __nv_bfloat16* p = static_cast<__nv_bfloat16*>(ws);
  r.ab = p;
  r.ab_shared = p + tk * 2 * I;
  r.h = r.ab_shared + T * Ns * 2 * I;
  r.h_shared = r.h + tk * I;
  return r;
}

// Row-major bf16 [rows, cols] with the 128-byte swizzle.
static CUresult encode_bf16_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                               uint32_t box_cols, uint32_t box_rows) {
  return encode_tensor_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(base), cols,
                              rows, cols * 2, box_cols, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

cudaError_t launch_experts_bwd_input_bf16(const ExpertsBwdArgs& a, cudaStream_t st) {
  using bwdgemm::BK;
  using bwdgemm::BM;
  const moe_cfg_t& c = *a.cfg;
  const uint64_t tk = static_cast<uint64_t>(c.T) * c.K;
  const int I = c.inter, Ns = c.n_shared, d = c.d;
  const bool has_shared = Ns > 0;
  const ExpertsBwdScratch w = a.scratch;

  // ---- 1. recompute [a | b] = x W13^T with the forward's plain grouped GEMM
  // (unless the training forward kept it)
  if (!a.ab_kept) {
    using namespace bf16gemm;
    Params g{};
    g.offsets = a.offsets; g.n_rows = static_cast<int>(tk); g.E = c.E; g.T = c.T; g.has_shared = has_shared ? 1 : 0;
    g.d = 2 * I;   // B rows of one routed matrix
    g.inter = d;   // K of one matrix
    // (each map also with half its box: the pair kernel's CTAs hold half a
    // B tile each, and 64 A rows each in a segment's last half tile)
    CUresult r = encode_bf16_2d(&g.a_map[0], a.x_perm, d, tk, BK, BM);
    if (r == CUDA_SUCCESS) r = encode_bf16_2d(&g.a_half[0], a.x_perm, d, tk, BK, BM / 2);
    if (r == CUDA_SUCCESS)
      r = encode_bf16_2d(&g.b_map[0], a.w13, d, static_cast<uint64_t>(c.E) * 2 * I, BK, BN);
    if (r == CUDA_SUCCESS)
      r = encode_bf16_2d(&g.b_half[0], a.w13, d, static_cast<uint64_t>(c.E) * 2 * I, BK, BN / 2);
    if (r == CUDA_SUCCESS && has_shared) {
      r = encode_bf16_2d(&g.a_map[1], a.x, d, c.T, BK, BM);
      if (r == CUDA_SUCCESS) r = encode_bf16_2d(&g.a_half[1], a.x, d, c.T, BK, BM / 2);
      if (r == CUDA_SUCCESS)
        r = encode_bf16_2d(&g.b_map[1], a.ws13, d, static_cast<uint64_t>(Ns) * 2 * I, BK, BN);
      if (r == CUDA_SUCCESS)
        r = encode_bf16_2d(&g.b_half[1], a.ws13, d, static_cast<uint64_t>(Ns) * 2 * I, BK, BN / 2);
    } else {
      g.a_map[1] = g.a_map[0];
      g.b_map[1] = g.b_map[0];
      g.a_half[1] = g.a_half[0];
      g.b_half[1] = g.b_half[0];
    }
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    g.cls[0] = ClassDesc{w.ab, 2 * I, 2 * I, d};
    g.cls[1] = ClassDesc{w.ab_shared, Ns * 2 * I, Ns * 2 * I, d};
    cudaError_t e = launch_bf16_pair_gemm<DOWN>(g, st);
    if (e != cudaSuccess) return e;
  }

  using namespace bwdgemm;
  // ---- 2. dh = dy W2; [da | db] over [a | b]; h
  Params p{};
  p.offsets = a.offsets; p.n_rows = static_cast<int>(static_cast<int64_t>(c.T) * c.K); p.E = c.E; p.T = c.T;
  p.n_sh = Ns;
  p.n_dim = I;
  CUresult r = encode_bf16_2d(&p.a_map[0], a.dy_perm, d, tk, BK, BM);
  if (r == CUDA_SUCCESS)
    r = encode_bf16_2d(&p.b_map[0], a.w2, I, static_cast<uint64_t>(c.E) * d, 64, BK);
  if (r == CUDA_SUCCESS && has_shared) {
    r = encode_bf16_2d(&p.a_map[1], a.dout, d, c.T, BK, BM);
    if (r == CUDA_SUCCESS)
      r = encode_bf16_2d(&p.b_map[1], a.ws2, I, static_cast<uint64_t>(Ns) * d, 64, BK);
  } else {
    p.a_map[1] = p.a_map[0];
    p.b_map[1] = p.b_map[0];
  }
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  p.cls[0] = ClassDesc{d, d, 0, 0, w.h, I, 0, 0, w.ab, 2 * I, 0};
  p.cls[1] = ClassDesc{d, d, 0, 0, w.h_shared, Ns * I, I, 0, w.ab_shared, Ns * 2 * I, 2 * I};
  cudaError_t e = launch_bwd_gemm<DG_SWIGLU>(p, st);
  if (e != cudaSuccess) return e;

  // ---- 3. dx = [da | db] W13 (routed rows; the shared experts' sum in one group)
  Params q{};
  q.offsets = a.offsets; q.n_rows = static_cast<int>(static_cast<int64_t>(c.T) * c.K); q.E = c.E; q.T = c.T;
  q.n_sh = has_shared ? 1 : 0;
  q.n_dim = d;
  r = encode_bf16_2d(&q.a_map[0], w.ab, 2 * I, tk, BK, BM);
  if (r == CUDA_SUCCESS)
    r = encode_bf16_2d(&q.b_map[0], a.w13, d, static_cast<uint64_t>(c.E) * 2 * I, 64, BK);
  if (r == CUDA_SUCCESS && has_shared) {
    r = encode_bf16_2d(&q.a_map[1], w.ab_shared, static_cast<uint64_t>(Ns) * 2 * I, c.T, BK, BM);
    if (r == CUDA_SUCCESS)
      r = encode_bf16_2d(&q.b_map[1], a.ws13, d, static_cast<uint64_t>(Ns) * 2 * I, 64, BK);
  } else {
    q.a_map[1] = q.a_map[0];
    q.b_map[1] = q.b_map[0];
  }
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  q.cls[0] = ClassDesc{2 * I, 2 * I, 0, 0, static_cast<__nv_bfloat16*>(a.dx_perm), d, 0, 0,
                       nullptr, 0, 0};
  q.cls[1] = ClassDesc{Ns * 2 * I, 0, 0, 0, static_cast<__nv_bfloat16*>(a.dx_shared), d, 0, 0,
                       nullptr, 0, 0};
  return launch_bwd_gemm<DG_PLAIN>(q, st);
}

// Wgrad output of a class: `groups` matrices [m, n] bf16 seen as a 3-D map
// with a 32-row x 64-column box (one epilogue warp's chunk, 128-byte swizzle).
static CUresult encode_wgrad_out(CUtensorMap* m, void* base, int rows, int cols, int groups) {
  const uint64_t dims[3] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                            static_cast<uint64_t>(groups)};
  const uint64_t strides[2] = {static_cast<uint64_t>(cols) * 2, static_cast<uint64_t>(rows) * cols * 2};
  const uint32_t box[3] = {64, 32, 1};
  return encode_tensor_map_nd(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, 3, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B);
}

cudaError_t launch_experts_bwd_weights_bf16(const ExpertsBwdArgs& a, cudaStream_t st) {
  using namespace bwdgemm;
  const moe_cfg_t& c = *a.cfg;
  const uint64_t tk = static_cast<uint64_t>(c.T) * c.K;
  const int I = c.inter, Ns = c.n_shared, d = c.d;
  const bool has_shared = Ns > 0;
  const ExpertsBwdScratch w = a.scratch;

  // ---- dW2 = dy^T h: M = d, N = I, K = the rows of the segment
  Params p{};
  p.offsets = a.offsets; p.n_rows = static_cast<int>(static_cast<int64_t>(c.T) * c.K); p.E = c.E; p.T = c.T;
  p.n_sh = Ns;
  p.m_dim = d;
  p.n_dim = I;
  CUresult r = encode_bf16_2d(&p.a_map[0], a.dy_perm, d, tk, 64, BK);
  if (r == CUDA_SUCCESS) r = encode_bf16_2d(&p.b_map[0], w.h, I, tk, 64, BK);
  if (r == CUDA_SUCCESS && has_shared) {
    r = encode_bf16_2d(&p.a_map[1], a.dout, d, c.T, 64, BK);
    if (r == CUDA_SUCCESS)
      r = encode_bf16_2d(&p.b_map[1], w.h_shared, static_cast<uint64_t>(Ns) * I, c.T, 64, BK);
  } else {
    p.a_map[1] = p.a_map[0];
    p.b_map[1] = p.b_map[0];
  }
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const size_t mat2 = static_cast<size_t>(d) * I;
  p.cls[0] = ClassDesc{0, 0, 0, 0, static_cast<__nv_bfloat16*>(a.dw2), 0, 0, mat2, nullptr, 0, 0};
  p.cls[1] = ClassDesc{0, 0, 0, I, static_cast<__nv_bfloat16*>(a.dws2), 0, 0, mat2, nullptr, 0, 0};
  r = encode_wgrad_out(&p.out_map[0], a.dw2, d, I, c.E);
  if (r == CUDA_SUCCESS)
    r = has_shared ? encode_wgrad_out(&p.out_map[1], a.dws2, d, I, Ns) : CUDA_SUCCESS;
  if (!has_shared) p.out_map[1] = p.out_map[0];
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  cudaError_t e = launch_bwd_gemm<WG>(p, st);
  if (e != cudaSuccess) return e;

  // ---- dW13 = [da | db]^T x: M = 2I, N = d
  Params q{};
  q.offsets = a.offsets; q.n_rows = static_cast<int>(static_cast<int64_t>(c.T) * c.K); q.E = c.E; q.T = c.T;
  q.n_sh = Ns;
  q.m_dim = 2 * I;
  q.n_dim = d;
  r = encode_bf16_2d(&q.a_map[0], w.ab, 2 * I, tk, 64, BK);
  if (r == CUDA_SUCCESS) r = encode_bf16_2d(&q.b_map[0], a.x_perm, d, tk, 64, BK);
  if (r == CUDA_SUCCESS && has_shared) {
    r = encode_bf16_2d(&q.a_map[1], w.ab_shared, static_cast<uint64_t>(Ns) * 2 * I, c.T, 64, BK);
    if (r == CUDA_SUCCESS) r = encode_bf16_2d(&q.b_map[1], a.x, d, c.T, 64, BK);
  } else {
    q.a_map[1] = q.a_map[0];
    q.b_map[1] = q.b_map[0];
  }
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const size_t mat13 = static_cast<size_t>(2) * I * d;
  q.cls[0] = ClassDesc{0, 0, 0, 0, static_cast<__nv_bfloat16*>(a.dw13), 0, 0, mat13, nullptr, 0, 0};
  q.cls[1] = ClassDesc{0, 0, 2 * I, 0, static_cast<__nv_bfloat16*>(a.dws13), 0, 0, mat13, nullptr,
                       0, 0};
  r = encode_wgrad_out(&q.out_map[0], a.dw13, 2 * I, d, c.E);
  if (r == CUDA_SUCCESS)
    r = has_shared ? encode_wgrad_out(&q.out_map[1], a.dws13, 2 * I, d, Ns) : CUDA_SUCCESS;
  if (!has_shared) q.out_map[1] = q.out_map[0];
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  return launch_bwd_gemm<WG>(q, st);
}

}  // namespace moe
