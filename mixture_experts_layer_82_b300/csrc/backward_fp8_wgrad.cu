// Backward for weights of the expert FFNs in FP8 E4M3 (the Wgrad GEMMs).
//
// "DeepSeek-V3 Technical Report", mixed precision framework paragraph
// (Figure 6): Wgrad runs in FP8 with fp32 accumulation; fine-grained
// quantisation paragraph: activation-like operands in tiles of 128 values
// with one fp32 scale each.  Wgrad contracts over the token rows of an
// expert's segment (dW2 = dy^T h, dW13 = [da | db]^T u), so both operands
// are quantised in 128 x 1 tiles: 128 consecutive rows of one column (a
// segment's last tile holds the rows that are left, the missing ones are
// zeros).  Per 128-row block of the segment the tensor cores form the
// block's partial product, and the promotion adds partial * sa[row] *
// sb[column] to fp32 registers: unlike the forward, B's scale varies along
// the output columns, so it is applied per element.
//
// Layout.  The operands are formed on the fly from what the FP8 backward
// for input left in the workspace (dy: the caller's rows; u: the dequantised
// forward codes; h = silu(a) b and [da | db] from [a | b] and dh, with the
// input side's formulas) and written row-major, every segment padded to
// whole 128-row tiles: codes [P_max, C] and scales [P_max / 128, C], where
// segment e occupies rows [poff_e, poff_e + 128 * ceil(n_e / 128)).  The
// GEMM reads both operands MN-major: a TMA box is one 128-row K block of
// 128 columns (128 bytes, the 128-byte swizzle), so no operand is ever
// transposed.  Its epilogue stages each bf16 tile in shared memory and
// writes it with a TMA store.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace wgfp8 {

constexpr int BM = 128, BN = 128, BK = 128;  // BK: rows of one 128 x 1 tile
constexpr int STAGES = 5;                            // operand ring
constexpr int A_BYTES = BM * BK, B_BYTES = BN * BK;  // 16 KiB each
constexpr int PARTS = 4;                             // TMEM partials of BN columns
constexpr int SLOTS = 8;                             // scale ring: a K block's sa and sb rows
constexpr uint32_t TMEM_COLS = PARTS * BN;           // 512
constexpr int EPI_WARP0 = 2;                         // warps 2..9: promotion + epilogue
constexpr int THREADS = (EPI_WARP0 + 8) * 32;        // 320
constexpr int MAX_GROUPS = 1025;
constexpr int HALF_BYTES = BM * 64 * 2;              // one 64-column bf16 half of a tile
constexpr uint32_t SCALE_BYTES = (BM + BN) * 4;
// E4M3 x E4M3 -> fp32; bits 15 and 16: A and B MN-major
constexpr uint32_t IDESC = idesc_f32acc(0, 0, BM, BN) | (1u << 15) | (1u << 16);

// The operand a quantise pass forms from the workspace.
enum Src { DY = 0, U = 1, H = 2, DAB = 3 };

// ------------------------------------------------------- padded segments
// poff[e] = 128 * sum_{e' < e} ceil(n_e' / 128), poff[E] = padded total;
// tile_rows[t] = (first row of segment e in padded tile t, rows of the
// segment in that tile) for every padded tile t < poff[E] / 128.
__global__ void pad_offsets_kernel(const int32_t* __restrict__ offsets, int E, int64_t n_rows,
                                   int32_t* __restrict__ poff, int2* __restrict__ tile_rows) {
  const int lane = threadIdx.x;
  const int per = ceil_div(E, 32);
  const int g0 = lane * per, g1 = min(E, g0 + per);
  int sum = 0;
  for (int g = g0; g < g1; ++g) {
    int o0;
    sum += ceil_div(checked_segment(offsets, g, n_rows, o0), 128) * 128;
  }
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  int run = incl - sum;
  for (int g = g0; g < g1; ++g) {
    poff[g] = run;
    int o0;
    const int n = checked_segment(offsets, g, n_rows, o0);
    for (int j = 0; j * 128 < n; ++j)
      tile_rows[run / 128 + j] = make_int2(o0 + 128 * j, min(128, n - 128 * j));
    run += ceil_div(n, 128) * 128;
  }
  if (lane == 31) poff[E] = incl;
}

// A quantise pass: the tile's source boxes (128 rows x 128 columns each) are
// copied by TMA into shared memory: dy; the forward's codes; a and b of
// [a | b]; a, b and dh.
struct QtParams {
  CUtensorMap src;           // DY: dy [rows, C]; U: codes [rows, C]; H, DAB: [a | b] [rows, 2I]
  CUtensorMap dh;            // DAB: dh [rows, I]
  const int2* tile_rows;     // routed: rows of every padded tile; null for the shared class
  const int32_t* poff;       // routed: padded starts
  int E;
  int n_rows;                // shared: T
  int C;                     // columns of X
  int inter;                 // I (H, DAB)
  const float* xs;           // U: the forward's 1 x 128 scales [rows, C / 128]
  uint8_t* q;                // out: codes [P, C], row-major
  float* s;                  // out: scales [P / 128, C]
};

template <int SRC>
struct QtLayout {
  static constexpr int ELEM = SRC == U ? 1 : 2;            // bytes of a source value
  static constexpr int BOX = 128 * 128 * ELEM;             // one 128 x 128 box
  static constexpr int BOXES = SRC == DAB ? 3 : (SRC == H ? 2 : 1);
  static constexpr int BYTES = BOX * BOXES;
};

__device__ __forceinline__ float4 bf16x4(const uint8_t* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}

__device__ __forceinline__ float4 sigmoid4(float4 a) {
  return make_float4(1.f / (1.f + __expf(-a.x)), 1.f / (1.f + __expf(-a.y)),
                     1.f / (1.f + __expf(-a.z)), 1.f / (1.f + __expf(-a.w)));
}

// Values of columns 4l .. 4l + 3 of the block's 128 (one 128-column group
// and one half of [da | db]) in row r of the staged tile.
template <int SRC>
__device__ __forceinline__ float4 staged_quad(const uint8_t* t, int r, int l, bool da, float xscale) {
  constexpr int RB = 128 * QtLayout<SRC>::ELEM;  // bytes of a staged row
  if (SRC == DY) return bf16x4(t + r * RB + 8 * l);
  if (SRC == U) {
    const uint32_t q4 = *reinterpret_cast<const uint32_t*>(t + r * RB + 4 * l);
    const __half2_raw lo =
        __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(q4 & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi =
        __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(q4 >> 16), __NV_E4M3);
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&lo));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&hi));
    return make_float4(f0.x * xscale, f0.y * xscale, f1.x * xscale, f1.y * xscale);
  }
  const float4 av = bf16x4(t + r * RB + 8 * l);
  const float4 bv = bf16x4(t + QtLayout<SRC>::BOX + r * RB + 8 * l);
  const float4 sg = sigmoid4(av);
  if (SRC == H)
    return make_float4(av.x * sg.x * bv.x, av.y * sg.y * bv.y, av.z * sg.z * bv.z, av.w * sg.w * bv.w);
  const float4 h = bf16x4(t + 2 * QtLayout<SRC>::BOX + r * RB + 8 * l);
  if (da)
    return make_float4(h.x * bv.x * (sg.x * (1.f + av.x * (1.f - sg.x))),
                       h.y * bv.y * (sg.y * (1.f + av.y * (1.f - sg.y))),
                       h.z * bv.z * (sg.z * (1.f + av.z * (1.f - sg.z))),
                       h.w * bv.w * (sg.w * (1.f + av.w * (1.f - sg.w))));
  return make_float4(h.x * (av.x * sg.x), h.y * (av.y * sg.y), h.z * (av.z * sg.z),
                     h.w * (av.w * sg.w));
}

// One block per (128-row tile of the padded layout, 128 columns).  Thread
// 0 copies the tile's source boxes into shared memory (rows past the
// segment are copied too and zeroed here); warp w then forms rows
// 16w .. 16w + 15, lane l columns 4l .. 4l + 3, the amax of each column over
// the 128 rows is reduced through shared memory, and every store of a warp
// covers one row's 128 codes.
template <int SRC>
__global__ void __launch_bounds__(256) quant_rows_kernel(const __grid_constant__ QtParams a) {
  extern __shared__ uint8_t qt_smem[];
  uint8_t* tile = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(qt_smem) + 127) & ~static_cast<uintptr_t>(127));
  __shared__ float4 red[8][32];
  __shared__ alignas(8) uint64_t bar;
  __shared__ int qt_abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int pt = blockIdx.x;  // padded row tile
  const int c0 = blockIdx.y * 128;
  const int p0 = pt * 128;
  // the rows of padded tile pt: [row0, row0 + count) of X
  int row0, count;
  if (a.tile_rows != nullptr) {
    if (p0 >= a.poff[a.E]) return;  // past the last segment (the whole block)
    const int2 tr = a.tile_rows[pt];
    row0 = tr.x;
    count = tr.y;
  } else {
    row0 = p0;
    count = min(128, a.n_rows - p0);
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    qt_abort = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t pol = l2_policy_evict_first();
    mbar_arrive_expect_tx(&bar, QtLayout<SRC>::BYTES);
    if (SRC == DY || SRC == U) {
      tma_load_2d(tile, &a.src, &bar, c0, row0, pol);
    } else {
      const int i0 = SRC == H || c0 < a.inter ? c0 : c0 - a.inter;
      tma_load_2d(tile, &a.src, &bar, i0, row0, pol);
      tma_load_2d(tile + QtLayout<SRC>::BOX, &a.src, &bar, a.inter + i0, row0, pol);
      if (SRC == DAB) tma_load_2d(tile + 2 * QtLayout<SRC>::BOX, &a.dh, &bar, i0, row0, pol);
    }
  }
  // U: the forward's scale of each of this thread's rows (while the copy runs)
  float xsc[16];
#pragma unroll
  for (int r = 0; r < 16; ++r)
    xsc[r] = SRC == U ? a.xs[static_cast<int64_t>(row0 + min(warp * 16 + r, count - 1)) * (a.C / 128) +
                             c0 / 128]
                      : 1.f;
  // A wait that gives up sets the error word; the whole block then leaves
  // together (nothing written) instead of some threads reaching a barrier.
  const bool landed = mbar_wait(&bar, 0, &qt_abort);
  if (__syncthreads_or(landed ? 0 : 1)) return;
  const bool da = c0 < a.inter;
  float4 v[16];
  float4 m = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int lr = warp * 16 + r;
    v[r] = lr < count ? staged_quad<SRC>(tile, lr, lane, da, xsc[r]) : make_float4(0.f, 0.f, 0.f, 0.f);
    m = make_float4(fmaxf(m.x, fabsf(v[r].x)), fmaxf(m.y, fabsf(v[r].y)),
                    fmaxf(m.z, fabsf(v[r].z)), fmaxf(m.w, fabsf(v[r].w)));
  }
  red[warp][lane] = m;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const float4 o = red[w][lane];
    m = make_float4(fmaxf(m.x, o.x), fmaxf(m.y, o.y), fmaxf(m.z, o.z), fmaxf(m.w, o.w));
  }
  const float4 sc = make_float4(fp8_scale_of(m.x), fp8_scale_of(m.y), fp8_scale_of(m.z),
                                fp8_scale_of(m.w));
  const float4 rc = make_float4(__frcp_rn(sc.x), __frcp_rn(sc.y), __frcp_rn(sc.z), __frcp_rn(sc.w));
  const int c = c0 + 4 * lane;
  uint8_t* dst = a.q + static_cast<int64_t>(p0 + warp * 16) * a.C + c;
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const uint32_t lo = e4m3x2_of_quotients(v[r].x, v[r].y, sc.x, sc.y, rc.x, rc.y);
    const uint32_t hi = e4m3x2_of_quotients(v[r].z, v[r].w, sc.z, sc.w, rc.z, rc.w);
    *reinterpret_cast<uint32_t*>(dst + static_cast<int64_t>(r) * a.C) = lo | (hi << 16);
  }
  if (warp == 0) *reinterpret_cast<float4*>(a.s + static_cast<int64_t>(pt) * a.C + c) = sc;
}

// ------------------------------------------------------------ Wgrad GEMM
struct ClassDesc {
  int m_total, n_total;  // dW rows (columns of A) and columns (columns of B)
  const float* sa;       // [P / 128, m_total]
  const float* sb;       // [P / 128, n_total]
};

struct Params {
  CUtensorMap a_map[2];    // [class] A codes [P, m_total]: box 128 rows x 128 columns
  CUtensorMap b_map[2];    // [class] B codes [P, n_total]
  CUtensorMap out_map[2];  // [class] dW bf16 [groups][m_total][n_total]: box 1 x 128 x 64
  ClassDesc cls[2];
  const int32_t* poff;     // routed padded starts [E + 1]
  int E;
  int has_shared;
  int p_shared;            // the shared class's padded rows
};

struct Smem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t pfull[PARTS];
  uint64_t pempty[PARTS];
  uint64_t sfull[SLOTS];  // the slot's scale rows have landed
  uint64_t sfree[SLOTS];  // the promotion has read them (8 warp arrivals)
  uint64_t stg_full[2];  // [half] the staging half is written (4 warp arrivals)
  uint64_t stg_free[2];  // [half] the last store of the half has read it
  uint64_t done;
  uint32_t tmem_base;
  int abort;
  int n_groups;
  alignas(16) float sa[SLOTS][BM];  // scale rows of K block j in slot j % SLOTS
  alignas(16) float sb[SLOTS][BN];
  int gstart[MAX_GROUPS + 1];  // first tile of every group
  int kbeg[MAX_GROUPS];        // padded rows [kbeg, kend) of every group
  int kend[MAX_GROUPS];
};

constexpr size_t kRingBytes = static_cast<size_t>(STAGES) * (A_BYTES + B_BYTES);
constexpr size_t kStageOutBytes = 2 * HALF_BYTES;
constexpr size_t kSmemBytes = 1024 + kRingBytes + kStageOutBytes + sizeof(Smem);
static_assert(kSmemBytes <= 232448, "above the 227 KiB of shared memory a block may use");

// Shared-memory descriptor of an MN-major E4M3 operand tile: K row r is the
// 128-byte line r (128 values of M or N, 128-byte swizzle, 8-row atoms
// 1024 bytes apart).  A tile is one atom wide, so the leading byte offset
// (the next 128 values of M or N) is never used.
__device__ __forceinline__ uint64_t sdesc_mn_fp8_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);       // start address
  d |= static_cast<uint64_t>(A_BYTES >> 4) << 16;            // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;               // stride byte offset: next 8 K rows
  d |= static_cast<uint64_t>(1) << 46;                       // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                       // 128-byte swizzle
  return d;
}

__device__ __forceinline__ int tiles_of(const Params& p, int cls) {
  return ceil_div(p.cls[cls].m_total, BM) * ceil_div(p.cls[cls].n_total, BN);
}

// Groups: the E routed experts, then the shared expert; every group has all
// its (M, N) tiles, with as many K blocks as its padded rows / 128 (none
// for an expert without rows: a zero tile).
__device__ void build_table(const Params& p, Smem& s) {
  const int lane = threadIdx.x % 32;
  const int G = p.E + (p.has_shared ? 1 : 0);
  const int per = ceil_div(G, 32);
  const int g0 = lane * per, g1 = min(G, g0 + per);
  int sum = 0;
  for (int g = g0; g < g1; ++g) sum += tiles_of(p, g < p.E ? 0 : 1);
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  int run = incl - sum;
  for (int g = g0; g < g1; ++g) {
    s.gstart[g] = run;
    run += tiles_of(p, g < p.E ? 0 : 1);
    s.kbeg[g] = g < p.E ? p.poff[g] : 0;
    s.kend[g] = g < p.E ? p.poff[g + 1] : p.p_shared;
  }
  if (lane == 31) {
    s.gstart[G] = incl;
    s.n_groups = G;
  }
}

struct Tile {
  int cls, group, mt, nt, k0, nk;  // k0: first padded row; nk: 128-row blocks
};

__device__ __forceinline__ Tile decode(const Params& p, const Smem& s, int t, int& g) {
  while (s.gstart[g + 1] <= t) ++g;
  Tile tl;
  tl.group = g;
  tl.cls = g < p.E ? 0 : 1;
  const int local = t - s.gstart[g];
  const int mtn = ceil_div(p.cls[tl.cls].m_total, BM);
  tl.mt = local % mtn;
  tl.nt = local / mtn;
  tl.k0 = s.kbeg[g];
  tl.nk = max(s.kend[g] - tl.k0, 0) / BK;
  return tl;
}

__global__ void __launch_bounds__(THREADS, 1) wgrad_fp8_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stage_out = ring + kRingBytes;  // two 64-column halves, 1024-byte aligned
  Smem& s = *reinterpret_cast<Smem*>(stage_out + kStageOutBytes);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  volatile int* abort_flag = &s.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      tma_prefetch_desc(&p.a_map[i]);
      tma_prefetch_desc(&p.b_map[i]);
      tma_prefetch_desc(&p.out_map[i]);
    }
    for (int i = 0; i < STAGES; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], 1); }
    for (int i = 0; i < PARTS; ++i) { mbar_init(&s.pfull[i], 1); mbar_init(&s.pempty[i], 8); }
    for (int i = 0; i < SLOTS; ++i) { mbar_init(&s.sfull[i], 1); mbar_init(&s.sfree[i], 8); }
    for (int i = 0; i < 2; ++i) { mbar_init(&s.stg_full[i], 4); mbar_init(&s.stg_free[i], 1); }
    mbar_init(&s.done, 1);
    s.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  if (warp == 0) build_table(p, s);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_base;
  const int total = s.gstart[s.n_groups];

  if (warp == 0) {
    // ----------------------------------------------------------- producer
    // K block j of the CTA: A and B boxes into ring stage j % STAGES, their
    // scale rows into slot j % SLOTS once the promotion has read that slot.
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_normal();
      uint32_t g = 0;  // K blocks of the CTA so far
      int gh = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < total && !stop && !*abort_flag; t += gridDim.x) {
        const Tile tl = decode(p, s, t, gh);
        const ClassDesc& cd = p.cls[tl.cls];
        for (int kb = 0; kb < tl.nk; ++kb, ++g) {
          const int stage = static_cast<int>(g % STAGES);
          const int slot = static_cast<int>(g % SLOTS);
          if (!mbar_wait(&s.empty[stage], ((g / STAGES) & 1u) ^ 1u, abort_flag)) { stop = true; break; }
          if (!mbar_wait(&s.sfree[slot], ((g / SLOTS) & 1u) ^ 1u, abort_flag)) { stop = true; break; }
          uint8_t* sa = ring + stage * A_BYTES;
          uint8_t* sb = ring + STAGES * A_BYTES + stage * B_BYTES;
          const int row = tl.k0 + kb * BK;
          const int64_t pt = row / BK;
          mbar_arrive_expect_tx(&s.full[stage], A_BYTES + B_BYTES);
          tma_load_2d(sa, &p.a_map[tl.cls], &s.full[stage], tl.mt * BM, row, pol);
          tma_load_2d(sb, &p.b_map[tl.cls], &s.full[stage], tl.nt * BN, row, pol);
          mbar_arrive_expect_tx(&s.sfull[slot], SCALE_BYTES);
          bulk_load(s.sa[slot], cd.sa + pt * cd.m_total + tl.mt * BM, BM * 4, &s.sfull[slot]);
          bulk_load(s.sb[slot], cd.sb + pt * cd.n_total + tl.nt * BN, BN * 4, &s.sfull[slot]);
        }
      }
      // Drain: the last copies of every stage and slot have landed (after an
      // abort too; in the normal path the MMA thread and the promotion have
      // waited for all of them).
      for (uint32_t i = 0; i < static_cast<uint32_t>(STAGES) && i < g; ++i) {
        const uint32_t j = g - 1 - i;
        mbar_wait_drain(&s.full[j % STAGES], (j / STAGES) & 1u);
      }
      for (uint32_t i = 0; i < static_cast<uint32_t>(SLOTS) && i < g; ++i) {
        const uint32_t j = g - 1 - i;
        mbar_wait_drain(&s.sfull[j % SLOTS], (j / SLOTS) & 1u);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    // K block j of the CTA goes to TMEM partial j % 4; the MMAs run up to
    // three blocks ahead of the promotion, the loads up to STAGES more.
    if (lane == 0) {
      uint32_t g = 0;
      int gh = 0;
      bool any = false, ok = true;
      for (int t = blockIdx.x; t < total && ok && !*abort_flag; t += gridDim.x) {
        const Tile tl = decode(p, s, t, gh);
        for (int kb = 0; kb < tl.nk; ++kb, ++g) {
          const int stage = static_cast<int>(g % STAGES);
          const int part = static_cast<int>(g % PARTS);
          if (!mbar_wait(&s.full[stage], (g / STAGES) & 1u, abort_flag)) { ok = false; break; }
          if (!mbar_wait(&s.pempty[part], ((g / PARTS) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = sdesc_mn_fp8_sw128(smem_u32(ring + stage * A_BYTES));
          const uint64_t bd = sdesc_mn_fp8_sw128(smem_u32(ring + STAGES * A_BYTES + stage * B_BYTES));
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(part * BN);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)  // +32 K rows = +4096 bytes = +256 in the address field
            mma_fp8_ss(d_tmem, ad + 256 * k, bd + 256 * k, IDESC, k != 0 ? 1u : 0u);
          any = true;
          mma_commit(&s.pfull[part]);
          mma_commit(&s.empty[stage]);
        }
      }
      if (any) {
        mma_commit(&s.done);
        mbar_wait_drain(&s.done, 0);
      }
    }
  } else {
    // ------------------------------------------------ promotion + epilogue
    // Warp w reads TMEM lanes 32 * (w % 4) .. +31 (its 32 rows of the tile);
    // warps 2..5 own columns 0..63 of a partial, warps 6..9 columns 64..127.
    // The warp with w % 4 == 0 of each half issues that half's TMA stores.
    const int q = warp & 3;
    const int hf = (warp - EPI_WARP0) >> 2;
    const bool issuer = q == 0 && lane == 0;
    const int mrow = q * 32 + lane;  // row of the tile
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    uint8_t* half = stage_out + hf * HALF_BYTES;
    uint32_t g = 0, it = 0;
    int gh = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
      const Tile tl = decode(p, s, t, gh);
      float acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = 0.f;
      for (int kb = 0; kb < tl.nk; ++kb, ++g) {
        const int part = static_cast<int>(g % PARTS);
        const int slot = static_cast<int>(g % SLOTS);
        if (!mbar_wait(&s.pfull[part], (g / PARTS) & 1u, abort_flag)) { ok = false; break; }
        if (!mbar_wait(&s.sfull[slot], (g / SLOTS) & 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t taddr = lane_addr + static_cast<uint32_t>(part * BN + hf * 64);
        const float sa = s.sa[slot][mrow];
        const float* sbp = &s.sb[slot][hf * 64];
        // two 32-column batches (one batch in registers at a time: 64
        // accumulators + 32 values fit the 168 registers of 10 warps)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float x[32];
          tmem_ld32(taddr + 32 * h, x);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            // acc += (x * sb) * sa, two lanes per packed instruction
            const float4 b = *reinterpret_cast<const float4*>(sbp + 32 * h + j);
            float p0, p1, p2, p3;
            fmul2(p0, p1, x[j + 0], x[j + 1], b.x, b.y);
            fmul2(p2, p3, x[j + 2], x[j + 3], b.z, b.w);
            ffma2_bcast(acc[32 * h + j + 0], acc[32 * h + j + 1], p0, p1, sa);
            ffma2_bcast(acc[32 * h + j + 2], acc[32 * h + j + 3], p2, p3, sa);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&s.pempty[part]);
          mbar_arrive(&s.sfree[slot]);
        }
      }
      if (!ok) break;
      // epilogue: the staging half is free once this half's previous store
      // has read it
      if (issuer) {
        bulk_wait_read_all();
        mbar_arrive(&s.stg_free[hf]);
      }
      if (!mbar_wait(&s.stg_free[hf], it & 1u, abort_flag)) break;
      uint8_t* rowp = half + mrow * 128;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 v = make_uint4(pack_bf16x2(acc[8 * j + 0], acc[8 * j + 1]),
                                   pack_bf16x2(acc[8 * j + 2], acc[8 * j + 3]),
                                   pack_bf16x2(acc[8 * j + 4], acc[8 * j + 5]),
                                   pack_bf16x2(acc[8 * j + 6], acc[8 * j + 7]));
        *reinterpret_cast<uint4*>(rowp + ((j ^ (mrow & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.stg_full[hf]);
      if (issuer) {
        if (!mbar_wait(&s.stg_full[hf], it & 1u, abort_flag)) break;
        tma_store_3d(&p.out_map[tl.cls], half, tl.nt * BN + hf * 64, tl.mt * BM,
                     tl.cls == 0 ? tl.group : 0);
        bulk_commit();
      }
    }
    if (issuer) bulk_wait_all();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Padded rows of the routed class at most: every segment rounded up to 128.
inline int64_t p_max(const moe_cfg_t& c) {
  return (static_cast<int64_t>(c.T) * c.K + 127 * static_cast<int64_t>(c.E) + 127) / 128 * 128;
}
inline int64_t p_shared(const moe_cfg_t& c) { return (static_cast<int64_t>(c.T) + 127) / 128 * 128; }

struct WgScratch {
  int32_t* poff;
  int2* tile_rows;  // [P / 128]
  uint8_t* q[4];   // dy [P, d], u [P, d], h [P, I], [da | db] [P, 2I]: codes
  float* s[4];     // and scales [P / 128, C]
  uint8_t* qs[4];  // the shared class's, [P_s, C]
  float* ss[4];
};

inline int cols_of(const moe_cfg_t& c, int src) {
  return src == H ? c.inter : (src == DAB ? 2 * c.inter : c.d);
}

inline size_t wg_bytes(const moe_cfg_t& c, WgScratch* out, void* base) {
  char* p = static_cast<char*>(base);
  size_t n = 0;
  auto take = [&](size_t bytes) {
    char* q = p == nullptr ? nullptr : p + n;
    n += align_up(bytes, 256);
    return q;
  };
  const int64_t P = p_max(c), Ps = p_shared(c);
  void* poff = take(static_cast<size_t>(c.E + 1) * 4);
  void* tile_rows = take(static_cast<size_t>(P / 128) * 8);
  if (out != nullptr) {
    out->poff = static_cast<int32_t*>(poff);
    out->tile_rows = static_cast<int2*>(tile_rows);
  }
  for (int src = 0; src < 4; ++src) {
    const size_t C = static_cast<size_t>(cols_of(c, src));
    void* q = take(C * P);
    void* s = take(static_cast<size_t>(P / 128) * C * 4);
    void* qs = take(c.n_shared ? C * Ps : 0);
    void* ss = take(c.n_shared ? static_cast<size_t>(Ps / 128) * C * 4 : 0);
    if (out != nullptr) {
      out->q[src] = static_cast<uint8_t*>(q);
      out->s[src] = static_cast<float*>(s);
      out->qs[src] = static_cast<uint8_t*>(qs);
      out->ss[src] = static_cast<float*>(ss);
    }
  }
  return n;
}

template <int SRC>
cudaError_t launch_quant_rows(const QtParams& q, dim3 grid, cudaStream_t st) {
  constexpr int bytes = QtLayout<SRC>::BYTES + 128;  // + alignment of the staged tile
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(quant_rows_kernel<SRC>), bytes);
  if (e != cudaSuccess) return e;
  quant_rows_kernel<SRC><<<grid, 256, bytes, st>>>(q);
  return cudaGetLastError();
}

// One quantise pass: operand `src` of class `cls` (0 routed, 1 shared).
cudaError_t quantise_operand(const ExpertsBwdWeightsFp8Args& a, const WgScratch& w, int src,
                             int cls, cudaStream_t st) {
  const moe_cfg_t& c = *a.cfg;
  const int64_t tk = static_cast<int64_t>(c.T) * c.K;
  const int I = c.inter, d = c.d;
  const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle NOSW = CU_TENSOR_MAP_SWIZZLE_NONE;
  QtParams q{};
  q.tile_rows = cls == 0 ? w.tile_rows : nullptr;
  q.poff = w.poff;
  q.E = c.E;
  q.n_rows = cls == 0 ? static_cast<int>(tk) : c.T;
  q.C = cols_of(c, src);
  q.inter = I;
  const uint64_t rows = cls == 0 ? static_cast<uint64_t>(tk) : static_cast<uint64_t>(c.T);
  CUresult r = CUDA_SUCCESS;
  if (src == DY) {
    void* dy = const_cast<void*>(cls == 0 ? a.dy_perm : a.dout);
    r = encode_tensor_map_2d(&q.src, BF, dy, d, rows, static_cast<uint64_t>(d) * 2, 128, 128, NOSW);
  } else if (src == U) {
    void* xq = const_cast<void*>(cls == 0 ? a.x_perm : a.x_q);
    r = encode_tensor_map_2d(&q.src, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, d, rows,
                             static_cast<uint64_t>(d), 128, 128, NOSW);
    q.xs = cls == 0 ? a.x_perm_scales : a.x_q_scales;
  } else {
    const __nv_bfloat16* ab = cls == 0 ? a.ab : a.ab + tk * 2 * I;
    const __nv_bfloat16* dh = cls == 0 ? a.dh : a.dh + tk * I;
    r = encode_tensor_map_2d(&q.src, BF, const_cast<__nv_bfloat16*>(ab), 2 * I, rows,
                             static_cast<uint64_t>(I) * 4, 128, 128, NOSW);
    if (r == CUDA_SUCCESS && src == DAB)
      r = encode_tensor_map_2d(&q.dh, BF, const_cast<__nv_bfloat16*>(dh), I, rows,
                               static_cast<uint64_t>(I) * 2, 128, 128, NOSW);
  }
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  q.q = cls == 0 ? w.q[src] : w.qs[src];
  q.s = cls == 0 ? w.s[src] : w.ss[src];
  const dim3 grid(static_cast<unsigned>((cls == 0 ? p_max(c) : p_shared(c)) / 128), q.C / 128);
  switch (src) {
    case DY: return launch_quant_rows<DY>(q, grid, st);
    case U: return launch_quant_rows<U>(q, grid, st);
    case H: return launch_quant_rows<H>(q, grid, st);
    default: return launch_quant_rows<DAB>(q, grid, st);
  }
}

}  // namespace wgfp8

cudaError_t launch_quantize_act_128x1(const void* x, int rows, int cols, uint8_t* q, float* scales,
                                      cudaStream_t st) {
  using namespace wgfp8;
  QtParams prm{};
  prm.tile_rows = nullptr;  // one segment: all rows
  prm.n_rows = rows;
  prm.C = cols;
  CUresult r = encode_tensor_map_2d(&prm.src, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(x),
                                    static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                                    static_cast<uint64_t>(cols) * 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  prm.q = q;
  prm.s = scales;
  return launch_quant_rows<DY>(prm, dim3(static_cast<unsigned>((rows + 127) / 128), cols / 128), st);
}

size_t experts_wgrad_fp8_scratch_bytes(const moe_cfg_t& c) {
  return wgfp8::wg_bytes(c, nullptr, nullptr);
}

cudaError_t launch_experts_bwd_weights_fp8(const ExpertsBwdWeightsFp8Args& a, cudaStream_t st) {
  using namespace wgfp8;
  const moe_cfg_t& c = *a.cfg;
  const int64_t tk = static_cast<int64_t>(c.T) * c.K;
  const int I = c.inter, d = c.d;
  const bool has_shared = c.n_shared > 0;
  if (d % 128 != 0 || I % 128 != 0) return cudaErrorInvalidValue;
  WgScratch w{};
  wg_bytes(c, &w, a.wg_ws);
  const int64_t P = p_max(c), Ps = p_shared(c);

  pad_offsets_kernel<<<1, 32, 0, st>>>(a.offsets, c.E, tk, w.poff, w.tile_rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // 1. the four operands, quantised in 128 x 1 tiles, row-major
  for (int src = 0; src < 4; ++src) {
    for (int cls = 0; cls < (has_shared ? 2 : 1); ++cls) {
      e = quantise_operand(a, w, src, cls, st);
      if (e != cudaSuccess) return e;
    }
  }

  e = ensure_smem_limit(reinterpret_cast<const void*>(wgrad_fp8_kernel), static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapSwizzle SW = CU_TENSOR_MAP_SWIZZLE_128B;
  // 2. dW2 = dy^T h  ([d, I]),  dW13 = [da | db]^T u  ([2I, d])
  const int A_SRC[2] = {DY, DAB}, B_SRC[2] = {H, U};
  void* outs[2] = {a.dw2, a.dw13};
  void* outs_sh[2] = {a.dws2, a.dws13};
  for (int gm = 0; gm < 2; ++gm) {
    const int as = A_SRC[gm], bs = B_SRC[gm];
    const int M = cols_of(c, as), N = cols_of(c, bs);
    Params p{};
    p.poff = w.poff;
    p.E = c.E;
    p.has_shared = has_shared ? 1 : 0;
    p.p_shared = static_cast<int>(Ps);
    const uint32_t obox[3] = {64, BM, 1};
    const uint64_t ostr[2] = {static_cast<uint64_t>(N) * 2, static_cast<uint64_t>(M) * N * 2};
    const uint64_t odim[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M),
                              static_cast<uint64_t>(c.E)};
    const uint64_t odim_sh[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M), 1};
    CUresult r = encode_tensor_map_2d(&p.a_map[0], U8, w.q[as], M, P, M, BM, BK, SW);
    if (r == CUDA_SUCCESS) r = encode_tensor_map_2d(&p.b_map[0], U8, w.q[bs], N, P, N, BN, BK, SW);
    if (r == CUDA_SUCCESS)
      r = encode_tensor_map_nd(&p.out_map[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, outs[gm], 3, odim,
                               ostr, obox, SW);
    if (r == CUDA_SUCCESS && has_shared) {
      r = encode_tensor_map_2d(&p.a_map[1], U8, w.qs[as], M, Ps, M, BM, BK, SW);
      if (r == CUDA_SUCCESS) r = encode_tensor_map_2d(&p.b_map[1], U8, w.qs[bs], N, Ps, N, BN, BK, SW);
      if (r == CUDA_SUCCESS)
        r = encode_tensor_map_nd(&p.out_map[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, outs_sh[gm], 3,
                                 odim_sh, ostr, obox, SW);
    } else {
      p.a_map[1] = p.a_map[0];
      p.b_map[1] = p.b_map[0];
      p.out_map[1] = p.out_map[0];
    }
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    p.cls[0] = ClassDesc{M, N, w.s[as], w.s[bs]};
    p.cls[1] = has_shared ? ClassDesc{M, N, w.ss[as], w.ss[bs]} : p.cls[0];
    wgrad_fp8_kernel<<<sm_count(), THREADS, kSmemBytes, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
