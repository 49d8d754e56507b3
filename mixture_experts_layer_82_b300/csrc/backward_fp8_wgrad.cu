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
// Layout.  A TMA copy must start on a 16-byte boundary along its inner
// dimension, and segments start anywhere, so every operand is first written
// transposed, with each segment padded to whole 128-row tiles: X^T codes
// [C, P_max] (column c of X is row c of X^T) and scales [P_max / 128, C],
// where segment e occupies columns [poff_e, poff_e + 128 * ceil(n_e / 128))
// of X^T.  The K blocks of the Wgrad GEMM are then plain 128-byte-aligned
// boxes.  The operands are formed on the fly from what the FP8 backward
// for input left in the workspace: dy (the caller's dy rows), u =
// dequantised forward codes, h = silu(a) b and [da | db] from [a | b] and dh,
// with the same formulas as the input side.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace wgfp8 {

constexpr int BM = 128, BN = 128, BK = 128;  // BK bytes: one 128-row tile of a segment
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK, B_BYTES = BN * BK;  // 16 KiB each
constexpr int PARTS = 4;                             // TMEM partials of BN columns
constexpr uint32_t TMEM_COLS = PARTS * BN;           // 512
constexpr int EPI_WARP0 = 2;                         // warps 2..9: promotion + epilogue
constexpr int THREADS = (EPI_WARP0 + 8) * 32;        // 320
constexpr int MAX_GROUPS = 1025;
constexpr uint32_t IDESC = idesc_f32acc(0, 0, BM, BN);  // E4M3 x E4M3 -> fp32

// The operand a quantise-transpose pass forms from the workspace.
enum Src { DY = 0, U = 1, H = 2, DAB = 3 };

// ------------------------------------------------------- padded segments
// poff[e] = 128 * sum_{e' < e} ceil(n_e' / 128), poff[E] = padded total.
__global__ void pad_offsets_kernel(const int32_t* __restrict__ offsets, int E, int64_t n_rows,
                                   int32_t* __restrict__ poff) {
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
    run += ceil_div(checked_segment(offsets, g, n_rows, o0), 128) * 128;
  }
  if (lane == 31) poff[E] = incl;
}

struct QtArgs {
  const int32_t* offsets;     // routed: segment starts; null for the shared class
  const int32_t* poff;        // routed: padded starts
  int E;
  int64_t n_rows;             // routed: T * K (segment bound); shared: T
  int C;                      // columns of X
  int inter;                  // I (H, DAB)
  int64_t p_stride;           // columns of X^T (P_max)
  const __nv_bfloat16* dy;    // DY: [rows, C]
  const uint8_t* xq;          // U: E4M3 codes [rows, C] and 1 x 128 scales
  const float* xs;
  const __nv_bfloat16* ab;    // H, DAB: [rows, 2I]
  const __nv_bfloat16* dh;    // DAB: [rows, I]
  uint8_t* xt;                // out: X^T codes [C, p_stride]
  float* st;                  // out: scales [p_stride / 128, C]
};

// One block per (128-row tile of the padded layout, 128 columns): thread j
// owns column c; it forms the tile's 128 values of its column, takes their
// amax, and writes the 128 codes as one contiguous 128-byte run of X^T.
template <int SRC>
__global__ void __launch_bounds__(128) quant_t_kernel(const QtArgs a) {
  const int pt = blockIdx.x;              // padded row tile
  const int c = blockIdx.y * 128 + threadIdx.x;
  const int p0 = pt * 128;
  // the segment holding padded rows [p0, p0 + 128)
  int row0, count, local0;
  if (a.offsets != nullptr) {
    if (p0 >= a.poff[a.E]) return;        // past the last segment
    int lo = 0, hi = a.E;                 // poff[lo] <= p0 < poff[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (a.poff[mid] <= p0) lo = mid; else hi = mid;
    }
    while (lo + 1 < a.E && a.poff[lo + 1] <= p0) ++lo;  // skip empty segments
    count = checked_segment(a.offsets, lo, a.n_rows, row0);
    local0 = p0 - a.poff[lo];
  } else {
    row0 = 0;
    count = static_cast<int>(a.n_rows);
    local0 = p0;
  }
  float v[128];
  float amax = 0.f;
#pragma unroll
  for (int r = 0; r < 128; ++r) {
    float x = 0.f;
    if (local0 + r < count) {
      const int64_t row = static_cast<int64_t>(row0) + local0 + r;
      if (SRC == DY) {
        x = __bfloat162float(a.dy[row * a.C + c]);
      } else if (SRC == U) {
        const __nv_fp8_e4m3 q = *reinterpret_cast<const __nv_fp8_e4m3*>(a.xq + row * a.C + c);
        x = static_cast<float>(q) * a.xs[row * (a.C / 128) + c / 128];
      } else {
        const int i = SRC == H || c < a.inter ? c : c - a.inter;
        const float av = __bfloat162float(a.ab[row * 2 * a.inter + i]);
        const float bv = __bfloat162float(a.ab[row * 2 * a.inter + a.inter + i]);
        const float s = 1.f / (1.f + __expf(-av));
        if (SRC == H) {
          x = av * s * bv;
        } else {
          const float h = __bfloat162float(a.dh[row * a.inter + i]);
          x = c < a.inter ? h * bv * (s * (1.f + av * (1.f - s))) : h * (av * s);
        }
      }
    }
    v[r] = x;
    amax = fmaxf(amax, fabsf(x));
  }
  const float scale = fp8_scale_of(amax);
  uint8_t* dst = a.xt + static_cast<int64_t>(c) * a.p_stride + p0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      w[k] = quant4_e4m3(v[16 * j + 4 * k], v[16 * j + 4 * k + 1], v[16 * j + 4 * k + 2],
                         v[16 * j + 4 * k + 3], scale);
    reinterpret_cast<uint4*>(dst)[j] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  a.st[static_cast<int64_t>(pt) * a.C + c] = scale;
}

// ------------------------------------------------------------ Wgrad GEMM
struct ClassDesc {
  int m_total, n_total;  // dW rows (rows of A^T) and columns (rows of B^T)
  const float* sa;       // [P / 128, m_total]
  const float* sb;       // [P / 128, n_total]
  __nv_bfloat16* out;    // [groups, m_total, n_total]
};

struct Params {
  CUtensorMap a_map[2];  // [class] A^T codes [m_total, P]: box 128 x 128
  CUtensorMap b_map[2];  // [class] B^T codes [n_total, P]
  ClassDesc cls[2];
  const int32_t* poff;   // routed padded starts [E + 1]
  int E;
  int has_shared;
  int p_shared;          // the shared class's padded rows
};

struct Smem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t pfull[PARTS];
  uint64_t pempty[PARTS];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
  int n_groups;
  int gstart[MAX_GROUPS + 1];  // first tile of every group
  int kbeg[MAX_GROUPS];        // padded rows [kbeg, kend) of every group
  int kend[MAX_GROUPS];
};

constexpr size_t kRingBytes = static_cast<size_t>(STAGES) * (A_BYTES + B_BYTES);
constexpr size_t kSmemBytes = 1024 + kRingBytes + sizeof(Smem);
static_assert(kSmemBytes <= 232448, "above the 227 KiB of shared memory a block may use");

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
  Smem& s = *reinterpret_cast<Smem*>(ring + kRingBytes);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  volatile int* abort_flag = &s.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) { tma_prefetch_desc(&p.a_map[i]); tma_prefetch_desc(&p.b_map[i]); }
    for (int i = 0; i < STAGES; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], 1); }
    for (int i = 0; i < PARTS; ++i) { mbar_init(&s.pfull[i], 1); mbar_init(&s.pempty[i], 8); }
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
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_normal();
      uint32_t g = 0;  // K blocks of the CTA so far
      int gh = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < total && !stop && !*abort_flag; t += gridDim.x) {
        const Tile tl = decode(p, s, t, gh);
        for (int kb = 0; kb < tl.nk; ++kb, ++g) {
          const int stage = static_cast<int>(g % STAGES);
          if (!mbar_wait(&s.empty[stage], ((g / STAGES) & 1u) ^ 1u, abort_flag)) { stop = true; break; }
          uint8_t* sa = ring + stage * A_BYTES;
          uint8_t* sb = ring + STAGES * A_BYTES + stage * B_BYTES;
          mbar_arrive_expect_tx(&s.full[stage], A_BYTES + B_BYTES);
          tma_load_2d(sa, &p.a_map[tl.cls], &s.full[stage], tl.k0 + kb * BK, tl.mt * BM, pol);
          tma_load_2d(sb, &p.b_map[tl.cls], &s.full[stage], tl.k0 + kb * BK, tl.nt * BN, pol);
        }
      }
      // (one producer uses every slot: without an abort the MMA thread has
      // waited for every stage, so every load has landed)
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    // K block j of the CTA goes to TMEM partial j % 4; the MMAs run up to
    // three blocks ahead of the promotion.
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
          const uint64_t ad = sdesc_kmajor_sw128(smem_u32(ring + stage * A_BYTES));
          const uint64_t bd = sdesc_kmajor_sw128(smem_u32(ring + STAGES * A_BYTES + stage * B_BYTES));
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(part * BN);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)  // +32 bytes along K = +2 in the address field
            mma_fp8_ss(d_tmem, ad + 2 * k, bd + 2 * k, IDESC, k != 0 ? 1u : 0u);
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
    const int q = warp & 3;
    const int hf = (warp - EPI_WARP0) >> 2;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t g = 0;
    int gh = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = decode(p, s, t, gh);
      const ClassDesc& cd = p.cls[tl.cls];
      const int m = tl.mt * BM + q * 32 + lane;  // dW row of this thread
      const int n0 = tl.nt * BN + hf * 64;       // first of its 64 columns
      const bool row_ok = m < cd.m_total;
      float acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = 0.f;
      for (int kb = 0; kb < tl.nk; ++kb, ++g) {
        const int part = static_cast<int>(g % PARTS);
        const int64_t pt = tl.k0 / BK + kb;  // padded row tile: the scales' row
        const float sa = row_ok ? __ldg(cd.sa + pt * cd.m_total + m) : 0.f;
        const float* sbp = cd.sb + pt * cd.n_total + n0;
        if (!mbar_wait(&s.pfull[part], (g / PARTS) & 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t taddr = lane_addr + static_cast<uint32_t>(part * BN + hf * 64);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float x[32];
          tmem_ld32(taddr + r * 32, x);
          tmem_ld_wait();
          if (r == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.pempty[part]);
          }
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            // column scales: the same for every lane (one broadcast load)
            const float4 sb = n0 + r * 32 + j < cd.n_total
                                  ? __ldg(reinterpret_cast<const float4*>(sbp + r * 32 + j))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            acc[r * 32 + j + 0] = fmaf(x[j + 0] * sb.x, sa, acc[r * 32 + j + 0]);
            acc[r * 32 + j + 1] = fmaf(x[j + 1] * sb.y, sa, acc[r * 32 + j + 1]);
            acc[r * 32 + j + 2] = fmaf(x[j + 2] * sb.z, sa, acc[r * 32 + j + 2]);
            acc[r * 32 + j + 3] = fmaf(x[j + 3] * sb.w, sa, acc[r * 32 + j + 3]);
          }
        }
      }
      if (!ok) break;
      if (row_ok) {
        __nv_bfloat16* orow = cd.out + (static_cast<size_t>(tl.cls == 0 ? tl.group : 0) * cd.m_total + m) *
                                           cd.n_total + n0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (n0 + c * 16 < cd.n_total) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 16);
            dst[0] = make_uint4(pack_bf16x2(acc[c * 16 + 0], acc[c * 16 + 1]),
                                pack_bf16x2(acc[c * 16 + 2], acc[c * 16 + 3]),
                                pack_bf16x2(acc[c * 16 + 4], acc[c * 16 + 5]),
                                pack_bf16x2(acc[c * 16 + 6], acc[c * 16 + 7]));
            dst[1] = make_uint4(pack_bf16x2(acc[c * 16 + 8], acc[c * 16 + 9]),
                                pack_bf16x2(acc[c * 16 + 10], acc[c * 16 + 11]),
                                pack_bf16x2(acc[c * 16 + 12], acc[c * 16 + 13]),
                                pack_bf16x2(acc[c * 16 + 14], acc[c * 16 + 15]));
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

}  // namespace wgfp8

// ------------------------------------------------------------------- host
namespace wgfp8 {

// Padded rows of the routed class at most: every segment rounded up to 128.
inline int64_t p_max(const moe_cfg_t& c) {
  return (static_cast<int64_t>(c.T) * c.K + 127 * static_cast<int64_t>(c.E) + 127) / 128 * 128;
}
inline int64_t p_shared(const moe_cfg_t& c) { return (static_cast<int64_t>(c.T) + 127) / 128 * 128; }

struct WgScratch {
  int32_t* poff;
  uint8_t* t[4];   // DY^T [d, P], U^T [d, P], H^T [I, P], DAB^T [2I, P]
  float* s[4];
  uint8_t* ts[4];  // the shared class's, [*, P_s]
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
  if (out != nullptr) out->poff = static_cast<int32_t*>(poff);
  for (int src = 0; src < 4; ++src) {
    const size_t C = static_cast<size_t>(cols_of(c, src));
    void* t = take(C * P);
    void* s = take(static_cast<size_t>(P / 128) * C * 4);
    void* ts = take(c.n_shared ? C * Ps : 0);
    void* ss = take(c.n_shared ? static_cast<size_t>(Ps / 128) * C * 4 : 0);
    if (out != nullptr) {
      out->t[src] = static_cast<uint8_t*>(t);
      out->s[src] = static_cast<float*>(s);
      out->ts[src] = static_cast<uint8_t*>(ts);
      out->ss[src] = static_cast<float*>(ss);
    }
  }
  return n;
}

}  // namespace wgfp8

size_t experts_wgrad_fp8_scratch_bytes(const moe_cfg_t& c) {
  return wgfp8::wg_bytes(c, nullptr, nullptr);
}

cudaError_t launch_experts_bwd_weights_fp8(const ExpertsBwdWeightsFp8Args& a, cudaStream_t st) {
  using namespace wgfp8;
  const moe_cfg_t& c = *a.cfg;
  const int64_t tk = static_cast<int64_t>(c.T) * c.K;
  const int I = c.inter, d = c.d;
  const bool has_shared = c.n_shared > 0;
  WgScratch w{};
  wg_bytes(c, &w, a.wg_ws);
  const int64_t P = p_max(c), Ps = p_shared(c);

  pad_offsets_kernel<<<1, 32, 0, st>>>(a.offsets, c.E, tk, w.poff);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // 1. the four operands, transposed and quantised in 128 x 1 tiles
  for (int src = 0; src < 4; ++src) {
    const int C = cols_of(c, src);
    for (int cls = 0; cls < (has_shared ? 2 : 1); ++cls) {
      QtArgs q{};
      q.offsets = cls == 0 ? a.offsets : nullptr;
      q.poff = w.poff;
      q.E = c.E;
      q.n_rows = cls == 0 ? tk : c.T;
      q.C = C;
      q.inter = I;
      q.p_stride = cls == 0 ? P : Ps;
      q.dy = static_cast<const __nv_bfloat16*>(cls == 0 ? a.dy_perm : a.dout);
      q.xq = static_cast<const uint8_t*>(cls == 0 ? a.x_perm : a.x_q);
      q.xs = cls == 0 ? a.x_perm_scales : a.x_q_scales;
      q.ab = cls == 0 ? a.ab : a.ab + tk * 2 * I;
      q.dh = cls == 0 ? a.dh : a.dh + tk * I;
      q.xt = cls == 0 ? w.t[src] : w.ts[src];
      q.st = cls == 0 ? w.s[src] : w.ss[src];
      const dim3 grid(static_cast<unsigned>((cls == 0 ? P : Ps) / 128), C / 128);
      switch (src) {
        case DY: quant_t_kernel<DY><<<grid, 128, 0, st>>>(q); break;
        case U: quant_t_kernel<U><<<grid, 128, 0, st>>>(q); break;
        case H: quant_t_kernel<H><<<grid, 128, 0, st>>>(q); break;
        default: quant_t_kernel<DAB><<<grid, 128, 0, st>>>(q); break;
      }
      e = cudaGetLastError();
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
    CUresult r = encode_tensor_map_2d(&p.a_map[0], U8, w.t[as], P, M, P, BK, BM, SW);
    if (r == CUDA_SUCCESS) r = encode_tensor_map_2d(&p.b_map[0], U8, w.t[bs], P, N, P, BK, BN, SW);
    if (r == CUDA_SUCCESS && has_shared) {
      r = encode_tensor_map_2d(&p.a_map[1], U8, w.ts[as], Ps, M, Ps, BK, BM, SW);
      if (r == CUDA_SUCCESS) r = encode_tensor_map_2d(&p.b_map[1], U8, w.ts[bs], Ps, N, Ps, BK, BN, SW);
    } else {
      p.a_map[1] = p.a_map[0];
      p.b_map[1] = p.b_map[0];
    }
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    p.cls[0] = ClassDesc{M, N, w.s[as], w.s[bs], static_cast<__nv_bfloat16*>(outs[gm])};
    p.cls[1] = has_shared ? ClassDesc{M, N, w.ss[as], w.ss[bs], static_cast<__nv_bfloat16*>(outs_sh[gm])}
                          : p.cls[0];
    wgrad_fp8_kernel<<<sm_count(), THREADS, kSmemBytes, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
