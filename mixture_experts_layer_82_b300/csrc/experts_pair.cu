// Grouped expert GEMMs for the bf16 kind on CTA pairs: every tcgen05.mma
// runs with cta_group::2 and spans the two SMs of a cluster.
//
// "DeepSeek-V3 Technical Report", DeepSeekMoE paragraph: each routed expert
// is a SwiGLU FFN applied to the tokens routed to it, the shared experts to
// every token; same two launches as experts_sm100.cu (gate/up with SwiGLU
// in the epilogue, down), same work list of (group, M tile, N tile).
//
// Why pairs.  A single-CTA 128 x 256 tile makes its SM take in 48 KiB of
// operands per 64-deep K block (A 16 KiB, B 32 KiB), and that intake, not
// the tensor pipe, bounds a dense GEMM of these shapes.  In a pair MMA each
// CTA holds its own A rows and only half of the B tile; the two SMs' tensor
// cores share the B halves, so an SM takes in 32 KiB per K block for the
// same MMA work.  (Measured on a dense 8192 x 4096 x 7168 GEMM: 0.71 of the
// bf16 peak with one CTA per tile, 0.80 with pairs.  In a routed layer
// whose experts are mostly small, streaming their weights bounds the GEMMs
// instead, and pairs then gain little.)
//
// Tiles.  An expert's segment is cut into 256-row pair tiles (M = 256: 128
// rows per CTA).  A segment's last tile is a half tile when at most 128
// rows are left (M = 128: 64 rows per CTA), so the rows padded to a tile
// boundary are the same as with 128-row tiles.  TMEM layout of the pair
// MMA (each CTA's share of D): M = 256 puts row r of the CTA in lane r with
// column n in TMEM column n; M = 128 puts row r (0..63) in lanes r and
// r + 64, with columns n < 128 in lane r and columns n >= 128 in lane
// r + 64, both at TMEM column n % 128.  So in a half gate/up tile each CTA
// loads 64 W1 rows followed by the matching 64 W3 rows (the a and b of 64
// h columns share a lane); in a full tile CTA 0 loads 128 W1 rows and CTA 1
// the matching 128 W3 rows.  Down tiles split B's 256 rows between the CTAs.
//
// Synchronisation.  Both CTAs' producers fill their own ring slots; their
// copies complete on the even CTA's full barrier, which expects both CTAs'
// bytes.  The even CTA's MMA thread issues the pair MMAs; its commits arrive
// on the empty and accumulator-full barriers of both CTAs.  Each CTA's
// epilogue drains its own TMEM; the even CTA's four warps arrive on its
// accumulator-empty barrier, the odd CTA's on a local one, which a relay
// thread passes on with one cluster-scope arrival (a warp's own
// cluster-scope release would wait for its outstanding output stores).
// Every wait is bounded.
//
// Roles (224 threads, one CTA per SM, clusters of two): warps 0 and 6 TMA
// producers (alternate stages of a 6-stage ring of 32 KiB), warp 1 TMEM
// allocation (both CTAs), the MMA thread (even CTA) or the relay (odd CTA),
// warps 2..5 the epilogue.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace bf16gemm {

constexpr int P2_STAGES = 6;                    // even: two producers take alternate stages
constexpr int P2_A_BYTES = BM * BK * 2;         // a CTA's A rows (128; 64 in a half tile)
constexpr int P2_B_BYTES = (BN / 2) * BK * 2;   // a CTA's half of the B tile
constexpr uint32_t P2_IDESC_FULL = idesc_f32acc(1, 1, 2 * BM, BN);  // M = 256 over the pair
constexpr uint32_t P2_IDESC_HALF = idesc_f32acc(1, 1, BM, BN);      // M = 128 over the pair

struct Smem2 {
  uint64_t full[P2_STAGES];   // even CTA: both CTAs' copies of the stage have landed
  uint64_t empty[P2_STAGES];  // both CTAs: the pair MMAs have read the stage
  uint64_t tfull[2];          // both CTAs: the accumulator holds the tile
  uint64_t tempty[2];         // even CTA: both epilogues have drained it (4 local warps + 1 relay)
  uint64_t tdrained[2];       // odd CTA: its 4 epilogue warps have drained it
  uint64_t done;
  uint32_t tmem_base;
  int abort;
  int n_groups;
  int gstart[MAX_GROUPS + 1];  // first tile of every group
  int mtiles[MAX_GROUPS];      // pair M tiles of every group
  int off[MAX_GROUPS];         // first row of every routed group (copy of offsets[0..E])
};

constexpr size_t kP2RingBytes = static_cast<size_t>(P2_STAGES) * (P2_A_BYTES + P2_B_BYTES);
constexpr size_t kP2SmemBytes = 1024 + kP2RingBytes + sizeof(Smem2);
static_assert(kP2SmemBytes <= 232448, "above the 227 KiB of shared memory a block may use");

struct Tile2 {
  int cls, group;  // class (0 routed, 1 shared), routed expert index
  int row0, rows;  // first row of the group in its class's row space, its rows
  int mt, nt;      // pair M tile (256 rows), N tile
  bool half;       // a last tile with at most 128 rows: M = 128 over the pair
};

__device__ __forceinline__ int pair_mtiles(int rows) { return rows > 0 ? ceil_div(rows, 2 * BM) : 0; }

template <int MODE>
__device__ void build_table2(const Params& p, Smem2& s) {
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
    s.mtiles[g] = pair_mtiles(rows);
    sum += s.mtiles[g] * n_tiles_of<MODE>(p, cls);
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
    run += s.mtiles[g] * n_tiles_of<MODE>(p, g < p.E ? 0 : 1);
  }
  if (lane == 31) {
    s.gstart[G] = incl;
    s.n_groups = G;
    s.off[p.E] = p.offsets[p.E];
  }
}

// Tile t of the cluster's work list; inside a group the M tile varies
// fastest, so the clusters running together share each weight tile in L2.
template <int MODE>
__device__ __forceinline__ Tile2 decode_tile2(const Params& p, const Smem2& s, int t) {
  int lo = 0, hi = s.n_groups;  // gstart[lo] <= t < gstart[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.gstart[mid] <= t) lo = mid; else hi = mid;
  }
  Tile2 tl;
  tl.cls = lo < p.E ? 0 : 1;
  tl.group = lo;
  const int local = t - s.gstart[lo];
  const int mtn = s.mtiles[lo];
  tl.mt = local % mtn;
  tl.nt = local / mtn;
  if (tl.cls == 0) { tl.row0 = s.off[lo]; tl.rows = s.off[lo + 1] - tl.row0; }
  else { tl.row0 = 0; tl.rows = p.T; }
  tl.half = tl.rows - tl.mt * 2 * BM <= BM;
  return tl;
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1) experts_bf16_pair_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Smem2& s = *reinterpret_cast<Smem2*>(ring + kP2RingBytes);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  volatile int* abort_flag = &s.abort;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      tma_prefetch_desc(&p.a_map[i]);
      tma_prefetch_desc(&p.a_half[i]);
      tma_prefetch_desc(&p.b_half[i]);
      if (MODE == GATEUP) tma_prefetch_desc(&p.b_mix[i]);
    }
    for (int i = 0; i < P2_STAGES; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], 5);
      mbar_init(&s.tdrained[i], 4);
    }
    mbar_init(&s.done, 1);
    s.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&s.tmem_base, TMEM_COLS);
    tmem_relinquish_pair();
    tc_fence_before();
  }
  if (warp == 2) build_table2<MODE>(p, s);
  __syncthreads();
  // both CTAs' barriers are initialised before either signals the other's
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_base;
  const int total = s.gstart[s.n_groups];
  const int w_first = static_cast<int>(blockIdx.x) >> 1;
  const int w_step = static_cast<int>(gridDim.x) >> 1;
  constexpr int HALF_RING = P2_STAGES / 2;

  if (warp == 0 || warp == PRODUCER2) {
    // ----------------------------------------------------------- producers
    // Warp 0 fills the even stages of the CTA's stage sequence (slots 0, 2,
    // 4), warp 6 the odd ones; a stage is this CTA's A rows and its half of
    // the B tile, completing on the even CTA's full barrier.
    if (lane == 0) {
      const uint32_t par = warp == 0 ? 0u : 1u;
      const uint64_t pol_a = l2_policy_evict_last();
      const uint64_t pol_b = l2_policy_evict_normal();
      uint32_t g = 0, mine = 0;
      bool stop = false;
      for (int t = w_first; t < total && !stop && !*abort_flag; t += w_step) {
        const Tile2 tl = decode_tile2<MODE>(p, s, t);
        const int nk = p.cls[tl.cls].k_dim / BK;
        const int rows_here = tl.half ? BM / 2 : BM;
        const int a_row = tl.row0 + tl.mt * 2 * BM + static_cast<int>(rank) * rows_here;
        const CUtensorMap* am = tl.half ? &p.a_half[tl.cls] : &p.a_map[tl.cls];
        const uint32_t stage_bytes = 2u * (rows_here * BK * 2 + P2_B_BYTES);
        // B coordinates as in experts_sm100.cu: gate/up (k, i0, matrix,
        // expert) in the [n][2][I][d] view, down (k, row) in [n * d, I]
        int bmat = 0, bi = 0, bxk = 0, brow = 0;
        if (MODE == GATEUP) {
          const int n0 = tl.nt * (BN / 2);
          bmat = tl.cls == 0 ? tl.group : n0 / p.inter;
          bi = n0 % p.inter;
        } else {
          brow = (tl.cls == 0 ? tl.group : 0) * p.d + tl.nt * BN + static_cast<int>(rank) * (BN / 2);
        }
        for (int kb = 0; kb < nk; ++kb, ++g) {
          if ((g & 1u) == par) {
            const int stage = static_cast<int>(par + 2 * (mine % HALF_RING));
            const uint32_t sphase = (mine / HALF_RING) & 1u;
            if (!mbar_wait(&s.empty[stage], sphase ^ 1u, abort_flag)) { stop = true; break; }
            uint8_t* sa = ring + stage * P2_A_BYTES;
            uint8_t* sb = ring + P2_STAGES * P2_A_BYTES + stage * P2_B_BYTES;
            const uint32_t full = cluster_addr(&s.full[stage], 0);
            if (rank == 0) mbar_arrive_expect_tx(&s.full[stage], stage_bytes);
            tma_load_2d_pair(sa, am, full, kb * BK, a_row, pol_a);
            if (MODE == GATEUP) {
              if (tl.half)  // 64 W1 rows, then the matching 64 W3 rows
                tma_load_4d_pair(sb, &p.b_mix[tl.cls], full, kb * BK, bi + static_cast<int>(rank) * 64, 0,
                                 bmat, pol_b);
              else  // 128 W1 rows (CTA 0) or the matching 128 W3 rows (CTA 1)
                tma_load_4d_pair(sb, &p.b_half[tl.cls], full, kb * BK, bi, static_cast<int>(rank), bmat,
                                 pol_b);
            } else {
              tma_load_2d_pair(sb, &p.b_half[tl.cls], full, bxk, brow, pol_b);
            }
            ++mine;
          }
          if (MODE == DOWN) {
            bxk += BK;
            if (bxk == p.inter) { bxk = 0; brow += p.d; }
          }
        }
      }
      // Drain: the pair MMAs that read this thread's last stages have
      // completed, so those copies have landed (their completion went to the
      // even CTA's barrier).
      for (uint32_t i = 0; i < static_cast<uint32_t>(HALF_RING) && i < mine; ++i) {
        const uint32_t j = mine - 1 - i;
        mbar_wait_drain(&s.empty[par + 2 * (j % HALF_RING)], (j / HALF_RING) & 1u);
      }
    }
  } else if (warp == 1 && rank != 0) {
    // ------------------------------------------- relay (odd CTA, warp 1)
    // Once the odd CTA's four epilogue warps have drained an accumulator
    // (CTA-scope arrivals), one cluster-scope arrival tells the even CTA's
    // MMA thread; this thread has no stores of its own to wait for.
    if (lane == 0) {
      const uint32_t tempty_even0 = cluster_addr(&s.tempty[0], 0);
      const uint32_t tempty_even1 = cluster_addr(&s.tempty[1], 0);
      int it = 0;
      for (int t = w_first; t < total; t += w_step, ++it) {
        const int acc = it & 1;
        if (!mbar_wait(&s.tdrained[acc], static_cast<uint32_t>(it >> 1) & 1u, abort_flag)) break;
        mbar_arrive_cluster(acc ? tempty_even1 : tempty_even0);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------- MMA (even CTA only)
    if (lane == 0 && rank == 0) {
      uint32_t stage = 0, phase = 0;
      int it = 0;
      bool any = false;
      for (int t = w_first; t < total && !*abort_flag; t += w_step, ++it) {
        const Tile2 tl = decode_tile2<MODE>(p, s, t);
        const int nk = p.cls[tl.cls].k_dim / BK;
        const int acc = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
        if (!mbar_wait(&s.tempty[acc], use ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        const uint32_t idesc = tl.half ? P2_IDESC_HALF : P2_IDESC_FULL;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&s.full[stage], phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(ring + stage * P2_A_BYTES);
          const uint32_t b0 = smem_u32(ring + P2_STAGES * P2_A_BYTES + stage * P2_B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_bf16_pair(d_tmem, sdesc_kmajor_sw128(a0 + k * 32), sdesc_kmajor_sw128(b0 + k * 32), idesc,
                          (kb | k) != 0 ? 1u : 0u);
          any = true;
          mma_commit_pair(&s.empty[stage], 0x3);
          if (++stage == P2_STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit_pair(&s.tfull[acc], 0x3);
      }
      // Drain: every pair MMA issued by this thread has completed after this.
      if (any) {
        mma_commit_pair(&s.done, 0x1);
        mbar_wait_drain(&s.done, 0);
      }
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int it = 0;
    for (int t = w_first; t < total; t += w_step, ++it) {
      const Tile2 tl = decode_tile2<MODE>(p, s, t);
      const ClassDesc& cd = p.cls[tl.cls];
      const int acc = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
      if (!mbar_wait(&s.tfull[acc], use, abort_flag)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + static_cast<uint32_t>(acc * BN) +
                             (static_cast<uint32_t>(q * 32) << 16);
      // this lane's row of the CTA's share and, in a half tile, its half of N
      const int rows_here = tl.half ? BM / 2 : BM;
      const int r = tl.half ? (q & 1) * 32 + lane : q * 32 + lane;
      const int nh = tl.half ? q >> 1 : 0;
      const int m = tl.mt * 2 * BM + static_cast<int>(rank) * rows_here + r;
      const bool valid = m < tl.rows;
      const int n_base = tl.nt * out_tile_cols<MODE>();
      __nv_bfloat16* orow = cd.out + static_cast<size_t>(tl.row0 + (valid ? m : 0)) * cd.ld_out + n_base;
      if (MODE == GATEUP) {
        // h columns of this lane: all 128 of the tile (a in TMEM columns
        // 0..127, b in 128..255), or 64 of them in a half tile (a in 0..63,
        // b in 64..127)
        const int hc = tl.half ? 64 : 128;
        const int h0 = nh * 64;
        __nv_bfloat16* abrow =
            cd.ab != nullptr && valid
                ? cd.ab + static_cast<size_t>(tl.row0 + m) * cd.ld_ab +
                      (n_base / p.inter) * 2 * p.inter + n_base % p.inter + h0
                : nullptr;
#pragma unroll 1
        for (int c = 0; c < hc / 16; ++c) {
          float a[16], b[16];
          tmem_ld16(taddr + c * 16, a);
          tmem_ld16(taddr + hc + c * 16, b);
          tmem_ld_wait();
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            pk[i] = pack_bf16x2(silu_f(a[2 * i]) * b[2 * i], silu_f(a[2 * i + 1]) * b[2 * i + 1]);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + h0 + c * 16);
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
        // output columns of this lane: all 256 (TMEM columns 0..255), or the
        // half nh of them in a half tile (TMEM columns 0..127)
        const int nc = tl.half ? 128 : 256;
        const int c0 = nh * 128;
        const float gm = cd.gate != nullptr && valid ? cd.gate[tl.row0 + m] : 1.f;
#pragma unroll 1
        for (int c = 0; c < nc / 16; ++c) {
          float v[16];
          tmem_ld16(taddr + c * 16, v);
          tmem_ld_wait();
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(v[2 * i] * gm, v[2 * i + 1] * gm);
          if (valid && n_base + c0 + c * 16 < cd.n_out) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c0 + c * 16);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      // (CTA scope: the even CTA's warps arrive on its own barrier, the odd
      // CTA's on theirs, which warp 1 relays)
      if (lane == 0) mbar_arrive(rank == 0 ? &s.tempty[acc] : &s.tdrained[acc]);
    }
  }
  __syncthreads();
  // neither CTA leaves while the other's MMAs may read its shared memory or
  // its epilogue may arrive on its barriers
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace bf16gemm

// Clusters of two CTAs that can be resident at once (one CTA per SM).
int experts_pair_clusters(const void* func, const cudaLaunchConfig_t& cfg);

template <int MODE>
cudaError_t launch_bf16_pair_gemm(const bf16gemm::Params& prm, cudaStream_t st) {
  using namespace bf16gemm;
  const void* func = reinterpret_cast<const void*>(experts_bf16_pair_kernel<MODE>);
  cudaError_t e = ensure_smem_limit(func, static_cast<int>(kP2SmemBytes));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = kP2SmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2);
  cfg.gridDim = dim3(2 * experts_pair_clusters(func, cfg));
  e = cudaLaunchKernelEx(&cfg, experts_bf16_pair_kernel<MODE>, prm);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
