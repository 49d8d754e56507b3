// Router product on the tensor cores for bf16 token rows.
//
// "DeepSeek-V3 Technical Report", mixed-precision framework paragraph: the
// MoE gating stays in high precision.  The token rows x are bf16 (exact in
// bf16); every fp32 centroid is split into three bf16 terms,
//     e = e_hi + e_mid + e_lo   (e_hi = bf16(e), e_mid = bf16(e - e_hi), ...)
// which carry 24 significand bits, so
//     x . e = x . e_hi + x . e_mid + x . e_lo
// is a sum of exact bf16 x bf16 products.  A long chain of tcgen05.mma
// accumulations loses precision (the same observation as the report's
// increased-precision accumulation paragraph), so the sum is promoted: the
// tensor cores accumulate one 128-element K chunk (all three terms) into a
// TMEM partial, and the epilogue warps add each chunk's partial to fp32
// registers in chunk order.  Two TMEM partials alternate so the MMAs never
// wait for the promotion.
//
// One 128 x 128 output tile per CTA (tokens x experts).  When the tiles do
// not fill the GPU (decode-sized T) the d range is split over CTAs; every
// split writes its fp32 partial and a second kernel adds the partials in
// split order (deterministic) and applies the sigmoid.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace routertc {

constexpr int BM = 128, BN = 128, BK = 64;
constexpr int KB_PER_CHUNK = 2;              // 128 K elements per promotion
constexpr int STAGES = 3;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_PART_BYTES = BN * BK * 2;
constexpr int B_BYTES = 3 * B_PART_BYTES;  // hi, mid, lo tiles
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 256;          // two 128-column partials
constexpr uint32_t IDESC = idesc_f32acc(1, 1, BM, BN);
constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(STAGES) * (A_BYTES + B_BYTES) + 256;

struct Params {
  CUtensorMap a_map;  // x [T, d] bf16
  CUtensorMap b_map;  // split centroids [E, 3d] bf16
  float* out;         // splits == 1: affinities [T, E]; else partials [splits, T, E]
  int T, E, d;
  int nkb;            // k blocks of d
  int kb_per_split;
  int splits;
};

struct Bars {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t pfull[2];
  uint64_t pempty[2];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(THREADS, 1) router_tc_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars& s = *reinterpret_cast<Bars*>(ring + STAGES * (A_BYTES + B_BYTES));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  volatile int* abort_flag = &s.abort;
  const int nt = blockIdx.x, mt = blockIdx.y, split = blockIdx.z;
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(p.nkb, kb0 + p.kb_per_split);
  const int n_chunks = ceil_div(kb1 - kb0, KB_PER_CHUNK);

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&p.a_map);
    tma_prefetch_desc(&p.b_map);
    for (int i = 0; i < STAGES; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&s.pfull[i], 1); mbar_init(&s.pempty[i], 4); }
    mbar_init(&s.done, 1);
    s.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_normal();
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&s.empty[stage], phase ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(&s.full[stage], A_BYTES + B_BYTES);
        tma_load_2d(ring + stage * A_BYTES, &p.a_map, &s.full[stage], kb * BK, mt * BM, pol);
        uint8_t* sb = ring + STAGES * A_BYTES + stage * B_BYTES;
#pragma unroll
        for (int part = 0; part < 3; ++part)
          tma_load_2d(sb + part * B_PART_BYTES, &p.b_map, &s.full[stage], part * p.d + kb * BK,
                      nt * BN, pol);
        ++issued;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      for (int i = 0; i < STAGES && i < issued; ++i) {  // drain own copies
        if (stage == 0) { stage = STAGES - 1; phase ^= 1u; } else { --stage; }
        mbar_wait_drain(&s.full[stage], phase);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool any = false;
      for (int c = 0; c < n_chunks && !*abort_flag; ++c) {
        const int buf = c & 1;
        if (!mbar_wait(&s.pempty[buf], ((c >> 1) & 1) ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * BN);
        const int kc0 = kb0 + c * KB_PER_CHUNK, kc1 = min(kb1, kc0 + KB_PER_CHUNK);
        bool ok = true;
        for (int kb = kc0; kb < kc1; ++kb) {
          if (!mbar_wait(&s.full[stage], phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(ring + stage * A_BYTES);
          const uint32_t b0 = smem_u32(ring + STAGES * A_BYTES + stage * B_BYTES);
#pragma unroll
          for (int part = 0; part < 3; ++part)
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              mma_bf16_ss(d_tmem, sdesc_kmajor_sw128(a0 + k * 32),
                          sdesc_kmajor_sw128(b0 + part * B_PART_BYTES + k * 32), IDESC,
                          (kb > kc0 || part > 0 || k > 0) ? 1u : 0u);
          any = true;
          mma_commit(&s.empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&s.pfull[buf]);
      }
      if (any) {  // drain: every MMA issued here has completed after this
        mma_commit(&s.done);
        mbar_wait_drain(&s.done, 0);
      }
    }
  } else {
    const int q = warp & 3;
    const int m = mt * BM + q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    float acc[BN];
#pragma unroll
    for (int i = 0; i < BN; ++i) acc[i] = 0.f;
    bool ok = true;
    for (int c = 0; c < n_chunks; ++c) {
      const int buf = c & 1;
      if (!mbar_wait(&s.pfull[buf], (c >> 1) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t taddr = tmem + static_cast<uint32_t>(buf * BN) + lane_off;
#pragma unroll
      for (int j = 0; j < BN / 16; ++j) {
        float v[16];
        tmem_ld16(taddr + j * 16, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[j * 16 + i] = __fadd_rn(acc[j * 16 + i], v[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.pempty[buf]);
    }
    if (ok && m < p.T) {
      float* orow = p.out + (static_cast<size_t>(split) * p.T + m) * p.E;
      const bool last = p.splits == 1;
#pragma unroll
      for (int i = 0; i < BN; ++i) {
        const int n = nt * BN + i;
        if (n < p.E) orow[n] = last ? 1.0f / (1.0f + expf(-acc[i])) : acc[i];
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// s[t, e] = sigmoid(sum over splits in order of partial[split, t, e])
__global__ void router_reduce_kernel(const float* __restrict__ part, float* __restrict__ s,
                                     int64_t n, int splits) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < splits; ++j) acc = __fadd_rn(acc, part[j * n + i]);
    s[i] = 1.0f / (1.0f + expf(-acc));
  }
}

// [E, d] fp32 -> [E, 3d] bf16: hi | mid | lo.
__global__ void router_split_kernel(const float* __restrict__ w, __nv_bfloat16* __restrict__ ws,
                                    int E, int d) {
  const int64_t n = static_cast<int64_t>(E) * d;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = i / d, k = i % d;
    const float v = w[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = __fsub_rn(v, __bfloat162float(hi));
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = __fsub_rn(r1, __bfloat162float(mid));
    __nv_bfloat16* row = ws + e * 3 * d;
    row[k] = hi;
    row[d + k] = mid;
    row[2 * d + k] = __float2bfloat16_rn(r2);
  }
}

}  // namespace routertc

// Number of K' splits for a T x E problem: enough CTAs to cover the SMs,
// at least 4 k blocks (of d) per split.
static int router_splits(const moe_cfg_t& c, int sms) {
  using namespace routertc;
  const int tiles = ceil_div(c.T, BM) * ceil_div(c.E, BN);
  const int nkb = c.d / BK;
  int s = sms / tiles;
  s = std::max(1, std::min(s, nkb / 4));
  return s;
}

size_t router_tc_scratch_bytes(const moe_cfg_t& c) {
  using namespace routertc;
  const size_t split_w = align_up(static_cast<size_t>(c.E) * 3 * c.d * 2, 256);
  const int s = router_splits(c, 148);
  const size_t part = s > 1 ? align_up(static_cast<size_t>(s) * c.T * c.E * 4, 256) : 0;
  return split_w + part;
}

cudaError_t launch_router_tc(const moe_cfg_t& c, const void* x, const float* w, float* affinity,
                             void* scratch, cudaStream_t st) {
  using namespace routertc;
  const cudaError_t ea = ensure_smem_limit(reinterpret_cast<const void*>(router_tc_kernel),
                                           static_cast<int>(kSmemBytes));
  if (ea != cudaSuccess) return ea;
  // The split count is fixed (148 SMs of a B300) so that the scratch size
  // is a function of the shape alone.
  const int splits = router_splits(c, 148);
  __nv_bfloat16* wsplit = static_cast<__nv_bfloat16*>(scratch);
  float* part = reinterpret_cast<float*>(static_cast<char*>(scratch) +
                                         align_up(static_cast<size_t>(c.E) * 3 * c.d * 2, 256));
  const int64_t nw = static_cast<int64_t>(c.E) * c.d;
  router_split_kernel<<<static_cast<int>(std::min<int64_t>((nw + 255) / 256, 148 * 8)), 256, 0, st>>>(
      w, wsplit, c.E, c.d);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  Params p{};
  CUresult r = encode_tensor_map_2d(&p.a_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(x),
                                    c.d, c.T, static_cast<uint64_t>(c.d) * 2, BK, BM,
                                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (r == CUDA_SUCCESS)
    r = encode_tensor_map_2d(&p.b_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, wsplit,
                             static_cast<uint64_t>(3) * c.d, c.E, static_cast<uint64_t>(3) * c.d * 2,
                             BK, BN, CU_TENSOR_MAP_SWIZZLE_128B);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  p.T = c.T; p.E = c.E; p.d = c.d;
  p.nkb = c.d / BK;
  p.kb_per_split = ceil_div(p.nkb, splits);
  p.splits = ceil_div(p.nkb, p.kb_per_split);  // no empty split
  p.out = p.splits == 1 ? affinity : part;
  dim3 grid(ceil_div(c.E, BN), ceil_div(c.T, BM), p.splits);
  router_tc_kernel<<<grid, THREADS, kSmemBytes, st>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.splits == 1) return e;
  const int64_t n = static_cast<int64_t>(c.T) * c.E;
  router_reduce_kernel<<<static_cast<int>(std::min<int64_t>((n + 255) / 256, 148 * 8)), 256, 0, st>>>(
      part, affinity, n, p.splits);
  return cudaGetLastError();
}

}  // namespace moe
