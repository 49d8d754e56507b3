// Routing of the DeepSeekMoE layer ("DeepSeek-V3 Technical Report",
// DeepSeekMoE paragraph and auxiliary-loss-free load balancing paragraph):
//   1. affinity  s = sigmoid(x e^T)                 (router product, fp32)
//   2. select    group-limited top-K on fl32(s + b), gates from s
//   3. scan      per-expert loads, segment offsets, per-tile bases
//   4. assign    permuted row of every (token, slot)
// plus the sign-rule bias update.  No atomic decides an output order: the
// within-segment rank of a token is a popcount over a per-tile bit mask
// (bit i set <=> token i of the tile chose the expert), so rows follow
// ascending token order and every run gives the same layout.
#include <float.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// ------------------------------------------------------------ scratch layout
size_t route_scratch_bytes(const moe_cfg_t& c, bool need_affinity) {
  const size_t ntile = ceil_div(c.T, kRouteTile);
  size_t b = align_up(ntile * c.E * sizeof(int32_t), 256);
  if (need_affinity) b += align_up(static_cast<size_t>(c.T) * c.E * sizeof(float), 256);
  if (c.dtype != MOE_DTYPE_FP32) b += router_tc_scratch_bytes(c);
  return b;
}

RouteScratch route_scratch_carve(const moe_cfg_t& c, void* ws, bool need_affinity) {
  char* p = static_cast<char*>(ws);
  RouteScratch r{};
  const size_t ntile = ceil_div(c.T, kRouteTile);
  r.tile_counts = reinterpret_cast<int32_t*>(p);
  p += align_up(ntile * c.E * sizeof(int32_t), 256);
  if (need_affinity) {
    r.affinity = reinterpret_cast<float*>(p);
    p += align_up(static_cast<size_t>(c.T) * c.E * sizeof(float), 256);
  }
  if (c.dtype != MOE_DTYPE_FP32) r.router = p;
  return r;
}

// ------------------------------------------------------- 1. router affinity
// logits[t, e] = sum_k x[t, k] w[e, k] in fp32 (FFMA, k ascending), then
// s = 1 / (1 + exp(-logit)).  64 x 64 output tile per block, 4 x 4 per thread.
constexpr int kAffBM = 64, kAffBN = 64, kAffBK = 32;

template <typename TX>
__device__ __forceinline__ float to_f32(TX v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename TX>
__global__ void __launch_bounds__(256) router_affinity_kernel(const TX* __restrict__ x,
                                                              const float* __restrict__ w,
                                                              float* __restrict__ s, int T,
                                                              int E, int d) {
  __shared__ float xs[kAffBK][kAffBM + 4];
  __shared__ float wsh[kAffBK][kAffBN + 4];
  const int t0 = blockIdx.y * kAffBM, e0 = blockIdx.x * kAffBN;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += kAffBK) {
    // 64 rows x 32 k of each operand: 2048 values / 256 threads = 8 each.
    for (int i = threadIdx.x; i < kAffBM * kAffBK; i += 256) {
      const int r = i / kAffBK, kk = i % kAffBK;
      const int t = t0 + r, e = e0 + r, k = k0 + kk;
      xs[kk][r] = (t < T && k < d) ? to_f32<TX>(x[static_cast<size_t>(t) * d + k]) : 0.f;
      wsh[kk][r] = (e < E && k < d) ? w[static_cast<size_t>(e) * d + k] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kAffBK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = wsh[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) s[static_cast<size_t>(t) * E + e] = 1.0f / (1.0f + expf(-acc[i][j]));
    }
  }
}

// fp32 token rows: CUDA-core product.  bf16 token rows: tensor cores with
// the centroids split into three bf16 terms (router_sm100.cu).
cudaError_t launch_router_affinity(const moe_cfg_t& c, const void* x, const float* w,
                                   float* affinity, const RouteScratch& rs, cudaStream_t st) {
  if (c.dtype != MOE_DTYPE_FP32) return launch_router_tc(c, x, w, affinity, rs.router, st);
  dim3 grid(ceil_div(c.E, kAffBN), ceil_div(c.T, kAffBM));
  router_affinity_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(x), w, affinity,
                                                      c.T, c.E, c.d);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- 2. select
// (value, index) order used everywhere: larger value first, then lower index.
__device__ __forceinline__ bool ranks_above(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__device__ __forceinline__ void warp_best(float& v, int& i) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, off);
    const int oi = __shfl_xor_sync(0xffffffffu, i, off);
    if (ranks_above(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

constexpr int kMaxTopn = 8;

// Warps per selection block: one token per warp when the per-warp buffers
// (2 E floats) fit in 64 KiB, fewer warps (several tokens each) otherwise.
static int select_warps(int E) {
  int w = 32;
  while (w > 1 && static_cast<size_t>(w) * 2 * E * sizeof(float) > 64 * 1024) w >>= 1;
  return w;
}

// One block per 32-token tile.  Per token: the biased scores go to shared
// memory; lane g scores group g; the kept groups and then the K experts come
// from repeated warp arg-max reductions.
__global__ void __launch_bounds__(1024) route_select_kernel(
    const float* __restrict__ affinity, const float* __restrict__ bias,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
    int32_t* __restrict__ local_rank, int32_t* __restrict__ tile_counts, int T, int E,
    int n_groups, int topk_groups, int K, int topn, float route_scale) {
  extern __shared__ float sel_smem[];
  float* biased = sel_smem + (threadIdx.x / 32) * 2 * E;  // per warp [E]
  float* sval = biased + E;                               // per warp [E]
  const int n_warps = blockDim.x / 32;
  uint32_t* mask = reinterpret_cast<uint32_t*>(sel_smem + n_warps * 2 * E);  // [E]
  int32_t* chosen = reinterpret_cast<int32_t*>(mask + E);                     // [32][K]
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int tile = blockIdx.x;
  const int per = E / n_groups;
  const int nj = ceil_div(E, 32);

  for (int e = threadIdx.x; e < E; e += blockDim.x) mask[e] = 0u;
  __syncthreads();

  for (int tl = warp; tl < kRouteTile; tl += n_warps) {
    const int t = tile * kRouteTile + tl;
    if (t >= T) break;
    const float* srow = affinity + static_cast<size_t>(t) * E;
    for (int e = lane; e < E; e += 32) {
      const float sv = srow[e];
      sval[e] = sv;
      biased[e] = __fadd_rn(sv, bias[e]);
    }
    __syncwarp();
    // group scores: the group's top-n biased values summed in descending order
    float gscore = -FLT_MAX;
    int gidx = 0x7fffffff;
    if (lane < n_groups) {
      float top[kMaxTopn];
      const int n = min(topn, per);
#pragma unroll
      for (int i = 0; i < kMaxTopn; ++i) top[i] = -FLT_MAX;
      for (int m = 0; m < per; ++m) {
        float v = biased[lane * per + m];
        // insertion into the descending list top[0..n)
#pragma unroll
        for (int i = 0; i < kMaxTopn; ++i) {
          if (i < n && v > top[i]) { const float tmp = top[i]; top[i] = v; v = tmp; }
        }
      }
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxTopn; ++i)
        if (i < n) acc = __fadd_rn(acc, top[i]);
      gscore = acc;
      gidx = lane;
    }
    uint32_t kept = 0u;
    bool taken_g = false;
    for (int r = 0; r < topk_groups; ++r) {
      float v = taken_g ? -FLT_MAX : gscore;
      int i = taken_g ? 0x7fffffff : gidx;
      warp_best(v, i);
      kept |= 1u << i;
      if (lane == i) taken_g = true;
    }
    // experts of the kept groups; lane holds experts lane + 32 j
    uint32_t taken = 0u;
    int my_pick = -1;
    for (int r = 0; r < K; ++r) {
      float v = -FLT_MAX;
      int i = 0x7fffffff;
      for (int j = 0; j < nj; ++j) {
        const int e = lane + 32 * j;
        if (e >= E || (taken >> j & 1u) || !(kept >> (e / per) & 1u)) continue;
        const float bv = biased[e];
        if (ranks_above(bv, e, v, i)) { v = bv; i = e; }
      }
      warp_best(v, i);
      if (i == 0x7fffffff) { i = 0; raise_error(kErrIndex); }  // host checks exclude this
      if ((i & 31) == lane) taken |= 1u << (i >> 5);
      if (lane == r) my_pick = i;
    }
    // gates from the unbiased affinities, summed in slot order
    float ssel = (lane < K) ? sval[my_pick] : 0.f;
    float sum = 0.f;
    for (int r = 0; r < K; ++r) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, ssel, r));
    if (lane < K) {
      const size_t o = static_cast<size_t>(t) * K + lane;
      topk_idx[o] = my_pick;
      topk_w[o] = route_scale * __fdiv_rn(ssel, sum);
      chosen[tl * K + lane] = my_pick;
      atomicOr(&mask[my_pick], 1u << tl);  // OR is order-free
    }
    __syncwarp();
  }
  __syncthreads();
  // per-tile loads and within-tile ranks
  int32_t* tc = tile_counts + static_cast<size_t>(tile) * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) tc[e] = __popc(mask[e]);
  for (int i = threadIdx.x; i < kRouteTile * K; i += blockDim.x) {
    const int tl = i / K;
    const int t = tile * kRouteTile + tl;
    if (t >= T) continue;
    const int e = chosen[i];
    local_rank[static_cast<size_t>(t) * K + (i % K)] = __popc(mask[e] & ((1u << tl) - 1u));
  }
}

cudaError_t launch_route_select(const moe_cfg_t& c, const float* affinity, const float* bias,
                                int32_t* topk_idx, float* topk_w, int32_t* local_rank,
                                int32_t* tile_counts, cudaStream_t st) {
  const int warps = select_warps(c.E);
  const size_t smem = static_cast<size_t>(warps) * 2 * c.E * sizeof(float) +
                      static_cast<size_t>(c.E) * sizeof(uint32_t) +
                      static_cast<size_t>(kRouteTile) * c.K * sizeof(int32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(route_select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  route_select_kernel<<<ceil_div(c.T, kRouteTile), warps * 32, smem, st>>>(
      affinity, bias, topk_idx, topk_w, local_rank, tile_counts, c.T, c.E, c.n_groups,
      c.topk_groups, c.K, c.group_score_topn, c.route_scale);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ 3. scan
// One block.  For each chunk of 256 experts: warp w sums the loads of its
// contiguous range of tiles; a scan over warps gives each warp's starting
// base; each warp then rewrites its tiles' loads as exclusive bases.  The
// per-expert totals are scanned into the segment offsets.
constexpr int kScanThreads = 1024;
constexpr int kScanWarps = kScanThreads / 32;
constexpr int kScanChunk = 256;

__global__ void __launch_bounds__(kScanThreads) route_scan_kernel(int32_t* __restrict__ tile_counts,
                                                                  int32_t* __restrict__ counts,
                                                                  int32_t* __restrict__ offsets,
                                                                  int ntile, int E) {
  __shared__ int32_t part[kScanWarps][kScanChunk];
  __shared__ int32_t total[1024];
  __shared__ int32_t warp_sums[kScanWarps];
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int per_warp = ceil_div(ntile, kScanWarps);
  const int tb = warp * per_warp, te = min(ntile, tb + per_warp);
  for (int c0 = 0; c0 < E; c0 += kScanChunk) {
    const int cn = min(kScanChunk, E - c0);
    for (int j = lane; j < cn; j += 32) {
      int32_t acc = 0;
      for (int tl = tb; tl < te; ++tl) acc += tile_counts[static_cast<size_t>(tl) * E + c0 + j];
      part[warp][j] = acc;
    }
    __syncthreads();
    if (threadIdx.x < cn) {
      int32_t run = 0;
      for (int w = 0; w < kScanWarps; ++w) {
        const int32_t v = part[w][threadIdx.x];
        part[w][threadIdx.x] = run;
        run += v;
      }
      total[c0 + threadIdx.x] = run;
    }
    __syncthreads();
    for (int j = lane; j < cn; j += 32) {
      int32_t run = part[warp][j];
      for (int tl = tb; tl < te; ++tl) {
        int32_t* p = tile_counts + static_cast<size_t>(tl) * E + c0 + j;
        const int32_t v = *p;
        *p = run;
        run += v;
      }
    }
    __syncthreads();
  }
  // exclusive scan of totals over experts (E <= 1024)
  const int e = threadIdx.x;
  int32_t v = (e < E) ? total[e] : 0;
  int32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t ws = warp_sums[lane];
    int32_t wi = ws;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    warp_sums[lane] = wi - ws;
  }
  __syncthreads();
  const int32_t excl = warp_sums[warp] + incl - v;
  if (e < E) {
    counts[e] = v;
    offsets[e] = excl;
    if (e == E - 1) offsets[E] = excl + v;
  }
}

cudaError_t launch_route_scan(const moe_cfg_t& c, int32_t* tile_counts, int32_t* counts,
                              int32_t* offsets, cudaStream_t st) {
  route_scan_kernel<<<1, kScanThreads, 0, st>>>(tile_counts, counts, offsets,
                                                ceil_div(c.T, kRouteTile), c.E);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- 4. assign
__global__ void route_assign_kernel(const int32_t* __restrict__ topk_idx,
                                    const int32_t* __restrict__ offsets,
                                    const int32_t* __restrict__ tile_base,
                                    int32_t* __restrict__ row_of_slot,
                                    int32_t* __restrict__ token_of_row, int T, int E, int K) {
  const int64_t n = static_cast<int64_t>(T) * K;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / K);
    const int e = topk_idx[i];
    if (e < 0 || e >= E) { raise_error(kErrIndex); continue; }
    const int64_t row = static_cast<int64_t>(offsets[e]) +
                        tile_base[static_cast<size_t>(t / kRouteTile) * E + e] + row_of_slot[i];
    if (row < 0 || row >= n) { raise_error(kErrIndex); continue; }
    row_of_slot[i] = static_cast<int32_t>(row);
    token_of_row[row] = t;
  }
}

cudaError_t launch_route_assign(const moe_cfg_t& c, const int32_t* topk_idx,
                                const int32_t* offsets, const int32_t* tile_base,
                                int32_t* row_of_slot, int32_t* token_of_row, cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(c.T) * c.K;
  const int blocks = static_cast<int>(std::min<int64_t>(ceil_div(static_cast<int>(n), 256), 148 * 8));
  route_assign_kernel<<<blocks, 256, 0, st>>>(topk_idx, offsets, tile_base, row_of_slot,
                                              token_of_row, c.T, c.E, c.K);
  return cudaGetLastError();
}

// ----------------------------------------------------------- bias update
__global__ void bias_update_kernel(const int32_t* __restrict__ counts, float* __restrict__ bias,
                                   int E, int64_t tk, float gamma) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const bool over = static_cast<int64_t>(counts[e]) * E > tk;
  bias[e] = over ? __fsub_rn(bias[e], gamma) : __fadd_rn(bias[e], gamma);
}

cudaError_t launch_bias_update(const moe_cfg_t& c, const int32_t* counts, float* bias,
                               cudaStream_t st) {
  bias_update_kernel<<<ceil_div(c.E, 256), 256, 0, st>>>(
      counts, bias, c.E, static_cast<int64_t>(c.T) * c.K, c.gamma);
  return cudaGetLastError();
}

// ------------------------------------------------ sequence-wise balance stat
// L_Bal = alpha * sum_i f_i P_i per sequence of L consecutive tokens
// ("DeepSeek-V3 Technical Report", auxiliary-loss-free paragraph: the
// complementary sequence-wise balance loss; alpha from the training
// hyper-parameters).  f_i = E / (K L) * selections of expert i in the
// sequence, P_i = mean over the sequence of s_i / sum_j s_j.
constexpr int kBalWarps = 8;
constexpr int kBalChunk = 256;  // tokens of a sequence per CTA

// Partial sums of one (sequence, 32-expert chunk, 256-token chunk): warp w
// takes tokens w, w + 8, ... of the token chunk; lane j owns expert
// 32 * blockIdx.y + j.  Writes sum_t s_e / sum_j s_j and the selection
// count of every owned expert to part_p / part_c [n_seq][chunks][E].
__global__ void __launch_bounds__(kBalWarps * 32) balance_partial_kernel(
    const float* __restrict__ s, const int32_t* __restrict__ topk_idx, int E, int K, int L,
    float* __restrict__ part_p, int* __restrict__ part_c) {
  __shared__ float ps[kBalWarps][32];
  __shared__ int cs[kBalWarps][32];
  const int q = blockIdx.x, e0 = blockIdx.y * 32, ch = blockIdx.z, nch = gridDim.z;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int e = e0 + lane;
  const int i0 = ch * kBalChunk, i1 = min(L, i0 + kBalChunk);
  float p = 0.f;
  int cnt = 0;
  for (int i = i0 + warp; i < i1; i += kBalWarps) {
    const size_t t = static_cast<size_t>(q) * L + i;
    const float* row = s + t * E;
    float rs = 0.f;
    for (int j = lane; j < E; j += 32) rs += row[j];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
    const int my_idx = lane < K ? topk_idx[t * K + lane] : -1;
    for (int k = 0; k < K; ++k) cnt += __shfl_sync(0xffffffffu, my_idx, k) == e ? 1 : 0;
    if (e < E) p += __fdiv_rn(row[e], rs);
  }
  ps[warp][lane] = p;
  cs[warp][lane] = cnt;
  __syncthreads();
  if (warp == 0 && e < E) {
    float pt = 0.f;
    int ct = 0;
    for (int w = 0; w < kBalWarps; ++w) { pt += ps[w][lane]; ct += cs[w][lane]; }
    const size_t o = (static_cast<size_t>(q) * nch + ch) * E + e;
    part_p[o] = pt;
    part_c[o] = ct;
  }
}

// One CTA per sequence: f and P of every expert from the partials (summed
// in chunk order), then loss = alpha * sum_i f_i P_i (each thread sums its
// experts in order, then a fixed reduction tree).
__global__ void __launch_bounds__(256) balance_final_kernel(
    const float* __restrict__ part_p, const int* __restrict__ part_c, int E, int K, int L, int nch,
    float alpha, float* __restrict__ f_out, float* __restrict__ p_out, float* __restrict__ loss) {
  __shared__ float red[256];
  const int q = blockIdx.x;
  float acc = 0.f;
  for (int e = threadIdx.x; e < E; e += 256) {
    float pt = 0.f;
    int ct = 0;
    for (int ch = 0; ch < nch; ++ch) {
      const size_t o = (static_cast<size_t>(q) * nch + ch) * E + e;
      pt += part_p[o];
      ct += part_c[o];
    }
    const float P = __fdiv_rn(pt, static_cast<float>(L));
    const float f = static_cast<float>(static_cast<double>(E) * ct / (static_cast<double>(K) * L));
    p_out[static_cast<size_t>(q) * E + e] = P;
    f_out[static_cast<size_t>(q) * E + e] = f;
    acc = fmaf(f, P, acc);
  }
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) loss[q] = alpha * red[0];
}

size_t balance_scratch_bytes(const moe_cfg_t& c, int seq_len) {
  const size_t n = static_cast<size_t>(c.T / seq_len) * ceil_div(seq_len, kBalChunk) * c.E;
  return align_up(n * 4, 256) * 2;
}

cudaError_t launch_balance_stat(const moe_cfg_t& c, const float* affinity, const int32_t* topk_idx,
                                int seq_len, float alpha, float* f_out, float* p_out, float* loss,
                                void* ws, cudaStream_t st) {
  const int n_seq = c.T / seq_len;
  const int nch = ceil_div(seq_len, kBalChunk);
  const size_t n = static_cast<size_t>(n_seq) * nch * c.E;
  float* part_p = static_cast<float*>(ws);
  int* part_c = reinterpret_cast<int*>(static_cast<char*>(ws) + align_up(n * 4, 256));
  dim3 grid(n_seq, ceil_div(c.E, 32), nch);
  balance_partial_kernel<<<grid, kBalWarps * 32, 0, st>>>(affinity, topk_idx, c.E, c.K, seq_len,
                                                          part_p, part_c);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  balance_final_kernel<<<n_seq, 256, 0, st>>>(part_p, part_c, c.E, c.K, seq_len, nch, alpha, f_out,
                                              p_out, loss);
  return cudaGetLastError();
}

}  // namespace moe
