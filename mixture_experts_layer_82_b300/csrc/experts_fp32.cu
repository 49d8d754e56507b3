// Expert FFNs of the fp32 kind: a plain CUDA-core grouped GEMM pair.
//
// Every routed expert e runs SwiGLU on its segment of the permuted rows,
//   h = silu(x W1_e^T) * (x W3_e^T),   y = h W2_e^T,
// and the N_s shared experts run on all T rows as one expert of
// intermediate N_s * I ("DeepSeek-V3 Technical Report", DeepSeekMoE
// paragraph).  This kind exists for exact small-shape checks; the bf16 and
// FP8 kinds use the tensor-core kernels.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kSBM = 64, kSBN = 64, kSBK = 16;

struct SimtGroup {
  int cls;        // 0 routed, 1 shared
  int expert;     // routed expert index (cls 0)
  int row0;       // first row of the group in its class's row space
  int rows;       // rows of the group
  int m_tile;     // tile index inside the group
};

// Maps a linear M-tile index to its group: routed experts first (offsets
// from device memory), then the shared class.  Returns false past the end.
__device__ bool simt_find_group(const int32_t* offsets, int E, int T, int n_rows, bool has_shared,
                                int lin, SimtGroup& g) {
  int acc = 0;
  for (int e = 0; e < E; ++e) {
    int row0;
    const int rows = checked_segment(offsets, e, n_rows, row0);
    const int nt = ceil_div(rows, kSBM);
    if (lin < acc + nt) {
      g = SimtGroup{0, e, row0, rows, lin - acc};
      return true;
    }
    acc += nt;
  }
  if (has_shared && lin < acc + ceil_div(T, kSBM)) {
    g = SimtGroup{1, 0, 0, T, lin - acc};
    return true;
  }
  return false;
}

// Gate/up projection + SwiGLU.  A: [rows, d]; h: [rows, n_cols].
__global__ void __launch_bounds__(256) simt_gateup_kernel(
    const float* __restrict__ x_perm, const float* __restrict__ x, const int32_t* __restrict__ offsets,
    const float* __restrict__ w13, const float* __restrict__ ws13, float* __restrict__ h_routed,
    float* __restrict__ h_shared, int E, int T, int n_rows, int d, int inter, int n_shared) {
  SimtGroup g;
  if (!simt_find_group(offsets, E, T, n_rows, n_shared > 0, blockIdx.y, g)) return;
  const int ncols = g.cls == 0 ? inter : n_shared * inter;
  const int n0 = blockIdx.x * kSBN;
  if (n0 >= ncols) return;
  const float* A = g.cls == 0 ? x_perm + static_cast<size_t>(g.row0) * d : x;
  float* H = g.cls == 0 ? h_routed + static_cast<size_t>(g.row0) * inter : h_shared;
  const int m0 = g.m_tile * kSBM;
  __shared__ float as[kSBK][kSBM + 1];
  __shared__ float gs[kSBK][kSBN + 1];
  __shared__ float us[kSBK][kSBN + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float ag[4][4] = {}, au[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += kSBK) {
    for (int i = threadIdx.x; i < kSBM * kSBK; i += 256) {
      const int r = i / kSBK, kk = i % kSBK, k = k0 + kk;
      const int m = m0 + r, n = n0 + r;
      as[kk][r] = (m < g.rows && k < d) ? A[static_cast<size_t>(m) * d + k] : 0.f;
      float gv = 0.f, uv = 0.f;
      if (n < ncols && k < d) {
        const int s = n / inter, i_loc = n % inter;
        const float* W = g.cls == 0 ? w13 + static_cast<size_t>(g.expert) * 2 * inter * d
                                    : ws13 + static_cast<size_t>(s) * 2 * inter * d;
        gv = W[static_cast<size_t>(i_loc) * d + k];
        uv = W[static_cast<size_t>(inter + i_loc) * d + k];
      }
      gs[kk][r] = gv;
      us[kk][r] = uv;
    }
    __syncthreads();
    for (int kk = 0; kk < kSBK; ++kk) {
      float a[4], bg[4], bu[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = as[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) { bg[j] = gs[kk][tx * 4 + j]; bu[j] = us[kk][tx * 4 + j]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          ag[i][j] = fmaf(a[i], bg[j], ag[i][j]);
          au[i][j] = fmaf(a[i], bu[j], au[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= g.rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < ncols) H[static_cast<size_t>(m) * ncols + n] = silu_f(ag[i][j]) * au[i][j];
    }
  }
}

// Down projection.  h: [rows, kdim]; y: [rows, d].
__global__ void __launch_bounds__(256) simt_down_kernel(
    const float* __restrict__ h_routed, const float* __restrict__ h_shared,
    const int32_t* __restrict__ offsets, const float* __restrict__ w2, const float* __restrict__ ws2,
    float* __restrict__ y_perm, float* __restrict__ y_shared, int E, int T, int n_rows, int d, int inter,
    int n_shared, const float* __restrict__ gate_of_row) {
  SimtGroup g;
  if (!simt_find_group(offsets, E, T, n_rows, n_shared > 0, blockIdx.y, g)) return;
  const int kdim = g.cls == 0 ? inter : n_shared * inter;
  const int n0 = blockIdx.x * kSBN;
  if (n0 >= d) return;
  const float* A = g.cls == 0 ? h_routed + static_cast<size_t>(g.row0) * inter : h_shared;
  float* Y = g.cls == 0 ? y_perm + static_cast<size_t>(g.row0) * d : y_shared;
  const int m0 = g.m_tile * kSBM;
  __shared__ float as[kSBK][kSBM + 1];
  __shared__ float bs[kSBK][kSBN + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < kdim; k0 += kSBK) {
    for (int i = threadIdx.x; i < kSBM * kSBK; i += 256) {
      const int r = i / kSBK, kk = i % kSBK, k = k0 + kk;
      const int m = m0 + r, n = n0 + r;
      as[kk][r] = (m < g.rows && k < kdim) ? A[static_cast<size_t>(m) * kdim + k] : 0.f;
      float bv = 0.f;
      if (n < d && k < kdim) {
        const int s = k / inter, i_loc = k % inter;
        const float* W = g.cls == 0 ? w2 + static_cast<size_t>(g.expert) * d * inter
                                    : ws2 + static_cast<size_t>(s) * d * inter;
        bv = W[static_cast<size_t>(n) * inter + i_loc];
      }
      bs[kk][r] = bv;
    }
    __syncthreads();
    for (int kk = 0; kk < kSBK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = as[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= g.rows) continue;
    // the routed rows' gate, folded in before the store
    const float gm = g.cls == 0 && gate_of_row != nullptr ? gate_of_row[g.row0 + m] : 1.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < d) Y[static_cast<size_t>(m) * d + n] = acc[i][j] * gm;
    }
  }
}

cudaError_t launch_experts_fp32(const ExpertsArgs& a, cudaStream_t st) {
  const moe_cfg_t& c = *a.cfg;
  // Upper bound of M tiles: every routed expert adds at most one ragged tile.
  const int64_t tk = static_cast<int64_t>(c.T) * c.K;
  const int m_tiles = static_cast<int>((tk + kSBM - 1) / kSBM) + c.E +
                      (c.n_shared > 0 ? ceil_div(c.T, kSBM) : 0);
  float* h_routed = static_cast<float*>(a.h);
  float* h_shared = h_routed + tk * c.inter;
  const int n_gate = std::max(c.inter, c.n_shared * c.inter);
  simt_gateup_kernel<<<dim3(ceil_div(n_gate, kSBN), m_tiles), 256, 0, st>>>(
      static_cast<const float*>(a.x_perm), static_cast<const float*>(a.x), a.offsets,
      static_cast<const float*>(a.w13), static_cast<const float*>(a.ws13), h_routed, h_shared, c.E,
      c.T, static_cast<int>(tk), c.d, c.inter, c.n_shared);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  simt_down_kernel<<<dim3(ceil_div(c.d, kSBN), m_tiles), 256, 0, st>>>(
      h_routed, h_shared, a.offsets, static_cast<const float*>(a.w2),
      static_cast<const float*>(a.ws2), static_cast<float*>(a.y_perm),
      static_cast<float*>(a.y_shared), c.E, c.T, static_cast<int>(tk), c.d, c.inter, c.n_shared,
      a.gate_of_row);
  return cudaGetLastError();
}

}  // namespace moe
