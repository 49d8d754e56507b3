// Dispatch and combine on one device, and the FP8 quantisers.
//
// permute: x_perm[r] = x[token_of_row[r]] (the single-device form of the
//   dispatch all-to-all, "DeepSeek-V3 Technical Report", cross-node
//   all-to-all paragraph); one warp per row, 16-byte vector copies.
// quantise: E4M3 with one fp32 scale per 1 x 128 tile (fine-grained
//   quantisation paragraph): scale = fl32(amax / 448), 1 for a zero tile;
//   code = E4M3(fl32(v / scale)), nearest-even, saturating.
// combine: out[t] = y_shared[t] + sum_k g[t,k] y_perm[row_of_slot[t,k]],
//   fp32 accumulation in exactly that order (DeepSeekMoE paragraph).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kRowWarps = 8;

// Row copy by one warp.  The destination rows are written once and read
// by a later kernel, so they are stored with the streaming hint (.cs): they
// should not push the source rows (each read K times) out of L2.
__device__ __forceinline__ void copy_row_bytes(char* __restrict__ dst, const char* __restrict__ src,
                                               size_t bytes, int lane) {
  const size_t nv = bytes / 16;
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (size_t i = lane; i < nv; i += 32) __stcs(d4 + i, __ldg(s4 + i));
  for (size_t i = nv * 16 + lane * 4; i < bytes; i += 128)
    *reinterpret_cast<uint32_t*>(dst + i) = *reinterpret_cast<const uint32_t*>(src + i);
}

__global__ void __launch_bounds__(kRowWarps * 32) permute_kernel(
    const char* __restrict__ x, const int32_t* __restrict__ token_of_row, char* __restrict__ x_perm,
    int64_t rows, int T, size_t row_bytes) {
  const int lane = threadIdx.x % 32;
  for (int64_t r = blockIdx.x * static_cast<int64_t>(kRowWarps) + threadIdx.x / 32; r < rows;
       r += static_cast<int64_t>(gridDim.x) * kRowWarps) {
    const int t = token_of_row[r];
    if (t < 0 || t >= T) { if (lane == 0) raise_error(kErrIndex); continue; }
    copy_row_bytes(x_perm + r * row_bytes, x + static_cast<size_t>(t) * row_bytes, row_bytes, lane);
  }
}

static int row_grid(int64_t rows) {
  return static_cast<int>(std::min<int64_t>((rows + kRowWarps - 1) / kRowWarps, 148 * 16));
}

cudaError_t launch_permute(const moe_cfg_t& c, const void* x, const int32_t* token_of_row,
                           void* x_perm, size_t elem_bytes, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(c.T) * c.K;
  permute_kernel<<<row_grid(rows), kRowWarps * 32, 0, st>>>(
      static_cast<const char*>(x), token_of_row, static_cast<char*>(x_perm), rows, c.T,
      static_cast<size_t>(c.d) * elem_bytes);
  return cudaGetLastError();
}

// ------------------------------------------------------------ FP8 quantiser
__device__ __forceinline__ float fp8_scale_of(float amax) {
  return amax == 0.f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

// E4M3 codes of fl32(a / scale) .. fl32(d / scale), packed (the exact
// quotients' codes, through the reciprocal with its exactness check).
__device__ __forceinline__ uint32_t quant4_e4m3(float a, float b, float c, float d, float scale) {
  const float r = __frcp_rn(scale);
  return e4m3x2_of_quotients(a, b, scale, scale, r, r) |
         (e4m3x2_of_quotients(c, d, scale, scale, r, r) << 16);
}

// E4M3 codes of a * rs ... d * rs (rs: a reciprocal scale), packed.
__device__ __forceinline__ uint32_t quant4_e4m3_mul(float a, float b, float c, float d, float rs) {
  const __nv_fp8x2_storage_t lo =
      __nv_cvt_float2_to_fp8x2(make_float2(a * rs, b * rs), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi =
      __nv_cvt_float2_to_fp8x2(make_float2(c * rs, d * rs), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// One warp per row; per 128-wide tile each lane holds 4 consecutive values.
__global__ void __launch_bounds__(kRowWarps * 32) quantize_act_kernel(
    const __nv_bfloat16* __restrict__ x, int rows, int cols, uint8_t* __restrict__ q,
    float* __restrict__ scales) {
  const int lane = threadIdx.x % 32;
  const int ntile = cols / 128;
  for (int64_t r = blockIdx.x * static_cast<int64_t>(kRowWarps) + threadIdx.x / 32; r < rows;
       r += static_cast<int64_t>(gridDim.x) * kRowWarps) {
    const __nv_bfloat16* xr = x + r * cols;
    for (int tb = 0; tb < ntile; ++tb) {
      const uint2 raw = *reinterpret_cast<const uint2*>(xr + tb * 128 + lane * 4);
      const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
      const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
      const float v0 = __low2float(p0), v1 = __high2float(p0);
      const float v2 = __low2float(p1), v3 = __high2float(p1);
      float amax = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const float scale = fp8_scale_of(amax);
      *reinterpret_cast<uint32_t*>(q + r * cols + tb * 128 + lane * 4) =
          quant4_e4m3(v0, v1, v2, v3, scale);
      if (lane == 0) scales[r * ntile + tb] = scale;
    }
  }
}

cudaError_t launch_quantize_act_fp8(const void* x_bf16, int rows, int cols, void* q,
                                    float* scales, cudaStream_t st) {
  quantize_act_kernel<<<row_grid(rows), kRowWarps * 32, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x_bf16), rows, cols, static_cast<uint8_t*>(q), scales);
  return cudaGetLastError();
}

__global__ void __launch_bounds__(kRowWarps * 32) permute_fp8_kernel(
    const char* __restrict__ xq, const float* __restrict__ xs,
    const int32_t* __restrict__ token_of_row, char* __restrict__ x_perm,
    float* __restrict__ x_perm_scales, int64_t rows, int T, int d) {
  const int lane = threadIdx.x % 32;
  const int ntile = d / 128;
  for (int64_t r = blockIdx.x * static_cast<int64_t>(kRowWarps) + threadIdx.x / 32; r < rows;
       r += static_cast<int64_t>(gridDim.x) * kRowWarps) {
    const int t = token_of_row[r];
    if (t < 0 || t >= T) { if (lane == 0) raise_error(kErrIndex); continue; }
    copy_row_bytes(x_perm + r * d, xq + static_cast<size_t>(t) * d, d, lane);
    for (int i = lane; i < ntile; i += 32) x_perm_scales[r * ntile + i] = xs[static_cast<size_t>(t) * ntile + i];
  }
}

cudaError_t launch_permute_fp8(const moe_cfg_t& c, const void* x_q, const float* x_scales,
                               const int32_t* token_of_row, void* x_perm, float* x_perm_scales,
                               cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(c.T) * c.K;
  permute_fp8_kernel<<<row_grid(rows), kRowWarps * 32, 0, st>>>(
      static_cast<const char*>(x_q), x_scales, token_of_row, static_cast<char*>(x_perm),
      x_perm_scales, rows, c.T, c.d);
  return cudaGetLastError();
}

// 128 x 128 weight blocks: one block of 256 threads per (matrix, row block,
// column block); each thread quantises 64 values.
__global__ void __launch_bounds__(256) quantize_weight_kernel(const __nv_bfloat16* __restrict__ w,
                                                             int rows, int cols,
                                                             uint8_t* __restrict__ q,
                                                             float* __restrict__ scales) {
  __shared__ float red[8];
  const int cb = blockIdx.x, rb = blockIdx.y, m = blockIdx.z;
  const int nrb = gridDim.y, ncb = gridDim.x;
  const size_t mat = static_cast<size_t>(m) * rows * cols;
  const int c = cb * 128 + (threadIdx.x % 32) * 4;  // 4 consecutive columns
  float amax = 0.f;
  for (int rr = threadIdx.x / 32; rr < 128; rr += 8) {
    const int r = rb * 128 + rr;
    if (r >= rows) break;
    const __nv_bfloat16* p = w + mat + static_cast<size_t>(r) * cols + c;
#pragma unroll
    for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(__bfloat162float(p[i])));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float scale = fp8_scale_of(amax);
  for (int rr = threadIdx.x / 32; rr < 128; rr += 8) {
    const int r = rb * 128 + rr;
    if (r >= rows) break;
    const __nv_bfloat16* p = w + mat + static_cast<size_t>(r) * cols + c;
    *reinterpret_cast<uint32_t*>(q + mat + static_cast<size_t>(r) * cols + c) =
        quant4_e4m3(__bfloat162float(p[0]), __bfloat162float(p[1]), __bfloat162float(p[2]),
                    __bfloat162float(p[3]), scale);
  }
  if (threadIdx.x == 0) scales[(static_cast<size_t>(m) * nrb + rb) * ncb + cb] = scale;
}

cudaError_t launch_quantize_weights_fp8(const void* w, int n_mats, int rows, int cols, void* q,
                                        float* scales, cudaStream_t st) {
  dim3 grid(cols / 128, ceil_div(rows, 128), n_mats);
  quantize_weight_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(w), rows, cols,
                                               static_cast<uint8_t*>(q), scales);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- combine
template <typename TY>
struct Vec16;
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int n = 8;
  __device__ static void load(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 r = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __low2float(h[i]);
      v[2 * i + 1] = __high2float(h[i]);
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float (&v)[8]) {
    uint4 r;
    r.x = pack_bf16x2(v[0], v[1]);
    r.y = pack_bf16x2(v[2], v[3]);
    r.z = pack_bf16x2(v[4], v[5]);
    r.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(p) = r;
  }
};
template <>
struct Vec16<float> {
  static constexpr int n = 4;
  __device__ static void load(const float* p, float (&v)[4]) {
    const float4 r = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w;
  }
  __device__ static void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};

constexpr int kMaxK = 32;
constexpr int kCombineVecs = 4;  // 16-byte vectors per lane and work item

// One warp per (token, column chunk of 32 * kCombineVecs vectors): enough
// independent warps for small T, several loads in flight per lane.
template <typename TY>
__global__ void __launch_bounds__(kRowWarps * 32) combine_kernel(
    const TY* __restrict__ y_perm, const TY* __restrict__ y_shared,
    const int32_t* __restrict__ row_of_slot, const float* __restrict__ topk_w, TY* __restrict__ out,
    int T, int K, int d, int64_t n_rows) {
  using V = Vec16<TY>;
  constexpr int n = V::n;
  constexpr int chunk = 32 * n * kCombineVecs;
  const int lane = threadIdx.x % 32;
  const int n_chunks = (d + chunk - 1) / chunk;
  const int64_t items = static_cast<int64_t>(T) * n_chunks;
  for (int64_t it = blockIdx.x * static_cast<int64_t>(kRowWarps) + threadIdx.x / 32; it < items;
       it += static_cast<int64_t>(gridDim.x) * kRowWarps) {
    const int64_t t = it / n_chunks;
    const int c0 = static_cast<int>(it % n_chunks) * chunk;
    // lane k < K holds slot k's row and gate
    int64_t my_row = 0;
    float my_g = 0.f;
    if (lane < K) {
      my_row = row_of_slot[t * K + lane];
      // no gates: the rows already hold gate * y (a plain ordered sum)
      my_g = topk_w != nullptr ? topk_w[t * K + lane] : 1.f;
      if (my_row < 0 || my_row >= n_rows) { raise_error(kErrIndex); my_row = 0; }
    }
    float acc[kCombineVecs][n];
#pragma unroll
    for (int v = 0; v < kCombineVecs; ++v) {
      const int c = c0 + (v * 32 + lane) * n;
      if (y_shared != nullptr && c < d) {
        V::load(y_shared + t * d + c, acc[v]);
      } else {
#pragma unroll
        for (int i = 0; i < n; ++i) acc[v][i] = 0.f;
      }
    }
    for (int k = 0; k < K; ++k) {
      const int64_t row = __shfl_sync(0xffffffffu, my_row, k);
      const float g = __shfl_sync(0xffffffffu, my_g, k);
#pragma unroll
      for (int v = 0; v < kCombineVecs; ++v) {
        const int c = c0 + (v * 32 + lane) * n;
        if (c < d) {
          float y[n];
          V::load(y_perm + row * d + c, y);
#pragma unroll
          for (int i = 0; i < n; ++i) acc[v][i] = fmaf(g, y[i], acc[v][i]);
        }
      }
    }
#pragma unroll
    for (int v = 0; v < kCombineVecs; ++v) {
      const int c = c0 + (v * 32 + lane) * n;
      if (c < d) V::store(out + t * d + c, acc[v]);
    }
  }
}

// Gate of every permuted row: the row of (token t, slot k) takes g[t, k]
// (the DeepSeekMoE paragraph's gate of that expert for that token).
__global__ void gate_rows_kernel(const int32_t* __restrict__ row_of_slot,
                                 const float* __restrict__ topk_w, float* __restrict__ gate_of_row,
                                 int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = row_of_slot[i];
    if (row < 0 || row >= n) { raise_error(kErrIndex); continue; }
    gate_of_row[row] = topk_w[i];
  }
}

cudaError_t launch_gate_rows(const moe_cfg_t& c, const int32_t* row_of_slot, const float* topk_w,
                             float* gate_of_row, cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(c.T) * c.K;
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 148 * 8));
  gate_rows_kernel<<<blocks, 256, 0, st>>>(row_of_slot, topk_w, gate_of_row, n);
  return cudaGetLastError();
}

cudaError_t launch_combine(const moe_cfg_t& c, const void* y_perm, const void* y_shared,
                           const int32_t* row_of_slot, const float* topk_w, void* out,
                           cudaStream_t st) {
  const int64_t n_rows = static_cast<int64_t>(c.T) * c.K;
  const int per = (c.dtype == MOE_DTYPE_FP32 ? 4 : 8) * 32 * kCombineVecs;
  const int64_t items = static_cast<int64_t>(c.T) * ((c.d + per - 1) / per);
  const int grid = row_grid(items);
  if (c.dtype == MOE_DTYPE_FP32)
    combine_kernel<float><<<grid, kRowWarps * 32, 0, st>>>(
        static_cast<const float*>(y_perm), static_cast<const float*>(y_shared), row_of_slot,
        topk_w, static_cast<float*>(out), c.T, c.K, c.d, n_rows);
  else
    combine_kernel<__nv_bfloat16><<<grid, kRowWarps * 32, 0, st>>>(
        static_cast<const __nv_bfloat16*>(y_perm), static_cast<const __nv_bfloat16*>(y_shared),
        row_of_slot, topk_w, static_cast<__nv_bfloat16*>(out), c.T, c.K, c.d, n_rows);
  return cudaGetLastError();
}

}  // namespace moe
