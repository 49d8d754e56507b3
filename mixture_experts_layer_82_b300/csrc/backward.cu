// Backward of the combine and of the router (bf16 kind), on the CUDA cores:
// both are a few flops per byte.
//
// "DeepSeek-V3 Technical Report", DeepSeekMoE paragraph: the output is
// y_t = shared(u_t) + sum_k g_{t,k} FFN_{e_k}(u_t) with g = rho s / S,
// S = sum over the selected experts of s = sigmoid(u . e).  With dL/dy given
// and the selection fixed:
//   combine backward: dy_perm[row(t,k)] = g_{t,k} dL/dy_t,
//                     dL/dg_{t,k} = dL/dy_t . y_perm[row(t,k)]
//   router backward:  dL/ds_k = rho / S (dL/dg_k - sum_j dL/dg_j s_j / S),
//                     dL/dl_k = dL/ds_k s_k (1 - s_k)    (l = u . e)
//                     dx_t = dx_shared_t + sum_k (dx_perm[row(t,k)] + dL/dl_k e_{e_k})
//                     de_i = sum over the rows r of expert i of dL/dl(r) u_{token(r)}
// Every sum runs in a fixed order (no atomics), so results are
// deterministic.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace bwd {

constexpr int kWarps = 8;

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 raw = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                            pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// One warp per token; each lane owns 8 consecutive columns of every
// 256-column chunk.
__global__ void __launch_bounds__(kWarps * 32) combine_backward_kernel(
    const __nv_bfloat16* __restrict__ dout, const __nv_bfloat16* __restrict__ y_perm,
    const int32_t* __restrict__ row_of_slot, const float* __restrict__ topk_w,
    __nv_bfloat16* __restrict__ dy_perm, float* __restrict__ dgate, int T, int K, int d,
    int64_t n_rows) {
  const int lane = threadIdx.x % 32;
  for (int64_t t = blockIdx.x * static_cast<int64_t>(kWarps) + threadIdx.x / 32; t < T;
       t += static_cast<int64_t>(gridDim.x) * kWarps) {
    const __nv_bfloat16* go = dout + t * d;
    for (int k = 0; k < K; ++k) {
      int64_t row = row_of_slot[t * K + k];
      const float g = topk_w[t * K + k];
      if (row < 0 || row >= n_rows) {
        if (lane == 0) raise_error(kErrIndex);
        continue;
      }
      const __nv_bfloat16* yr = y_perm + row * d;
      __nv_bfloat16* dr = dy_perm + row * d;
      float dot = 0.f;
      for (int c = lane * 8; c < d; c += 256) {
        float o[8], y[8], w[8];
        load8(go + c, o);
        load8(yr + c, y);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          dot = fmaf(o[i], y[i], dot);
          w[i] = g * o[i];
        }
        store8(dr + c, w);
      }
      dot = warp_sum(dot);
      if (lane == 0) dgate[t * K + k] = dot;
    }
  }
}

// One warp per token: lanes k < K hold slot k.
__global__ void __launch_bounds__(kWarps * 32) route_backward_kernel(
    const float* __restrict__ affinity, const float* __restrict__ router_w,
    const int32_t* __restrict__ topk_idx, const float* __restrict__ dgate,
    const int32_t* __restrict__ row_of_slot, const __nv_bfloat16* __restrict__ dx_perm,
    const __nv_bfloat16* __restrict__ dx_shared, float* __restrict__ dlogit,
    float* __restrict__ dlogit_row, __nv_bfloat16* __restrict__ dx, int T, int E, int K, int d,
    float rho, int64_t n_rows) {
  const int lane = threadIdx.x % 32;
  for (int64_t t = blockIdx.x * static_cast<int64_t>(kWarps) + threadIdx.x / 32; t < T;
       t += static_cast<int64_t>(gridDim.x) * kWarps) {
    int e = 0;
    int64_t row = 0;
    float sv = 0.f, dg = 0.f;
    if (lane < K) {
      e = topk_idx[t * K + lane];
      row = row_of_slot[t * K + lane];
      if (e < 0 || e >= E || row < 0 || row >= n_rows) {
        raise_error(kErrIndex);
        e = 0;
        row = -1;
      } else {
        sv = affinity[t * E + e];
        dg = dgate[t * K + lane];
      }
    }
    const float S = warp_sum(sv);
    const float inner = warp_sum(dg * sv) / S;
    const float ds = rho / S * (dg - inner);
    const float dl = lane < K ? ds * sv * (1.0f - sv) : 0.f;
    if (lane < K) {
      dlogit[t * K + lane] = dl;
      if (row >= 0) dlogit_row[row] = dl;
    }
    for (int c = lane * 8; c < d; c += 256) {
      float acc[8];
      if (dx_shared != nullptr) {
        load8(dx_shared + t * d + c, acc);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      }
      for (int k = 0; k < K; ++k) {
        const int64_t rk = __shfl_sync(0xffffffffu, row, k);
        const int ek = __shfl_sync(0xffffffffu, e, k);
        const float lk = __shfl_sync(0xffffffffu, dl, k);
        if (rk < 0) continue;
        float v[8];
        load8(dx_perm + rk * d + c, v);
        const float4 w0 = *reinterpret_cast<const float4*>(router_w + static_cast<int64_t>(ek) * d + c);
        const float4 w1 = *reinterpret_cast<const float4*>(router_w + static_cast<int64_t>(ek) * d + c + 4);
        const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(lk, w[i], acc[i] + v[i]);
      }
      store8(dx + t * d + c, acc);
    }
  }
}

// Router weight gradient: block (expert i, 256-column chunk).  Warp w sums
// the rows w, w + 8, ... of the expert's segment; the eight partial rows are
// then added in warp order.
__global__ void __launch_bounds__(kWarps * 32) router_wgrad_kernel(
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ token_of_row,
    const int32_t* __restrict__ offsets, const float* __restrict__ dlogit_row,
    float* __restrict__ drouter_w, int T, int n_rows, int d) {
  __shared__ float part[kWarps][256];
  const int e = blockIdx.x;
  const int c0 = blockIdx.y * 256;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int r0;
  const int nr = checked_segment(offsets, e, n_rows, r0);
  const int r1 = r0 + nr;
  const int c = c0 + lane * 8;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (c < d) {
    for (int r = r0 + warp; r < r1; r += kWarps) {
      const int t = token_of_row[r];
      if (t < 0 || t >= T) {
        if (lane == 0) raise_error(kErrIndex);
        continue;
      }
      const float l = dlogit_row[r];
      float v[8];
      load8(x + static_cast<int64_t>(t) * d + c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(l, v[i], acc[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) part[warp][lane * 8 + i] = acc[i];
  __syncthreads();
  const int j = threadIdx.x;
  if (c0 + j < d) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += part[w][j];
    drouter_w[static_cast<int64_t>(e) * d + c0 + j] = s;
  }
}

int token_grid(int64_t T) {
  return static_cast<int>(std::min<int64_t>((T + kWarps - 1) / kWarps, 148 * 16));
}

}  // namespace bwd

cudaError_t launch_combine_backward(const moe_cfg_t& c, const void* dout, const void* y_perm,
                                    const int32_t* row_of_slot, const float* topk_w,
                                    void* dy_perm, float* dgate, cudaStream_t st) {
  using namespace bwd;
  combine_backward_kernel<<<token_grid(c.T), kWarps * 32, 0, st>>>(
      static_cast<const __nv_bfloat16*>(dout), static_cast<const __nv_bfloat16*>(y_perm),
      row_of_slot, topk_w, static_cast<__nv_bfloat16*>(dy_perm), dgate, c.T, c.K, c.d,
      static_cast<int64_t>(c.T) * c.K);
  return cudaGetLastError();
}

cudaError_t launch_route_backward(const moe_cfg_t& c, const RouteBwdArgs& a, cudaStream_t st) {
  using namespace bwd;
  route_backward_kernel<<<token_grid(c.T), kWarps * 32, 0, st>>>(
      a.affinity, a.router_w, a.topk_idx, a.dgate, a.row_of_slot,
      static_cast<const __nv_bfloat16*>(a.dx_perm), static_cast<const __nv_bfloat16*>(a.dx_shared),
      a.dlogit, a.dlogit_row, static_cast<__nv_bfloat16*>(a.dx), c.T, c.E, c.K, c.d,
      c.route_scale, static_cast<int64_t>(c.T) * c.K);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid(c.E, (c.d + 255) / 256);
  router_wgrad_kernel<<<grid, kWarps * 32, 0, st>>>(static_cast<const __nv_bfloat16*>(a.x),
                                                     a.token_of_row, a.offsets, a.dlogit_row,
                                                     a.drouter_w, c.T,
                                                     static_cast<int>(static_cast<int64_t>(c.T) * c.K), c.d);
  return cudaGetLastError();
}

}  // namespace moe
