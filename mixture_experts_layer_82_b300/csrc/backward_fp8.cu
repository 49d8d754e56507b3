// Backward for input of the expert FFNs in FP8 E4M3 (the Dgrad GEMMs).
//
// "DeepSeek-V3 Technical Report", mixed precision framework paragraph
// (Figure 6): every linear's Dgrad runs in FP8 with fp32 accumulation;
// fine-grained quantisation paragraph: activation-like operands in 1 x 128
// tiles, weights in 128 x 128 blocks, fp32 scales.  A scale factors out of a
// dot product only if it is constant along the contraction, so the gradient
// rows are tiled along their columns (the contraction of Dgrad) and the
// weights keep their forward blocks, which a square block serves in either
// orientation.  Per routed row (per token for the shared expert), with
// dy = dL/d(expert output) in bf16:
//   [a | b] = u W13^T        recomputed from the forward's E4M3 codes of u
//   dh      = q(dy) W2       dy quantised in 1 x 128 tiles along d
//   da = dh b silu'(a),  db = dh silu(a)      fp32, then 1 x 128 tiles along 2I
//   du      = q([da | db]) W13
// All three GEMMs are the forward's FP8 grouped GEMM (experts_fp8.cu, plain
// bf16 output): Dgrad contracts a weight over its other dimension, so it
// reads K-major transposed copies of the weight codes (W2^T [I, d],
// W13^T [d, 2I]) made once by moe_transpose_weights_fp8 from the forward's
// codes and block scales; their blocks are the forward's blocks.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace bwdfp8 {

// ---------------------------------------------------------- weight transpose
// codes [n, R, C] -> [n, C, R]: 64 x 64-byte tiles through shared memory.
__global__ void __launch_bounds__(256) transpose_codes_kernel(const uint8_t* __restrict__ in,
                                                              uint8_t* __restrict__ out, int R,
                                                              int C) {
  __shared__ uint8_t tile[64][65];
  const int mat = blockIdx.z;
  const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
  const uint8_t* src = in + static_cast<size_t>(mat) * R * C;
  uint8_t* dst = out + static_cast<size_t>(mat) * R * C;
  const int tx = threadIdx.x % 64, ty = threadIdx.x / 64;  // 64 x 4 threads
  for (int i = ty; i < 64; i += 4) {
    const int r = r0 + i, c = c0 + tx;
    tile[i][tx] = (r < R && c < C) ? src[static_cast<size_t>(r) * C + c] : 0;
  }
  __syncthreads();
  for (int i = ty; i < 64; i += 4) {
    const int c = c0 + i, r = r0 + tx;
    if (c < C && r < R) dst[static_cast<size_t>(c) * R + r] = tile[tx][i];
  }
}

// scales [n, Rb, Cb] -> [n, Cb, Rb]
__global__ void transpose_scales_kernel(const float* __restrict__ in, float* __restrict__ out,
                                        int n, int Rb, int Cb) {
  const int64_t total = static_cast<int64_t>(n) * Rb * Cb;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t mat = i / (static_cast<int64_t>(Rb) * Cb);
    const int rem = static_cast<int>(i % (static_cast<int64_t>(Rb) * Cb));
    const int rb = rem / Cb, cb = rem % Cb;
    out[mat * Rb * Cb + static_cast<int64_t>(cb) * Rb + rb] = in[i];
  }
}

// --------------------------------------------- SwiGLU backward + quantisation
// One warp per row: from [a | b] (bf16, 2I columns) and dh (bf16, I columns),
// da = dh b silu'(a) and db = dh silu(a) in fp32, silu'(a) = s (1 + a (1 - s))
// with s = sigmoid(a); then [da | db] in 1 x 128 tiles along its 2I columns:
// scale fl32(amax / 448) (1 for an all-zero tile), codes E4M3(v / scale).
__global__ void __launch_bounds__(kRowWarps * 32) swiglu_bwd_quant_kernel(
    const __nv_bfloat16* __restrict__ ab, const __nv_bfloat16* __restrict__ dh, int64_t rows,
    int inter, uint8_t* __restrict__ q, float* __restrict__ scales) {
  const int lane = threadIdx.x % 32;
  const int nt = inter / 128;
  for (int64_t r = blockIdx.x * static_cast<int64_t>(kRowWarps) + threadIdx.x / 32; r < rows;
       r += static_cast<int64_t>(gridDim.x) * kRowWarps) {
    const __nv_bfloat16* ar = ab + r * 2 * inter;
    const __nv_bfloat16* hr = dh + r * inter;
    uint8_t* qr = q + r * 2 * inter;
    float* sr = scales + r * 2 * nt;
    for (int tb = 0; tb < nt; ++tb) {
      const int c = tb * 128 + lane * 4;
      float da[4], db[4];
      {
        const uint2 ra = *reinterpret_cast<const uint2*>(ar + c);
        const uint2 rb = *reinterpret_cast<const uint2*>(ar + inter + c);
        const uint2 rh = *reinterpret_cast<const uint2*>(hr + c);
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&ra);
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&rb);
        const __nv_bfloat162* ph = reinterpret_cast<const __nv_bfloat162*>(&rh);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float2 a = __bfloat1622float2(pa[j]), b = __bfloat1622float2(pb[j]);
          const float2 h = __bfloat1622float2(ph[j]);
          const float s0 = 1.f / (1.f + __expf(-a.x)), s1 = 1.f / (1.f + __expf(-a.y));
          da[2 * j] = h.x * b.x * (s0 * (1.f + a.x * (1.f - s0)));
          da[2 * j + 1] = h.y * b.y * (s1 * (1.f + a.y * (1.f - s1)));
          db[2 * j] = h.x * (a.x * s0);
          db[2 * j + 1] = h.y * (a.y * s1);
        }
      }
      float ma = fmaxf(fmaxf(fabsf(da[0]), fabsf(da[1])), fmaxf(fabsf(da[2]), fabsf(da[3])));
      float mb = fmaxf(fmaxf(fabsf(db[0]), fabsf(db[1])), fmaxf(fabsf(db[2]), fabsf(db[3])));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, off));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
      }
      const float sa = fp8_scale_of(ma), sb = fp8_scale_of(mb);
      *reinterpret_cast<uint32_t*>(qr + c) = quant4_e4m3(da[0], da[1], da[2], da[3], sa);
      *reinterpret_cast<uint32_t*>(qr + inter + c) = quant4_e4m3(db[0], db[1], db[2], db[3], sb);
      if (lane == 0) {
        sr[tb] = sa;
        sr[nt + tb] = sb;
      }
    }
  }
}

}  // namespace bwdfp8

// ------------------------------------------------------------------- host
cudaError_t launch_transpose_weights_fp8(const void* w_q, const float* w_scales, int n_mats,
                                         int rows, int cols, void* wt_q, float* wt_scales,
                                         cudaStream_t st) {
  using namespace bwdfp8;
  const dim3 grid(ceil_div(cols, 64), ceil_div(rows, 64), n_mats);
  transpose_codes_kernel<<<grid, 256, 0, st>>>(static_cast<const uint8_t*>(w_q),
                                               static_cast<uint8_t*>(wt_q), rows, cols);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int rb = ceil_div(rows, 128), cb = cols / 128;
  const int64_t n = static_cast<int64_t>(n_mats) * rb * cb;
  transpose_scales_kernel<<<static_cast<int>(std::min<int64_t>((n + 255) / 256, 1184)), 256, 0,
                            st>>>(w_scales, wt_scales, n_mats, rb, cb);
  return cudaGetLastError();
}

size_t experts_bwd_fp8_scratch_bytes(const moe_cfg_t& c) {
  const size_t tk = static_cast<size_t>(c.T) * c.K, T = c.T, I = c.inter, d = c.d;
  const size_t rows = tk + T;  // routed rows, then the shared expert's T rows
  return align_up(rows * d, 256) + align_up(rows * (d / 128) * 4, 256) +  // q(dy)
         align_up(rows * 2 * I * 2, 256) +                                 // [a | b]
         align_up(rows * I * 2, 256) +                                     // dh
         align_up(rows * 2 * I, 256) + align_up(rows * (2 * I / 128) * 4, 256);  // q([da | db])
}

namespace bwdfp8 {

struct Fp8BwdScratch {
  uint8_t* dyq;
  float* dys;
  __nv_bfloat16* ab;
  __nv_bfloat16* dh;
  uint8_t* dabq;
  float* dabs;
};

Fp8BwdScratch carve_fp8_bwd(const moe_cfg_t& c, void* ws) {
  const size_t tk = static_cast<size_t>(c.T) * c.K, T = c.T, I = c.inter, d = c.d;
  const size_t rows = tk + T;
  char* p = static_cast<char*>(ws);
  Fp8BwdScratch s;
  s.dyq = reinterpret_cast<uint8_t*>(p); p += align_up(rows * d, 256);
  s.dys = reinterpret_cast<float*>(p); p += align_up(rows * (d / 128) * 4, 256);
  s.ab = reinterpret_cast<__nv_bfloat16*>(p); p += align_up(rows * 2 * I * 2, 256);
  s.dh = reinterpret_cast<__nv_bfloat16*>(p); p += align_up(rows * I * 2, 256);
  s.dabq = reinterpret_cast<uint8_t*>(p); p += align_up(rows * 2 * I, 256);
  s.dabs = reinterpret_cast<float*>(p);
  return s;
}

// One FP8 grouped GEMM y = A B^T (bf16 y), routed class over the segments
// of `offsets` and, with a shared expert, the shared class over T rows:
// A codes [rows, K] with 1 x 128 scales, B codes [n, N, K] with 128 x 128
// block scales [n, N/128, K/128]; y [rows, N].
struct Fp8Gemm {
  const void* a;           // routed A codes [T*K, k]
  const float* a_scales;
  const void* a_sh;        // shared A codes [T, k]
  const float* a_sh_scales;
  const void* b;           // routed B codes [E, n, k]
  const float* b_scales;
  const void* b_sh;        // shared B codes [1, n, k]
  const float* b_sh_scales;
  void* y;                 // [T*K, n]
  void* y_sh;              // [T, n]
  int n, k;
};

cudaError_t run_fp8_gemm(const moe_cfg_t& c, const int32_t* offsets, const Fp8Gemm& g,
                         cudaStream_t st) {
  using namespace fp8gemm;
  const int64_t tk = static_cast<int64_t>(c.T) * c.K;
  const bool has_shared = c.n_shared > 0;
  const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapSwizzle SW = CU_TENSOR_MAP_SWIZZLE_128B;
  Params p{};
  p.offsets = offsets;
  p.n_rows = static_cast<int>(tk);
  p.E = c.E;
  p.T = c.T;
  p.has_shared = has_shared ? 1 : 0;
  p.d = g.n;      // B rows of one matrix (the down mode's output width)
  p.inter = g.k;  // K of one matrix
  CUresult r = encode_tensor_map_2d(&p.a_map[0], U8, const_cast<void*>(g.a), g.k, tk,
                                    static_cast<uint64_t>(g.k), BK, BM, SW);
  if (r == CUDA_SUCCESS)
    r = encode_tensor_map_2d(&p.b_map[0], U8, const_cast<void*>(g.b), g.k,
                             static_cast<uint64_t>(c.E) * g.n, static_cast<uint64_t>(g.k), BK,
                             BN, SW);
  if (r == CUDA_SUCCESS && has_shared) {
    r = encode_tensor_map_2d(&p.a_map[1], U8, const_cast<void*>(g.a_sh), g.k, c.T,
                             static_cast<uint64_t>(g.k), BK, BM, SW);
    if (r == CUDA_SUCCESS)
      r = encode_tensor_map_2d(&p.b_map[1], U8, const_cast<void*>(g.b_sh), g.k, g.n,
                               static_cast<uint64_t>(g.k), BK, BN, SW);
  } else {
    p.a_map[1] = p.a_map[0];
    p.b_map[1] = p.b_map[0];
  }
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const auto al32 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 31u) == 0; };
  p.out32 = al32(g.y) && (!has_shared || al32(g.y_sh)) ? 1 : 0;
  p.cls[0] = ClassDesc{g.y, nullptr, g.a_scales, g.b_scales, g.n, g.k, nullptr};
  p.cls[1] = has_shared ? ClassDesc{g.y_sh, nullptr, g.a_sh_scales, g.b_sh_scales, g.n, g.k, nullptr}
                        : p.cls[0];
  return launch_fp8_gemm<DOWN>(p, st);
}

}  // namespace bwdfp8

void experts_bwd_fp8_ab_dh(const moe_cfg_t& c, void* ws, const __nv_bfloat16** ab,
                           const __nv_bfloat16** dh) {
  const bwdfp8::Fp8BwdScratch s = bwdfp8::carve_fp8_bwd(c, ws);
  *ab = s.ab;
  *dh = s.dh;
}

cudaError_t launch_experts_bwd_input_fp8(const ExpertsBwdFp8Args& a, cudaStream_t st) {
  using namespace bwdfp8;
  const moe_cfg_t& c = *a.cfg;
  const int64_t tk = static_cast<int64_t>(c.T) * c.K;
  const int I = c.inter, d = c.d;
  const bool has_shared = c.n_shared > 0;
  Fp8BwdScratch s = carve_fp8_bwd(c, a.ws);
  // shared rows follow the routed ones in every scratch buffer
  uint8_t* dyq_sh = s.dyq + tk * d;
  float* dys_sh = s.dys + tk * (d / 128);
  __nv_bfloat16* ab_sh = s.ab + tk * 2 * I;
  __nv_bfloat16* dh_sh = s.dh + tk * I;
  uint8_t* dabq_sh = s.dabq + tk * 2 * I;
  float* dabs_sh = s.dabs + tk * (2 * I / 128);

  // 1. dy in 1 x 128 tiles along d (routed rows; the shared expert's dout)
  cudaError_t e = launch_quantize_act_fp8(a.dy_perm, static_cast<int>(tk), d, s.dyq, s.dys, st);
  if (e == cudaSuccess && has_shared)
    e = launch_quantize_act_fp8(a.dout, c.T, d, dyq_sh, dys_sh, st);
  if (e != cudaSuccess) return e;
  // 2. [a | b] = u W13^T from the forward's codes (unless the training
  //    forward kept it)
  Fp8Gemm g{a.x_perm, a.x_perm_scales, a.x_q, a.x_q_scales, a.w13, a.w13_scales,
            a.ws13, a.ws13_scales, s.ab, ab_sh, 2 * I, d};
  if (!a.ab_kept) {
    e = run_fp8_gemm(c, a.offsets, g, st);
    if (e != cudaSuccess) return e;
  }
  // 3. dh = q(dy) W2, through W2^T [I, d]
  g = Fp8Gemm{s.dyq, s.dys, dyq_sh, dys_sh, a.w2t, a.w2t_scales, a.ws2t, a.ws2t_scales,
              s.dh, dh_sh, I, d};
  e = run_fp8_gemm(c, a.offsets, g, st);
  if (e != cudaSuccess) return e;
  // 4. [da | db] and its 1 x 128 codes
  const int64_t rows = tk + (has_shared ? c.T : 0);
  swiglu_bwd_quant_kernel<<<static_cast<int>(std::min<int64_t>((rows + kRowWarps - 1) / kRowWarps,
                                                               148 * 16)),
                            kRowWarps * 32, 0, st>>>(s.ab, s.dh, rows, I, s.dabq, s.dabs);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // 5. du = q([da | db]) W13, through W13^T [d, 2I]
  g = Fp8Gemm{s.dabq, s.dabs, dabq_sh, dabs_sh, a.w13t, a.w13t_scales, a.ws13t, a.ws13t_scales,
              a.dx_perm, a.dx_shared, d, 2 * I};
  return run_fp8_gemm(c, a.offsets, g, st);
}

}  // namespace moe
