// The C ABI of libmoe (declared in include/moe.h): host-side argument
// checks, workspace layout and kernel dispatch.  Nothing here allocates
// device memory; the only library state is the per-device error word.
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

using namespace moe;

namespace {

constexpr int32_t kVersion = 100;  // 0.1.0

// Failure-detection self test: thread 0 waits, with the bounded wait of the
// GEMM kernels, on a barrier that nothing arrives on, so the wait gives up
// after limit_ns and sets the timeout bit of the error word.
__global__ void selftest_wait_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, limit_ns);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

const char* moe_status_str(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_SHAPE: return "unsupported shape";
    case MOE_ERR_ALIGN: return "pointer not 16-byte aligned";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE: return "device-side check failed";
    case MOE_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

int32_t moe_version(void) { return kVersion; }

moe_status_t moe_check_cfg(const moe_cfg_t* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->T < 1 || c->d < 1 || c->E < 1 || c->K < 1 || c->inter < 1 || c->n_shared < 0 ||
      c->n_groups < 1 || c->topk_groups < 1 || c->group_score_topn < 1)
    return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_DTYPE_FP32 && c->dtype != MOE_DTYPE_BF16 && c->dtype != MOE_DTYPE_FP8_E4M3)
    return MOE_ERR_INVALID_ARG;
  if (c->E % c->n_groups != 0 || c->topk_groups > c->n_groups || c->K > c->E)
    return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(c->topk_groups) * (c->E / c->n_groups) < c->K) return MOE_ERR_INVALID_ARG;
  if (!(c->route_scale == c->route_scale) || !(c->gamma == c->gamma)) return MOE_ERR_INVALID_ARG;
  if (c->T > (1 << 22) || c->E > 1024 || c->K > 32 || c->n_groups > 32 || c->group_score_topn > 8)
    return MOE_ERR_SHAPE;
  const int64_t tk = static_cast<int64_t>(c->T) * c->K;
  if (tk >= (int64_t{1} << 31)) return MOE_ERR_SHAPE;
  if (c->dtype == MOE_DTYPE_FP32) {
    if (c->d % 4 != 0) return MOE_ERR_SHAPE;
    const int64_t m_tiles = (tk + 63) / 64 + c->E + (c->T + 63) / 64;
    if (m_tiles >= 65535) return MOE_ERR_SHAPE;
  } else {
    if (c->d % 128 != 0 || c->inter % 128 != 0) return MOE_ERR_SHAPE;
  }
  return MOE_OK;
}

size_t moe_workspace_bytes(const moe_cfg_t* c) {
  if (moe_check_cfg(c) != MOE_OK) return 0;
  const size_t r = route_scratch_bytes(*c, true);
  const size_t e = experts_scratch_bytes(*c);
  return r > e ? r : e;
}

moe_status_t moe_route(const moe_cfg_t* cfg, const void* x, const float* router_w,
                       const float* bias, const float* affinity_in, float* affinity_out,
                       int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                       int32_t* row_of_slot, int32_t* token_of_row, void* ws, size_t ws_bytes,
                       void* stream) {
  moe_status_t st = moe_check_cfg(cfg);
  if (st != MOE_OK) return st;
  const moe_cfg_t& c = *cfg;
  if (bias == nullptr || topk_idx == nullptr || topk_w == nullptr || counts == nullptr ||
      offsets == nullptr || row_of_slot == nullptr || token_of_row == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (affinity_in == nullptr && (x == nullptr || router_w == nullptr)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, router_w, bias, affinity_in, affinity_out, topk_idx, topk_w,
                        counts, offsets, row_of_slot, token_of_row, ws};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_ALIGN;
  const bool need_aff = affinity_in == nullptr && affinity_out == nullptr;
  if (ws_bytes < route_scratch_bytes(c, need_aff)) return MOE_ERR_WORKSPACE;
  const RouteScratch rs = route_scratch_carve(c, ws, need_aff);
  cudaStream_t s = as_stream(stream);
  const float* aff = affinity_in;
  if (aff == nullptr) {
    float* dst = affinity_out != nullptr ? affinity_out : rs.affinity;
    cudaError_t e = launch_router_affinity(c, x, router_w, dst, rs, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    aff = dst;
  } else if (affinity_out != nullptr && affinity_out != affinity_in) {
    cudaError_t e = cudaMemcpyAsync(affinity_out, affinity_in,
                                    static_cast<size_t>(c.T) * c.E * sizeof(float),
                                    cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  cudaError_t e = launch_route_select(c, aff, bias, topk_idx, topk_w, row_of_slot, rs.tile_counts, s);
  if (e == cudaSuccess) e = launch_route_scan(c, rs.tile_counts, counts, offsets, s);
  if (e == cudaSuccess)
    e = launch_route_assign(c, topk_idx, offsets, rs.tile_counts, row_of_slot, token_of_row, s);
  return from_cuda(e);
}

moe_status_t moe_permute(const moe_cfg_t* cfg, const void* x, const int32_t* token_of_row,
                         void* x_perm, float* x_perm_scales, void* x_q, float* x_q_scales,
                         void* stream) {
  moe_status_t st = moe_check_cfg(cfg);
  if (st != MOE_OK) return st;
  const moe_cfg_t& c = *cfg;
  if (x == nullptr || token_of_row == nullptr || x_perm == nullptr) return MOE_ERR_INVALID_ARG;
  const bool fp8 = c.dtype == MOE_DTYPE_FP8_E4M3;
  if (fp8 && (x_perm_scales == nullptr || x_q == nullptr || x_q_scales == nullptr))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, token_of_row, x_perm, x_perm_scales, x_q, x_q_scales};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_ALIGN;
  cudaStream_t s = as_stream(stream);
  cudaError_t e;
  if (fp8) {
    e = launch_quantize_act_fp8(x, c.T, c.d, x_q, x_q_scales, s);
    if (e == cudaSuccess) e = launch_permute_fp8(c, x_q, x_q_scales, token_of_row, x_perm, x_perm_scales, s);
  } else {
    e = launch_permute(c, x, token_of_row, x_perm, c.dtype == MOE_DTYPE_FP32 ? 4 : 2, s);
  }
  return from_cuda(e);
}

}  // extern "C"

// moe_experts_grouped, and with row_of_slot / topk_w given, its gated form.
static moe_status_t experts_grouped(const moe_cfg_t* cfg, const void* x_perm,
                                    const float* x_perm_scales, const void* x,
                                    const float* x_scales, const int32_t* offsets, const void* w13,
                                    const float* w13_scales, const void* w2,
                                    const float* w2_scales, const void* ws13,
                                    const float* ws13_scales, const void* ws2,
                                    const float* ws2_scales, const int32_t* row_of_slot,
                                    const float* topk_w, void* y_perm, void* y_shared, void* ws,
                                    size_t ws_bytes, void* stream,
                                    __nv_bfloat16* ab = nullptr,
                                    __nv_bfloat16* ab_shared = nullptr) {
  moe_status_t st = moe_check_cfg(cfg);
  if (st != MOE_OK) return st;
  const moe_cfg_t& c = *cfg;
  if (x_perm == nullptr || offsets == nullptr || w13 == nullptr || w2 == nullptr ||
      y_perm == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && (x == nullptr || ws13 == nullptr || ws2 == nullptr || y_shared == nullptr))
    return MOE_ERR_INVALID_ARG;
  const bool fp8 = c.dtype == MOE_DTYPE_FP8_E4M3;
  if (fp8 && (x_perm_scales == nullptr || w13_scales == nullptr || w2_scales == nullptr ||
              (c.n_shared > 0 && (x_scales == nullptr || ws13_scales == nullptr ||
                                  ws2_scales == nullptr))))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x_perm, x_perm_scales, x, x_scales, offsets, w13, w13_scales, w2,
                        w2_scales, ws13, ws13_scales, ws2, ws2_scales, y_perm, y_shared, ws,
                        row_of_slot, topk_w};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_ALIGN;
  if (ws_bytes < experts_scratch_bytes(c)) return MOE_ERR_WORKSPACE;
  ExpertsArgs a{};
  a.cfg = &c;
  a.x_perm = x_perm; a.x_perm_scales = x_perm_scales; a.x = x; a.x_scales = x_scales;
  a.offsets = offsets;
  a.w13 = w13; a.w13_scales = w13_scales; a.w2 = w2; a.w2_scales = w2_scales;
  a.ws13 = ws13; a.ws13_scales = ws13_scales; a.ws2 = ws2; a.ws2_scales = ws2_scales;
  a.y_perm = y_perm; a.y_shared = c.n_shared > 0 ? y_shared : nullptr;
  a.ab = ab;
  a.ab_shared = c.n_shared > 0 ? ab_shared : nullptr;
  experts_scratch_carve(c, ws, &a.h, &a.h_scales);
  cudaStream_t s = as_stream(stream);
  cudaError_t e;
  if (row_of_slot != nullptr) {
    float* gate_rows = experts_gate_rows(c, ws);
    e = launch_gate_rows(c, row_of_slot, topk_w, gate_rows, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    a.gate_of_row = gate_rows;
  }
  switch (c.dtype) {
    case MOE_DTYPE_FP32: e = launch_experts_fp32(a, s); break;
    case MOE_DTYPE_BF16: e = launch_experts_bf16(a, s); break;
    default: e = launch_experts_fp8(a, s); break;
  }
  return from_cuda(e);
}

extern "C" {

moe_status_t moe_experts_grouped(const moe_cfg_t* cfg, const void* x_perm,
                                 const float* x_perm_scales, const void* x, const float* x_scales,
                                 const int32_t* offsets, const void* w13, const float* w13_scales,
                                 const void* w2, const float* w2_scales, const void* ws13,
                                 const float* ws13_scales, const void* ws2, const float* ws2_scales,
                                 void* y_perm, void* y_shared, void* ws, size_t ws_bytes,
                                 void* stream) {
  return experts_grouped(cfg, x_perm, x_perm_scales, x, x_scales, offsets, w13, w13_scales, w2,
                         w2_scales, ws13, ws13_scales, ws2, ws2_scales, nullptr, nullptr, y_perm,
                         y_shared, ws, ws_bytes, stream);
}

moe_status_t moe_experts_grouped_gated(const moe_cfg_t* cfg, const void* x_perm,
                                       const float* x_perm_scales, const void* x,
                                       const float* x_scales, const int32_t* offsets,
                                       const void* w13, const float* w13_scales, const void* w2,
                                       const float* w2_scales, const void* ws13,
                                       const float* ws13_scales, const void* ws2,
                                       const float* ws2_scales, const int32_t* row_of_slot,
                                       const float* topk_w, void* y_perm, void* y_shared,
                                       void* ws, size_t ws_bytes, void* stream) {
  if (row_of_slot == nullptr || topk_w == nullptr) return MOE_ERR_INVALID_ARG;
  return experts_grouped(cfg, x_perm, x_perm_scales, x, x_scales, offsets, w13, w13_scales, w2,
                         w2_scales, ws13, ws13_scales, ws2, ws2_scales, row_of_slot, topk_w,
                         y_perm, y_shared, ws, ws_bytes, stream);
}

moe_status_t moe_experts_grouped_gather(const moe_cfg_t* cfg, const void* x,
                                        const float* x_scales, const int32_t* token_of_row,
                                        const int32_t* offsets, const void* w13,
                                        const float* w13_scales, const void* w2,
                                        const float* w2_scales, const void* ws13,
                                        const float* ws13_scales, const void* ws2,
                                        const float* ws2_scales, void* y_perm, void* y_shared,
                                        void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = moe_check_cfg(cfg);
  if (st != MOE_OK) return st;
  const moe_cfg_t& c = *cfg;
  if (c.dtype != MOE_DTYPE_BF16) return MOE_ERR_SHAPE;
  if (x == nullptr || token_of_row == nullptr || offsets == nullptr || w13 == nullptr ||
      w2 == nullptr || y_perm == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && (ws13 == nullptr || ws2 == nullptr || y_shared == nullptr))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, x_scales, token_of_row, offsets, w13, w13_scales, w2, w2_scales,
                        ws13, ws13_scales, ws2, ws2_scales, y_perm, y_shared, ws};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_ALIGN;
  if (ws_bytes < experts_scratch_bytes(c)) return MOE_ERR_WORKSPACE;
  ExpertsArgs a{};
  a.cfg = &c;
  a.x = x;
  a.token_of_row = token_of_row;
  a.offsets = offsets;
  a.w13 = w13; a.w2 = w2; a.ws13 = ws13; a.ws2 = ws2;
  a.y_perm = y_perm; a.y_shared = c.n_shared > 0 ? y_shared : nullptr;
  experts_scratch_carve(c, ws, &a.h, &a.h_scales);
  return from_cuda(launch_experts_bf16(a, as_stream(stream)));
}

moe_status_t moe_combine(const moe_cfg_t* cfg, const void* y_perm, const void* y_shared,
                         const int32_t* row_of_slot, const float* topk_w, void* out, void* stream) {
  moe_status_t st = moe_check_cfg(cfg);
  if (st != MOE_OK) return st;
  const moe_cfg_t& c = *cfg;
  // topk_w NULL: the rows already carry their gates (moe_experts_grouped_gated)
  if (y_perm == nullptr || row_of_slot == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {y_perm, y_shared, row_of_slot, topk_w, out};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_ALIGN;
  return from_cuda(launch_combine(c, y_perm, c.n_shared > 0 ? y_shared : nullptr, row_of_slot,
                                  topk_w, out, as_stream(stream)));
}

moe_status_t moe_bias_update(const moe_cfg_t* cfg, const int32_t* counts, float* bias,
                             void* stream) {
  // The sign rule reads E, K, T and gamma only: the whole-batch T of
  // data-parallel replicas may exceed what one routing call accepts.
  if (cfg == nullptr) return MOE_ERR_INVALID_ARG;
  if (cfg->E < 1 || cfg->K < 1 || cfg->K > cfg->E || cfg->T < 1 || !(cfg->gamma == cfg->gamma))
    return MOE_ERR_INVALID_ARG;
  if (cfg->E > 1024 || cfg->K > 32) return MOE_ERR_SHAPE;
  if (counts == nullptr || bias == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(counts) || !aligned16(bias)) return MOE_ERR_ALIGN;
  return from_cuda(launch_bias_update(*cfg, counts, bias, as_stream(stream)));
}

moe_status_t moe_balance_stat(const moe_cfg_t* cfg, const float* affinity,
                              const int32_t* topk_idx, int32_t seq_len, float alpha, float* f_out,
                              float* p_out, float* loss_out, void* ws, size_t ws_bytes,
                              void* stream) {
  moe_status_t st = moe_check_cfg(cfg);
  if (st != MOE_OK) return st;
  const moe_cfg_t& c = *cfg;
  if (affinity == nullptr || topk_idx == nullptr || f_out == nullptr || p_out == nullptr ||
      loss_out == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (seq_len < 1 || c.T % seq_len != 0 || !(alpha == alpha)) return MOE_ERR_INVALID_ARG;
  if (c.T / seq_len > 65535) return MOE_ERR_SHAPE;
  const void* ptrs[] = {affinity, topk_idx, f_out, p_out, loss_out, ws};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_ALIGN;
  if (ws_bytes < balance_scratch_bytes(c, seq_len)) return MOE_ERR_WORKSPACE;
  return from_cuda(launch_balance_stat(c, affinity, topk_idx, seq_len, alpha, f_out, p_out,
                                       loss_out, ws, as_stream(stream)));
}

// ------------------------------------------------------------ backward pass
namespace {

// The backward calls: the bf16 kind (up to 64 shared experts) and, for the
// calls that handle it, the FP8 kind (at most one shared expert).
moe_status_t check_backward_cfg(const moe_cfg_t* cfg) {
  moe_status_t st = moe_check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (cfg->dtype == MOE_DTYPE_BF16) return cfg->n_shared > 64 ? MOE_ERR_SHAPE : MOE_OK;
  if (cfg->dtype == MOE_DTYPE_FP8_E4M3) return cfg->n_shared > 1 ? MOE_ERR_SHAPE : MOE_OK;
  return MOE_ERR_SHAPE;
}

// Bytes of the expert part of the backward workspace (the routing part follows).
size_t backward_experts_bytes(const moe_cfg_t& c) {
  return c.dtype == MOE_DTYPE_FP8_E4M3
             ? experts_bwd_fp8_scratch_bytes(c) + experts_wgrad_fp8_scratch_bytes(c)
             : experts_bwd_scratch_bytes(c);
}

size_t backward_route_bytes(const moe_cfg_t& c) {
  return align_up(static_cast<size_t>(c.T) * c.K * 4, 256);
}

}  // namespace

size_t moe_backward_workspace_bytes(const moe_cfg_t* c) {
  if (check_backward_cfg(c) != MOE_OK) return 0;
  return backward_experts_bytes(*c) + backward_route_bytes(*c);
}

moe_status_t moe_combine_backward(const moe_cfg_t* cfg, const void* dout, const void* y_perm,
                                  const int32_t* row_of_slot, const float* topk_w,
                                  void* dy_perm, float* dgate, void* stream) {
  moe_status_t st = check_backward_cfg(cfg);
  if (st != MOE_OK) return st;
  if (dout == nullptr || y_perm == nullptr || row_of_slot == nullptr || topk_w == nullptr ||
      dy_perm == nullptr || dgate == nullptr)
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {dout, y_perm, row_of_slot, topk_w, dy_perm, dgate};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_ALIGN;
  return from_cuda(launch_combine_backward(*cfg, dout, y_perm, row_of_slot, topk_w, dy_perm,
                                           dgate, as_stream(stream)));
}

moe_status_t moe_experts_grouped_train(const moe_cfg_t* cfg, const void* x_perm, const void* x,
                                       const int32_t* offsets, const void* w13, const void* w2,
                                       const void* ws13, const void* ws2, void* y_perm,
                                       void* y_shared, void* ws, size_t ws_bytes, void* bws,
                                       size_t bws_bytes, void* stream) {
  moe_status_t st = check_backward_cfg(cfg);
  if (st == MOE_OK && cfg->dtype != MOE_DTYPE_BF16) st = MOE_ERR_SHAPE;  // bf16 kind only
  if (st != MOE_OK) return st;
  const moe_cfg_t& c = *cfg;
  if (x_perm == nullptr || offsets == nullptr || w13 == nullptr || w2 == nullptr ||
      y_perm == nullptr || ws == nullptr || bws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && (x == nullptr || ws13 == nullptr || ws2 == nullptr || y_shared == nullptr))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x_perm, x, offsets, w13, w2, ws13, ws2, y_perm, y_shared, ws, bws};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_ALIGN;
  if (ws_bytes < experts_scratch_bytes(c) || bws_bytes < moe_backward_workspace_bytes(cfg))
    return MOE_ERR_WORKSPACE;
  ExpertsArgs a{};
  a.cfg = &c;
  a.x_perm = x_perm; a.x = x; a.offsets = offsets;
  a.w13 = w13; a.w2 = w2; a.ws13 = ws13; a.ws2 = ws2;
  a.y_perm = y_perm; a.y_shared = c.n_shared > 0 ? y_shared : nullptr;
  experts_scratch_carve(c, ws, &a.h, &a.h_scales);
  const ExpertsBwdScratch w = experts_bwd_scratch_carve(c, bws);
  a.ab = w.ab;
  a.ab_shared = w.ab_shared;
  return from_cuda(launch_experts_bf16(a, as_stream(stream)));
}

moe_status_t moe_experts_backward_input(const moe_cfg_t* cfg, const void* x_perm,
                                        const void* x, const int32_t* offsets, const void* w13,
                                        const void* w2, const void* ws13, const void* ws2,
                                        const void* dy_perm, const void* dout, void* dx_perm,
                                        void* dx_shared, int32_t ab_kept, void* ws,
                                        size_t ws_bytes, void* stream) {
  moe_status_t st = check_backward_cfg(cfg);
  if (st == MOE_OK && cfg->dtype != MOE_DTYPE_BF16) st = MOE_ERR_SHAPE;  // bf16 kind only
  if (st != MOE_OK) return st;
  const moe_cfg_t& c = *cfg;
  if (x_perm == nullptr || offsets == nullptr || w13 == nullptr || w2 == nullptr ||
      dy_perm == nullptr || dx_perm == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && (x == nullptr || ws13 == nullptr || ws2 == nullptr || dout == nullptr ||
                         dx_shared == nullptr))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x_perm, x, offsets, w13, w2, ws13, ws2, dy_perm, dout, dx_perm,
                        dx_shared, ws};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_ALIGN;
  if (ws_bytes < moe_backward_workspace_bytes(cfg)) return MOE_ERR_WORKSPACE;
  ExpertsBwdArgs a{};
  a.cfg = &c;
  a.x_perm = x_perm; a.x = x; a.offsets = offsets;
  a.w13 = w13; a.w2 = w2; a.ws13 = ws13; a.ws2 = ws2;
  a.dy_perm = dy_perm; a.dout = dout;
  a.dx_perm = dx_perm; a.dx_shared = c.n_shared > 0 ? dx_shared : nullptr;
  a.ab_kept = ab_kept != 0;
  a.scratch = experts_bwd_scratch_carve(c, ws);
  return from_cuda(launch_experts_bwd_input_bf16(a, as_stream(stream)));
}

moe_status_t moe_experts_backward_weights(const moe_cfg_t* cfg, const void* x_perm,
                                          const void* x, const int32_t* offsets,
                                          const void* dy_perm, const void* dout, void* dw13,
                                          void* dw2, void* dws13, void* dws2, void* ws,
                                          size_t ws_bytes, void* stream) {
  moe_status_t st = check_backward_cfg(cfg);
  if (st == MOE_OK && cfg->dtype != MOE_DTYPE_BF16) st = MOE_ERR_SHAPE;  // bf16 kind only
  if (st != MOE_OK) return st;
  const moe_cfg_t& c = *cfg;
  if (x_perm == nullptr || offsets == nullptr || dy_perm == nullptr || dw13 == nullptr ||
      dw2 == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && (x == nullptr || dout == nullptr || dws13 == nullptr || dws2 == nullptr))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x_perm, x, offsets, dy_perm, dout, dw13, dw2, dws13, dws2, ws};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_ALIGN;
  if (ws_bytes < moe_backward_workspace_bytes(cfg)) return MOE_ERR_WORKSPACE;
  ExpertsBwdArgs a{};
  a.cfg = &c;
  a.x_perm = x_perm; a.x = x; a.offsets = offsets;
  a.dy_perm = dy_perm; a.dout = dout;
  a.dw13 = dw13; a.dw2 = dw2;
  a.dws13 = c.n_shared > 0 ? dws13 : nullptr;
  a.dws2 = c.n_shared > 0 ? dws2 : nullptr;
  a.scratch = experts_bwd_scratch_carve(c, ws);
  return from_cuda(launch_experts_bwd_weights_bf16(a, as_stream(stream)));
}

moe_status_t moe_route_backward(const moe_cfg_t* cfg, const void* x, const float* router_w,
                                const float* affinity, const int32_t* topk_idx,
                                const float* dgate, const int32_t* row_of_slot,
                                const int32_t* token_of_row, const int32_t* offsets,
                                const void* dx_perm, const void* dx_shared, float* dlogit,
                                void* dx, float* drouter_w, void* ws, size_t ws_bytes,
                                void* stream) {
  moe_status_t st = check_backward_cfg(cfg);
  if (st != MOE_OK) return st;
  const moe_cfg_t& c = *cfg;
  if (x == nullptr || router_w == nullptr || affinity == nullptr || topk_idx == nullptr ||
      dgate == nullptr || row_of_slot == nullptr || token_of_row == nullptr ||
      offsets == nullptr || dx_perm == nullptr || dlogit == nullptr || dx == nullptr ||
      drouter_w == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && dx_shared == nullptr) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, router_w, affinity, topk_idx, dgate, row_of_slot, token_of_row,
                        offsets, dx_perm, dx_shared, dlogit, dx, drouter_w, ws};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_ALIGN;
  if (ws_bytes < moe_backward_workspace_bytes(cfg)) return MOE_ERR_WORKSPACE;
  RouteBwdArgs a{};
  a.x = x; a.router_w = router_w; a.affinity = affinity; a.topk_idx = topk_idx;
  a.dgate = dgate; a.row_of_slot = row_of_slot; a.token_of_row = token_of_row;
  a.offsets = offsets; a.dx_perm = dx_perm;
  a.dx_shared = c.n_shared > 0 ? dx_shared : nullptr;
  a.dlogit = dlogit;
  a.dlogit_row = reinterpret_cast<float*>(static_cast<char*>(ws) + backward_experts_bytes(c));
  a.dx = dx; a.drouter_w = drouter_w;
  return from_cuda(launch_route_backward(c, a, as_stream(stream)));
}

moe_status_t moe_transpose_weights_fp8(const void* w_q, const float* w_scales, int32_t n_mats,
                                       int32_t rows, int32_t cols, void* wt_q, float* wt_scales,
                                       void* stream) {
  if (w_q == nullptr || w_scales == nullptr || wt_q == nullptr || wt_scales == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (n_mats < 1 || rows < 1 || cols < 1) return MOE_ERR_INVALID_ARG;
  if (rows % 128 != 0 || cols % 128 != 0) return MOE_ERR_SHAPE;
  const void* ptrs[] = {w_q, w_scales, wt_q, wt_scales};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_ALIGN;
  return from_cuda(launch_transpose_weights_fp8(w_q, w_scales, n_mats, rows, cols, wt_q, wt_scales,
                                                as_stream(stream)));
}

moe_status_t moe_quantize_act_fp8_128x1(const void* x, int32_t rows, int32_t cols, void* q,
                                        float* scales, void* stream) {
  if (x == nullptr || q == nullptr || scales == nullptr) return MOE_ERR_INVALID_ARG;
  if (rows < 1 || cols < 1) return MOE_ERR_INVALID_ARG;
  if (cols % 128 != 0 || cols / 128 > 65535) return MOE_ERR_SHAPE;
  const void* ptrs[] = {x, q, scales};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_ALIGN;
  return from_cuda(launch_quantize_act_128x1(x, rows, cols, static_cast<uint8_t*>(q), scales,
                                             as_stream(stream)));
}

moe_status_t moe_experts_backward_input_fp8(
    const moe_cfg_t* cfg, const void* x_perm, const float* x_perm_scales, const void* x_q,
    const float* x_q_scales, const int32_t* offsets, const void* w13, const float* w13_scales,
    const void* w13t, const float* w13t_scales, const void* w2t, const float* w2t_scales,
    const void* ws13, const float* ws13_scales, const void* ws13t, const float* ws13t_scales,
    const void* ws2t, const float* ws2t_scales, const void* dy_perm, const void* dout,
    void* dx_perm, void* dx_shared, int32_t ab_kept, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = moe_check_cfg(cfg);
  if (st != MOE_OK) return st;
  const moe_cfg_t& c = *cfg;
  if (c.dtype != MOE_DTYPE_FP8_E4M3 || c.n_shared > 1) return MOE_ERR_SHAPE;
  // (its scratch is the expert part of the backward workspace)
  const void* need[] = {x_perm, x_perm_scales, offsets, w13, w13_scales, w13t, w13t_scales,
                        w2t, w2t_scales, dy_perm, dx_perm, ws};
  for (const void* p : need)
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0) {
    const void* need_sh[] = {x_q, x_q_scales, ws13, ws13_scales, ws13t, ws13t_scales, ws2t,
                             ws2t_scales, dout, dx_shared};
    for (const void* p : need_sh)
      if (p == nullptr) return MOE_ERR_INVALID_ARG;
  }
  const void* ptrs[] = {x_perm, x_perm_scales, x_q, x_q_scales, offsets, w13, w13_scales,
                        w13t, w13t_scales, w2t, w2t_scales, ws13, ws13_scales, ws13t,
                        ws13t_scales, ws2t, ws2t_scales, dy_perm, dout, dx_perm, dx_shared, ws};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_ALIGN;
  if (ws_bytes < experts_bwd_fp8_scratch_bytes(c)) return MOE_ERR_WORKSPACE;
  ExpertsBwdFp8Args a{};
  a.cfg = &c;
  a.x_perm = x_perm; a.x_perm_scales = x_perm_scales; a.x_q = x_q; a.x_q_scales = x_q_scales;
  a.offsets = offsets;
  a.w13 = w13; a.w13_scales = w13_scales; a.w13t = w13t; a.w13t_scales = w13t_scales;
  a.w2t = w2t; a.w2t_scales = w2t_scales;
  a.ws13 = ws13; a.ws13_scales = ws13_scales; a.ws13t = ws13t; a.ws13t_scales = ws13t_scales;
  a.ws2t = ws2t; a.ws2t_scales = ws2t_scales;
  a.dy_perm = dy_perm; a.dout = dout; a.dx_perm = dx_perm;
  a.dx_shared = c.n_shared > 0 ? dx_shared : nullptr;
  a.ws = ws;
  a.ab_kept = ab_kept != 0;
  return from_cuda(launch_experts_bwd_input_fp8(a, as_stream(stream)));
}

moe_status_t moe_experts_grouped_train_fp8(
    const moe_cfg_t* cfg, const void* x_perm, const float* x_perm_scales, const void* x,
    const float* x_scales, const int32_t* offsets, const void* w13, const float* w13_scales,
    const void* w2, const float* w2_scales, const void* ws13, const float* ws13_scales,
    const void* ws2, const float* ws2_scales, void* y_perm, void* y_shared, void* ws,
    size_t ws_bytes, void* bws, size_t bws_bytes, void* stream) {
  moe_status_t st = moe_check_cfg(cfg);
  if (st != MOE_OK) return st;
  const moe_cfg_t& c = *cfg;
  if (c.dtype != MOE_DTYPE_FP8_E4M3 || c.n_shared > 1) return MOE_ERR_SHAPE;
  if (bws == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(bws)) return MOE_ERR_ALIGN;
  if (bws_bytes < moe_backward_workspace_bytes(cfg)) return MOE_ERR_WORKSPACE;
  const __nv_bfloat16 *ab = nullptr, *dh = nullptr;
  experts_bwd_fp8_ab_dh(c, bws, &ab, &dh);
  __nv_bfloat16* abw = const_cast<__nv_bfloat16*>(ab);
  return experts_grouped(cfg, x_perm, x_perm_scales, x, x_scales, offsets, w13, w13_scales, w2,
                         w2_scales, ws13, ws13_scales, ws2, ws2_scales, nullptr, nullptr, y_perm,
                         y_shared, ws, ws_bytes, stream, abw,
                         abw + static_cast<size_t>(c.T) * c.K * 2 * c.inter);
}

moe_status_t moe_experts_backward_weights_fp8(
    const moe_cfg_t* cfg, const void* x_perm, const float* x_perm_scales, const void* x_q,
    const float* x_q_scales, const int32_t* offsets, const void* dy_perm, const void* dout,
    void* dw13, void* dw2, void* dws13, void* dws2, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = moe_check_cfg(cfg);
  if (st != MOE_OK) return st;
  const moe_cfg_t& c = *cfg;
  if (c.dtype != MOE_DTYPE_FP8_E4M3 || c.n_shared > 1) return MOE_ERR_SHAPE;
  const void* need[] = {x_perm, x_perm_scales, offsets, dy_perm, dw13, dw2, ws};
  for (const void* p : need)
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0) {
    const void* need_sh[] = {x_q, x_q_scales, dout, dws13, dws2};
    for (const void* p : need_sh)
      if (p == nullptr) return MOE_ERR_INVALID_ARG;
  }
  const void* ptrs[] = {x_perm, x_perm_scales, x_q, x_q_scales, offsets, dy_perm, dout,
                        dw13, dw2, dws13, dws2, ws};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_ALIGN;
  if (ws_bytes < moe_backward_workspace_bytes(cfg)) return MOE_ERR_WORKSPACE;
  ExpertsBwdWeightsFp8Args a{};
  a.cfg = &c;
  a.x_perm = x_perm; a.x_perm_scales = x_perm_scales; a.x_q = x_q; a.x_q_scales = x_q_scales;
  a.offsets = offsets; a.dy_perm = dy_perm; a.dout = dout;
  experts_bwd_fp8_ab_dh(c, ws, &a.ab, &a.dh);
  a.dw13 = dw13; a.dw2 = dw2;
  a.dws13 = c.n_shared > 0 ? dws13 : nullptr;
  a.dws2 = c.n_shared > 0 ? dws2 : nullptr;
  a.wg_ws = static_cast<char*>(ws) + experts_bwd_fp8_scratch_bytes(c);
  return from_cuda(launch_experts_bwd_weights_fp8(a, as_stream(stream)));
}

moe_status_t moe_quantize_weights_fp8(const void* w_bf16, int32_t n_mats, int32_t rows,
                                      int32_t cols, void* q, float* scales, void* stream) {
  if (w_bf16 == nullptr || q == nullptr || scales == nullptr) return MOE_ERR_INVALID_ARG;
  if (n_mats < 1 || rows < 1 || cols < 1) return MOE_ERR_INVALID_ARG;
  if (cols % 128 != 0 || n_mats > 65535 || (rows + 127) / 128 > 65535) return MOE_ERR_SHAPE;
  if (!aligned16(w_bf16) || !aligned16(q) || !aligned16(scales)) return MOE_ERR_ALIGN;
  return from_cuda(launch_quantize_weights_fp8(w_bf16, n_mats, rows, cols, q, scales,
                                               as_stream(stream)));
}

moe_status_t moe_selftest_wait(int64_t limit_ns, void* stream) {
  if (limit_ns < 1 || limit_ns > 10000000000LL) return MOE_ERR_INVALID_ARG;
  selftest_wait_kernel<<<1, 32, 0, as_stream(stream)>>>(static_cast<uint64_t>(limit_ns));
  return from_cuda(cudaGetLastError());
}

moe_status_t moe_get_device_error(void* stream) {
  cudaStream_t s = as_stream(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word)) != cudaSuccess) return MOE_ERR_CUDA;
  const uint32_t zero = 0;
  if (word != 0 && cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (word & kErrTimeout) return MOE_ERR_TIMEOUT;
  if (word != 0) return MOE_ERR_DEVICE;
  return MOE_OK;
}

}  // extern "C"
