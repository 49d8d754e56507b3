// moe_route_static_scratch: the routing call of moe_route with its scratch
// memory taken from a fixed array inside the library instead of a
// caller-provided workspace, for callers that cannot allocate device memory.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kStaticScratchBytes of it until the process exits.  Host code
// must not pass the array's name to a kernel (on the host it is only a
// stand-in symbol); the device address is looked up once per device with
// cudaGetSymbolAddress, on the first call made on that device.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr size_t kStaticScratchBytes = size_t{32} << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_route_scratch[kStaticScratchBytes];

static void* g_static_scratch_addr[kMaxDevices] = {};
static std::mutex g_static_scratch_mu;

// Device address of the static scratch on the current device.
static cudaError_t static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_scratch_mu);
  if (g_static_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_route_scratch);
    if (e != cudaSuccess) return e;
    g_static_scratch_addr[dev] = p;
  }
  *out = g_static_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace moe

extern "C" moe_status_t moe_route_static_scratch(
    const moe_cfg_t* cfg, const void* x, const float* router_w, const float* bias,
    const float* affinity_in, float* affinity_out, int32_t* topk_idx, float* topk_w,
    int32_t* counts, int32_t* offsets, int32_t* row_of_slot, int32_t* token_of_row,
    void* stream) {
  using namespace moe;
  moe_status_t st = moe_check_cfg(cfg);
  if (st != MOE_OK) return st;
  const moe_cfg_t& c = *cfg;
  if (bias == nullptr || topk_idx == nullptr || topk_w == nullptr || counts == nullptr ||
      offsets == nullptr || row_of_slot == nullptr || token_of_row == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (affinity_in == nullptr && (x == nullptr || router_w == nullptr)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, router_w, bias, affinity_in, affinity_out, topk_idx, topk_w,
                        counts, offsets, row_of_slot, token_of_row};
  for (const void* p : ptrs)
    if (p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) != 0) return MOE_ERR_ALIGN;
  const bool need_aff = affinity_in == nullptr && affinity_out == nullptr;
  if (route_scratch_bytes(c, need_aff) > kStaticScratchBytes) return MOE_ERR_WORKSPACE;
  void* ws = nullptr;
  if (static_scratch_address(&ws) != cudaSuccess) return MOE_ERR_CUDA;
  // Every scratch word the kernels read is written earlier in the same call
  // (per-tile loads by the selection kernel, affinities by the router), so
  // nothing has to be cleared between calls.
  const RouteScratch rs = route_scratch_carve(c, ws, need_aff);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float* aff = affinity_in;
  if (aff == nullptr) {
    float* dst = affinity_out != nullptr ? affinity_out : rs.affinity;
    if (launch_router_affinity(c, x, router_w, dst, rs, s) != cudaSuccess) return MOE_ERR_CUDA;
    aff = dst;
  } else if (affinity_out != nullptr && affinity_out != affinity_in) {
    if (cudaMemcpyAsync(affinity_out, affinity_in, static_cast<size_t>(c.T) * c.E * sizeof(float),
                        cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  cudaError_t e = launch_route_select(c, aff, bias, topk_idx, topk_w, row_of_slot, rs.tile_counts, s);
  if (e == cudaSuccess) e = launch_route_scan(c, rs.tile_counts, counts, offsets, s);
  if (e == cudaSuccess)
    e = launch_route_assign(c, topk_idx, offsets, rs.tile_counts, row_of_slot, token_of_row, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
