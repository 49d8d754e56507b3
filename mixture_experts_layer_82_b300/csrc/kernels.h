// Host-side launchers of the libmoe kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Tokens per routing tile: the unit of the per-expert histogram and of the
// within-segment rank (one 32-bit mask per expert and tile).
constexpr int kRouteTile = 32;

struct RouteScratch {
  float* affinity;        // [T, E] when the caller keeps none
  int32_t* tile_counts;   // [ceil(T/32), E], later the per-tile segment base
  void* router;           // bf16 kinds: split centroids and split-K partials
};

// Layout of the routing scratch inside a workspace buffer.
size_t route_scratch_bytes(const moe_cfg_t& c, bool need_affinity);
RouteScratch route_scratch_carve(const moe_cfg_t& c, void* ws, bool need_affinity);

cudaError_t launch_router_affinity(const moe_cfg_t& c, const void* x, const float* w,
                                   float* affinity, const RouteScratch& rs, cudaStream_t s);
size_t router_tc_scratch_bytes(const moe_cfg_t& c);
cudaError_t launch_router_tc(const moe_cfg_t& c, const void* x, const float* w, float* affinity,
                             void* scratch, cudaStream_t s);
cudaError_t launch_route_select(const moe_cfg_t& c, const float* affinity, const float* bias,
                                int32_t* topk_idx, float* topk_w, int32_t* local_rank,
                                int32_t* tile_counts, cudaStream_t s);
cudaError_t launch_route_scan(const moe_cfg_t& c, int32_t* tile_counts, int32_t* counts,
                              int32_t* offsets, cudaStream_t s);
cudaError_t launch_route_assign(const moe_cfg_t& c, const int32_t* topk_idx,
                                const int32_t* offsets, const int32_t* tile_base,
                                int32_t* row_of_slot /* in: local rank, out: row */,
                                int32_t* token_of_row, cudaStream_t s);
cudaError_t launch_bias_update(const moe_cfg_t& c, const int32_t* counts, float* bias,
                               cudaStream_t s);
size_t balance_scratch_bytes(const moe_cfg_t& c, int seq_len);
cudaError_t launch_balance_stat(const moe_cfg_t& c, const float* affinity, const int32_t* topk_idx,
                                int seq_len, float alpha, float* f_out, float* p_out, float* loss,
                                void* ws, cudaStream_t s);

// permute / combine / quantise
cudaError_t launch_permute(const moe_cfg_t& c, const void* x, const int32_t* token_of_row,
                           void* x_perm, size_t elem_bytes, cudaStream_t s);
cudaError_t launch_quantize_act_fp8(const void* x_bf16, int rows, int cols, void* q,
                                    float* scales, cudaStream_t s);
cudaError_t launch_permute_fp8(const moe_cfg_t& c, const void* x_q, const float* x_scales,
                               const int32_t* token_of_row, void* x_perm, float* x_perm_scales,
                               cudaStream_t s);
// gate_of_row[row_of_slot[i]] = topk_w[i] for every (token, slot) i.
cudaError_t launch_gate_rows(const moe_cfg_t& c, const int32_t* row_of_slot, const float* topk_w,
                             float* gate_of_row, cudaStream_t s);
cudaError_t launch_combine(const moe_cfg_t& c, const void* y_perm, const void* y_shared,
                           const int32_t* row_of_slot, const float* topk_w, void* out,
                           cudaStream_t s);
cudaError_t launch_quantize_weights_fp8(const void* w, int n_mats, int rows, int cols, void* q,
                                        float* scales, cudaStream_t s);

// expert GEMMs
struct ExpertsArgs {
  const moe_cfg_t* cfg;
  const void* x_perm;
  const float* x_perm_scales;
  const void* x;
  const float* x_scales;
  const int32_t* offsets;
  const void* w13;
  const float* w13_scales;
  const void* w2;
  const float* w2_scales;
  const void* ws13;
  const float* ws13_scales;
  const void* ws2;
  const float* ws2_scales;
  void* y_perm;
  void* y_shared;
  const int32_t* token_of_row;  // non-null: gate/up gathers its routed A rows from x
  void* h;            // workspace: routed rows [T*K, I] then shared rows [T, Ns*I]
  float* h_scales;    // FP8: [T*K, I/128] then [T, Ns*I/128]
  __nv_bfloat16* ab;         // training forward, optional: [a | b] rows kept for the
  __nv_bfloat16* ab_shared;  // backward ([T*K, 2I] and [T, Ns*2I]; FP8: Ns <= 1)
  const float* gate_of_row;  // optional [T*K]: the down projection writes gate * y
};

size_t experts_scratch_bytes(const moe_cfg_t& c);
void experts_scratch_carve(const moe_cfg_t& c, void* ws, void** h, float** h_scales);
// The gate of every permuted row ([T*K] fp32) in the experts' scratch.
float* experts_gate_rows(const moe_cfg_t& c, void* ws);

cudaError_t launch_experts_fp32(const ExpertsArgs& a, cudaStream_t s);
cudaError_t launch_experts_bf16(const ExpertsArgs& a, cudaStream_t s);
cudaError_t launch_experts_fp8(const ExpertsArgs& a, cudaStream_t s);

// backward (BF16 kind)
struct ExpertsBwdScratch {
  __nv_bfloat16* ab;         // [T*K, 2I]: [a | b], then [da | db]
  __nv_bfloat16* ab_shared;  // [T, N_s * 2I]: per shared expert [a | b], then [da | db]
  __nv_bfloat16* h;          // [T*K, I]
  __nv_bfloat16* h_shared;   // [T, N_s * I]
};

struct ExpertsBwdArgs {
  const moe_cfg_t* cfg;
  const void* x_perm;
  const void* x;
  const int32_t* offsets;
  const void* w13;
  const void* w2;
  const void* ws13;
  const void* ws2;
  const void* dy_perm;
  const void* dout;
  void* dx_perm;
  void* dx_shared;
  void* dw13;
  void* dw2;
  void* dws13;
  void* dws2;
  bool ab_kept;  // the forward kept [a | b] in the scratch: no recomputation
  ExpertsBwdScratch scratch;
};

// Backward for input of the FP8 expert FFNs (backward_fp8.cu).
struct ExpertsBwdFp8Args {
  const moe_cfg_t* cfg;
  const void* x_perm;          // forward's E4M3 rows [T*K, d] and 1 x 128 scales
  const float* x_perm_scales;
  const void* x_q;             // forward's E4M3 token rows [T, d] (shared expert)
  const float* x_q_scales;
  const int32_t* offsets;
  const void* w13;             // [E, 2I, d] codes, [E, 2I/128, d/128] scales
  const float* w13_scales;
  const void* w13t;            // [E, d, 2I] transposed codes and block scales
  const float* w13t_scales;
  const void* w2t;             // [E, I, d] transposed W2 codes and block scales
  const float* w2t_scales;
  const void* ws13;            // the shared expert's: [1, 2I, d], [1, d, 2I], [1, I, d]
  const float* ws13_scales;
  const void* ws13t;
  const float* ws13t_scales;
  const void* ws2t;
  const float* ws2t_scales;
  const void* dy_perm;         // [T*K, d] bf16
  const void* dout;            // [T, d] bf16
  void* dx_perm;               // [T*K, d] bf16 out
  void* dx_shared;             // [T, d] bf16 out
  void* ws;                    // experts_bwd_fp8_scratch_bytes
  bool ab_kept;                // ws already holds [a | b] from the training forward
};
size_t experts_bwd_fp8_scratch_bytes(const moe_cfg_t& c);

// Backward for weights of the FP8 expert FFNs (backward_fp8_wgrad.cu): from
// the forward's codes, the caller's dy and the [a | b] and dh the input
// side left in its scratch.
struct ExpertsBwdWeightsFp8Args {
  const moe_cfg_t* cfg;
  const void* x_perm;
  const float* x_perm_scales;
  const void* x_q;
  const float* x_q_scales;
  const int32_t* offsets;
  const void* dy_perm;
  const void* dout;
  const __nv_bfloat16* ab;  // [T*K + T, 2I]
  const __nv_bfloat16* dh;  // [T*K + T, I]
  void* dw13;               // [E, 2I, d] bf16 out
  void* dw2;                // [E, d, I] bf16 out
  void* dws13;              // [1, 2I, d], [1, d, I] (N_s = 1)
  void* dws2;
  void* wg_ws;              // experts_wgrad_fp8_scratch_bytes
};
size_t experts_wgrad_fp8_scratch_bytes(const moe_cfg_t& c);
// bf16 x [rows, cols] (cols % 128 == 0) in 128 x 1 tiles along the rows:
// codes [round128(rows), cols] (rows past `rows` zero), scales [rows/128 up, cols].
cudaError_t launch_quantize_act_128x1(const void* x, int rows, int cols, uint8_t* q, float* scales,
                                      cudaStream_t s);
cudaError_t launch_experts_bwd_weights_fp8(const ExpertsBwdWeightsFp8Args& a, cudaStream_t s);
// [a | b] and dh of the routed rows in the FP8 input side's scratch (the
// shared expert's rows follow them).
void experts_bwd_fp8_ab_dh(const moe_cfg_t& c, void* ws, const __nv_bfloat16** ab,
                           const __nv_bfloat16** dh);
cudaError_t launch_experts_bwd_input_fp8(const ExpertsBwdFp8Args& a, cudaStream_t s);
cudaError_t launch_transpose_weights_fp8(const void* w_q, const float* w_scales, int n_mats,
                                         int rows, int cols, void* wt_q, float* wt_scales,
                                         cudaStream_t s);

struct RouteBwdArgs {
  const void* x;
  const float* router_w;
  const float* affinity;
  const int32_t* topk_idx;
  const float* dgate;
  const int32_t* row_of_slot;
  const int32_t* token_of_row;
  const int32_t* offsets;
  const void* dx_perm;
  const void* dx_shared;
  float* dlogit;
  float* dlogit_row;  // scratch [T*K]
  void* dx;
  float* drouter_w;
};

size_t experts_bwd_scratch_bytes(const moe_cfg_t& c);
ExpertsBwdScratch experts_bwd_scratch_carve(const moe_cfg_t& c, void* ws);
cudaError_t launch_experts_bwd_input_bf16(const ExpertsBwdArgs& a, cudaStream_t s);
cudaError_t launch_experts_bwd_weights_bf16(const ExpertsBwdArgs& a, cudaStream_t s);
cudaError_t launch_combine_backward(const moe_cfg_t& c, const void* dout, const void* y_perm,
                                    const int32_t* row_of_slot, const float* topk_w,
                                    void* dy_perm, float* dgate, cudaStream_t s);
cudaError_t launch_route_backward(const moe_cfg_t& c, const RouteBwdArgs& a, cudaStream_t s);

// Driver entry point of cuTensorMapEncodeTiled (resolved once).
CUresult encode_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, void* base,
                              uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                              uint32_t box_inner, uint32_t box_outer,
                              CUtensorMapSwizzle swizzle);
// Rank-n map: dims and box innermost first; strides_bytes[i] is the stride
// of dimension i + 1.
CUresult encode_tensor_map_nd(CUtensorMap* m, CUtensorMapDataType dt, void* base, int rank,
                              const uint64_t* dims, const uint64_t* strides_bytes,
                              const uint32_t* box, CUtensorMapSwizzle swizzle);

// The gate/up weights [n, 2I, d] seen as [n][2][I][d]: one box of
// box_k x box_rows x 2 x 1 is box_rows W1 rows followed by the matching
// box_rows W3 rows (box_mats = 2); with box_mats = 1 a box is the W1 or the
// W3 rows alone.
CUresult encode_gate_up_map(CUtensorMap* m, CUtensorMapDataType dt, const void* w13, int n,
                            int inter, int d, size_t elem_bytes, uint32_t box_k,
                            uint32_t box_mats = 2, uint32_t box_rows = 128);

// The gate/up weights [n, 2I, d] seen as [n][I/64][2][64][d]: one box of
// box_k x 64 x 2 x 2 x 1 is 64 W1 rows, the matching 64 W3 rows, the next
// 64 W1 rows and their 64 W3 rows (I % 128 == 0).
CUresult encode_gate_up_map_interleaved(CUtensorMap* m, CUtensorMapDataType dt, const void* w13,
                                        int n, int inter, int d, size_t elem_bytes,
                                        uint32_t box_k);

}  // namespace moe
