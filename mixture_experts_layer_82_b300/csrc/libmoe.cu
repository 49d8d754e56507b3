// Single translation unit of libmoe: the per-device error word and the
// kernels that set it live in one module (no relocatable device code).
#include "moe_api.cu"
#include "route.cu"
#include "router_sm100.cu"
#include "permute.cu"
#include "experts_fp32.cu"
#include "experts_sm100.cu"
#include "experts_fp8.cu"
#include "backward_sm100.cu"
#include "backward.cu"
#include "backward_fp8.cu"
#include "tma.cu"
#include "route_static.cu"
