// Decode-kernel instantiations of plain decode for groups of 5-8 query heads per
// kv head on 16-bit caches (the tensor-core path that merges the warps'
// partials four heads per round): bf16 and fp16, head_dim 64/128/256, output
// in the cache type or fp32. Split and suffix mode use the kPathMma kernels.
#include "pa_decode_launch.cuh"

PA_INSTANTIATE_DECODE(__nv_bfloat16, __nv_bfloat16, __nv_bfloat16, 64, pa::kPathMmaG8)
PA_INSTANTIATE_DECODE(__nv_bfloat16, __nv_bfloat16, float, 64, pa::kPathMmaG8)
PA_INSTANTIATE_DECODE(__nv_bfloat16, __nv_bfloat16, __nv_bfloat16, 128, pa::kPathMmaG8)
PA_INSTANTIATE_DECODE(__nv_bfloat16, __nv_bfloat16, float, 128, pa::kPathMmaG8)
PA_INSTANTIATE_DECODE(__nv_bfloat16, __nv_bfloat16, __nv_bfloat16, 256, pa::kPathMmaG8)
PA_INSTANTIATE_DECODE(__nv_bfloat16, __nv_bfloat16, float, 256, pa::kPathMmaG8)
PA_INSTANTIATE_DECODE(__half, __half, __half, 64, pa::kPathMmaG8)
PA_INSTANTIATE_DECODE(__half, __half, float, 64, pa::kPathMmaG8)
PA_INSTANTIATE_DECODE(__half, __half, __half, 128, pa::kPathMmaG8)
PA_INSTANTIATE_DECODE(__half, __half, float, 128, pa::kPathMmaG8)
PA_INSTANTIATE_DECODE(__half, __half, __half, 256, pa::kPathMmaG8)
PA_INSTANTIATE_DECODE(__half, __half, float, 256, pa::kPathMmaG8)
