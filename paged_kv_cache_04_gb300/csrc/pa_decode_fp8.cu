// Decode-kernel instantiations for FP8 (E4M3) caches: bf16 or fp16 queries, head_dim
// 128, plain and split mode, on the tensor-core path at every group (in fp16).
#include "pa_decode_launch.cuh"

PA_INSTANTIATE_DECODE(pa::fp8e4m3, __nv_bfloat16, __nv_bfloat16, 128, pa::kPathMma)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __nv_bfloat16, float, 128, pa::kPathMma)
PA_INSTANTIATE_SPLIT(pa::fp8e4m3, __nv_bfloat16, 128, pa::kPathMma)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __half, __half, 128, pa::kPathMma)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __half, float, 128, pa::kPathMma)
PA_INSTANTIATE_SPLIT(pa::fp8e4m3, __half, 128, pa::kPathMma)
// plain decode at groups of 5-8 (merge in rounds of four heads)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __nv_bfloat16, __nv_bfloat16, 128, pa::kPathMmaG8)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __nv_bfloat16, float, 128, pa::kPathMmaG8)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __half, __half, 128, pa::kPathMmaG8)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __half, float, 128, pa::kPathMmaG8)
