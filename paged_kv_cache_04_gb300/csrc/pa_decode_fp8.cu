// Decode-kernel instantiations for FP8 (E4M3) caches: bf16 or fp16 queries, the
// three compute paths (tensor cores in fp16), head_dim 128, plain and split mode.
#include "pa_decode_launch.cuh"

PA_INSTANTIATE_DECODE(pa::fp8e4m3, __nv_bfloat16, __nv_bfloat16, 128, pa::kPathVec)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __nv_bfloat16, float, 128, pa::kPathVec)
PA_INSTANTIATE_SPLIT(pa::fp8e4m3, __nv_bfloat16, 128, pa::kPathVec)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __nv_bfloat16, __nv_bfloat16, 128, pa::kPathVecMha)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __nv_bfloat16, float, 128, pa::kPathVecMha)
PA_INSTANTIATE_SPLIT(pa::fp8e4m3, __nv_bfloat16, 128, pa::kPathVecMha)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __nv_bfloat16, __nv_bfloat16, 128, pa::kPathMma)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __nv_bfloat16, float, 128, pa::kPathMma)
PA_INSTANTIATE_SPLIT(pa::fp8e4m3, __nv_bfloat16, 128, pa::kPathMma)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __half, __half, 128, pa::kPathVec)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __half, float, 128, pa::kPathVec)
PA_INSTANTIATE_SPLIT(pa::fp8e4m3, __half, 128, pa::kPathVec)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __half, __half, 128, pa::kPathVecMha)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __half, float, 128, pa::kPathVecMha)
PA_INSTANTIATE_SPLIT(pa::fp8e4m3, __half, 128, pa::kPathVecMha)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __half, __half, 128, pa::kPathMma)
PA_INSTANTIATE_DECODE(pa::fp8e4m3, __half, float, 128, pa::kPathMma)
PA_INSTANTIATE_SPLIT(pa::fp8e4m3, __half, 128, pa::kPathMma)
