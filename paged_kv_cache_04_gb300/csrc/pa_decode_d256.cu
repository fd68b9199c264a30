// Decode-kernel instantiations for head_dim 256 (bf16, fp16, fp32 caches): the
// vector path (q in shared memory: MHA on 16-bit caches, every group on fp32) and,
// for 16-bit caches with a group of >= 2, the tensor-core path; plain and split
// mode, and the reduce. The shared-prefix suffix pass and the E4M3 caches stop at
// head_dim 128.
#include "pa_decode_launch.cuh"

PA_INSTANTIATE_DECODE(__nv_bfloat16, __nv_bfloat16, __nv_bfloat16, 256, pa::kPathVec)
PA_INSTANTIATE_DECODE(__nv_bfloat16, __nv_bfloat16, float, 256, pa::kPathVec)
PA_INSTANTIATE_SPLIT(__nv_bfloat16, __nv_bfloat16, 256, pa::kPathVec)
PA_INSTANTIATE_DECODE(__nv_bfloat16, __nv_bfloat16, __nv_bfloat16, 256, pa::kPathMma)
PA_INSTANTIATE_DECODE(__nv_bfloat16, __nv_bfloat16, float, 256, pa::kPathMma)
PA_INSTANTIATE_SPLIT(__nv_bfloat16, __nv_bfloat16, 256, pa::kPathMma)
PA_INSTANTIATE_DECODE(__half, __half, __half, 256, pa::kPathVec)
PA_INSTANTIATE_DECODE(__half, __half, float, 256, pa::kPathVec)
PA_INSTANTIATE_SPLIT(__half, __half, 256, pa::kPathVec)
PA_INSTANTIATE_DECODE(__half, __half, __half, 256, pa::kPathMma)
PA_INSTANTIATE_DECODE(__half, __half, float, 256, pa::kPathMma)
PA_INSTANTIATE_SPLIT(__half, __half, 256, pa::kPathMma)
PA_INSTANTIATE_DECODE(float, float, float, 256, pa::kPathVec)
PA_INSTANTIATE_SPLIT(float, float, 256, pa::kPathVec)

template pa_status pa::launch_lse_reduce<__nv_bfloat16, 256>(const pa::DecodeParams&, cudaStream_t);
template pa_status pa::launch_lse_reduce<__half, 256>(const pa::DecodeParams&, cudaStream_t);
template pa_status pa::launch_lse_reduce<float, 256>(const pa::DecodeParams&, cudaStream_t);
