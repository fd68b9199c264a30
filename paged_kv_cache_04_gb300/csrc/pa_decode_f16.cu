// Decode-kernel instantiations for fp16 caches, head_dim 64/128: the MHA vector
// path (group 1) and the tensor-core path (groups 2-8; plain decode at groups 5-8
// is in pa_decode_g8.cu), output in the cache type or fp32, plain, split and
// shared-prefix suffix mode.
#include "pa_decode_launch.cuh"

PA_INSTANTIATE_DECODE(__half, __half, __half, 64, pa::kPathVecMha)
PA_INSTANTIATE_DECODE(__half, __half, float, 64, pa::kPathVecMha)
PA_INSTANTIATE_SPLIT(__half, __half, 64, pa::kPathVecMha)
PA_INSTANTIATE_SUFFIX(__half, __half, 64, pa::kPathVecMha)
PA_INSTANTIATE_DECODE(__half, __half, __half, 64, pa::kPathMma)
PA_INSTANTIATE_DECODE(__half, __half, float, 64, pa::kPathMma)
PA_INSTANTIATE_SPLIT(__half, __half, 64, pa::kPathMma)
PA_INSTANTIATE_SUFFIX(__half, __half, 64, pa::kPathMma)
PA_INSTANTIATE_DECODE(__half, __half, __half, 128, pa::kPathVecMha)
PA_INSTANTIATE_DECODE(__half, __half, float, 128, pa::kPathVecMha)
PA_INSTANTIATE_SPLIT(__half, __half, 128, pa::kPathVecMha)
PA_INSTANTIATE_SUFFIX(__half, __half, 128, pa::kPathVecMha)
PA_INSTANTIATE_DECODE(__half, __half, __half, 128, pa::kPathMma)
PA_INSTANTIATE_DECODE(__half, __half, float, 128, pa::kPathMma)
PA_INSTANTIATE_SPLIT(__half, __half, 128, pa::kPathMma)
PA_INSTANTIATE_SUFFIX(__half, __half, 128, pa::kPathMma)

template pa_status pa::launch_lse_reduce<__half, 64>(const pa::DecodeParams&, cudaStream_t);
template pa_status pa::launch_lse_reduce<__half, 128>(const pa::DecodeParams&, cudaStream_t);
