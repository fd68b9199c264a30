// Decode-kernel instantiations for bf16 caches: both compute paths, head_dim 64/128,
// output in the cache type or fp32, plain and split mode.
#include "pa_decode_launch.cuh"

PA_INSTANTIATE_DECODE(__nv_bfloat16, __nv_bfloat16, 64, true)
PA_INSTANTIATE_DECODE(__nv_bfloat16, float, 64, true)
PA_INSTANTIATE_SPLIT(__nv_bfloat16, 64, true)
PA_INSTANTIATE_DECODE(__nv_bfloat16, __nv_bfloat16, 64, false)
PA_INSTANTIATE_DECODE(__nv_bfloat16, float, 64, false)
PA_INSTANTIATE_SPLIT(__nv_bfloat16, 64, false)
PA_INSTANTIATE_DECODE(__nv_bfloat16, __nv_bfloat16, 128, true)
PA_INSTANTIATE_DECODE(__nv_bfloat16, float, 128, true)
PA_INSTANTIATE_SPLIT(__nv_bfloat16, 128, true)
PA_INSTANTIATE_DECODE(__nv_bfloat16, __nv_bfloat16, 128, false)
PA_INSTANTIATE_DECODE(__nv_bfloat16, float, 128, false)
PA_INSTANTIATE_SPLIT(__nv_bfloat16, 128, false)

template pa_status pa::launch_lse_reduce<__nv_bfloat16, 64>(const pa::DecodeParams&, cudaStream_t);
template pa_status pa::launch_lse_reduce<__nv_bfloat16, 128>(const pa::DecodeParams&, cudaStream_t);
