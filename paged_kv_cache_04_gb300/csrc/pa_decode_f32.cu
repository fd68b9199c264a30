// Decode-kernel instantiations for fp32 caches (vector paths), head_dim 64/128,
// plain and split mode, plus the fp32-output reduce.
#include "pa_decode_launch.cuh"

PA_INSTANTIATE_DECODE(float, float, float, 64, pa::kPathVec)
PA_INSTANTIATE_SPLIT(float, float, 64, pa::kPathVec)
PA_INSTANTIATE_DECODE(float, float, float, 64, pa::kPathVecMha)
PA_INSTANTIATE_SPLIT(float, float, 64, pa::kPathVecMha)
PA_INSTANTIATE_DECODE(float, float, float, 128, pa::kPathVec)
PA_INSTANTIATE_SPLIT(float, float, 128, pa::kPathVec)
PA_INSTANTIATE_DECODE(float, float, float, 128, pa::kPathVecMha)
PA_INSTANTIATE_SPLIT(float, float, 128, pa::kPathVecMha)

template pa_status pa::launch_lse_reduce<float, 64>(const pa::DecodeParams&, cudaStream_t);
template pa_status pa::launch_lse_reduce<float, 128>(const pa::DecodeParams&, cudaStream_t);
