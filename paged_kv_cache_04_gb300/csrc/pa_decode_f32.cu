// Decode-kernel instantiations for fp32 caches (vector path), head_dim 64/128,
// plain and split mode, plus the fp32-output reduce.
#include "pa_decode_launch.cuh"

PA_INSTANTIATE_DECODE(float, float, 64, false)
PA_INSTANTIATE_SPLIT(float, 64, false)
PA_INSTANTIATE_DECODE(float, float, 128, false)
PA_INSTANTIATE_SPLIT(float, 128, false)

template pa_status pa::launch_lse_reduce<float, 64>(const pa::DecodeParams&, cudaStream_t);
template pa_status pa::launch_lse_reduce<float, 128>(const pa::DecodeParams&, cudaStream_t);
