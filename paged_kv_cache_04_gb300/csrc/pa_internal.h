// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>

#include "pa.h"

namespace pa {

struct DecodeParams;

// Per-device state, set up on the first call on a device: the device address
// of the error word and the SM count. Returns PA_ERR_CUDA if CUDA fails.
pa_status device_state(unsigned** err, int* num_sms);

// Launchers, one per (cache type, query type, output type, head_dim, path,
// split) combination, instantiated in pa_decode_{f32,f16,bf16,fp8}.cu.
template <typename DT, typename QT, typename OT, int D, int PATH, int MODE>
pa_status launch_decode(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                        int num_sms, long long max_items, cudaStream_t stream);

template <typename OT, int D>
pa_status launch_lse_reduce(const DecodeParams& p, cudaStream_t stream);

// Prefix pass of the shared-prefix decode (pa_cascade.cu).
template <typename DT, int D, int NT>
pa_status launch_cascade_prefix(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                                int num_sms, long long max_items, cudaStream_t stream);

// The same pass on tcgen05 tensor cores (pa_cascade.cu).
template <typename DT, int D, int MR>
pa_status launch_cascade_prefix_tc(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                                   int num_sms, long long max_items, cudaStream_t stream);

}  // namespace pa
