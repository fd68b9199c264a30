// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>

#include "pa.h"

namespace pa {

struct DecodeParams;

// Every argument check of pa_decode_split except those on the workspace itself
// (pa_api.cu); *need receives the workspace size (0 for an empty batch).
pa_status check_split_call(const void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                           int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                           pa_kv_layout layout, int64_t num_blocks, float scale, pa_dtype dtype, pa_dtype out_dtype,
                           int max_context_len, int partition_tokens, size_t* need);

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

// The same pass on tcgen05 tensor cores (pa_cascade.cu); qmap views q as
// [S][H][D] with a box of MR / group sequences x group heads x 64 columns.
template <typename DT, int D, int MR>
pa_status launch_cascade_prefix_tc(const CUtensorMap& kmap, const CUtensorMap& vmap, const CUtensorMap& qmap,
                                   const DecodeParams& p, int num_sms, long long max_items, cudaStream_t stream);

}  // namespace pa
