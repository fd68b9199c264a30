// pa_decode_split_static: the split decode with its scratch built into the
// library, for callers that cannot allocate device memory themselves.
//
// The partition results of the split path need somewhere to live between its
// two launches. pa_decode_split takes that space from the caller; this entry
// point instead uses one fixed array in the library's device memory, so a call
// allocates nothing (no cudaMalloc, no cudaFree, no allocating library call).
#include <cstdint>
#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace {

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_split_scratch[PA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// The array's device address on the current device. In host code the symbol
// is only a stand-in, so the address is looked up (once per device, with that
// device current) and cached.
pa_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_split_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" size_t pa_static_scratch_bytes(void) { return (size_t)PA_STATIC_SCRATCH_BYTES; }

extern "C" pa_status pa_decode_split_static(void* out, const void* q, const void* k_cache, const void* v_cache,
                                            const int32_t* block_tables, int max_blocks_per_seq,
                                            const int32_t* context_lens, int num_seqs, int num_heads,
                                            int num_kv_heads, int head_dim, int block_size, pa_kv_layout layout,
                                            int64_t num_blocks, float scale, pa_dtype dtype, pa_dtype out_dtype, int max_context_len,
                                            int partition_tokens, cudaStream_t stream) {
  // The same argument checks as pa_decode_split, in the same order, so that a bad
  // call gets the same status from both; the size limit comes after them.
  size_t need = 0;
  const pa_status chk = pa::check_split_call(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                             num_seqs, num_heads, num_kv_heads, head_dim, block_size, layout,
                                             num_blocks, scale, dtype, out_dtype, max_context_len, partition_tokens,
                                             &need);
  if (chk != PA_OK || num_seqs == 0) return chk;
  if (need > (size_t)PA_STATIC_SCRATCH_BYTES) return PA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const pa_status s = scratch_address(&scratch);
  if (s != PA_OK) return s;
  // Nothing in the scratch has to start at zero: the first launch writes every
  // partition entry that the second launch reads.
  return pa_decode_split(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                         num_heads, num_kv_heads, head_dim, block_size, layout, num_blocks, scale, dtype,
                         out_dtype, max_context_len, partition_tokens, scratch, (size_t)PA_STATIC_SCRATCH_BYTES,
                         stream);
}
