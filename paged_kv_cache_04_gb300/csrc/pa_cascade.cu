// Launcher and instantiations of the shared-prefix (cascade) prefix pass.
#include <mutex>

#include "pa_cascade.cuh"
#include "pa_cascade_tc.cuh"
#include "pa_internal.h"

namespace pa {

template <typename DT, int D, int NT>
pa_status launch_cascade_prefix(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                                int num_sms, long long max_items, cudaStream_t stream) {
  auto kern = cascade_prefix_kernel<DT, D, NT>;
  const CascadeLayout L = cascade_layout(D, (int)sizeof(DT), p.num_groups);
  if (L.total > 227u * 1024u) return PA_ERR_UNSUPPORTED;
  static std::mutex mu;
  static unsigned set_bytes[64] = {0};
  static unsigned occ_bytes[64] = {0};
  static int occ_blocks[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
  int per_sm = 1;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (set_bytes[dev] < L.total) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total) != cudaSuccess)
        return PA_ERR_CUDA;
      set_bytes[dev] = L.total;
    }
    if (occ_bytes[dev] != L.total) {
      int n = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, (kCascadeConsumers + 1) * 32, L.total) !=
          cudaSuccess)
        return PA_ERR_CUDA;
      occ_bytes[dev] = L.total;
      occ_blocks[dev] = n;
    }
    per_sm = occ_blocks[dev];
  }
  if (per_sm < 1) return PA_ERR_UNSUPPORTED;
  // Three CTAs per SM: a fourth (which fits when the kernel needs under 100
  // registers) measured 6% slower on the 64 x 8-sample shared-prefix batch.
  if (per_sm > 3) per_sm = 3;
  long long grid = (long long)num_sms * per_sm;
  if (max_items < grid) grid = max_items;
  if (grid <= 0) return PA_OK;
  return launch_pdl(kern, dim3((unsigned)grid), dim3((kCascadeConsumers + 1) * 32), L.total, stream, kmap, vmap, p) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

template <typename DT, int D, int MR>
pa_status launch_cascade_prefix_tc(const CUtensorMap& kmap, const CUtensorMap& vmap, const CUtensorMap& qmap,
                                   const DecodeParams& p, int num_sms, long long max_items, cudaStream_t stream) {
  auto kern = cascade_prefix_tc_kernel<DT, D, MR>;
  const TcLayout L = tc_layout(D, p.num_groups, MR);
  if (L.total > 227u * 1024u) return PA_ERR_UNSUPPORTED;
  static std::mutex mu;
  static unsigned set_bytes[64] = {0};
  static unsigned occ_bytes[64] = {0};
  static int occ_blocks[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
  int per_sm = 1;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (set_bytes[dev] < L.total) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total) != cudaSuccess)
        return PA_ERR_CUDA;
      set_bytes[dev] = L.total;
    }
    if (occ_bytes[dev] != L.total) {
      // CTAs per SM from this kernel's own budget: shared memory (plus the 1 KiB
      // the driver reserves per CTA) within the SM's, and at most two, since two
      // CTAs' tensor-memory allocations fill the SM's 512 columns. (The runtime's
      // occupancy query answers 1 for this kernel although two fit.)
      int sm_bytes = 0;
      if (cudaDeviceGetAttribute(&sm_bytes, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess)
        return PA_ERR_CUDA;
      int n = sm_bytes / (int)(L.total + 1024u);
      occ_bytes[dev] = L.total;
      occ_blocks[dev] = n < 2 ? n : 2;
    }
    per_sm = occ_blocks[dev];
  }
  if (per_sm < 1) return PA_ERR_UNSUPPORTED;
  long long grid = (long long)num_sms * per_sm;
  if (max_items < grid) grid = max_items;
  if (grid <= 0) return PA_OK;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kTcThreads), L.total, stream, kmap, vmap, qmap, p) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

#define PA_INSTANTIATE_CASCADE_TC(DT, D, MR)                                                                \
  template pa_status launch_cascade_prefix_tc<DT, D, MR>(const CUtensorMap&, const CUtensorMap&,               \
                                                         const CUtensorMap&, const DecodeParams&, int, long long, \
                                                         cudaStream_t);
PA_INSTANTIATE_CASCADE_TC(__nv_bfloat16, 128, 64)
PA_INSTANTIATE_CASCADE_TC(__nv_bfloat16, 128, 128)
PA_INSTANTIATE_CASCADE_TC(__nv_bfloat16, 64, 64)
PA_INSTANTIATE_CASCADE_TC(__nv_bfloat16, 64, 128)
PA_INSTANTIATE_CASCADE_TC(__half, 128, 64)
PA_INSTANTIATE_CASCADE_TC(__half, 128, 128)
PA_INSTANTIATE_CASCADE_TC(__half, 64, 64)
PA_INSTANTIATE_CASCADE_TC(__half, 64, 128)

#define PA_INSTANTIATE_CASCADE(DT, D, NT)                                                                   \
  template pa_status launch_cascade_prefix<DT, D, NT>(const CUtensorMap&, const CUtensorMap&, const DecodeParams&, \
                                                      int, long long, cudaStream_t);
PA_INSTANTIATE_CASCADE(__nv_bfloat16, 128, 1)
PA_INSTANTIATE_CASCADE(__nv_bfloat16, 64, 1)
PA_INSTANTIATE_CASCADE(__half, 128, 1)
PA_INSTANTIATE_CASCADE(__half, 64, 1)

}  // namespace pa
