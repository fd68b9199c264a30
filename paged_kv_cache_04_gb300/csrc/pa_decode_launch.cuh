// Host launchers for the decode kernels (included by the per-dtype units).
#pragma once

#include <mutex>

#include "pa_decode.cuh"
#include "pa_internal.h"

namespace pa {

template <typename DT, typename QT, typename OT, int D, int PATH, int MODE>
pa_status launch_decode(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                        int num_sms, long long max_items, cudaStream_t stream) {
  using Cfg = StageCfg<DT, D, PATH, MODE>;
  auto kern = paged_decode_kernel<DT, QT, OT, D, PATH, MODE>;
  DecodeParams q = p;
  q.order_cap = MODE == kModePlain ? plain_order_cap(p.S, p.G, num_sms) : 0;
  const SmemLayout L =
      make_layout(Cfg::W, Cfg::R, D, Cfg::E, (int)sizeof(QT), p.group, PATH, MODE == kModeSplit, p.S, Cfg::JPS,
                  MODE == kModeSuffix, q.order_cap);
  if (L.total > 227u * 1024u) return PA_ERR_UNSUPPORTED;

  // Opt in to the dynamic shared memory once per device, and remember the
  // occupancy for the last shared-memory size seen on that device.
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
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Cfg::W * 32, L.total) != cudaSuccess)
        return PA_ERR_CUDA;
      occ_bytes[dev] = L.total;
      occ_blocks[dev] = n;
    }
    per_sm = occ_blocks[dev];
  }
  if (per_sm < 1) return PA_ERR_UNSUPPORTED;
  long long grid = (long long)num_sms * per_sm;
  // the suffix pass deals items to warps, the other modes to CTAs
  const long long ctas = MODE == kModeSuffix ? (max_items + Cfg::W - 1) / Cfg::W : max_items;
  if (ctas < grid) grid = ctas;
  if (grid <= 0) return PA_OK;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(Cfg::W * 32), L.total, stream, kmap, vmap, q) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

template <typename OT, int D>
pa_status launch_lse_reduce(const DecodeParams& p, cudaStream_t stream) {
  const long long rows = (long long)p.S * p.H;
  if (rows <= 0) return PA_OK;
  const cudaError_t e =
      p.max_partitions <= 32
          ? launch_pdl(lse_reduce_small_kernel<OT, D>, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, stream, p)
          : launch_pdl(lse_reduce_kernel<OT, D>, dim3((unsigned)rows), dim3(256), 0, stream, p);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa

// Explicit instantiations for one element type DT (the tensor-core path only
// exists for 16-bit types).
#define PA_INSTANTIATE_DECODE(DT, QT, OT, D, PATH)                                                        \
  template pa_status pa::launch_decode<DT, QT, OT, D, PATH, pa::kModePlain>(                               \
      const CUtensorMap&, const CUtensorMap&, const pa::DecodeParams&, int, long long, cudaStream_t);
#define PA_INSTANTIATE_SPLIT(DT, QT, D, PATH)                                                               \
  template pa_status pa::launch_decode<DT, QT, float, D, PATH, pa::kModeSplit>(                            \
      const CUtensorMap&, const CUtensorMap&, const pa::DecodeParams&, int, long long, cudaStream_t);
#define PA_INSTANTIATE_SUFFIX(DT, QT, D, PATH)                                                              \
  template pa_status pa::launch_decode<DT, QT, float, D, PATH, pa::kModeSuffix>(                           \
      const CUtensorMap&, const CUtensorMap&, const pa::DecodeParams&, int, long long, cudaStream_t);
