// The kernels that keep the paged KV cache current (CS349E Lecture 7 notes,
// §4.3: one fused write of new tokens into their block slots, one batched copy
// of the blocks copy-on-write must duplicate; §6.2: swapping a preempted
// sequence's blocks to CPU memory and back). All are pure data movement:
// 16-byte vector loads and stores, bit-exact, bounds-checked against the pools.
#include <algorithm>
#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// Row of the pool that holds (slot, kv head h): HND [blocks][G][B] rows, NHD
// [blocks][B][G] rows (where slot * G + h is the row).
__device__ __forceinline__ long long pool_row(long long slot, int h, int G, int BS, int nhd) {
  if (nhd) return slot * G + h;
  const long long blk = slot / BS, row = slot - blk * BS;
  return (blk * G + h) * BS + row;
}

// One thread per VPT consecutive 16-byte vectors of a (token, K-or-V, kv head)
// row; its VPT loads (which do not depend on the slot) are all in flight before
// the stores.
template <int VPT>
__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value, uint4* k_cache,
                             uint4* v_cache, const int64_t* __restrict__ slot_mapping, int num_tokens, int G,
                             int vpr, int BS, int nhd, long long num_slots, unsigned* err) {
  pdl_begin();
  const int gpr = vpr / VPT;  // vector groups per row
  const long long total = (long long)num_tokens * 2 * G * gpr;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int v0 = (int)(idx % gpr) * VPT;
    long long rest = idx / gpr;
    const int h = (int)(rest % G);
    rest /= G;
    const int which = (int)(rest & 1);
    const long long t = rest >> 1;
    const long long slot = __ldg(slot_mapping + t);
    const uint4* src = (which ? value : key) + (t * G + h) * vpr + v0;
    uint4 r[VPT];
#pragma unroll
    for (int u = 0; u < VPT; ++u) r[u] = __ldg(src + u);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (v0 == 0 && h == 0 && which == 0) atomicOr(err, kErrSlot);
      continue;
    }
    uint4* dst = (which ? v_cache : k_cache) + pool_row(slot, h, G, BS, nhd) * vpr + v0;
#pragma unroll
    for (int u = 0; u < VPT; ++u) dst[u] = r[u];
  }
}

constexpr int kMaxLayersPerLaunch = 64;
struct LayerPtrs {
  uint4* k[kMaxLayersPerLaunch];
  uint4* v[kMaxLayersPerLaunch];
};

// grid = (pairs, layers, 2): one CTA copies one K or V block of one layer.
template <int VPT>
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(const LayerPtrs ptrs, const int64_t* __restrict__ pairs, long long num_blocks,
                       int vpb, unsigned* err) {
  pdl_begin();
  const long long src = __ldg(pairs + 2 * (long long)blockIdx.x);
  const long long dst = __ldg(pairs + 2 * (long long)blockIdx.x + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) atomicOr(err, kErrPair);
    return;
  }
  uint4* base = blockIdx.z ? ptrs.v[blockIdx.y] : ptrs.k[blockIdx.y];
  const uint4* s = base + src * vpb;
  uint4* d = base + dst * vpb;
  for (int i0 = threadIdx.x; i0 < vpb; i0 += 256 * VPT) {
    uint4 r[VPT];
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
      const int i = i0 + u * 256;
      if (i < vpb) r[u] = __ldcs(s + i);
    }
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
      const int i = i0 + u * 256;
      if (i < vpb) __stcs(d + i, r[u]);
    }
  }
}

constexpr int kMaxSwapLayers = 32;
struct SwapPtrs {
  const uint4* src_k[kMaxSwapLayers];
  const uint4* src_v[kMaxSwapLayers];
  uint4* dst_k[kMaxSwapLayers];
  uint4* dst_v[kMaxSwapLayers];
};

// grid = (pairs, layers, 2): one CTA moves one K or V block of one layer from
// the source pool to the destination pool (either may be pinned host memory,
// reached directly through the unified address space).
template <int VPT>
__global__ void __launch_bounds__(256)
    swap_blocks_kernel(const SwapPtrs ptrs, const int64_t* __restrict__ pairs, long long src_blocks,
                       long long dst_blocks, int vpb, unsigned* err) {
  pdl_begin();
  const long long src = __ldg(pairs + 2 * (long long)blockIdx.x);
  const long long dst = __ldg(pairs + 2 * (long long)blockIdx.x + 1);
  if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) atomicOr(err, kErrPair);
    return;
  }
  const uint4* s = (blockIdx.z ? ptrs.src_v[blockIdx.y] : ptrs.src_k[blockIdx.y]) + src * vpb;
  uint4* d = (blockIdx.z ? ptrs.dst_v[blockIdx.y] : ptrs.dst_k[blockIdx.y]) + dst * vpb;
  for (int i0 = threadIdx.x; i0 < vpb; i0 += 256 * VPT) {
    uint4 r[VPT];
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
      const int i = i0 + u * 256;
      if (i < vpb) r[u] = __ldcs(s + i);
    }
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
      const int i = i0 + u * 256;
      if (i < vpb) __stcs(d + i, r[u]);
    }
  }
}

int esize(pa_dtype dt) { return dt == PA_F32 ? 4 : (dt == PA_FP8_E4M3 ? 1 : 2); }
bool valid_dtype(pa_dtype dt) { return dt == PA_F32 || dt == PA_F16 || dt == PA_BF16 || dt == PA_FP8_E4M3; }

// FP8 cache write: one thread quantises and stores 16 consecutive elements of a
// (token, K-or-V, kv head) row: code = E4M3(x / scale), fp32 division, round to
// nearest even, saturating.
template <typename IT>
__global__ void __launch_bounds__(256)
    reshape_and_cache_fp8_kernel(const IT* __restrict__ key, const IT* __restrict__ value, uint8_t* k_cache,
                                 uint8_t* v_cache, const int64_t* __restrict__ slot_mapping, int num_tokens, int G,
                                 int D, int BS, int nhd, long long num_slots, float k_scale, float v_scale,
                                 unsigned* err) {
  pdl_begin();
  const int cpr = D / 16;  // 16-element chunks per row
  const long long total = (long long)num_tokens * 2 * G * cpr;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(idx % cpr);
    long long rest = idx / cpr;
    const int h = (int)(rest % G);
    rest /= G;
    const int which = (int)(rest & 1);
    const long long t = rest >> 1;
    const long long slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (c == 0 && h == 0 && which == 0) atomicOr(err, kErrSlot);
      continue;
    }
    const IT* src = (which ? value : key) + (t * G + h) * D + c * 16;
    const float sc = which ? v_scale : k_scale;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a0 = __fdiv_rn(to_f32(src[4 * i + 0]), sc), a1 = __fdiv_rn(to_f32(src[4 * i + 1]), sc);
      const float a2 = __fdiv_rn(to_f32(src[4 * i + 2]), sc), a3 = __fdiv_rn(to_f32(src[4 * i + 3]), sc);
      w[i] = f32x2_to_e4m3x2(a0, a1) | (f32x2_to_e4m3x2(a2, a3) << 16);
    }
    uint8_t* dst = (which ? v_cache : k_cache) + pool_row(slot, h, G, BS, nhd) * D + c * 16;
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace pa

extern "C" pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                                          const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                          int head_dim, int block_size, pa_kv_layout layout, int64_t num_blocks,
                                          pa_dtype dtype, cudaStream_t stream) {
  using namespace pa;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0 ||
      !valid_dtype(dtype) || (layout != PA_LAYOUT_HND && layout != PA_LAYOUT_NHD))
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PA_ERR_INVALID_ARG;
  const int row_bytes = head_dim * esize(dtype);
  if (row_bytes % 16) return PA_ERR_UNSUPPORTED;
  unsigned* err = nullptr;
  int sms = 0;
  pa_status st = device_state(&err, &sms);
  if (st != PA_OK) return st;
  const int vpr = row_bytes / 16;
  const int vpt = vpr % 4 == 0 ? 4 : (vpr % 2 == 0 ? 2 : 1);
  const long long total = (long long)num_tokens * 2 * num_kv_heads * (vpr / vpt);
  const long long want = (total + 255) / 256;
  const unsigned grid = (unsigned)std::min<long long>(want, (long long)sms * 16);
  auto kern = vpt == 4 ? reshape_and_cache_kernel<4> : (vpt == 2 ? reshape_and_cache_kernel<2> : reshape_and_cache_kernel<1>);
  const cudaError_t e =
      launch_pdl(kern, dim3(grid), dim3(256), 0, stream, static_cast<const uint4*>(key),
                 static_cast<const uint4*>(value), static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                 slot_mapping, num_tokens, num_kv_heads, vpr, block_size, layout == PA_LAYOUT_NHD ? 1 : 0,
                 (long long)num_blocks * block_size, err);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status pa_copy_blocks(void* const* k_caches, void* const* v_caches, int num_layers,
                                    const int64_t* block_pairs, int num_pairs, int num_kv_heads, int head_dim,
                                    int block_size, int64_t num_blocks, pa_dtype dtype, cudaStream_t stream) {
  using namespace pa;
  if (num_layers < 0 || num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_blocks <= 0 || !valid_dtype(dtype))
    return PA_ERR_INVALID_ARG;
  if (num_layers == 0 || num_pairs == 0) return PA_OK;
  if (!k_caches || !v_caches || !block_pairs || (reinterpret_cast<uintptr_t>(block_pairs) & 7u))
    return PA_ERR_INVALID_ARG;
  for (int l = 0; l < num_layers; ++l)
    if (!k_caches[l] || !v_caches[l] || !aligned16(k_caches[l]) || !aligned16(v_caches[l]))
      return PA_ERR_INVALID_ARG;
  const long long block_bytes = (long long)num_kv_heads * block_size * head_dim * esize(dtype);
  if (block_bytes % 16 || block_bytes / 16 > (1LL << 30) || num_pairs > 0x7fffffff / 2) return PA_ERR_UNSUPPORTED;
  unsigned* err = nullptr;
  int sms = 0;
  pa_status st = device_state(&err, &sms);
  if (st != PA_OK) return st;
  const int vpb = (int)(block_bytes / 16);
  for (int l0 = 0; l0 < num_layers; l0 += kMaxLayersPerLaunch) {
    const int nl = std::min(kMaxLayersPerLaunch, num_layers - l0);
    LayerPtrs ptrs;
    for (int i = 0; i < kMaxLayersPerLaunch; ++i) {
      ptrs.k[i] = i < nl ? static_cast<uint4*>(k_caches[l0 + i]) : nullptr;
      ptrs.v[i] = i < nl ? static_cast<uint4*>(v_caches[l0 + i]) : nullptr;
    }
    dim3 grid((unsigned)num_pairs, (unsigned)nl, 2);
    if (launch_pdl(copy_blocks_kernel<8>, grid, dim3(256), 0, stream, ptrs, block_pairs, (long long)num_blocks, vpb,
                   err) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  return PA_OK;
}

extern "C" pa_status pa_swap_blocks(void* const* dst_k_caches, void* const* dst_v_caches,
                                    const void* const* src_k_caches, const void* const* src_v_caches,
                                    int num_layers, const int64_t* block_pairs, int num_pairs, int num_kv_heads,
                                    int head_dim, int block_size, int64_t dst_num_blocks, int64_t src_num_blocks,
                                    pa_dtype dtype, cudaStream_t stream) {
  using namespace pa;
  if (num_layers < 0 || num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      dst_num_blocks <= 0 || src_num_blocks <= 0 || !valid_dtype(dtype))
    return PA_ERR_INVALID_ARG;
  if (num_layers == 0 || num_pairs == 0) return PA_OK;
  if (!dst_k_caches || !dst_v_caches || !src_k_caches || !src_v_caches || !block_pairs ||
      (reinterpret_cast<uintptr_t>(block_pairs) & 7u))
    return PA_ERR_INVALID_ARG;
  for (int l = 0; l < num_layers; ++l)
    if (!dst_k_caches[l] || !dst_v_caches[l] || !src_k_caches[l] || !src_v_caches[l] ||
        !aligned16(dst_k_caches[l]) || !aligned16(dst_v_caches[l]) || !aligned16(src_k_caches[l]) ||
        !aligned16(src_v_caches[l]))
      return PA_ERR_INVALID_ARG;
  const long long block_bytes = (long long)num_kv_heads * block_size * head_dim * esize(dtype);
  if (block_bytes % 16 || block_bytes / 16 > (1LL << 30) || num_pairs > 0x7fffffff / 2) return PA_ERR_UNSUPPORTED;
  unsigned* err = nullptr;
  int sms = 0;
  pa_status st = device_state(&err, &sms);
  if (st != PA_OK) return st;
  const int vpb = (int)(block_bytes / 16);
  for (int l0 = 0; l0 < num_layers; l0 += kMaxSwapLayers) {
    const int nl = std::min(kMaxSwapLayers, num_layers - l0);
    SwapPtrs ptrs;
    for (int i = 0; i < kMaxSwapLayers; ++i) {
      ptrs.src_k[i] = i < nl ? static_cast<const uint4*>(src_k_caches[l0 + i]) : nullptr;
      ptrs.src_v[i] = i < nl ? static_cast<const uint4*>(src_v_caches[l0 + i]) : nullptr;
      ptrs.dst_k[i] = i < nl ? static_cast<uint4*>(dst_k_caches[l0 + i]) : nullptr;
      ptrs.dst_v[i] = i < nl ? static_cast<uint4*>(dst_v_caches[l0 + i]) : nullptr;
    }
    dim3 grid((unsigned)num_pairs, (unsigned)nl, 2);
    if (launch_pdl(swap_blocks_kernel<8>, grid, dim3(256), 0, stream, ptrs, block_pairs, (long long)src_num_blocks,
                   (long long)dst_num_blocks, vpb, err) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  return PA_OK;
}

extern "C" pa_status pa_reshape_and_cache_fp8(const void* key, const void* value, void* k_cache, void* v_cache,
                                              const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                              int head_dim, int block_size, pa_kv_layout layout,
                                              int64_t num_blocks, pa_dtype in_dtype, float k_scale, float v_scale,
                                              cudaStream_t stream) {
  using namespace pa;
  if (layout != PA_LAYOUT_HND && layout != PA_LAYOUT_NHD) return PA_ERR_INVALID_ARG;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0 ||
      !(in_dtype == PA_F32 || in_dtype == PA_F16 || in_dtype == PA_BF16) || !(k_scale > 0.f) ||
      !(v_scale > 0.f) || k_scale == INFINITY || v_scale == INFINITY)
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PA_ERR_INVALID_ARG;
  if (head_dim % 16) return PA_ERR_UNSUPPORTED;
  unsigned* err = nullptr;
  int sms = 0;
  pa_status st = device_state(&err, &sms);
  if (st != PA_OK) return st;
  const long long total = (long long)num_tokens * 2 * num_kv_heads * (head_dim / 16);
  const unsigned grid = (unsigned)std::min<long long>((total + 255) / 256, (long long)sms * 16);
  uint8_t* kc = static_cast<uint8_t*>(k_cache);
  uint8_t* vc = static_cast<uint8_t*>(v_cache);
  const long long nslots = (long long)num_blocks * block_size;
  const int nhd = layout == PA_LAYOUT_NHD ? 1 : 0;
  cudaError_t e;
  switch (in_dtype) {
    case PA_F32:
      e = launch_pdl(reshape_and_cache_fp8_kernel<float>, dim3(grid), dim3(256), 0, stream,
                     static_cast<const float*>(key), static_cast<const float*>(value), kc, vc, slot_mapping,
                     num_tokens, num_kv_heads, head_dim, block_size, nhd, nslots, k_scale, v_scale, err);
      break;
    case PA_F16:
      e = launch_pdl(reshape_and_cache_fp8_kernel<__half>, dim3(grid), dim3(256), 0, stream,
                     static_cast<const __half*>(key), static_cast<const __half*>(value), kc, vc, slot_mapping,
                     num_tokens, num_kv_heads, head_dim, block_size, nhd, nslots, k_scale, v_scale, err);
      break;
    default:
      e = launch_pdl(reshape_and_cache_fp8_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, stream,
                     static_cast<const __nv_bfloat16*>(key), static_cast<const __nv_bfloat16*>(value), kc, vc,
                     slot_mapping, num_tokens, num_kv_heads, head_dim, block_size, nhd, nslots, k_scale, v_scale,
                     err);
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
