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

constexpr int kMaxLayersPerLaunch = 32;
// Per-layer pools of one launch: the source and destination of layer l's K and
// V blocks (the same pools for copy-on-write, two pools for a swap).
struct MovePtrs {
  const uint4* src_k[kMaxLayersPerLaunch];
  const uint4* src_v[kMaxLayersPerLaunch];
  uint4* dst_k[kMaxLayersPerLaunch];
  uint4* dst_v[kMaxLayersPerLaunch];
};

// Whether pair `me` (src, dst) races with another pair of the list: two copies
// writing one block, or one copy writing a block that another reads. With
// same_pool (copy-on-write inside one pool, or a swap whose two pools are the
// same memory) source and destination ids name the same blocks, so a
// destination may also not be any pair's source (its own included). Pairs with
// ids outside their pools are skipped by every CTA and race with nothing. All
// threads of the CTA take part; every thread gets the same answer.
__device__ __forceinline__ bool pair_races(const int64_t* __restrict__ pairs, int num_pairs, int me, long long src,
                                           long long dst, long long src_blocks, long long dst_blocks,
                                           bool same_pool) {
  bool bad = same_pool && src == dst;
  for (int q = threadIdx.x; q < num_pairs; q += blockDim.x) {
    if (q == me) continue;
    const long long sq = __ldg(pairs + 2 * (long long)q), dq = __ldg(pairs + 2 * (long long)q + 1);
    if (sq < 0 || sq >= src_blocks || dq < 0 || dq >= dst_blocks) continue;
    bad |= dq == dst;
    if (same_pool) bad |= (sq == dst) | (dq == src);
  }
  return __syncthreads_or(bad) != 0;
}

// grid = (pairs, layer chunks, 2): one CTA moves the K (z = 0) or V (z = 1) block
// of one pair for layers [y * layers_per_cta, ...) of the launch, from the source
// pool to the destination pool (either may be pinned host memory, reached
// directly through the unified address space). Every CTA first checks its pair
// against the whole list, so a racing pair is skipped in all of its CTAs. The
// first chunk's loads go out before that check (reading a racing pair's source
// is harmless; only its stores are skipped), so the check's latency hides behind
// them.
template <int VPT>
__global__ void __launch_bounds__(256)
    move_blocks_kernel(const MovePtrs ptrs, const int64_t* __restrict__ pairs, int num_pairs, long long src_blocks,
                       long long dst_blocks, int vpb, int num_layers, int layers_per_cta, int same_pool,
                       unsigned* err) {
  pdl_begin();
  const int me = blockIdx.x;
  const long long src = __ldg(pairs + 2 * (long long)me);
  const long long dst = __ldg(pairs + 2 * (long long)me + 1);
  const bool first = threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
  if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
    if (first) atomicOr(err, kErrPair);
    return;
  }
  const int l0 = blockIdx.y * layers_per_cta, l1 = min(num_layers, l0 + layers_per_cta);
  uint4 r[VPT];
  auto load = [&](int l, int i0) {
    const uint4* s = (blockIdx.z ? ptrs.src_v[l] : ptrs.src_k[l]) + src * vpb;
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
      const int i = i0 + u * 256;
      if (i < vpb) r[u] = __ldcs(s + i);
    }
  };
  auto store = [&](int l, int i0) {
    uint4* d = (blockIdx.z ? ptrs.dst_v[l] : ptrs.dst_k[l]) + dst * vpb;
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
      const int i = i0 + u * 256;
      if (i < vpb) __stcs(d + i, r[u]);
    }
  };
  load(l0, threadIdx.x);
  if (pair_races(pairs, num_pairs, me, src, dst, src_blocks, dst_blocks, same_pool != 0)) {
    if (first) atomicOr(err, kErrPairAlias);
    return;
  }
  for (int l = l0; l < l1; ++l) {
    for (int i0 = threadIdx.x; i0 < vpb; i0 += 256 * VPT) {
      if (l != l0 || i0 != (int)threadIdx.x) load(l, i0);
      store(l, i0);
    }
  }
}

// Launch the moves of `num_layers` layers in chunks of kMaxLayersPerLaunch. Each
// CTA takes several layers of its pair when there are many CTAs, so that the
// per-CTA pair check is paid once for many blocks (about two waves of eight
// CTAs per SM).
template <typename SK, typename SV, typename DK, typename DV>
pa_status launch_moves(SK src_k, SV src_v, DK dst_k, DV dst_v, int num_layers, const int64_t* pairs,
                       int num_pairs, long long src_blocks, long long dst_blocks, int vpb, bool same_pool, int sms,
                       unsigned* err, cudaStream_t stream) {
  for (int b = 0; b < num_layers; b += kMaxLayersPerLaunch) {
    const int nl = std::min(kMaxLayersPerLaunch, num_layers - b);
    MovePtrs ptrs;
    for (int i = 0; i < kMaxLayersPerLaunch; ++i) {
      ptrs.src_k[i] = i < nl ? static_cast<const uint4*>(src_k[b + i]) : nullptr;
      ptrs.src_v[i] = i < nl ? static_cast<const uint4*>(src_v[b + i]) : nullptr;
      ptrs.dst_k[i] = i < nl ? static_cast<uint4*>(dst_k[b + i]) : nullptr;
      ptrs.dst_v[i] = i < nl ? static_cast<uint4*>(dst_v[b + i]) : nullptr;
    }
    const long long all = (long long)num_pairs * nl * 2, target = (long long)sms * 16;
    const int lpc = (int)std::max(1LL, std::min<long long>(nl, all / std::max(1LL, target)));
    dim3 grid((unsigned)num_pairs, (unsigned)((nl + lpc - 1) / lpc), 2);
    if (launch_pdl(move_blocks_kernel<8>, grid, dim3(256), 0, stream, ptrs, pairs, num_pairs, src_blocks,
                   dst_blocks, vpb, nl, lpc, same_pool ? 1 : 0, err) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  return PA_OK;
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
  return launch_moves(k_caches, v_caches, k_caches, v_caches, num_layers, block_pairs, num_pairs,
                      (long long)num_blocks, (long long)num_blocks, vpb, true, sms, err, stream);
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
  // ids name blocks of one id space only where a source and a destination pool are the same memory
  bool same_pool = false;
  for (int l = 0; l < num_layers; ++l)
    same_pool |= dst_k_caches[l] == src_k_caches[l] || dst_v_caches[l] == src_v_caches[l];
  return launch_moves(src_k_caches, src_v_caches, dst_k_caches, dst_v_caches, num_layers, block_pairs, num_pairs,
                      (long long)src_num_blocks, (long long)dst_num_blocks, vpb, same_pool, sms, err, stream);
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
