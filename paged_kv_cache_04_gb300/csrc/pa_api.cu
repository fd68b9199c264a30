// C ABI entry points for decode attention, argument checks, TMA descriptor set-up
// and the device error word.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "pa_cascade.cuh"
#include "pa_cascade_tc.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// The device error word: kernels OR PA_DEVERR_* bits into it; pa_get_error
// reads and clears it. One copy per device that loads the library.
__device__ unsigned g_error_word;

constexpr int kMaxDevices = 64;
struct DeviceState {
  bool ready = false;
  unsigned* err = nullptr;
  int sms = 0;
};
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int esize(pa_dtype dt) { return dt == PA_F32 ? 4 : (dt == PA_FP8_E4M3 ? 1 : 2); }
bool valid_dtype(pa_dtype dt) { return dt == PA_F32 || dt == PA_F16 || dt == PA_BF16; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

pa_status encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return PA_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = g_encode;
  return PA_OK;
}

// The TMA view of a KV pool. A box is 16 tokens of one (block, kv head) tile
// (one job), staged in 128-byte column regions ([regions][16 rows][128 B]),
// with 128-byte swizzling.
//   HND [num_blocks][G][B][D]: rows = num_blocks * G * B of D elements;
//   NHD [num_blocks][B][G][D]: (D, G, num_blocks * B), so a box takes one kv
//   head of 16 consecutive tokens (rows G * D elements apart).
//   regions: with a row wider than 128 bytes, a last dimension of extent
//   D * e / 128 and stride 128 bytes lets one box take every region of the
//   job (plain decode); without it a box is one region, placed by its column
//   coordinate (split decode, the shared-prefix passes).
//   swizzle: 128-byte swizzled stages (read by ldmatrix / by columns), or plain
//   row-major stages (V of the vector paths, whose lanes read one row at a time).
pa_status make_pool_map(CUtensorMap* map, const void* base, pa_dtype dt, int D, int G, int BS, long long num_blocks,
                        pa_kv_layout layout, bool swizzle, bool regions) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  pa_status st = encoder(&enc);
  if (st != PA_OK) return st;
  const int e = esize(dt);
  const CUtensorMapDataType t = dt == PA_F32          ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                : dt == PA_F16        ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                : dt == PA_FP8_E4M3   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const bool nhd = layout == PA_LAYOUT_NHD;
  const int nreg = regions ? D * e / 128 : 1;
  const bool rdim = nreg > 1;  // a region dimension after the row dimension(s)
  cuuint64_t dims[4] = {(cuuint64_t)(rdim ? 128 / e : D), (cuuint64_t)(num_blocks * G * BS), 1, 1};
  cuuint64_t strides[3] = {(cuuint64_t)D * e, 0, 0};
  cuuint32_t box[4] = {(cuuint32_t)(128 / e), (cuuint32_t)kJobTokens, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  int rank = 2;
  if (nhd) {
    dims[1] = (cuuint64_t)G;
    dims[2] = (cuuint64_t)(num_blocks * BS);
    strides[1] = (cuuint64_t)G * D * e;
    box[1] = 1;
    box[2] = (cuuint32_t)kJobTokens;
    rank = 3;
  }
  if (rdim) {
    dims[rank] = (cuuint64_t)nreg;
    strides[rank - 1] = 128;
    box[rank] = (cuuint32_t)nreg;
    ++rank;
  }
  // NHD rows of one kv head are G * D elements apart: promote only the 128 bytes a box reads, so a
  // 128-byte row does not drag its neighbour head's row into L2.
  CUresult r = enc(map, t, rank, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   nhd ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// The TMA view of q [S][H][D] (16-bit) for the tcgen05 prefix pass: one box is
// 64 columns of `group` consecutive heads (one kv head's queries) of
// `members` consecutive sequences, rows in (sequence, head) order, 128-byte
// swizzle; rows past the batch read as zeros.
pa_status make_q_map(CUtensorMap* map, const void* q, pa_dtype dt, int D, int H, int S, int group, int members) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  pa_status st = encoder(&enc);
  if (st != PA_OK) return st;
  if (members < 1 || members > 256 || group < 1 || group > 256) return PA_ERR_UNSUPPORTED;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)members};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dt == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

struct DecodeArgs {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  int max_blocks;
  const int32_t* context_lens;
  int S, H, G, D, BS;
  long long num_blocks;
  float scale;
  pa_dtype dt, odt;
  pa_dtype qdt = PA_F32;        // FP8 caches: the query type
  float k_scale = 1.f, v_scale = 1.f;
  pa_kv_layout layout = PA_LAYOUT_HND;
};

pa_status check_decode(const DecodeArgs& a) {
  if (a.S < 0 || a.H <= 0 || a.G <= 0 || a.D <= 0 || a.BS <= 0 || a.num_blocks <= 0 || a.max_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (a.H % a.G || !valid_dtype(a.dt) || !valid_dtype(a.odt) || !std::isfinite(a.scale)) return PA_ERR_INVALID_ARG;
  if (a.layout != PA_LAYOUT_HND && a.layout != PA_LAYOUT_NHD) return PA_ERR_INVALID_ARG;
  if (a.S == 0) return PA_OK;
  if (!a.out || !a.q || !a.k_cache || !a.v_cache || !a.block_tables || !a.context_lens) return PA_ERR_INVALID_ARG;
  if (!aligned16(a.out) || !aligned16(a.q) || !aligned16(a.k_cache) || !aligned16(a.v_cache) ||
      (reinterpret_cast<uintptr_t>(a.block_tables) & 3u) || (reinterpret_cast<uintptr_t>(a.context_lens) & 3u))
    return PA_ERR_INVALID_ARG;
  if ((a.D != 64 && a.D != 128 && a.D != 256) || (a.BS != 16 && a.BS != 32) || a.H / a.G > kMaxGroup)
    return PA_ERR_UNSUPPORTED;
  if (a.odt != a.dt && a.odt != PA_F32) return PA_ERR_UNSUPPORTED;
  // TMA row coordinates are 32-bit
  if ((long long)a.num_blocks * a.G * a.BS > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

template <typename DT, typename QT, typename OT, int D, int PATH>
pa_status dispatch_mode(const CUtensorMap& km, const CUtensorMap& vm, const DecodeParams& p, int sms,
                        long long items, int mode, cudaStream_t st) {
  if (mode == kModeSplit) return launch_decode<DT, QT, float, D, PATH, kModeSplit>(km, vm, p, sms, items, st);
  if (mode == kModeSuffix) {
    if constexpr (sizeof(DT) == 2 && D <= 128)  // the shared-prefix decode: 16-bit caches, head_dim <= 128
      return launch_decode<DT, QT, float, D, PATH, kModeSuffix>(km, vm, p, sms, items, st);
    return PA_ERR_UNSUPPORTED;
  }
  return launch_decode<DT, QT, OT, D, PATH, kModePlain>(km, vm, p, sms, items, st);
}

// Whether a decode launch takes the tensor-core path (mma.sync; V staged with
// the 128-byte swizzle) rather than a vector path (lanes split head_dim). A
// group of >= 2 query heads per kv head on 16-bit or E4M3 data: tensor cores
// (groups of 2-3 leave most of the MMA's 8 head columns empty, yet issue far
// fewer instructions per job than the vector path: measured 0.98 against 0.76
// of peak at group 2 and 0.97 against 0.57 at group 3 on 16-bit caches, 0.84
// against 0.53 / 0.32 over E4M3, 1.13x at head_dim 256). MHA (group 1) takes
// them over E4M3 caches (0.86 against 0.82) and in 16-bit split decode (0.97
// against 0.90 on 32K-128K contexts); 16-bit plain and suffix-pass MHA keep the
// vector path, which measured as fast or faster there (OPT-13B batch within 1%,
// head_dim 64 +2%) at three CTAs per SM. fp32 data: vector paths.
bool tensor_core_path(int esize_bytes, int group, int D, int mode) {
  if (esize_bytes > 2) return false;
  if (group >= 2 || esize_bytes == 1) return true;
  return mode == kModeSplit && D <= 128;
}

template <typename DT, typename QT, typename OT, int D>
pa_status dispatch_path(const CUtensorMap& km, const CUtensorMap& vm, const DecodeParams& p, int sms,
                        long long items, int mode, cudaStream_t st) {
  // Tensor cores (see tensor_core_path) or the vector paths. Plain decode at
  // groups of 5-8 merges in rounds (kPathMmaG8); split and suffix mode do not
  // merge inside the CTA and take kPathMma at every group.
  if constexpr (sizeof(DT) <= 2) {
    if (p.group > kMergeHeads && mode == kModePlain)
      return launch_decode<DT, QT, OT, D, kPathMmaG8, kModePlain>(km, vm, p, sms, items, st);
    if (tensor_core_path(sizeof(DT), p.group, D, mode))
      return dispatch_mode<DT, QT, OT, D, kPathMma>(km, vm, p, sms, items, mode, st);
    if constexpr (sizeof(DT) == 1) {
      return PA_ERR_UNSUPPORTED;  // (E4M3 always takes the tensor cores)
    } else if constexpr (D <= 128) {
      return dispatch_mode<DT, QT, OT, D, kPathVecMha>(km, vm, p, sms, items, mode, st);
    } else {
      // head_dim 256: q stays in shared memory; a lane's half of a 256-wide row in registers would spill
      return dispatch_mode<DT, QT, OT, D, kPathVec>(km, vm, p, sms, items, mode, st);
    }
  } else {  // fp32 data: the vector paths at every group
    if constexpr (D <= 128) {
      if (p.group == 1) return dispatch_mode<DT, QT, OT, D, kPathVecMha>(km, vm, p, sms, items, mode, st);
    }
    return dispatch_mode<DT, QT, OT, D, kPathVec>(km, vm, p, sms, items, mode, st);
  }
}

template <typename DT, typename OT>
pa_status dispatch_shape(const CUtensorMap& km, const CUtensorMap& vm, const DecodeParams& p, int D, int sms,
                         long long items, int mode, cudaStream_t st) {
  if (D == 64) return dispatch_path<DT, DT, OT, 64>(km, vm, p, sms, items, mode, st);
  if (D == 128) return dispatch_path<DT, DT, OT, 128>(km, vm, p, sms, items, mode, st);
  if (D == 256) return dispatch_path<DT, DT, OT, 256>(km, vm, p, sms, items, mode, st);
  return PA_ERR_UNSUPPORTED;
}

template <typename OT>
pa_status dispatch_reduce(const DecodeParams& p, int D, cudaStream_t st) {
  if (D == 64) return launch_lse_reduce<OT, 64>(p, st);
  return D == 128 ? launch_lse_reduce<OT, 128>(p, st) : launch_lse_reduce<OT, 256>(p, st);
}

// Shared-prefix groups for pa_decode_cascade (all null / zero otherwise).
struct CascadeArgs {
  const int32_t* group_starts = nullptr;
  const int32_t* prefix_lens = nullptr;
  int num_groups = 0;
  int prefix_slots = 0;  // workspace slots reserved for prefix partitions
  int rows = 0;          // query rows per group (members x query heads), at most 128
};

pa_status run_decode(const DecodeArgs& a, bool split, int partition, int max_partitions, void* ws,
                     cudaStream_t st, const CascadeArgs& c = CascadeArgs()) {
  unsigned* err = nullptr;
  int sms = 0;
  pa_status s = device_state(&err, &sms);
  if (s != PA_OK) return s;
  // tensor-core path or vector path: see tensor_core_path (the mode is set below)
  const int launch_mode = !split ? kModePlain : (c.group_starts ? kModeSuffix : kModeSplit);
  const bool mma_path = tensor_core_path(esize(a.dt), a.H / a.G, a.D, launch_mode);
  CUtensorMap km, vm;
  const bool whole = launch_mode == kModePlain;  // one box per job tile (see tma_load_job)
  if ((s = make_pool_map(&km, a.k_cache, a.dt, a.D, a.G, a.BS, a.num_blocks, a.layout, true, whole)) != PA_OK)
    return s;
  if ((s = make_pool_map(&vm, a.v_cache, a.dt, a.D, a.G, a.BS, a.num_blocks, a.layout, mma_path, whole)) != PA_OK)
    return s;

  DecodeParams p{};
  p.out = a.out;
  p.q = a.q;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.max_blocks = a.max_blocks;
  p.block_size = a.BS;
  p.block_shift = a.BS == 32 ? 5 : 4;
  p.S = a.S;
  p.H = a.H;
  p.G = a.G;
  p.group = a.H / a.G;
  p.num_blocks = a.num_blocks;
  p.scale_log2 = a.scale * a.k_scale * 1.4426950408889634f;
  p.v_scale = a.v_scale;
  p.nhd = a.layout == PA_LAYOUT_NHD;
  p.k_cache = a.k_cache;
  p.v_cache = a.v_cache;
  p.err = err;
  long long items = (long long)a.S * a.G;
  if (split) {
    p.partition = partition;
    p.max_partitions = max_partitions;
    const size_t o_bytes = (size_t)a.S * a.H * max_partitions * a.D * 4;
    const size_t m_bytes = (size_t)a.S * a.H * max_partitions * 4;
    p.ws_o = static_cast<float*>(ws);
    p.ws_m = reinterpret_cast<float*>(static_cast<char*>(ws) + align256(o_bytes));
    p.ws_l = reinterpret_cast<float*>(static_cast<char*>(ws) + align256(o_bytes) + align256(m_bytes));
    if (c.group_starts && c.prefix_slots > 0 && c.rows > 16 && a.S <= kSuffixStartMaxSeqs) {
      // the tcgen05 prefix pass computes the suffix pass's schedule (suffix_schedule)
      char* sched = static_cast<char*>(ws) + align256(o_bytes) + 2 * align256(m_bytes);
      p.sfx_order = reinterpret_cast<uint16_t*>(sched);
      p.sfx_start = reinterpret_cast<int*>(sched + align256((size_t)a.S * 2));
    }
    if (!c.group_starts) items *= max_partitions;  // the suffix pass has one item per (sequence, kv head)
  }
  const int mode = launch_mode;
  if (c.group_starts) {
    p.group_starts = c.group_starts;
    p.prefix_lens = c.prefix_lens;
    p.num_groups = c.num_groups;
    p.suffix_slot = c.prefix_slots;
    p.suffix_single = 1;
    const long long lim_ws = (long long)c.prefix_slots * partition, lim_bt = (long long)a.max_blocks * a.BS;
    p.prefix_limit = (int)(lim_ws < lim_bt ? lim_ws : lim_bt);
    if (c.prefix_slots > 0) {  // prefix pass: every group's query rows over its shared blocks
      const long long pitems = (long long)c.num_groups * a.G * c.prefix_slots;
      CUtensorMap vsw = vm;  // the prefix passes read V from swizzled stages
      if (!mma_path &&
          (s = make_pool_map(&vsw, a.v_cache, a.dt, a.D, a.G, a.BS, a.num_blocks, a.layout, true, false)) != PA_OK)
        return s;
      // Groups of 17-64 query rows take the M = 64 tile of the tcgen05 pass and
      // groups of 65-128 its M = 128 tile; up to 16 rows, the mma.sync pass (four
      // warps of 8 rows). The tcgen05 pass is bound by its per-tile chain, not by
      // its rows, so at 32 rows (8 samples of a GQA-4 model) a half-empty M = 64
      // tile still beats the mma.sync pass (3-3.5% per step on 64 prompts x 8
      // samples, measured).
      const bool bf = a.dt == PA_BF16;
      CUtensorMap qm;
      if (c.rows > 16 &&
          (s = make_q_map(&qm, a.q, a.dt, a.D, a.H, a.S, p.group, (c.rows > 64 ? 128 : 64) / p.group)) != PA_OK)
        return s;
      if (c.rows > 64) {
        if (a.D == 128)
          s = bf ? launch_cascade_prefix_tc<__nv_bfloat16, 128, 128>(km, vsw, qm, p, sms, pitems, st)
                 : launch_cascade_prefix_tc<__half, 128, 128>(km, vsw, qm, p, sms, pitems, st);
        else
          s = bf ? launch_cascade_prefix_tc<__nv_bfloat16, 64, 128>(km, vsw, qm, p, sms, pitems, st)
                 : launch_cascade_prefix_tc<__half, 64, 128>(km, vsw, qm, p, sms, pitems, st);
      } else if (c.rows > 16) {
        if (a.D == 128)
          s = bf ? launch_cascade_prefix_tc<__nv_bfloat16, 128, 64>(km, vsw, qm, p, sms, pitems, st)
                 : launch_cascade_prefix_tc<__half, 128, 64>(km, vsw, qm, p, sms, pitems, st);
        else
          s = bf ? launch_cascade_prefix_tc<__nv_bfloat16, 64, 64>(km, vsw, qm, p, sms, pitems, st)
                 : launch_cascade_prefix_tc<__half, 64, 64>(km, vsw, qm, p, sms, pitems, st);
      } else if (a.D == 128) {
        s = bf ? launch_cascade_prefix<__nv_bfloat16, 128, 1>(km, vsw, p, sms, pitems, st)
               : launch_cascade_prefix<__half, 128, 1>(km, vsw, p, sms, pitems, st);
      } else {
        s = bf ? launch_cascade_prefix<__nv_bfloat16, 64, 1>(km, vsw, p, sms, pitems, st)
               : launch_cascade_prefix<__half, 64, 1>(km, vsw, p, sms, pitems, st);
      }
      if (s != PA_OK) return s;
    }
  }
  switch (a.dt) {
    case PA_FP8_E4M3:
      if (a.D != 128) return PA_ERR_UNSUPPORTED;
      if (a.qdt == PA_BF16)
        s = a.odt == PA_F32
                ? dispatch_path<fp8e4m3, __nv_bfloat16, float, 128>(km, vm, p, sms, items, mode, st)
                : dispatch_path<fp8e4m3, __nv_bfloat16, __nv_bfloat16, 128>(km, vm, p, sms, items, mode, st);
      else
        s = a.odt == PA_F32 ? dispatch_path<fp8e4m3, __half, float, 128>(km, vm, p, sms, items, mode, st)
                            : dispatch_path<fp8e4m3, __half, __half, 128>(km, vm, p, sms, items, mode, st);
      break;
    case PA_BF16:
      s = a.odt == PA_F32 ? dispatch_shape<__nv_bfloat16, float>(km, vm, p, a.D, sms, items, mode, st)
                          : dispatch_shape<__nv_bfloat16, __nv_bfloat16>(km, vm, p, a.D, sms, items, mode, st);
      break;
    case PA_F16:
      s = a.odt == PA_F32 ? dispatch_shape<__half, float>(km, vm, p, a.D, sms, items, mode, st)
                          : dispatch_shape<__half, __half>(km, vm, p, a.D, sms, items, mode, st);
      break;
    default:
      s = dispatch_shape<float, float>(km, vm, p, a.D, sms, items, mode, st);
  }
  if (s != PA_OK || !split) return s;
  switch (a.odt) {
    case PA_BF16: return dispatch_reduce<__nv_bfloat16>(p, a.D, st);
    case PA_F16: return dispatch_reduce<__half>(p, a.D, st);
    default: return dispatch_reduce<float>(p, a.D, st);
  }
}

}  // namespace

pa_status device_state(unsigned** err, int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_error_word) != cudaSuccess) return PA_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return PA_ERR_CUDA;
    d.err = static_cast<unsigned*>(ptr);
    d.sms = sms;
    d.ready = true;
  }
  *err = d.err;
  *num_sms = d.sms;
  return PA_OK;
}

}  // namespace pa

extern "C" pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                               int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size, pa_kv_layout layout,
                               int64_t num_blocks, float scale, pa_dtype dtype, pa_dtype out_dtype,
                               cudaStream_t stream) {
  using namespace pa;
  DecodeArgs a{out,      q,         k_cache,      v_cache,  block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                     (long long)num_blocks, scale, dtype, out_dtype};
  a.layout = layout;
  pa_status s = check_decode(a);
  if (s != PA_OK || num_seqs == 0) return s;
  return run_decode(a, false, 0, 0, nullptr, stream);
}

extern "C" size_t pa_decode_split_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                                  int partition_tokens) {
  if (num_seqs < 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0 || partition_tokens <= 0) return 0;
  const long long P = std::max(1LL, ((long long)max_context_len + partition_tokens - 1) / partition_tokens);
  const size_t rows = (size_t)num_seqs * num_heads * P;
  return pa::align256(rows * head_dim * 4) + 2 * pa::align256(rows * 4);
}

namespace pa {
// Every check of pa_decode_split except those on the workspace itself; *need
// receives the workspace size (0 when num_seqs == 0).
pa_status check_split_call(const void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                           int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                           pa_kv_layout layout, int64_t num_blocks, float scale, pa_dtype dtype, pa_dtype out_dtype,
                           int max_context_len, int partition_tokens, size_t* need) {
  DecodeArgs a{const_cast<void*>(out), q,         k_cache,      v_cache,  block_tables, max_blocks_per_seq,
               context_lens,           num_seqs, num_heads, num_kv_heads, head_dim, block_size,
               (long long)num_blocks,  scale,     dtype,     out_dtype};
  a.layout = layout;
  *need = 0;
  pa_status s = check_decode(a);
  if (s != PA_OK) return s;
  if (max_context_len < 0 || partition_tokens <= 0 || partition_tokens % block_size) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (num_seqs > kSplitMaxSeqs) return PA_ERR_UNSUPPORTED;
  const long long P = std::max(1LL, ((long long)max_context_len + partition_tokens - 1) / partition_tokens);
  if ((long long)num_seqs * num_kv_heads * P > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  *need = pa_decode_split_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, partition_tokens);
  return *need == 0 ? PA_ERR_INVALID_ARG : PA_OK;
}
}  // namespace pa

extern "C" pa_status pa_decode_split(void* out, const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, int max_blocks_per_seq,
                                     const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                                     int head_dim, int block_size, pa_kv_layout layout, int64_t num_blocks, float scale,
                                     pa_dtype dtype, pa_dtype out_dtype, int max_context_len,
                                     int partition_tokens, void* workspace, size_t workspace_bytes,
                                     cudaStream_t stream) {
  using namespace pa;
  size_t need = 0;
  pa_status s = check_split_call(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                 num_heads, num_kv_heads, head_dim, block_size, layout, num_blocks, scale, dtype,
                                 out_dtype, max_context_len, partition_tokens, &need);
  if (s != PA_OK || num_seqs == 0) return s;
  if (!workspace || !aligned16(workspace) || workspace_bytes < need) return PA_ERR_INVALID_ARG;
  DecodeArgs a{out,      q,         k_cache,      v_cache,  block_tables, max_blocks_per_seq,
               context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
               (long long)num_blocks, scale, dtype, out_dtype};
  a.layout = layout;
  const long long P = std::max(1LL, ((long long)max_context_len + partition_tokens - 1) / partition_tokens);
  return run_decode(a, true, partition_tokens, (int)P, workspace, stream);
}

namespace {
// FP8 entry points: the cache is E4M3 codes, q is bf16 or fp16, out is q's type or fp32.
pa_status check_fp8(const pa::DecodeArgs& a) {
  if (a.qdt != PA_F16 && a.qdt != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (a.odt != a.qdt && a.odt != PA_F32) return PA_ERR_UNSUPPORTED;
  if (!std::isfinite(a.k_scale) || !std::isfinite(a.v_scale) || a.k_scale <= 0.f || a.v_scale <= 0.f)
    return PA_ERR_INVALID_ARG;
  if (a.D != 128) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}
}  // namespace

extern "C" pa_status pa_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                                   int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size, pa_kv_layout layout,
                                   int64_t num_blocks, float scale, float k_scale, float v_scale, pa_dtype q_dtype,
                                   pa_dtype out_dtype, cudaStream_t stream) {
  using namespace pa;
  DecodeArgs a{out,      q,         k_cache,      v_cache,  block_tables, max_blocks_per_seq,
               context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
               (long long)num_blocks, scale, q_dtype, out_dtype};
  a.layout = layout;
  pa_status s = check_decode(a);  // shapes, pointers, alignment (q / out type as the 16-bit type)
  if (s != PA_OK || num_seqs == 0) return s;
  a.dt = PA_FP8_E4M3;
  a.qdt = q_dtype;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  if ((s = check_fp8(a)) != PA_OK) return s;
  return run_decode(a, false, 0, 0, nullptr, stream);
}

extern "C" pa_status pa_decode_split_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, int max_blocks_per_seq,
                                         const int32_t* context_lens, int num_seqs, int num_heads,
                                         int num_kv_heads, int head_dim, int block_size, pa_kv_layout layout, int64_t num_blocks,
                                         float scale, float k_scale, float v_scale, pa_dtype q_dtype,
                                         pa_dtype out_dtype, int max_context_len, int partition_tokens,
                                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  using namespace pa;
  DecodeArgs a{out,      q,         k_cache,      v_cache,  block_tables, max_blocks_per_seq,
               context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
               (long long)num_blocks, scale, q_dtype, out_dtype};
  a.layout = layout;
  pa_status s = check_decode(a);
  if (s != PA_OK) return s;
  if (max_context_len < 0 || partition_tokens <= 0 || partition_tokens % block_size) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  a.dt = PA_FP8_E4M3;
  a.qdt = q_dtype;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  if ((s = check_fp8(a)) != PA_OK) return s;
  if (num_seqs > kSplitMaxSeqs) return PA_ERR_UNSUPPORTED;
  const size_t need =
      pa_decode_split_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, partition_tokens);
  if (!workspace || !aligned16(workspace) || workspace_bytes < need || need == 0) return PA_ERR_INVALID_ARG;
  const long long P = std::max(1LL, ((long long)max_context_len + partition_tokens - 1) / partition_tokens);
  if ((long long)num_seqs * num_kv_heads * P > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  return run_decode(a, true, partition_tokens, (int)P, workspace, stream);
}

extern "C" size_t pa_decode_cascade_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_prefix_len,
                                                    int max_context_len, int partition_tokens) {
  if (num_seqs < 0 || num_heads <= 0 || head_dim <= 0 || max_prefix_len < 0 || max_context_len < 0 ||
      partition_tokens <= 0)
    return 0;
  const long long P = ((long long)max_prefix_len + partition_tokens - 1) / partition_tokens + 1;
  const size_t rows = (size_t)num_seqs * num_heads * P;
  // then the suffix pass's schedule: the sequence order (2 bytes each) and their
  // first own tokens (4 bytes each)
  return pa::align256(rows * head_dim * 4) + 2 * pa::align256(rows * 4) + pa::align256((size_t)num_seqs * 2) +
         pa::align256((size_t)num_seqs * 4);
}

extern "C" pa_status pa_decode_cascade(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, int max_blocks_per_seq,
                                       const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                                       int head_dim, int block_size, pa_kv_layout layout, int64_t num_blocks, float scale,
                                       pa_dtype dtype, pa_dtype out_dtype, const int32_t* group_starts,
                                       const int32_t* prefix_lens, int num_groups, int max_group_size,
                                       int max_prefix_len, int max_context_len, int partition_tokens,
                                       void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  using namespace pa;
  DecodeArgs a{out,      q,         k_cache,      v_cache,  block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                     (long long)num_blocks, scale, dtype, out_dtype};
  a.layout = layout;
  pa_status s = check_decode(a);
  if (s != PA_OK) return s;
  if (max_context_len < 0 || max_prefix_len < 0 || partition_tokens <= 0 || partition_tokens % block_size ||
      num_groups <= 0 || max_group_size <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!group_starts || !prefix_lens || (reinterpret_cast<uintptr_t>(group_starts) & 3u) ||
      (reinterpret_cast<uintptr_t>(prefix_lens) & 3u))
    return PA_ERR_INVALID_ARG;
  if (dtype != PA_BF16 && dtype != PA_F16) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;  // the prefix pass: head_dim <= 128
  if (num_seqs > kSplitMaxSeqs || num_groups > kSplitMaxSeqs) return PA_ERR_UNSUPPORTED;
  const long long rows_per_group = (long long)max_group_size * (num_heads / num_kv_heads);
  if (rows_per_group > kTcMaxRows) return PA_ERR_UNSUPPORTED;
  const size_t need = pa_decode_cascade_workspace_bytes(num_seqs, num_heads, head_dim, max_prefix_len,
                                                        max_context_len, partition_tokens);
  if (!workspace || !aligned16(workspace) || workspace_bytes < need || need == 0) return PA_ERR_INVALID_ARG;
  CascadeArgs c;
  c.group_starts = group_starts;
  c.prefix_lens = prefix_lens;
  c.num_groups = num_groups;
  c.prefix_slots = (max_prefix_len + partition_tokens - 1) / partition_tokens;
  c.rows = (int)rows_per_group;
  const long long P = c.prefix_slots + 1;  // prefix partitions, then one slot for each sequence's own tokens
  if ((long long)num_seqs * num_kv_heads * P > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  return run_decode(a, true, partition_tokens, (int)P, workspace, stream, c);
}

extern "C" pa_status pa_get_error(uint32_t* error_bits, cudaStream_t stream) {
  if (!error_bits) return PA_ERR_INVALID_ARG;
  unsigned* err = nullptr;
  int sms = 0;
  pa_status s = pa::device_state(&err, &sms);
  if (s != PA_OK) return s;
  unsigned host = 0;
  if (cudaMemcpyAsync(&host, err, sizeof(unsigned), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaMemsetAsync(err, 0, sizeof(unsigned), stream) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PA_ERR_CUDA;
  *error_bits = host;
  return host ? PA_ERR_OUT_OF_RANGE : PA_OK;
}

extern "C" pa_status pa_debug_check(cudaStream_t stream) {
  uint32_t bits = 0;
  return pa_get_error(&bits, stream);
}

extern "C" const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_OUT_OF_RANGE: return "device-side value out of range";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_NO_BLOCKS: return "no free block";
  }
  return "unknown status";
}

extern "C" const char* pa_status_str(pa_status status) { return pa_status_string(status); }

extern "C" int pa_version(void) { return 200; }
