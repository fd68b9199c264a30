// Paged decode attention: one query token per sequence attends to its whole
// context, whose K/V rows sit in fixed-size physical blocks reached through a
// per-sequence block table.
//
// What is computed (Month 2 · PagedAttention, infra learning path, §2.1 and
// §5.4; CS349E Lecture 7 notes, §4.2): for sequence s, query head h and kv head
// kv = h / (H / G),
//     out[s][h] = sum_t softmax_t(scale * q[s][h] . K[s][t]) V[s][t],  t < ctx[s],
// where K[s][t] = k_cache[block_tables[s][t / B]][kv][t % B] (HND pool layout;
// NHD swaps the last two indices before head_dim). Blockwise evaluation with an
// online softmax merge gives the same result as a contiguous cache (CMU 15-779
// Lecture 16 notes, §3.3).
//
// Design (one launch, persistent CTAs):
//   * the unit of data movement is a 16-token job: one (K, V) pair of TMA
//     boxes of 16 rows x head_dim, taken from one physical block (a 32-token
//     block is two jobs). Each warp owns R job stages in shared memory, filled
//     by TMA tensor copies (2-D over HND rows, 3-D for NHD; the box lands the
//     same way) that complete on the stage's K and V mbarriers; the warp's lane
//     0 issues the copy of the job R ahead each time it finishes one, so a warp
//     always has R - 1 jobs in flight while it computes one (R - 2 while it
//     computes two: the tensor-core path of E4M3 and of 16-bit plain decode
//     takes two jobs per softmax step; a single producer warp feeding all four
//     rings measured 45% slower: its serial block-table and context-length
//     loads at item boundaries stall every ring at once);
//   * plain mode: a work item is (sequence, kv head); items are dealt to CTAs
//     in a serpentine order, longest contexts first (ties in batch order), and
//     an item's jobs go round-robin to the CTA's W warps, whose partial (max,
//     sum, output) triples are merged through shared memory at the end of the
//     item;
//   * split mode: an item is (sequence, kv head, W consecutive partitions) and
//     warp w handles partition w of it alone, writing its normalised partial
//     output and (max, sum) to the caller's workspace -- no merge or barrier
//     inside the CTA (a shared-partition variant with a per-partition merge
//     measured 40% slower on 32K-128K contexts); a second kernel merges
//     partitions with log-sum-exp weights;
//   * suffix mode (shared-prefix decode): items (sequence, kv head) over each
//     sequence's own tokens are dealt to single warps, which write one partial
//     each into the slot after the prefix partitions;
//   * a KV job is read once for all H / G query heads of its kv head: with a
//     group of >= 2 heads on 16-bit or E4M3 data the step is a small dense
//     contraction and runs on mma.sync m16n8k16 (tokens x heads for q K^T, d x
//     heads for P V; E4M3 codes are converted to fp16 on the way into the
//     fragments); otherwise (MHA, fp32) lanes split head_dim and use
//     FFMA, with V staged unswizzled so a token row sits at fixed offsets;
//   * the softmax is online, in fp32, base 2, with warp shuffles for the maxima;
//     the output accumulators are rescaled only when a running max grew; in
//     plain mode (and E4M3 split mode) the running max may also lag the true
//     one by up to kLazyTau
//     (see below);
//   * every kernel waits for the grid before it (programmatic dependent launch)
//     before touching global memory.
#pragma once

#include "pa_device.cuh"

namespace pa {

constexpr int kMaxGroup = 8;          // query heads per kv head
// Plain mode keeps a stale running max m while no new score exceeds it by more
// than kLazyTau (base 2): weights exp2(z - m) then stay below 2^kLazyTau, which
// fp32 sums and the hi + lo 16-bit split of P carry without loss, and the job
// skips the max shuffles and the accumulator rescale. The result is the same
// softmax (numerator and denominator share the stale reference); only the
// rounding differs. Plain mode uses it, and so does E4M3 split decode; 16-bit
// split decode and the suffix pass keep the exact per-partition max (a lagging
// max measured slower there). A split partial's (m, l) then describe the same
// log-sum-exp, m + log2 l, whichever reference m is.
constexpr float kLazyTau = 8.f;
constexpr int kSortMaxSeqs = 2048;    // longest-first ordering up to this batch size
// The suffix pass keeps each sequence's first own token in shared memory up to
// this batch size (4 bytes a sequence; above it, the MHA suffix pass would lose
// its third CTA per SM), and searches the groups per item beyond.
constexpr int kSuffixStartMaxSeqs = 1024;
constexpr int kSplitMaxSeqs = 2048;   // split mode keeps per-sequence offsets in shared memory
// Sort key of a length: about 8 log2(len) (the exponent and the top three
// mantissa bits), so lengths within ~9% of each other share a bucket: fine
// enough for the longest-first deal to balance the CTAs, coarse enough that
// samples of one prompt (equal prefixes, similar tails) mostly stay next to
// each other in batch order.
__device__ __forceinline__ int length_key(int len) {
  if (len <= 0) return 0;
  const int e = 31 - __clz(len);
  const int frac = e >= 3 ? (len >> (e - 3)) & 7 : (len << (3 - e)) & 7;
  return 1 + e * 8 + frac;
}
constexpr int kNumBuckets = 1024;     // sort buckets: length_key() < 256, length / 512 capped
constexpr int kJobTokens = 16;        // tokens per TMA job

// Compute paths of the decode kernel.
constexpr int kPathVec = 0;     // lanes split head_dim, FFMA; any group, q staged in shared memory
constexpr int kPathVecMha = 1;  // the same for group 1 (MHA), q held in registers
constexpr int kPathMma = 2;     // group >= 2 on 16-bit or E4M3 data: mma.sync m16n8k16
constexpr int kPathMmaG8 = 3;   // the same for groups of 5-8 in plain mode, merging heads in rounds
__host__ __device__ constexpr bool is_mma_path(int path) { return path == kPathMma || path == kPathMmaG8; }

// Plain mode merges the warps' fp32 partial outputs of an item through shared
// memory. kPathMmaG8 merges at most kMergeHeads heads per round (a group of 8 in
// two rounds), so its merge area stays W x 4 x head_dim floats: at group 8 the
// whole-group area (16 KiB at head_dim 128) would leave room for one CTA per SM
// instead of two. The other paths merge their whole group in one round.
constexpr int kMergeHeads = 4;
__host__ __device__ inline int merge_heads(int group, int path) {
  return path == kPathMmaG8 && group > kMergeHeads ? kMergeHeads : group;
}

// What a launch writes.
constexpr int kModePlain = 0;   // the attention output
constexpr int kModeSplit = 1;   // per-partition partials; each warp owns whole partitions
constexpr int kModeSuffix = 2;  // one partial per (sequence, head) over its own tokens after the
                                // shared prefix (cascade decode), at workspace slot suffix_slot

struct DecodeParams {
  void* out;                    // [S][H][D] out dtype (plain mode)
  const void* q;                // [S][H][D]
  const int32_t* block_tables;  // [S][max_blocks]
  const int32_t* context_lens;  // [S]
  int max_blocks;
  int block_size;               // 16 or 32
  int block_shift;              // log2(block_size)
  int S, H, G, group;
  long long num_blocks;
  float scale_log2;             // scale * log2(e)
  int partition;                // split mode: tokens per partition (multiple of the block size)
  int max_partitions;           // split mode: workspace partition dimension
  float* ws_o;                  // [S][H][P][D]
  float* ws_m;                  // [S][H][P]  (max score, base-2 units)
  float* ws_l;                  // [S][H][P]
  float v_scale;                // FP8 caches: V scale applied to the output (1 otherwise)
  // Shared-prefix (cascade) decode: sequences [group_starts[g], group_starts[g+1])
  // share their first prefix_lens[g] tokens (rounded down to whole blocks). The
  // split pass then covers only each sequence's own tokens, writing its
  // partitions from slot suffix_slot on; null group_starts: no shared prefixes.
  const int32_t* group_starts;  // [num_groups + 1]
  const int32_t* prefix_lens;   // [num_groups]
  int num_groups;
  int suffix_slot;
  int suffix_single;            // 1: one suffix partial per row (kModeSuffix)
  int prefix_limit;             // longest usable shared prefix: suffix_slot x partition, table width
  int nhd;                      // pool layout: 0 [blocks][G][B][d], 1 [blocks][B][G][d]
  const void* k_cache;          // the pools (for L2 prefetches of whole HND tiles)
  const void* v_cache;
  unsigned* err;
  // Shared-prefix decode with the tcgen05 prefix pass (S <= kSuffixStartMaxSeqs):
  // the suffix pass's schedule in the workspace, written by one CTA of the prefix
  // pass (suffix_schedule) and read by every CTA of the suffix pass; null: the
  // suffix pass sorts for itself.
  uint16_t* sfx_order;          // [S] sequences, longest own length first
  int* sfx_start;               // [S] each sequence's first own token
  // Plain mode: entries of the longest-first order a CTA keeps in shared memory,
  // one per item of its own (at least ceil(S G / grid)); set by the launcher.
  int order_cap;
};

// TMA copy of 16 rows (tokens r0 .. r0 + 15 of physical block phys, kv head kv)
// and 128 bytes of head_dim starting at element x, into a 16 x 128-byte
// swizzled stage. HND pools are a 2-D map over rows ((phys * G + kv) * B + r);
// NHD pools a 3-D map (head_dim, kv head, phys * B + r). The box lands in shared
// memory in the same order either way, so the consumers do not see the layout.
__device__ __forceinline__ void tma_load_tile(void* dst, const CUtensorMap* map, const DecodeParams& p, int x,
                                              long long phys, int kv, int r0, uint64_t* bar) {
  if (p.nhd)
    tma_load_3d(dst, map, x, kv, (int)(phys << p.block_shift) + r0, bar);
  else
    tma_load_2d(dst, map, x, (int)((phys * p.G + kv) << p.block_shift) + r0, bar);
}

// One job's K or V rows with all of head_dim in one box, for a pool map with a
// region dimension (128-byte column regions as a third / fourth coordinate,
// stride 128 bytes): the same [regions][16 rows][128 B] stage image as one box
// per region, from one copy instead of several. Plain decode takes its tiles
// this way (NHD batch +1%, OPT-13B MHA +1.3%); split decode measured 5% slower
// with it (0.863 against 0.910 on 32K-128K contexts) and, like the suffix pass
// (no change), keeps one box per region.
__device__ __forceinline__ void tma_load_job(void* dst, const CUtensorMap* map, const DecodeParams& p,
                                             long long phys, int kv, int r0, uint64_t* bar) {
  if (p.nhd)
    tma_load_4d(dst, map, 0, kv, (int)(phys << p.block_shift) + r0, 0, bar);
  else
    tma_load_3d(dst, map, 0, (int)((phys * p.G + kv) << p.block_shift) + r0, 0, bar);
}

// A job's tile of NREG 128-byte regions (BOX_X elements each): one box over a
// map with a region dimension (WHOLE), else one box per region.
template <int NREG, int BOX_X, bool WHOLE>
__device__ __forceinline__ void tma_load_rows(uint8_t* dst, const CUtensorMap* map, const DecodeParams& p,
                                              long long phys, int kv, int r0, uint64_t* bar) {
  if constexpr (WHOLE && NREG > 1) {
    tma_load_job(dst, map, p, phys, kv, r0, bar);
  } else {
#pragma unroll
    for (int rg = 0; rg < NREG; ++rg) tma_load_tile(dst + rg * kJobTokens * 128, map, p, rg * BOX_X, phys, kv, r0, bar);
  }
}

struct SmemLayout {
  unsigned stage_bytes, bars_off, ok_off, merge_off, q_off, wts_off, sched_off, misc_off, total;
};

__host__ __device__ inline unsigned round_up(unsigned x, unsigned a) { return (x + a - 1) / a * a; }

// Shared-memory map, computed identically on the host (launch size) and device.
// suffix: the shared-prefix suffix pass, which merges nothing inside the CTA
// and keeps each sequence's first own token beside the sort order.
// order_cap: plain mode's entries of the sort order per CTA (-1: the whole batch).
__host__ __device__ inline SmemLayout make_layout(int W, int R, int D, int esize, int qsize, int group, int path,
                                                  bool split, int S, int jps = 1, bool suffix = false,
                                                  int order_cap = -1) {
  SmemLayout L;
  L.stage_bytes = jps * 2u * kJobTokens * D * esize;  // jps jobs of K and V tiles
  unsigned off = W * R * L.stage_bytes;
  L.bars_off = off;
  off += W * R * 16;  // per stage: K barrier, V barrier
  L.ok_off = off;
  off = round_up(off + W * R * jps, 16);  // per job: its block id was in the pool
  L.merge_off = off;
  if (!split && !suffix) off += W * merge_heads(group, path) * D * 4 + W * kMaxGroup * 2 * 4;
  L.q_off = off;
  if (path == kPathVec) off += W * group * D * 4;            // fp32 q rows per warp
  if (path == kPathVecMha) off += round_up(W * D * qsize, 16);  // raw q row per warp
  L.wts_off = off;
  if (!is_mma_path(path)) off += W * kJobTokens * 4;          // vector paths: one job's weights per warp
  L.sched_off = off;
  if (split)
    off += (S + 1) * 4;
  else if (S <= kSortMaxSeqs && suffix)
    off += S * 2 + (S <= kSuffixStartMaxSeqs ? round_up(S * 2, 16) - S * 2 + S * 4 : 0);  // order [, starts]
  else if (S <= kSortMaxSeqs)
    off += (order_cap >= 0 ? order_cap : S) * 2;  // the sequences of this CTA's items
  off = round_up(off, 16);
  L.misc_off = off;
  off += 16;
  L.total = off + 1024;  // slack to align the dynamic window to 1024 bytes
  return L;
}

// Entries of the sort order a plain-mode CTA keeps: the launcher's grid holds at
// least min(num_sms, S G) CTAs, so no CTA deals itself more than this many items.
// (Capped at S, the whole order's size: a CTA with more items than that, at more
// than num_sms kv heads, takes the batch order.)
__host__ __device__ inline int plain_order_cap(int S, int G, int num_sms) {
  const long long items = (long long)S * G;
  const long long cap = items <= num_sms ? 1 : (items + num_sms - 1) / num_sms;
  return (int)(cap < S ? cap : (S > 1 ? S : 1));
}

template <typename DT, int D, int PATH, int MODE = kModePlain>
struct StageCfg {
  static constexpr int E = sizeof(DT);
  static constexpr int TILE = kJobTokens * D * E;  // one K (or V) job tile
  static constexpr int kJob = 2 * TILE;            // K and V of one job
  static constexpr int W = 4;
  // Tensor-core steps of two jobs each (see the kernel): E4M3 in every mode,
  // 16-bit data in plain mode at head_dim <= 128.
  static constexpr bool PAIRED = is_mma_path(PATH) && D <= 128 && (E == 1 || MODE == kModePlain);
  // Jobs of 4 KiB (E4M3 at head_dim 128, 16-bit data at 64) taken two per step
  // also travel two per stage: one barrier, one wait and one refill for both.
  // A copy-only build of the one-job-per-stage schedule topped out at 0.87-0.92
  // of the copy peak with such jobs (0.998 with 8 KiB jobs): per-job overheads.
  static constexpr int JPS = PAIRED && kJob <= 4096 ? 2 : 1;
  // The MHA path is bound by instruction latency with 2 CTAs per SM: two 8 KiB
  // stages per warp let 3 CTAs fit (50% more warps, the same bytes in flight).
  // head_dim 256 makes a job 16 KiB (16-bit) or 32 KiB (fp32): one stage per
  // warp, so that two CTAs (eight warps) share an SM instead of one. Four 4 KiB
  // jobs per warp: four stages, or two stages of two jobs.
  static constexpr int R = (D > 128 ? 1 : (kJob <= 4096 ? 4 : (PATH == kPathVecMha ? 2 : 3))) / JPS;
  // Minimum CTAs per SM for the register allocator (0: unspecified). The E4M3
  // tensor-core kernels fit 3 CTAs per SM by shared memory; saying so gives them
  // the registers of that occupancy (left alone, the compiler settles for 128
  // registers and spills in split mode). head_dim 256 runs two CTAs per SM.
  static constexpr int MINB = E == 1 && is_mma_path(PATH) ? 3 : (D > 128 ? 2 : 0);
};

struct Item {
  int s, kv, part;   // part: split mode, this warp's partition (-1: none)
  int t0, t1;        // this warp's token range (plain mode: the whole context)
};

// Context length of sequence s, clamped to what the table (and, in split mode,
// the workspace) can describe; out-of-range values are recorded.
__device__ __forceinline__ int clamp_ctx(const DecodeParams& p, int s, bool split) {
  int c = __ldg(p.context_lens + s);
  long long lim = (long long)p.max_blocks * p.block_size;
  if (split) {
    long long lp = (long long)p.max_partitions * p.partition;
    lim = lp < lim ? lp : lim;
  }
  if (c < 0 || c > lim) {
    atomicOr(p.err, kErrContext);
    c = c < 0 ? 0 : (int)lim;
  }
  return c;
}

// Group of sequence s (largest g with group_starts[g] <= s).
__device__ __forceinline__ int group_of(const DecodeParams& p, int s) {
  int lo = 0, hi = p.num_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.group_starts + mid) <= s) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Shared prefix length of group g in whole blocks, clamped to what the
// workspace's prefix slots and the block table can hold (prefix_limit; the
// prefix passes record a longer value, see check_group_prefix).
__device__ __forceinline__ int group_prefix(const DecodeParams& p, int g) {
  const int pl = min(max(0, __ldg(p.prefix_lens + g)), p.prefix_limit);
  return pl - (pl & (p.block_size - 1));
}

__device__ __forceinline__ void check_group_prefix(const DecodeParams& p, int g) {
  if (__ldg(p.prefix_lens + g) > p.prefix_limit) atomicOr(p.err, kErrContext);
}

// First token of sequence s that is its own (after its group's shared prefix).
__device__ __forceinline__ int seq_start(const DecodeParams& p, int s, int ctx) {
  if (p.group_starts == nullptr) return 0;
  const int st = group_prefix(p, group_of(p, s));
  if (st > ctx) {
    atomicOr(p.err, kErrContext);
    return ctx;
  }
  return st;
}

// Suffix pass: a row's prefix slots past its group's prefix partitions get a
// zero sum, so the reduce merges slots [0, suffix_slot] without looking the
// group up (the prefix pass writes the slots below; the reduce skips a zero
// sum). rbase: the row's first slot; t0: the sequence's first own token; the
// calling threads split the slots (thread i of n).
__device__ __forceinline__ void clear_prefix_slots(const DecodeParams& p, long long rbase, int t0, int i, int n) {
  for (int q = (t0 + p.partition - 1) / p.partition + i; q < p.suffix_slot; q += n) p.ws_l[rbase + q] = 0.f;
}

// ---- the stable counting sort of the sequences (every mode's schedule) --------
// Scratch: kNumBuckets counters (bucket b's at b + b / 32, so that lane l's 32
// consecutive buckets in the prefix pass fall in 32 different banks), then each
// sequence's bucket; order[] receives the sequences by ascending bucket, ties in
// batch order. Every thread of the block calls it; warp 0 ranks, then runs
// after_rank(lane) (order[] complete and visible to warp 0), before the block's
// closing barrier.
constexpr int kSortBaseWords = kNumBuckets + kNumBuckets / 32;
constexpr unsigned kSortScratchBytes = kSortBaseWords * 4 + kSortMaxSeqs * 2;
__device__ __forceinline__ int sort_bidx(int b) { return b + (b >> 5); }

template <typename BucketFn, typename AfterRank>
__device__ __forceinline__ void stable_sort_sequences(int S, uint8_t* scratch, uint16_t* order, BucketFn bucket_of,
                                                      int tid, int nthreads, AfterRank after_rank) {
  int* base = reinterpret_cast<int*>(scratch);
  uint16_t* keys = reinterpret_cast<uint16_t*>(scratch + kSortBaseWords * 4);
  const int warp = tid >> 5, lane = tid & 31;
  for (int b = tid; b < kSortBaseWords; b += nthreads) base[b] = 0;
  __syncthreads();
  for (int s = tid; s < S; s += nthreads) {
    const int b = bucket_of(s);
    keys[s] = (uint16_t)b;
    atomicAdd(&base[sort_bidx(b)], 1);
  }
  __syncthreads();
  if (warp == 0) {
    constexpr int PER = kNumBuckets / 32;
    int local = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) local += base[sort_bidx(lane * PER + i)];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int c = base[sort_bidx(lane * PER + i)];
      base[sort_bidx(lane * PER + i)] = run;
      run += c;
    }
    __syncwarp();
    const unsigned lt = (1u << lane) - 1u;
    for (int c0 = 0; c0 < S; c0 += 32) {
      const int s = c0 + lane;
      const int key = s < S ? (int)keys[s] : -1 - lane;  // padding lanes: keys of their own
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      if (s < S) order[base[sort_bidx(key)] + __popc(peers & lt)] = (uint16_t)s;
      __syncwarp();
      if (s < S && (peers & lt) == 0) base[sort_bidx(key)] += __popc(peers);
      __syncwarp();
    }
    after_rank(lane);
  }
  __syncthreads();
}

template <typename BucketFn>
__device__ __forceinline__ void stable_sort_sequences(int S, uint8_t* scratch, uint16_t* order, BucketFn bucket_of,
                                                      int tid, int nthreads) {
  stable_sort_sequences(S, scratch, order, bucket_of, tid, nthreads, [](int) {});
}

// The shared-prefix suffix pass's schedule (S <= kSuffixStartMaxSeqs): sstart[s],
// each sequence's first own token (its group's shared prefix, from one pass over
// the groups' member ranges; a sequence outside every range, with group_starts
// off its contract, is looked up), and order[], the sequences by descending own
// length (buckets of about 8 log2(length): the short suffix items balance better
// with the finer log-scale order). Every thread of the block calls it.
static __device__ __noinline__ void suffix_schedule(const DecodeParams& p, uint8_t* scratch, uint16_t* order, int* sstart,
                                             int tid, int nthreads) {
  for (int s = tid; s < p.S; s += nthreads) sstart[s] = -1;
  __syncthreads();
  for (int g = tid; g < p.num_groups; g += nthreads) {
    const int b = max(__ldg(p.group_starts + g), 0), e = min(__ldg(p.group_starts + g + 1), p.S);
    const int st = group_prefix(p, g);
    for (int s = b; s < e; ++s) sstart[s] = st;
  }
  __syncthreads();
  stable_sort_sequences(p.S, scratch, order, [&](int s) {
    const int c = clamp_ctx(p, s, false);
    int st = sstart[s];
    if (st < 0) {
      st = seq_start(p, s, c);
    } else if (st > c) {  // as seq_start: a prefix longer than the context
      atomicOr(p.err, kErrContext);
      st = c;
    }
    sstart[s] = st;
    return kNumBuckets - 1 - min(length_key(c - st), kNumBuckets - 1);
  }, tid, nthreads);
}

template <int MODE, int W>
struct Schedule {
  // plain mode: the sequence of this CTA's k-th item; suffix mode: the sequences
  // longest-first (nullptr: batch order)
  const uint16_t* order;
  const int* pstart;      // split mode: first item of each sequence, [S + 1]
  const int* sstart;      // suffix mode: each sequence's first own token (nullptr: look it up)
  int num_items;

  // k-th item of this CTA (serpentine deal over the grid), as seen by `warp`. The
  // suffix pass deals items to warps (each warp attends one sequence's short tail
  // alone and writes its partial), the other modes to whole CTAs.
  __device__ __forceinline__ bool get(const DecodeParams& p, int k, int warp, Item& it) const {
    const int pos = (k & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x;
    const long long i = MODE == kModeSuffix ? ((long long)k * gridDim.x + pos) * W + warp
                                            : (long long)k * gridDim.x + pos;
    if (i >= num_items) return false;
    const int ii = (int)i;
    it.kv = ii % p.G;
    const int qi = ii / p.G;
    if (MODE == kModeSplit) {
      int lo = 0, hi = p.S - 1;  // last s with pstart[s] <= qi
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pstart[mid] <= qi) lo = mid; else hi = mid - 1;
      }
      it.s = lo;
      const int c = clamp_ctx(p, lo, true);
      const int st = seq_start(p, lo, c);
      const int nparts = (c - st + p.partition - 1) / p.partition;
      const int part = (qi - pstart[lo]) * W + warp;
      if (part < nparts) {
        it.part = p.suffix_slot + part;  // workspace slot
        it.t0 = st + part * p.partition;
        it.t1 = min(it.t0 + p.partition, c);
      } else {
        it.part = -1;
        it.t0 = it.t1 = 0;
      }
    } else {
      it.s = order ? (int)order[MODE == kModePlain ? k : qi] : qi;  // plain mode: the CTA's own list
      it.t1 = clamp_ctx(p, it.s, false);
      if (MODE == kModeSuffix)
        it.t0 = sstart ? min(sstart[it.s], it.t1) : seq_start(p, it.s, it.t1);
      else
        it.t0 = 0;
      it.part = MODE == kModeSuffix ? p.suffix_slot : 0;
    }
    return true;
  }
};

// DT: cache element type (float, __half, __nv_bfloat16 or fp8e4m3); QT: query
// type (DT, or a 16-bit type over an FP8 cache); OT: output type.
template <typename DT, typename QT, typename OT, int D, int PATH, int MODE>
__global__ void __launch_bounds__(StageCfg<DT, D, PATH, MODE>::W * 32, StageCfg<DT, D, PATH, MODE>::MINB)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const DecodeParams p) {
  pdl_begin();
  using Cfg = StageCfg<DT, D, PATH, MODE>;
  constexpr bool MMA = is_mma_path(PATH);
  constexpr bool ROUNDS = PATH == kPathMmaG8;  // plain mode, groups of 5-8: merge four heads per round
  static_assert(!ROUNDS || MODE == kModePlain, "only plain mode merges inside the CTA");
  constexpr bool SPLIT = MODE == kModeSplit;
  constexpr bool SUFFIX = MODE == kModeSuffix;
  constexpr bool F8 = std::is_same<DT, fp8e4m3>::value;
  // Tensor-core path: two jobs per softmax step (one max / rescale per 32 tokens,
  // two independent score chains in flight). E4M3 in every mode; 16-bit data in
  // plain mode at head_dim <= 128, where it replaced the split refill below and,
  // with one barrier per stage, measured 0.967 -> 0.993 of the copy peak on the
  // Llama batch, 0.92 -> 0.95 at group 8, 1.2x on plain shared-prefix decode and
  // +6-10% at head_dim 64 (A/B on one GPU); 16-bit split decode and the suffix
  // pass gained nothing (0.942 vs 0.945; within 1%) and keep one job per step.
  constexpr bool PAIR = F8 || (MMA && D <= 128 && MODE == kModePlain);
  static_assert(PAIR == Cfg::PAIRED, "the stage configuration follows the step");
  constexpr int JPS = Cfg::JPS;  // jobs per stage
  // stale running max (see kLazyTau): plain mode, and E4M3 split mode (+2.8%
  // there; 16-bit split decode measured 6% slower with it)
  constexpr bool LAZY = MODE == kModePlain || (F8 && MODE == kModeSplit);
  // A one-job tensor-core step on 16-bit data in plain mode (head_dim 256) refills
  // a stage's K tile right after q K^T and its V tile after P V (two barriers per
  // stage): +2.7% on the Llama batch when one job per step was the plain-mode
  // form; the same split in split mode, in the suffix pass and on the MHA vector
  // path was 2-4% slower, so those refill whole stages.
  constexpr bool KV_SPLIT = MMA && !PAIR && MODE == kModePlain;
  // The one-job 16-bit tensor-core steps land K and V on separate barriers
  // (split decode measured +2% with it); the two-job steps (E4M3, 16-bit plain
  // mode) and the vector paths keep one barrier for both (two measured 1.5-2.5%
  // slower on E4M3, 0.5% on 16-bit plain decode, 1.4% on the one-stage
  // head_dim-256 vector path).
  constexpr bool TWO_BARS = MMA && !PAIR;
  static_assert(!KV_SPLIT || TWO_BARS, "a split refill needs a barrier per half");
  static_assert(!PAIR || Cfg::R * JPS >= 2, "two jobs per step need two staged jobs");
  using MT = typename std::conditional<F8, __half, DT>::type;  // tensor-core operand type
  static_assert(!F8 || D % 64 == 0, "FP8 caches need head_dim a multiple of 64");
  constexpr int W = Cfg::W, R = Cfg::R, E = Cfg::E, TILE = Cfg::TILE, JT = kJobTokens;
  constexpr int NCH = D * E / 16;     // 16-byte chunks per row
  constexpr int NREG = D * E / 128;   // 128-byte column regions
  constexpr int BOX_X = 128 / E;      // elements of a region
  // plain mode's pool maps carry a region dimension: one box per job tile
  constexpr bool WHOLE_ROWS = MODE == kModePlain;
  static_assert(NREG >= 1 && D * E % 128 == 0, "head_dim * element size must be a multiple of 128 bytes");
  static_assert(!MMA || ((sizeof(DT) == 2 || F8) && D % 16 == 0), "mma path needs 16-bit or FP8 data");

  extern __shared__ uint8_t smem_raw[];
  // TMA 128-byte swizzling needs 1024-byte aligned destinations: align the shared-window offset.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const SmemLayout L = make_layout(W, R, D, E, (int)sizeof(QT), p.group, PATH, SPLIT, p.S, JPS, SUFFIX, p.order_cap);
  static_assert(W * R * JPS * Cfg::kJob >= kSortScratchBytes + 16 + 2 * kSortMaxSeqs,
                "the sort's scratch and the whole batch's order fit in the stage memory");
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars_off);
  volatile uint8_t* stage_ok = smem + L.ok_off;                        // [W][R][JPS]
  const int MH = merge_heads(p.group, PATH);                           // heads per merge round
  float* mrg_o = reinterpret_cast<float*>(smem + L.merge_off);        // [W][MH][D] (plain mode)
  float* mrg_ml = mrg_o + W * MH * D;                                  // [W][kMaxGroup][2]
  float* qs_all = reinterpret_cast<float*>(smem + L.q_off);            // [W][group][D] (vector path)
  uint8_t* qraw_all = smem + L.q_off;                                  // [W][D] raw (MHA path)
  float* wts_all = reinterpret_cast<float*>(smem + L.wts_off);         // [W][JT] (vector paths)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x, nthreads = W * 32;

  if (tid == 0) {
    for (int i = 0; i < 2 * W * R; ++i) mbar_init(&bars[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (tid == 32) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }

  // ---- schedule tables (the stage buffers are free until the first copy) ------
  Schedule<MODE, W> sch;
  sch.order = nullptr;
  sch.pstart = nullptr;
  sch.sstart = nullptr;
  if (SPLIT) {
    int* pstart = reinterpret_cast<int*>(smem + L.sched_off);
    if (warp == 0) {
      // exclusive scan over sequences of ceil(partitions / W), lane-chunked
      const int per = (p.S + 31) / 32;
      const int b = lane * per, e = min(p.S, b + per);
      auto items_of = [&](int s) {
        const int c = clamp_ctx(p, s, true);
        const int st = seq_start(p, s, c);
        return ((c - st + p.partition - 1) / p.partition + W - 1) / W;
      };
      int local = 0;
      for (int s = b; s < e; ++s) local += items_of(s);
      int incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int run = incl - local;
      for (int s = b; s < e; ++s) {
        pstart[s] = run;
        run += items_of(s);
      }
      if (lane == 31) pstart[p.S] = incl;
    }
    __syncthreads();
    sch.pstart = pstart;
    sch.num_items = pstart[p.S] * p.G;
  } else {
    sch.num_items = p.S * p.G;
    // plain mode: the most items the serpentine deal gives one CTA
    const int kmax = (sch.num_items + (int)gridDim.x - 1) / (int)gridDim.x;
    if (p.S <= kSortMaxSeqs && (SUFFIX || kmax <= p.order_cap)) {
      // stable counting sort of the sequences by length bucket, longest first
      constexpr bool FINE_ORDER = !MMA || F8 || SUFFIX;
      // (plain mode: order[k] is the sequence of this CTA's k-th item; the suffix
      // pass, which deals to warps, keeps the whole order)
      uint16_t* order = reinterpret_cast<uint16_t*>(smem + L.sched_off);
      // suffix mode: each sequence's first own token (its group's prefix), found
      // once here instead of by a search over the groups at every item
      int* sstart = SUFFIX && p.S <= kSuffixStartMaxSeqs
                        ? reinterpret_cast<int*>(smem + L.sched_off + round_up(p.S * 2, 16))
                        : nullptr;
      // the counters and buckets in stage memory (at least 32 KiB, free until the
      // first copy); the shared-pair check's two counters after them
      int* shared_pairs = reinterpret_cast<int*>(smem + kSortScratchBytes);
      int* longest = shared_pairs + 1;
      bool sorted = false;
      if constexpr (SUFFIX) {
        if (sstart != nullptr) {
          if (p.sfx_order != nullptr) {
            // the schedule one CTA of the tcgen05 prefix pass wrote: checked, then
            // used (a value out of range, left by a prefix pass that stopped early,
            // and this CTA sorts for itself)
            int bad = 0;
            for (int s = tid; s < p.S; s += nthreads) {
              const int o = __ldg(p.sfx_order + s), st = __ldg(p.sfx_start + s);
              order[s] = (uint16_t)o;
              sstart[s] = st;
              bad |= (o >= p.S || st < 0) ? 1 : 0;
            }
            sorted = !__syncthreads_or(bad);
          }
          if (!sorted) suffix_schedule(p, smem, order, sstart, tid, nthreads);
          sorted = true;
        }
      }
      if (!sorted) {
        // The 16-bit tensor-core path sorts in 16-token buckets, which balances the
        // CTAs best (0.937 -> 0.945 of peak on the Llama batch), unless neighbours in
        // the batch share their first physical block (samples or beams of one prompt,
        // at least one pair in eight): then 512-token buckets keep a prompt's members
        // together, so its shared blocks are read while they are still in L2 (fine
        // buckets measured 10% slower there).
        // (Longer contexts widen the fine buckets so that the longest still gets a
        // bucket of its own.)
        int coarse_shift = 9;
        if constexpr (!FINE_ORDER) {
          if (tid == 0) *shared_pairs = *longest = 0;
          __syncthreads();
          int local = 0, cmax = 0;
          for (int s = tid; s < p.S; s += nthreads) {
            // the four loads go out together (a table's first entry is readable
            // whatever the context length; it is compared only for two live rows)
            const bool nxt = s + 1 < p.S;
            const int32_t* row = p.block_tables + (long long)s * p.max_blocks;
            const int c = __ldg(p.context_lens + s);
            const int c1 = nxt ? __ldg(p.context_lens + s + 1) : 0;
            const int32_t b0 = __ldg(row), b1 = nxt ? __ldg(row + p.max_blocks) : -1;
            cmax = max(cmax, c);
            if (nxt && c > 0 && c1 > 0 && b0 == b1) ++local;
          }
          if (local) atomicAdd(shared_pairs, local);
          if (cmax) atomicMax(longest, cmax);
          __syncthreads();
          if (*shared_pairs * 8 < p.S) coarse_shift = max(4, 32 - __clz(max(*longest, 1)) - 10);
        }
        // Plain mode ranks the whole batch in stage memory, after the sort's
        // scratch, and keeps only its own items' sequences (order_cap entries
        // instead of S: three E4M3 CTAs per SM still fit at 2,048 sequences).
        uint16_t* ranked = SUFFIX ? order : reinterpret_cast<uint16_t*>(smem + kSortScratchBytes + 16);
        stable_sort_sequences(p.S, smem, ranked, [&](int s) {  // ascending bucket = descending length
          const int c = clamp_ctx(p, s, false);
          // Paths that run below their share of the bandwidth (vector, FP8, the short
          // suffix items, here above the start cache's batch size) balance better
          // with the finer log-scale order.
          const int st = SUFFIX ? seq_start(p, s, c) : 0;
          const int key = FINE_ORDER ? min(length_key(c - st), kNumBuckets - 1)
                                     : min(c >> coarse_shift, kNumBuckets - 1);
          return kNumBuckets - 1 - key;
        }, tid, nthreads, [&](int ln) {
          if constexpr (!SUFFIX) {
            for (int k = ln; k < kmax; k += 32) {
              const int i = k * (int)gridDim.x + ((k & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x);
              if (i < sch.num_items) order[k] = ranked[i / p.G];
            }
          }
        });
      }
      sch.order = order;
      sch.sstart = sstart;
    } else {
      __syncthreads();
    }
  }

  // ---- per-warp issue cursor over this warp's jobs ---------------------------
  uint8_t* my_stages = smem + warp * R * L.stage_bytes;
  uint64_t* my_bars = bars + warp * 2 * R;  // [0, R): K tiles, [R, 2R): V tiles
  volatile uint8_t* my_ok = stage_ok + warp * R * JPS;
  // split mode: each warp owns whole partitions; suffix mode: each warp owns items
  constexpr bool WARP_PARTS = SPLIT || SUFFIX;
  // A warp that streams its own partition also asks L2 for the K and V tiles of
  // its job two after the one it issues (16-bit HND pools, where a tile is one
  // contiguous run): +3.5% on 32K-128K-token split decode. Plain mode deals an
  // item's jobs round-robin to four warps, and there (as for E4M3 caches, bound
  // by issue) the prefetch measured slower.
  constexpr bool PREFETCH = WARP_PARTS && E == 2;
  constexpr int PF_AHEAD = 2;
  const int job_step = WARP_PARTS ? 1 : W;

  struct Cursor {
    int k, u, ue;
    long long phys;  // block-table entry of job u, loaded one job ahead of its issue
    long long phys2; // JPS == 2: block-table entry of the warp's next job in the item (if has2)
    long long pf;    // PREFETCH: block-table entry of job u + PF_AHEAD in the same item, or -1
    Item it;
    bool valid, has2;
  };
  auto cursor_range = [&](Cursor& c) {
    c.u = c.it.t0 / JT + (WARP_PARTS ? 0 : warp);
    c.ue = (c.it.t1 + JT - 1) / JT;
  };
  auto cursor_settle = [&](Cursor& c) {
    while (c.valid && c.u >= c.ue) {
      ++c.k;
      c.valid = sch.get(p, c.k, warp, c.it);
      if (c.valid) cursor_range(c);
    }
    if (c.valid) {
      const int32_t* table = p.block_tables + (long long)c.it.s * p.max_blocks;
      c.phys = __ldg(table + ((c.u * JT) >> p.block_shift));
      if constexpr (JPS == 2) {
        const int u2 = c.u + job_step;
        c.has2 = u2 < c.ue;
        c.phys2 = c.has2 ? (long long)__ldg(table + ((u2 * JT) >> p.block_shift)) : -1;
      }
      if constexpr (PREFETCH) {
        const int uf = c.u + PF_AHEAD;
        c.pf = !p.nhd && uf < c.ue ? (long long)__ldg(table + ((uf * JT) >> p.block_shift)) : -1;
      }
    }
  };
  Cursor ic;
  ic.k = 0;
  ic.valid = sch.get(p, 0, warp, ic.it);
  if (ic.valid) {
    cursor_range(ic);
    cursor_settle(ic);
  }

  // part: kPartK (the K tile and the stage's ok flag), kPartV, or both
  constexpr int kPartK = 1, kPartV = 2;
  auto issue = [&](const Cursor& c, int n, int part) {
    if (lane == 0) {
      const int stage = n % R;
      uint64_t* kbar = &my_bars[stage];
      uint64_t* vbar = TWO_BARS ? &my_bars[R + stage] : kbar;
      const int tok = c.u * JT;
      const int blk = tok >> p.block_shift;
      const long long phys = c.phys;
      if (phys < 0 || phys >= p.num_blocks) {
        // complete the phases with no data; the consumer skips the job
        if (part & kPartK) {
          atomicOr(p.err, kErrBlockId);
          my_ok[stage] = 0;
          mbar_arrive(kbar);
        }
        if (TWO_BARS && (part & kPartV)) mbar_arrive(vbar);
      } else {
        uint8_t* kdst = my_stages + stage * L.stage_bytes;
        uint8_t* vdst = kdst + TILE;
        const int r0 = tok - (blk << p.block_shift);
        if (part & kPartK) my_ok[stage] = 1;
        fence_proxy_async_smem();
        if (part & kPartK) {
          mbar_arrive_expect_tx(kbar, TWO_BARS ? TILE : 2 * TILE);
          tma_load_rows<NREG, BOX_X, WHOLE_ROWS>(kdst, &kmap, p, phys, c.it.kv, r0, kbar);
        }
        if (part & kPartV) {
          if (TWO_BARS) mbar_arrive_expect_tx(vbar, TILE);
          tma_load_rows<NREG, BOX_X, WHOLE_ROWS>(vdst, &vmap, p, phys, c.it.kv, r0, vbar);
        }
        if (PREFETCH && (part & kPartV)) {
          if (c.pf >= 0 && c.pf < p.num_blocks) {  // [pf][kv][rows of job u + PF_AHEAD]: 16 x D contiguous
            const int tokf = (c.u + PF_AHEAD) * JT;
            const size_t off =
                (size_t)(((c.pf * p.G + c.it.kv) << p.block_shift) + (tokf & (p.block_size - 1))) * D * E;
            l2_prefetch(static_cast<const uint8_t*>(p.k_cache) + off, TILE);
            l2_prefetch(static_cast<const uint8_t*>(p.v_cache) + off, TILE);
          }
        }
      }
    }
  };

  // JPS == 2: stage n % R takes the cursor's job and, when the item has one, the
  // warp's next job (so an item's jobs pair up from its first one, as the
  // consumer takes them); one barrier counts both. The cursor moves past both.
  auto issue2 = [&](Cursor& c, int n) {
    const int stage = n % R;
    if (lane == 0) {
      uint64_t* bar = &my_bars[stage];
      uint8_t* base = my_stages + stage * L.stage_bytes;
      const long long ph[2] = {c.phys, c.phys2};
      bool ok[2];
      unsigned bytes = 0;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const bool real = j == 0 || c.has2;
        ok[j] = real && ph[j] >= 0 && ph[j] < p.num_blocks;
        if (real && !ok[j]) atomicOr(p.err, kErrBlockId);  // skipped; the consumer skips the job
        my_ok[stage * 2 + j] = ok[j] ? 1 : 0;
        bytes += ok[j] ? 2u * TILE : 0u;
      }
      fence_proxy_async_smem();
      if (bytes == 0) {
        mbar_arrive(bar);  // complete the phase with no data
      } else {
        mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (!ok[j]) continue;
          const int tok = (c.u + j * job_step) * JT;
          const int r0 = tok - ((tok >> p.block_shift) << p.block_shift);
          uint8_t* kdst = base + j * 2 * TILE;
          tma_load_rows<NREG, BOX_X, WHOLE_ROWS>(kdst, &kmap, p, ph[j], c.it.kv, r0, bar);
          tma_load_rows<NREG, BOX_X, WHOLE_ROWS>(kdst + TILE, &vmap, p, ph[j], c.it.kv, r0, bar);
        }
      }
    }
    c.u += (c.has2 ? 2 : 1) * job_step;
    cursor_settle(c);
  };

  fence_proxy_async_smem();  // generic writes to stage memory (sort counters) before TMA reuses it
  __syncthreads();            // barrier inits and schedule tables visible; stage memory free again

  int n_issue = 0;
#pragma unroll 1
  for (int r = 0; r < R && ic.valid; ++r) {
    if constexpr (JPS == 2) {
      issue2(ic, n_issue++);
    } else {
      issue(ic, n_issue++, kPartK | kPartV);
      ic.u += job_step;
      cursor_settle(ic);
    }
  }

  // ---- consume -----------------------------------------------------------------
  int n_done = 0;
  const float NEG_INF = -__int_as_float(0x7f800000);
  // wait for this warp's next job (ahead = 1: the one after it, still unreleased)
  auto next_job = [&](int& stage_out, int ahead) -> bool {
    const int n = n_done + ahead;
    stage_out = n % R;
    bool ok = mbar_wait_bounded(&my_bars[stage_out], (n / R) & 1, abort_flag, p.err, kWaitLimitNs);
    if (TWO_BARS && !KV_SPLIT && ok)
      ok = mbar_wait_bounded(&my_bars[R + stage_out], (n / R) & 1, abort_flag, p.err, kWaitLimitNs);
    ok = __all_sync(0xffffffffu, ok);
    return ok && my_ok[stage_out];
  };
  // KV_SPLIT: the current job's V tile, waited for only before P V
  auto wait_v = [&]() -> bool {
    if constexpr (!KV_SPLIT) return true;  // next_job waited for the whole stage
    const int n = n_done;
    const bool ok = mbar_wait_bounded(&my_bars[R + n % R], (n / R) & 1, abort_flag, p.err, kWaitLimitNs);
    return __all_sync(0xffffffffu, ok);
  };
  // KV_SPLIT: the current job's K tile is read; refill it with the K of the job R
  // ahead now, and its V after P V (job_done). After an abort no new half goes
  // out; a K half already out without its V is drained on its own at the end.
  auto aborted = [&]() -> bool { return __shfl_sync(0xffffffffu, *abort_flag, 0) != 0; };
  bool v_pending = false, k_orphan = false;
  auto k_done = [&]() {
    if constexpr (!KV_SPLIT) return;  // the stage is refilled whole by job_done
    __syncwarp();
    v_pending = ic.valid && !aborted();
    if (v_pending) issue(ic, n_issue, kPartK);
  };
  auto job_done = [&]() {  // release the stage and refill it with the job R ahead
    __syncwarp();
    ++n_done;
    if constexpr (KV_SPLIT) {
      if (v_pending) {
        v_pending = false;
        if (aborted()) {
          k_orphan = true;  // job n_issue: K in flight, V never issued
        } else {
          issue(ic, n_issue++, kPartV);
          ic.u += job_step;
          cursor_settle(ic);
        }
      }
    } else if (ic.valid && !*abort_flag) {
      if constexpr (JPS == 2) {
        issue2(ic, n_issue++);
      } else {
        issue(ic, n_issue++, kPartK | kPartV);
        ic.u += job_step;
        cursor_settle(ic);
      }
    }
  };
  // Plain mode: merge the W warps' partials of heads h0 .. h0 + MH - 1 of the
  // current item (at mrg_o[w][h - h0]) and write them.
  auto merge_and_write = [&](const Item& x, int h0) {
    asm volatile("bar.sync 1, %0;" ::"n"(W * 32) : "memory");
    const int hq0 = x.kv * p.group;
    const int nh = min(MH, p.group - h0);
    for (int idx = tid; idx < nh * D; idx += nthreads) {
      const int hh = idx / D, i = idx - hh * D, h = h0 + hh;
      float M = NEG_INF;
#pragma unroll
      for (int w = 0; w < W; ++w) {
        if (mrg_ml[(w * kMaxGroup + h) * 2 + 1] > 0.f) M = fmaxf(M, mrg_ml[(w * kMaxGroup + h) * 2 + 0]);
      }
      float Lsum = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float l = mrg_ml[(w * kMaxGroup + h) * 2 + 1];
        if (l > 0.f) {
          const float f = exp2f(mrg_ml[(w * kMaxGroup + h) * 2 + 0] - M);
          Lsum = fmaf(l, f, Lsum);
          O = fmaf(mrg_o[(w * MH + hh) * D + i], f, O);
        }
      }
      reinterpret_cast<OT*>(p.out)[((long long)x.s * p.H + hq0 + h) * D + i] =
          from_f32<OT>(Lsum > 0.f ? O * p.v_scale / Lsum : 0.f);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(W * 32) : "memory");
  };

  Item it;
  if constexpr (MMA) {
    // ---------------- tensor-core path: group >= 2, 16-bit or E4M3 data ----------------
    const int g = lane >> 2, t4 = lane & 3;
    uint32_t qf[D / 16][2], qn[D / 16][2];
    // FP8 caches permute head_dim inside each 64-wide slice so that a thread's
    // K bytes for four k-steps are 16 contiguous bytes: k-step ks = 4 kb + j,
    // MMA k-columns {2t, 2t+1, 2t+8, 2t+9} <-> d = 64 kb + 16 t + 4 j + {0,1,2,3};
    // q takes the same permutation, so q . K is unchanged.
    auto load_q = [&](const Item& x, uint32_t (&dst)[D / 16][2]) {
      const QT* qrow = reinterpret_cast<const QT*>(p.q) + ((long long)x.s * p.H + x.kv * p.group) * D;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        if (g < p.group) {
          if constexpr (F8) {
            const QT* qr = qrow + (long long)g * D + 64 * (ks >> 2) + 16 * t4 + 4 * (ks & 3);
            dst[ks][0] = Mma<__half>::pack(to_f32(qr[0]), to_f32(qr[1]));
            dst[ks][1] = Mma<__half>::pack(to_f32(qr[2]), to_f32(qr[3]));
          } else {
            const QT* qr = qrow + (long long)g * D + ks * 16 + 2 * t4;
            dst[ks][0] = __ldg(reinterpret_cast<const uint32_t*>(qr));
            dst[ks][1] = __ldg(reinterpret_cast<const uint32_t*>(qr + 8));
          }
        } else {
          dst[ks][0] = 0u;
          dst[ks][1] = 0u;
        }
      }
    };
    // FP8: MMA row r holds token tr(r) = (r & 7) / 2 + 4 (r & 1) + (r & 8), so the
    // eight lanes of a quarter-warp read rows tr(2i), tr(2i+1) = i, i + 4, whose
    // swizzled 16-byte chunks fall in different halves of the banks. K rows, V
    // rows (hence P) and the masks all use the same order, so the sums are the
    // same; 16-bit caches keep tr(r) = r (ldmatrix reads conflict-free already).
    auto tr = [](int r) -> int {
      if constexpr (F8) return ((r & 7) >> 1) + 4 * (r & 1) + (r & 8);
      else return r;
    };
    bool have = sch.get(p, 0, warp, it);
    if (have) load_q(it, qn);
#pragma unroll 1
    for (int k = 0; have; ++k) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qf[ks][0] = qn[ks][0];
        qf[ks][1] = qn[ks][1];
      }
      Item nx;
      const bool have_next = sch.get(p, k + 1, warp, nx);
      if (have_next) load_q(nx, qn);  // in flight while this item streams

      float o[D / 16][4];
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
      const int ub = it.t0 / JT + (WARP_PARTS ? 0 : warp), ue = (it.t1 + JT - 1) / JT;
      // Scores of one job: z[e] = scale_log2 * q . k for token tr(g + 8 (e >> 1)),
      // head 2 t4 + (e & 1); NEG_INF past the context.
      auto job_scores = [&](const uint8_t* ktp, int nv, float (&z)[4]) {
        const uint32_t kt = smem_u32(ktp);
        // two independent accumulator chains over head_dim halve the MMA latency chain
        float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (F8) {
#pragma unroll
          for (int kb = 0; kb < D / 64; ++kb) {
            const uint4 r0 = *reinterpret_cast<const uint4*>(ktp + sw128_offset(tr(g), 4 * kb + t4, JT));
            const uint4 r1 = *reinterpret_cast<const uint4*>(ktp + sw128_offset(tr(g + 8), 4 * kb + t4, JT));
            const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w}, w1[4] = {r1.x, r1.y, r1.z, r1.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t a[4];
              e4m3x4_to_f16x2x2(w0[j], a[0], a[2]);
              e4m3x4_to_f16x2x2(w1[j], a[1], a[3]);
              const int ks = 4 * kb + j;
              Mma<MT>::run((j & 1) ? sd : sc, a, qf[ks][0], qf[ks][1]);
            }
          }
        } else {
#pragma unroll
          for (int ks = 0; ks < D / 16; ks += 2) {
            uint32_t a[4], b[4];
            ldsm_x4(a, kt + sw128_offset(lane & 15, ks * 2 + (lane >> 4), JT));
            ldsm_x4(b, kt + sw128_offset(lane & 15, ks * 2 + 2 + (lane >> 4), JT));
            Mma<MT>::run(sc, a, qf[ks][0], qf[ks][1]);
            Mma<MT>::run(sd, b, qf[ks + 1][0], qf[ks + 1][1]);
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = tr(g + ((e >> 1) << 3));
          z[e] = tok < nv ? (sc[e] + sd[e]) * p.scale_log2 : NEG_INF;
        }
      };
      // P V of one job into o. P (this job's weights w, same order as z) enters as a
      // 16-bit operand (both operands of one MMA share a type). Rounding P to bf16
      // alone costs up to 2^-9 relative per weight, too coarse for a 2e-3 bound when
      // a few tokens dominate, so P is split into hi + lo 16-bit parts (P - hi - lo
      // is below 2^-17 P) and each part gets its own MMA into the same accumulator.
      auto job_pv = [&](const uint8_t* ktp, int nv, const float (&w)[4]) {
        const uint32_t h01 = Mma<MT>::pack(w[0], w[1]);
        const uint32_t h23 = Mma<MT>::pack(w[2], w[3]);
        float r0, r1, r2, r3;
        unpack2(h01, (MT*)nullptr, r0, r1);
        unpack2(h23, (MT*)nullptr, r2, r3);
        const uint32_t b0 = movmatrix_trans(h01);
        const uint32_t b1 = movmatrix_trans(h23);
        const uint32_t e0 = movmatrix_trans(Mma<MT>::pack(w[0] - r0, w[1] - r1));
        const uint32_t e1 = movmatrix_trans(Mma<MT>::pack(w[2] - r2, w[3] - r3));
        // tokens held by this lane's A fragments: lo pair (a0, a1), hi pair (a2, a3);
        // rows past the context are zeroed so that 0 * (stale or NaN) cannot leak in
        const int tlo = 2 * t4;
        const uint32_t mlo = (tr(tlo) < nv ? 0x0000ffffu : 0u) | (tr(tlo + 1) < nv ? 0xffff0000u : 0u);
        const uint32_t mhi = (tr(tlo + 8) < nv ? 0x0000ffffu : 0u) | (tr(tlo + 9) < nv ? 0xffff0000u : 0u);
        const bool full = nv == JT;  // every job but a sequence's last: no rows to mask
        if constexpr (F8) {
          // V^T fragments straight from the codes. The A fragment of m-tile mt
          // pairs, per register, two tokens at one head_dim index: k = 2 t4, 2 t4 + 1
          // (a0, a1) or 2 t4 + 8, 2 t4 + 9 (a2, a3), i.e. token rows t4 + 4j
          // (j = 0..3) in the tr() order. The lane reads 16 bytes (chunk vchunk(g))
          // of each of those four rows, interleaves two rows' bytes with one byte
          // permute and converts the pairs: accumulator row r of m-tile mt is head_dim
          // 16 vchunk(r & 7) + 2 mt + (r >> 3) (see drow()). vchunk puts lanes g and
          // g + 1 in opposite halves of the row, so a quarter-warp reads 8 bank groups.
          static_assert(!F8 || D == 128, "the FP8 V fragments cover 128 head_dim bytes");
          const uint8_t* vtp = ktp + TILE;
          const int vch = ((g & 1) << 2) | (g >> 1);
          uint4 rv[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            rv[j] = *reinterpret_cast<const uint4*>(vtp + sw128_offset(t4 + 4 * j, vch, JT));
          auto word = [](const uint4& v, int i) -> uint32_t {
            return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
          };
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            // bytes 2 mt, 2 mt + 1 of two rows, interleaved row by row
            const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
            uint32_t a[4];
            e4m3x4_to_f16x2x2(__byte_perm(word(rv[0], mt >> 1), word(rv[1], mt >> 1), sel), a[0], a[1]);
            e4m3x4_to_f16x2x2(__byte_perm(word(rv[2], mt >> 1), word(rv[3], mt >> 1), sel), a[2], a[3]);
            if (!full) {
              a[0] &= mlo;
              a[1] &= mlo;
              a[2] &= mhi;
              a[3] &= mhi;
            }
            Mma<MT>::run(o[mt], a, b0, b1);
            Mma<MT>::run(o[mt], a, e0, e1);
          }
        } else {
          const uint32_t vt = smem_u32(ktp) + TILE;
          const int vtok = ((lane >> 4) << 3) + (lane & 7);
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            uint32_t a[4];
            ldsm_x4_trans(a, vt + sw128_offset(vtok, mt * 2 + ((lane >> 3) & 1), JT));
            if (!full) {
              a[0] &= mlo;
              a[1] &= mlo;
              a[2] &= mhi;
              a[3] &= mhi;
            }
            Mma<MT>::run(o[mt], a, b0, b1);
            Mma<MT>::run(o[mt], a, e0, e1);
          }
        }
      };
      // Online-softmax step over N jobs' scores: update the running max (m0, m1)
      // and sums (l0, l1), rescale o if a max grew, turn z into weights in place.
      auto softmax_step = [&](float (*z)[4], int N) {
        bool up = false;  // some head's new score passes its running max by > kLazyTau
#pragma unroll
        for (int n = 0; n < N; ++n)
          up |= (fmaxf(z[n][0], z[n][2]) > m0 + kLazyTau) | (fmaxf(z[n][1], z[n][3]) > m1 + kLazyTau);
        if (LAZY && !__any_sync(0xffffffffu, up)) {
          // the first job of an item always takes the exact branch (m0 = m1 = -inf)
#pragma unroll
          for (int n = 0; n < N; ++n) {
            z[n][0] = exp2f(z[n][0] - m0);
            z[n][1] = exp2f(z[n][1] - m1);
            z[n][2] = exp2f(z[n][2] - m0);
            z[n][3] = exp2f(z[n][3] - m1);
            l0 += z[n][0] + z[n][2];
            l1 += z[n][1] + z[n][3];
          }
          return;
        }
        float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
        for (int n = 0; n < N; ++n) {
          mx0 = fmaxf(mx0, fmaxf(z[n][0], z[n][2]));
          mx1 = fmaxf(mx1, fmaxf(z[n][1], z[n][3]));
        }
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        // the accumulators need rescaling only when some head's running max grew
        // (otherwise the factor is exactly 1); after the first jobs it seldom does
        const bool grew = __any_sync(0xffffffffu, (mn0 != m0) | (mn1 != m1));
        const float c0 = exp2f(m0 - mn0), c1 = exp2f(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        l0 *= c0;
        l1 *= c1;
#pragma unroll
        for (int n = 0; n < N; ++n) {
          z[n][0] = exp2f(z[n][0] - mn0);
          z[n][1] = exp2f(z[n][1] - mn1);
          z[n][2] = exp2f(z[n][2] - mn0);
          z[n][3] = exp2f(z[n][3] - mn1);
          l0 += z[n][0] + z[n][2];
          l1 += z[n][1] + z[n][3];
        }
        if (grew) {
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            o[mt][0] *= c0;
            o[mt][2] *= c0;
            o[mt][1] *= c1;
            o[mt][3] *= c1;
          }
        }
      };
      if constexpr (PAIR) {
        // two jobs per step: one softmax update per 32 tokens, and two independent
        // score chains in flight (the FP8 path is bound by instruction latency)
#pragma unroll 1
        for (int u = ub; u < ue; u += 2 * job_step) {
          const bool two = u + job_step < ue;
          int sa = 0, sb = 0;
          bool oka, okb;
          const uint8_t *ka, *kb;
          if constexpr (JPS == 2) {  // both jobs in one stage, behind one barrier
            sa = n_done % R;
            bool ok = mbar_wait_bounded(&my_bars[sa], (n_done / R) & 1, abort_flag, p.err, kWaitLimitNs);
            ok = __all_sync(0xffffffffu, ok);
            oka = ok && my_ok[sa * 2];
            okb = ok && two && my_ok[sa * 2 + 1];
            ka = my_stages + sa * L.stage_bytes;
            kb = ka + 2 * TILE;
          } else {
            oka = next_job(sa, 0);
            okb = two && next_job(sb, 1);
            ka = my_stages + sa * L.stage_bytes;
            kb = my_stages + sb * L.stage_bytes;
          }
          const int nva = min(JT, it.t1 - u * JT), nvb = min(JT, it.t1 - (u + job_step) * JT);
          float z[2][4];
#pragma unroll
          for (int e = 0; e < 4; ++e) z[0][e] = z[1][e] = NEG_INF;
          if (oka) job_scores(ka, nva, z[0]);
          if (okb) job_scores(kb, nvb, z[1]);
          if (oka || okb) {
            softmax_step(z, 2);
            if (oka) job_pv(ka, nva, z[0]);
            if (okb) job_pv(kb, nvb, z[1]);
          }
          job_done();
          if (JPS == 1 && two) job_done();
        }
      } else {
#pragma unroll 1
        for (int u = ub; u < ue; u += job_step) {
          int stage;
          if (next_job(stage, 0)) {
            const uint8_t* ktp = my_stages + stage * L.stage_bytes;
            const int nv = min(JT, it.t1 - u * JT);
            float z[1][4];
            job_scores(ktp, nv, z[0]);
            k_done();
            softmax_step(z, 1);
            if (wait_v()) job_pv(ktp, nv, z[0]);
          } else {
            k_done();
          }
          job_done();
        }
      }
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o2);
      }
      const int hA = 2 * t4, hB = hA + 1;
      // head_dim index of accumulator row r (0..15) of m-tile mt
      auto drow = [&](int mt, int r) -> int {
        if constexpr (F8) {
          const int rr = r & 7;
          return 16 * (((rr & 1) << 2) | (rr >> 1)) + 2 * mt + (r >> 3);
        } else {
          return mt * 16 + r;
        }
      };
      if (WARP_PARTS) {
        if (it.part >= 0) {
          const long long rowA = ((long long)it.s * p.H + it.kv * p.group + hA) * p.max_partitions + it.part;
          const long long rowB = rowA + p.max_partitions;
          const float iA = l0 > 0.f ? p.v_scale / l0 : 0.f, iB = l1 > 0.f ? p.v_scale / l1 : 0.f;
          if (hA < p.group) {
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
              p.ws_o[rowA * D + drow(mt, g)] = o[mt][0] * iA;
              p.ws_o[rowA * D + drow(mt, g + 8)] = o[mt][2] * iA;
            }
            if (g == 0) {
              p.ws_m[rowA] = m0;
              p.ws_l[rowA] = l0;
            }
            if (SUFFIX) clear_prefix_slots(p, rowA - it.part, it.t0, g, 8);
          }
          if (hB < p.group) {
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
              p.ws_o[rowB * D + drow(mt, g)] = o[mt][1] * iB;
              p.ws_o[rowB * D + drow(mt, g + 8)] = o[mt][3] * iB;
            }
            if (g == 0) {
              p.ws_m[rowB] = m1;
              p.ws_l[rowB] = l1;
            }
            if (SUFFIX) clear_prefix_slots(p, rowB - it.part, it.t0, g, 8);
          }
        }
      } else {
        float* mo = mrg_o + warp * MH * D;
        if (g == 0) {
          float* ml = mrg_ml + warp * kMaxGroup * 2;
          ml[hA * 2 + 0] = m0;
          ml[hA * 2 + 1] = l0;
          ml[hB * 2 + 0] = m1;
          ml[hB * 2 + 1] = l1;
        }
        // Heads [h0, h0 + MH) of this lane's pair (hA, hB) go to the merge area,
        // then the CTA merges them. One round at groups of up to four; kPathMmaG8
        // takes two rounds of four heads, lanes t4 = 0, 1 in the first and
        // t4 = 2, 3 in the second.
        auto stage_heads = [&](int h0) {
          if (hA >= h0 && hA < h0 + MH && hA < p.group) {
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
              mo[(hA - h0) * D + drow(mt, g)] = o[mt][0];
              mo[(hA - h0) * D + drow(mt, g + 8)] = o[mt][2];
            }
          }
          if (hB >= h0 && hB < h0 + MH && hB < p.group) {
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
              mo[(hB - h0) * D + drow(mt, g)] = o[mt][1];
              mo[(hB - h0) * D + drow(mt, g + 8)] = o[mt][3];
            }
          }
          merge_and_write(it, h0);
        };
        if constexpr (ROUNDS) {
          stage_heads(0);
          stage_heads(kMergeHeads);
        } else {
          stage_heads(0);
        }
      }
      have = have_next;
      it = nx;
    }
  } else {
    // ---------------- vector path: lanes split head_dim, FFMA ----------------
    constexpr bool MHA = PATH == kPathVecMha;
    constexpr int GM = MHA ? 1 : kMaxGroup;  // heads held per warp
    constexpr int LPT = 32 / JT;             // lanes per token in q K^T (2)
    constexpr int CPL = NCH / LPT;           // 16-byte K chunks per lane
    constexpr int EPC = 16 / E;              // elements per 16-byte chunk
    constexpr int EPL = D / 32;              // output elements per lane in P V
    constexpr int VB = EPL * E;              // V bytes per lane per row
    constexpr int QE = (int)sizeof(QT);
    constexpr int QCH = D * QE / 16;         // 16-byte chunks of one q row
    float* qs = qs_all + warp * p.group * D;
    uint8_t* qraw = qraw_all + warp * D * QE;
    const int t = lane % JT, part = lane / JT;
    float qreg[MHA ? CPL * EPC : 1];  // MHA: this lane's half of the q row
    // MHA: an item's q row -> shared memory, async. One buffer a warp: the row is
    // read into registers (qreg) before the next item's row is fetched into it.
    auto fetch_q_raw = [&](const Item& x) {
      const uint8_t* src = reinterpret_cast<const uint8_t*>(p.q) + ((long long)x.s * p.H + x.kv) * D * QE;
      for (int c = lane; c < QCH; c += 32) cp_async16(qraw + c * 16, src + c * 16);
      cp_async_commit();
    };
    if constexpr (MHA) {
      if (sch.get(p, 0, warp, it)) fetch_q_raw(it);
    }
#pragma unroll 1
    for (int k = 0; sch.get(p, k, warp, it); ++k) {
      if constexpr (MHA) {
        cp_async_wait_all();
        __syncwarp();
        const QT* qr = reinterpret_cast<const QT*>(qraw);
#pragma unroll
        for (int c = 0; c < CPL; ++c)
#pragma unroll
          for (int e = 0; e < EPC; ++e) qreg[c * EPC + e] = to_f32(qr[(part * CPL + c) * EPC + e]);
        __syncwarp();  // every lane has its part of the row before the next one lands
        Item nx;
        if (sch.get(p, k + 1, warp, nx)) fetch_q_raw(nx);
      } else {
        const QT* qrow = reinterpret_cast<const QT*>(p.q) + ((long long)it.s * p.H + it.kv * p.group) * D;
        for (int i = lane; i < p.group * D; i += 32) qs[i] = to_f32(qrow[i]);
        __syncwarp();
      }
      float o[GM][EPL];
      float mr[GM], lr[GM];
#pragma unroll
      for (int h = 0; h < GM; ++h) {
        mr[h] = NEG_INF;
        lr[h] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[h][e] = 0.f;
      }
      const int ub = it.t0 / JT + (WARP_PARTS ? 0 : warp), ue = (it.t1 + JT - 1) / JT;
#pragma unroll 1
      for (int u = ub; u < ue; u += job_step) {
        int stage;
        if (next_job(stage, 0)) {
          const uint8_t* kt = my_stages + stage * L.stage_bytes;
          const uint8_t* vt = kt + TILE;
          const int nv = min(JT, it.t1 - u * JT);
#pragma unroll
          for (int h = 0; h < GM; ++h) {
            if (h >= p.group) break;
            const float* qh = qs + h * D;
            float zc[CPL];  // one partial sum per chunk: short, independent FMA chains
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
              float z = 0.f;
              const int ch = part * CPL + c;
              const uint4 raw = *reinterpret_cast<const uint4*>(kt + sw128_offset(t, ch, JT));
              float qv[EPC];
              if constexpr (MHA) {
#pragma unroll
                for (int e = 0; e < EPC; ++e) qv[e] = qreg[c * EPC + e];
              } else {
#pragma unroll
                for (int e = 0; e < EPC; e += 4) {
                  const float4 q4 = *reinterpret_cast<const float4*>(qh + ch * EPC + e);
                  qv[e] = q4.x;
                  qv[e + 1] = q4.y;
                  qv[e + 2] = q4.z;
                  qv[e + 3] = q4.w;
                }
              }
              if constexpr (E == 4) {
                z = fmaf(qv[0], __uint_as_float(raw.x), z);
                z = fmaf(qv[1], __uint_as_float(raw.y), z);
                z = fmaf(qv[2], __uint_as_float(raw.z), z);
                z = fmaf(qv[3], __uint_as_float(raw.w), z);
              } else if constexpr (E == 1) {
                const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int w4 = 0; w4 < 4; ++w4) {
                  float f0, f1, f2, f3;
                  e4m3x4_to_f32(wd[w4], f0, f1, f2, f3);
                  z = fmaf(qv[4 * w4 + 0], f0, z);
                  z = fmaf(qv[4 * w4 + 1], f1, z);
                  z = fmaf(qv[4 * w4 + 2], f2, z);
                  z = fmaf(qv[4 * w4 + 3], f3, z);
                }
              } else {
                float f0, f1, f2, f3, f4, f5, f6, f7;
                unpack2(raw.x, (DT*)nullptr, f0, f1);
                unpack2(raw.y, (DT*)nullptr, f2, f3);
                unpack2(raw.z, (DT*)nullptr, f4, f5);
                unpack2(raw.w, (DT*)nullptr, f6, f7);
                z = fmaf(qv[0], f0, z);
                z = fmaf(qv[1], f1, z);
                z = fmaf(qv[2], f2, z);
                z = fmaf(qv[3], f3, z);
                z = fmaf(qv[4], f4, z);
                z = fmaf(qv[5], f5, z);
                z = fmaf(qv[6], f6, z);
                z = fmaf(qv[7], f7, z);
              }
              zc[c] = z;
            }
#pragma unroll
            for (int w2 = 1; w2 < CPL; w2 <<= 1)
#pragma unroll
              for (int c = 0; c + w2 < CPL; c += 2 * w2) zc[c] += zc[c + w2];
            float z = zc[0];
            if (LPT == 2) z += __shfl_xor_sync(0xffffffffu, z, 16);
            z = t < nv ? z * p.scale_log2 : NEG_INF;
            float pt;
            if (!LAZY || __any_sync(0xffffffffu, z > mr[h] + kLazyTau)) {
              float mx = z;
#pragma unroll
              for (int o2 = 1; o2 < 16; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
              const float mn = fmaxf(mr[h], mx);
              const float corr = exp2f(mr[h] - mn);
              mr[h] = mn;
              pt = exp2f(z - mn);
              lr[h] = lr[h] * corr + (part == 0 ? pt : 0.f);
#pragma unroll
              for (int e = 0; e < EPL; ++e) o[h][e] *= corr;
            } else {  // stale max within kLazyTau of every score: no rescale
              pt = exp2f(z - mr[h]);
              lr[h] += part == 0 ? pt : 0.f;
            }
            // P V: the job's 16 weights go through shared memory (4 broadcast loads
            // instead of 16 shuffles); V tiles of the vector paths are staged without
            // swizzling, so token tt of this lane's columns is at a fixed offset.
            float* wb = wts_all + warp * JT;
            if (lane < JT) wb[lane] = pt;
            __syncwarp();
            const int byte = lane * VB;
            const uint8_t* vsrc = vt + (byte >> 7) * JT * 128 + (byte & 127);
            auto pv_token = [&](int tt, float w) {
              const uint8_t* src = vsrc + tt * 128;
              if constexpr (E == 1) {
                static_assert(VB == 4, "FP8 vector path reads 4 codes per lane");
                const uint32_t raw = *reinterpret_cast<const uint32_t*>(src);
                float f0, f1, f2, f3;
                e4m3x4_to_f32(raw, f0, f1, f2, f3);
                o[h][0] = fmaf(w, f0, o[h][0]);
                o[h][1] = fmaf(w, f1, o[h][1]);
                o[h][2] = fmaf(w, f2, o[h][2]);
                o[h][3] = fmaf(w, f3, o[h][3]);
              } else if constexpr (E == 4) {
                if constexpr (VB == 32) {
                  const float4 v0 = *reinterpret_cast<const float4*>(src);
                  const float4 v1 = *reinterpret_cast<const float4*>(src + 16);
                  o[h][0] = fmaf(w, v0.x, o[h][0]);
                  o[h][1] = fmaf(w, v0.y, o[h][1]);
                  o[h][2] = fmaf(w, v0.z, o[h][2]);
                  o[h][3] = fmaf(w, v0.w, o[h][3]);
                  o[h][4] = fmaf(w, v1.x, o[h][4]);
                  o[h][5] = fmaf(w, v1.y, o[h][5]);
                  o[h][6] = fmaf(w, v1.z, o[h][6]);
                  o[h][7] = fmaf(w, v1.w, o[h][7]);
                } else if constexpr (VB == 16) {
                  const float4 v = *reinterpret_cast<const float4*>(src);
                  o[h][0] = fmaf(w, v.x, o[h][0]);
                  o[h][1] = fmaf(w, v.y, o[h][1]);
                  o[h][2] = fmaf(w, v.z, o[h][2]);
                  o[h][3] = fmaf(w, v.w, o[h][3]);
                } else {
                  const float2 v = *reinterpret_cast<const float2*>(src);
                  o[h][0] = fmaf(w, v.x, o[h][0]);
                  o[h][1] = fmaf(w, v.y, o[h][1]);
                }
              } else {
                if constexpr (VB == 16) {
                  const uint4 raw = *reinterpret_cast<const uint4*>(src);
                  const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    float f0, f1;
                    unpack2(wd[i], (DT*)nullptr, f0, f1);
                    o[h][2 * i] = fmaf(w, f0, o[h][2 * i]);
                    o[h][2 * i + 1] = fmaf(w, f1, o[h][2 * i + 1]);
                  }
                } else if constexpr (VB == 8) {
                  const uint2 raw = *reinterpret_cast<const uint2*>(src);
                  float f0, f1, f2, f3;
                  unpack2(raw.x, (DT*)nullptr, f0, f1);
                  unpack2(raw.y, (DT*)nullptr, f2, f3);
                  o[h][0] = fmaf(w, f0, o[h][0]);
                  o[h][1] = fmaf(w, f1, o[h][1]);
                  o[h][2] = fmaf(w, f2, o[h][2]);
                  o[h][3] = fmaf(w, f3, o[h][3]);
                } else {
                  const uint32_t raw = *reinterpret_cast<const uint32_t*>(src);
                  float f0, f1;
                  unpack2(raw, (DT*)nullptr, f0, f1);
                  o[h][0] = fmaf(w, f0, o[h][0]);
                  o[h][1] = fmaf(w, f1, o[h][1]);
                }
              }
            };
            if (nv == JT) {  // every job but a sequence's last: fully unrolled
              float wv[JT];
#pragma unroll
              for (int i = 0; i < JT; i += 4) {
                const float4 w4 = *reinterpret_cast<const float4*>(wb + i);
                wv[i] = w4.x;
                wv[i + 1] = w4.y;
                wv[i + 2] = w4.z;
                wv[i + 3] = w4.w;
              }
#pragma unroll
              for (int tt = 0; tt < JT; ++tt) pv_token(tt, wv[tt]);
            } else {
#pragma unroll 4
              for (int tt = 0; tt < nv; ++tt) pv_token(tt, wb[tt]);
            }
            __syncwarp();  // the weights are read before the next head or job rewrites them
          }
        }
        job_done();
      }
      float* mo = mrg_o + warp * MH * D;  // vector paths: MH = group, one merge round
      float* ml = mrg_ml + warp * kMaxGroup * 2;
#pragma unroll
      for (int h = 0; h < GM; ++h) {
        if (h >= p.group) break;
        float l = lr[h];
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o2);
        if (WARP_PARTS) {
          if (it.part >= 0) {
            const long long row = ((long long)it.s * p.H + it.kv * p.group + h) * p.max_partitions + it.part;
            const float inv = l > 0.f ? p.v_scale / l : 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) p.ws_o[row * D + lane * EPL + e] = o[h][e] * inv;
            if (lane == 0) {
              p.ws_m[row] = mr[h];
              p.ws_l[row] = l;
            }
            if (SUFFIX) clear_prefix_slots(p, row - it.part, it.t0, lane, 32);
          }
        } else {
#pragma unroll
          for (int e = 0; e < EPL; ++e) mo[h * D + lane * EPL + e] = o[h][e];
          if (lane == 0) {
            ml[h * 2 + 0] = mr[h];
            ml[h * 2 + 1] = l;
          }
        }
      }
      if (!WARP_PARTS) merge_and_write(it, 0);
    }
    if constexpr (MHA) cp_async_wait_all();
  }

  // ---- let every copy this warp started land before the block exits ------------
  if (lane == 0) {
    const int first = n_issue - R > 0 ? n_issue - R : 0;
    for (int n = first; n < n_issue; ++n) {
      mbar_wait_bounded(&my_bars[n % R], (n / R) & 1, nullptr, p.err, kDrainLimitNs);
      if (TWO_BARS) mbar_wait_bounded(&my_bars[R + n % R], (n / R) & 1, nullptr, p.err, kDrainLimitNs);
    }
    if (k_orphan) mbar_wait_bounded(&my_bars[n_issue % R], (n_issue / R) & 1, nullptr, p.err, kDrainLimitNs);
  }
  __syncwarp();
}

// Slots the reduce merges for sequence s: split decode, the partitions of its
// context; shared-prefix decode, slots [0, suffix_slot) of prefix partitions
// (those past the group's prefix hold a zero sum, see clear_prefix_slots) and
// slot suffix_slot of its own tokens.
__device__ __forceinline__ int merged_slots(const DecodeParams& p, int s) {
  if (p.group_starts != nullptr) return p.suffix_slot + 1;
  return (clamp_ctx(p, s, true) + p.partition - 1) / p.partition;
}

// Pass 2 of split mode: merge the partitions of one (sequence, head) row with
// log-sum-exp weights, M = max_p m_p, w_p = l_p * 2^(m_p - M),
// out = sum_p w_p o_p / sum_p w_p. One CTA per row: thread (v, pg) owns float4
// column v of the partitions p = pg (mod PG) and merges them online as their
// loads arrive (a running max, rescaling its sum and accumulator when the max
// grows), BATCH partitions' loads in flight at a time; the PG partial merges of
// each column are then combined through shared memory. No pass is spent finding
// the row's maximum first.
template <typename OT, int D>
__global__ void __launch_bounds__(256) lse_reduce_kernel(const DecodeParams p) {
  pdl_begin();
  constexpr int NT = 256;
  constexpr int VPR = D / 4;        // float4 vectors per partial row
  constexpr int PG = NT / VPR;      // partition groups (8 for D = 128, 16 for D = 64)
  constexpr int BATCH = 8;          // partitions in flight per thread
  const int row = blockIdx.x;       // s * H + h
  const int s = row / p.H;
  const int tid = threadIdx.x;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const int P = merged_slots(p, s);
  auto slot = [](int q) { return q; };
  const long long base = (long long)row * p.max_partitions;
  const int v = tid % VPR, pg = tid / VPR;
  const float4* src = reinterpret_cast<const float4*>(p.ws_o + base * D) + v;

  float M = NEG_INF, W = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q0 = pg; q0 < P; q0 += PG * BATCH) {
    float4 x[BATCH];
    float mq[BATCH], lq[BATCH];
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      const int q = q0 + b * PG;
      if (q < P) {
        const int sl = slot(q);
        x[b] = __ldg(src + (long long)sl * VPR);
        mq[b] = __ldg(p.ws_m + base + sl);
        lq[b] = __ldg(p.ws_l + base + sl);
      } else {
        lq[b] = 0.f;
      }
    }
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      if (!(lq[b] > 0.f)) continue;  // empty partition
      const float Mn = fmaxf(M, mq[b]);
      const float r = exp2f(M - Mn), w = lq[b] * exp2f(mq[b] - Mn);
      acc.x = fmaf(w, x[b].x, acc.x * r);
      acc.y = fmaf(w, x[b].y, acc.y * r);
      acc.z = fmaf(w, x[b].z, acc.z * r);
      acc.w = fmaf(w, x[b].w, acc.w * r);
      W = fmaf(W, r, w);
      M = Mn;
    }
  }
  __shared__ float sh_m[PG][VPR], sh_w[PG][VPR];
  __shared__ float4 sh_acc[PG][VPR];
  sh_m[pg][v] = M;
  sh_w[pg][v] = W;
  sh_acc[pg][v] = acc;
  __syncthreads();
  if (pg == 0) {
    float Mt = NEG_INF;
#pragma unroll
    for (int gi = 0; gi < PG; ++gi)
      if (sh_w[gi][v] > 0.f) Mt = fmaxf(Mt, sh_m[gi][v]);
    float Wt = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int gi = 0; gi < PG; ++gi) {
      const float wg = sh_w[gi][v];
      if (!(wg > 0.f)) continue;
      const float r = exp2f(sh_m[gi][v] - Mt);
      const float4 a = sh_acc[gi][v];
      O.x = fmaf(r, a.x, O.x);
      O.y = fmaf(r, a.y, O.y);
      O.z = fmaf(r, a.z, O.z);
      O.w = fmaf(r, a.w, O.w);
      Wt = fmaf(r, wg, Wt);
    }
    const float inv = Wt > 0.f ? 1.f / Wt : 0.f;
    OT* out = reinterpret_cast<OT*>(p.out) + (long long)row * D + 4 * v;
    out[0] = from_f32<OT>(O.x * inv);
    out[1] = from_f32<OT>(O.y * inv);
    out[2] = from_f32<OT>(O.z * inv);
    out[3] = from_f32<OT>(O.w * inv);
  }
}

// Pass 2 for rows with few partitions (at most 32 slots): one warp per row.
template <typename OT, int D>
__global__ void __launch_bounds__(256) lse_reduce_small_kernel(const DecodeParams p) {
  pdl_begin();
  constexpr int EPL = D / 32;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.S * p.H) return;
  const int s = row / p.H;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const int P = min(merged_slots(p, s), 32);
  const long long base = (long long)row * p.max_partitions;
  // lane q holds slot q's (max, sum)
  const int sl = lane;
  const float lq = lane < P ? __ldg(p.ws_l + base + sl) : 0.f;
  const float mq = lane < P ? __ldg(p.ws_m + base + sl) : NEG_INF;
  float M = lq > 0.f ? mq : NEG_INF;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float w = lq > 0.f ? lq * exp2f(mq - M) : 0.f;
  float W = w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  for (int q = 0; q < P; ++q) {
    const float wq = __shfl_sync(0xffffffffu, w, q);
    const int slq = __shfl_sync(0xffffffffu, sl, q);
    if (wq == 0.f) continue;
    const float* oq = p.ws_o + (base + slq) * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = fmaf(wq, __ldg(oq + e), acc[e]);
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e)
    reinterpret_cast<OT*>(p.out)[(long long)row * D + lane * EPL + e] = from_f32<OT>(W > 0.f ? acc[e] / W : 0.f);
}

}  // namespace pa
