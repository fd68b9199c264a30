// Shared-prefix (cascade) decode, prefix pass on the fifth-generation tensor
// cores (tcgen05, accumulators in tensor memory).
//
// What is computed is the same as for the other prefix pass: every query row of
// a group (member x query head of one kv head) attends the group's shared
// prefix, partition by partition, and writes the partition's normalised
// partial output with its (max, sum) (CS349E Lecture 7 notes §5.1 and §5.3 for
// the shared blocks; CMU 15-779 Lecture 16 notes §3.3 for the merge). Here the
// group's rows form the M side (64 or 128, padded) of real matrix products:
//   S = Q K^T   M rows, N = 32 tokens, K = head_dim
//   O += P V    M rows, N = head_dim, K = 32 tokens
// Warp roles (256 threads):
//   warps 0-3  softmax: each thread owns one query row, or half of one (M = 64:
//              row 16 w + t of warp w sits in tensor-memory lane 32 w + t and
//              threads t and t + 16 take its two column halves; M = 128:
//              thread t of warp w owns row 32 w + t, in that lane); it reads
//              its part of S, keeps the running (max, sum), writes its part of
//              P (16-bit hi + lo parts) to tensor memory and, at the end of an
//              item, reads its part of O;
//   warp 4     K producer: TMA copies of two 16-token jobs' keys per slot
//              (128-byte swizzle) into a ring of K slots; a slot is free once
//              the softmax warps have read the tile's scores;
//   warp 7     V producer: the same jobs' values into a ring of V slots; a slot
//              is free once the tile's P V has completed (five K and five V
//              slots measured 2-3% faster than four and six);
//   warp 5     owns the tensor memory (allocation, release); its lane 0 issues
//              the score MMAs and commits them to mbarriers, and loads an
//              item's Q tile by TMA as soon as the last item's score MMAs have
//              completed (so the tile is there before the softmax warps are
//              done with the last item);
//   warp 6     its lane 0 issues the P V MMAs and commits them.
// Separate K and V rings keep every byte of shared memory busy: a K slot lives
// from its copy to the score MMAs, a V slot from its copy to the P V, instead
// of a combined stage living until the later of the two.
// S and P are double-buffered in tensor memory: the scores of a tile are
// computed while the softmax warps work on the one before, and the softmax
// writes a tile's weights while the P V of the one before runs. P is the A
// operand of P V straight from tensor memory (a row of P sits in the lane of
// its accumulator row, two 16-bit weights per column: checked on the GB300
// against the same product with P in shared memory), so it costs no shared
// memory and no proxy fence; shared memory goes to K and V slots. The
// accumulator O is rescaled lazily: a row's reference max moves only when a
// score exceeds it by more than kTcRescale (log2 units); weights then stay
// below 2^kTcRescale and the result is the same softmax (numerator and
// denominator share the reference).
// Every wait is time-bounded; on a timeout all roles stop, the copies and
// MMAs in flight are waited for, and the tensor memory is released.
#pragma once

#include "pa_decode.cuh"

namespace pa {

constexpr int kTcMaxRows = 128;    // query rows of one group (members x heads) the pass takes
constexpr int kTcTokens = 32;      // N of S, K of P V: tokens per slot (two TMA jobs)
// M of the tiles is 64 (groups of 17-64 query rows) or 128 (65-128); the
// larger Q tile of M = 128 leaves room for eight slots instead of ten.
__host__ __device__ constexpr int tc_kslots(int MR) { return MR == 64 ? 5 : 4; }
__host__ __device__ constexpr int tc_vslots(int MR) { return MR == 64 ? 5 : 4; }
constexpr int kTcThreads = 256;
constexpr float kTcRescale = 8.f;

struct TcLayout {
  unsigned q_bytes, k_off, v_off, slot_bytes, bar_off, misc_off, sched_off, total;
};

// Offsets from the 1024-byte aligned base: the Q tile, the K slots and the V
// slots (each [head_dim / 64 regions][32 tokens][128 B]), mbarriers, the
// tensor-memory base, the abort flag, per-K-slot job flags and the group scan.
__host__ __device__ inline TcLayout tc_layout(int D, int num_groups, int MR) {
  TcLayout L;
  L.q_bytes = MR * D * 2;
  L.slot_bytes = kTcTokens * D * 2;
  L.k_off = L.q_bytes;
  L.v_off = L.k_off + tc_kslots(MR) * L.slot_bytes;
  L.bar_off = L.v_off + tc_vslots(MR) * L.slot_bytes;
  L.misc_off = L.bar_off + (2 * tc_kslots(MR) + 2 * tc_vslots(MR) + 13) * 8;
  L.sched_off = round_up(L.misc_off + 16, 16);
  L.total = round_up(L.sched_off + (num_groups + 1) * 4, 16) + 1024;
  return L;
}

// ---- tcgen05 ------------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading and
// stride byte offsets (>> 4 each), descriptor version 1, layout type 2.
//   K-major tile ([rows][64-element regions]): stride offset = 1024 (one group
//   of 8 rows), leading offset unused;
//   MN-major tile (rows along K): leading offset = the stride between
//   64-element regions along MN, stride offset = 1024 (8 rows along K).
__device__ __forceinline__ uint64_t tc_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// The descriptor of addr + off, from the descriptor of addr: the start address
// field is addr >> 4 in the low 14 bits, and shared-memory addresses stay below
// 2^18, so adding off >> 4 (off a multiple of 16) never carries out of it.
__device__ __forceinline__ uint64_t tc_desc_add(uint64_t desc, uint32_t off) { return desc + (off >> 4); }

// Instruction descriptor of kind::f16 with an fp32 accumulator: operand format
// (0 fp16, 1 bf16) for A and B, B MN-major or K-major, N >> 3, M >> 4.
template <typename DT>
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N, bool b_mn_major) {
  return (1u << 4) | ((std::is_same<DT, __nv_bfloat16>::value ? 1u : 0u) << 7) |
         ((std::is_same<DT, __nv_bfloat16>::value ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// The same with A in tensor memory at a_tmem: row m of A in the lane that holds
// row m of an M-row accumulator, K elements two to a 32-bit column.
__device__ __forceinline__ void tc_mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                              bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// Arrive on `bar` once every MMA this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive 32-bit columns of this thread's lane (warp-collective).
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16 consecutive 32-bit columns of 16 lanes, twice (warp-collective, shape
// 16x32bx2): threads 0-15 read lanes 0-15 of the warp's quarter at columns
// taddr + j, threads 16-31 the same lanes at columns taddr + OFF + j (measured on
// the GB300 with known values stored through the 32x32b shape).
template <int OFF>
__device__ __forceinline__ void tc_ld16x2(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], %17;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr), "n"(OFF)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

template <int OFF>
__device__ __forceinline__ void tc_st16x2(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], %1, {%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17};" ::"r"(
          taddr),
      "n"(OFF), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Bounded wait whose polls suspend the thread for up to `hint_ns` while the
// phase is incomplete, so a waiting role leaves the issue slots to the others;
// otherwise as mbar_wait_bounded.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                unsigned* err, unsigned long long limit_ns) {
  constexpr uint32_t hint_ns = 2000;
  auto poll = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
  };
  if (poll()) return true;
  const unsigned long long t0 = globaltimer();
  for (;;) {
    if (poll()) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (globaltimer() - t0 > limit_ns) {
      if (abort_flag != nullptr) *abort_flag = 1;
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}

// 2^x on the special-function unit (inputs below -126 give 0).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// A box of fill values (zeros) for a job that does not exist: every row of the
// box lies before the start of the pool.
__device__ __forceinline__ void tma_load_zero_tile(void* dst, const CUtensorMap* map, const DecodeParams& p, int x,
                                                   uint64_t* bar) {
  if (p.nhd)
    tma_load_3d(dst, map, x, 0, -kJobTokens, bar);
  else
    tma_load_2d(dst, map, x, -kJobTokens, bar);
}

template <typename DT, int D, int MR>
__global__ void __launch_bounds__(kTcThreads, 2)
    cascade_prefix_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                             const __grid_constant__ CUtensorMap qmap, const DecodeParams p) {
  pdl_begin();
  static_assert(sizeof(DT) == 2 && (D == 64 || D == 128), "tensor-core prefix pass: 16-bit caches, head_dim 64/128");
  static_assert(MR == 64 || MR == 128, "tiles of 64 or 128 query rows");
  constexpr int RK = tc_kslots(MR), RV = tc_vslots(MR), NT = kTcTokens, JT = kJobTokens, M = MR;
  constexpr int NREG = D / 64;            // 128-byte regions of a row
  constexpr int TILE = NT * D * 2;        // K (or V) bytes of one slot
  constexpr int REG_BYTES = NT * 128;     // one region of a slot: [32 tokens][128 B]
  constexpr int KSTEPS = D / 16;
  // tensor-memory columns: O (D), two S buffers (NT each), two P buffers (NT each:
  // a row's NT hi and NT lo weights, two to a column)
  constexpr uint32_t TCOLS = 256u;
  constexpr uint32_t O_COL = 0, S_COL = D, P_COL = D + 2 * NT;
  static_assert(P_COL + 2 * NT <= TCOLS, "tensor-memory columns");
  constexpr uint32_t ID_S = tc_idesc<DT>(M, NT, false);
  constexpr uint32_t ID_PV = tc_idesc<DT>(M, D, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const TcLayout L = tc_layout(D, p.num_groups, MR);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* k_full = bars;                 // [RK] K copied -> score MMAs
  uint64_t* k_empty = bars + RK;           // [RK] scores read by the softmax -> K producer
  uint64_t* v_full = bars + 2 * RK;        // [RV] V copied -> P V MMAs
  uint64_t* v_empty = bars + 2 * RK + RV;  // [RV] P V done -> V producer
  uint64_t* s_full = bars + 2 * RK + 2 * RV;  // [2] S written -> softmax
  uint64_t* s_free = s_full + 2;      // [2] S read -> MMA
  uint64_t* q_full = s_full + 4;      // the item's Q tile landed -> score MMAs
  uint64_t* q_free = s_full + 5;      // the last item's score MMAs done -> Q tile reloaded
  uint64_t* p_full = s_full + 6;      // [2] P written -> MMA
  uint64_t* pv_done = s_full + 8;     // [2] P V done -> softmax (that P buffer free, O current)
  uint64_t* o_free = s_full + 10;     // O read at the end of an item -> MMA
  uint64_t* fin = s_full + 11;        // every score MMA done (teardown)
  uint64_t* fin_pv = s_full + 12;     // every P V MMA done (teardown)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc_off + 4);
  // [RK] bit j: job j of the K slot comes from a block in the pool. Written before
  // the K producer's arrive on k_full[slot] and read after a wait on it (the
  // softmax releases the slot after reading it).
  volatile uint8_t* job_ok = smem + L.misc_off + 8;
  int* pstart = reinterpret_cast<int*>(smem + L.sched_off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < RK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 4);
    }
    for (int i = 0; i < RV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 4);
      mbar_init(&q_full[b], 1);  // q_full, q_free
      mbar_init(&p_full[b], 4);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(o_free, 4);
    mbar_init(fin, 1);
    mbar_init(fin_pv, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    prefetch_tensormap(&qmap);
  }
  // Q rows past the box (group x (M / group) rows) stay zero; the box rows past
  // the group's members hold other sequences' queries (or zeros past the batch):
  // those rows' scores and outputs are computed and never written
  for (int i = threadIdx.x; i < (int)(L.q_bytes / 16); i += kTcThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TCOLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (warp == 0) {  // exclusive scan over groups of their prefix partitions
    const int per = (p.num_groups + 31) / 32;
    const int b = lane * per, e = min(p.num_groups, b + per);
    auto parts = [&](int g) { return (group_prefix(p, g) + p.partition - 1) / p.partition; };
    int local = 0;
    for (int g = b; g < e; ++g) {
      if (blockIdx.x == 0) check_group_prefix(p, g);
      local += parts(g);
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int g = b; g < e; ++g) {
      pstart[g] = run;
      run += parts(g);
    }
    if (lane == 31) pstart[p.num_groups] = incl;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const int num_items = pstart[p.num_groups] * p.G;

  struct PItem {
    int g, kv, part, s0, members, t0, t1;
  };
  auto get = [&](int k, PItem& it) -> bool {  // k-th item of this CTA (serpentine deal)
    const int pos = (k & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x;
    const long long i = (long long)k * gridDim.x + pos;
    if (i >= num_items) return false;
    it.kv = (int)(i % p.G);
    const int qi = (int)(i / p.G);
    int lo = 0, hi = p.num_groups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pstart[mid] <= qi) lo = mid; else hi = mid - 1;
    }
    it.g = lo;
    it.part = qi - pstart[lo];
    it.s0 = __ldg(p.group_starts + lo);
    it.members = __ldg(p.group_starts + lo + 1) - it.s0;
    it.t0 = it.part * p.partition;
    it.t1 = min(it.t0 + p.partition, group_prefix(p, lo));
    return true;
  };
  auto num_tiles = [&](const PItem& it) { return ((it.t1 - it.t0 + JT - 1) / JT + 1) / 2; };
  const uint32_t q_base = smem_u32(smem);
  const uint32_t k_base = smem_u32(smem + L.k_off);
  const uint32_t v_base = smem_u32(smem + L.v_off);

  if (warp == 4 || warp == 7) {
    // ------------------------------- producers ------------------------------
    // Warp 4 copies the keys, warp 7 the values of the same tiles, each into its
    // own ring. A warp reads the block ids of 32 jobs at a time (one per lane) and
    // lane 0 takes them by shuffle, so no table load waits between two copies.
    const bool is_v = warp == 7;
    const int R = is_v ? RV : RK;
    uint64_t* full = is_v ? v_full : k_full;
    uint64_t* empty = is_v ? v_empty : k_empty;
    uint8_t* ring = smem + (is_v ? L.v_off : L.k_off);
    const CUtensorMap* map = is_v ? &vmap : &kmap;
    int n = 0;
    PItem it;
    for (int k = 0; get(k, it); ++k) {
      if (__shfl_sync(0xffffffffu, (int)*abort_flag, 0)) break;
      const int32_t* table = p.block_tables + (long long)it.s0 * p.max_blocks;
      const int u0 = it.t0 / JT, ue = (it.t1 + JT - 1) / JT;  // the item's jobs
      const int nt = num_tiles(it);
      int wbase = u0;
      long long wphys = u0 + lane < ue ? (long long)__ldg(table + (((u0 + lane) * JT) >> p.block_shift)) : -1;
      bool stop = false;
      for (int i = 0; i < nt; ++i, ++n) {
        const int ua = u0 + 2 * i;
        if (ua + 1 >= wbase + 32) {  // the window moves to this tile
          wbase = ua;
          wphys = ua + lane < ue ? (long long)__ldg(table + (((ua + lane) * JT) >> p.block_shift)) : -1;
        }
        long long ph[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          ph[j] = __shfl_sync(0xffffffffu, wphys, ua + j - wbase);
          if (ua + j >= ue) ph[j] = -2;  // no such job in this item
        }
        // lane 0 waits for the slot and announces its bytes; lanes 0 .. 2 NREG - 1
        // then issue one box each (job j, region rg): a single thread issuing all
        // of a tile's boxes in turn measured slower than the copy itself
        const int slot = n % R;
        int ok = 1;
        if (lane == 0) {
          ok = mbar_wait_sleep(&empty[slot], ((n / R) & 1) ^ 1, abort_flag, p.err, kWaitLimitNs);
          if (ok) {
            if (!is_v) {
              job_ok[slot] = (uint8_t)((ph[0] >= 0 && ph[0] < p.num_blocks ? 1 : 0) |
                                       (ph[1] >= 0 && ph[1] < p.num_blocks ? 2 : 0));
#pragma unroll
              for (int j = 0; j < 2; ++j)
                if (ph[j] != -2 && (ph[j] < 0 || ph[j] >= p.num_blocks)) atomicOr(p.err, kErrBlockId);
            }
            mbar_arrive_expect_tx(&full[slot], TILE);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok && lane < 2 * NREG) {
          const int j = lane / NREG, rg = lane % NREG;
          long long phys = j ? ph[1] : ph[0];  // (a select: no local-memory array)
          if (phys >= p.num_blocks) phys = -1;
          const int tok = (ua + j) * JT;
          const int r0 = tok - ((tok >> p.block_shift) << p.block_shift);
          uint8_t* dst = ring + slot * L.slot_bytes + rg * REG_BYTES + j * JT * 128;
          if (phys >= 0)
            tma_load_tile(dst, map, p, rg * 64, phys, it.kv, r0, &full[slot]);
          else  // absent or out-of-pool job: zeros (the softmax masks its tokens)
            tma_load_zero_tile(dst, map, p, rg * 64, &full[slot]);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          stop = true;
          break;
        }
      }
      if (stop) break;
    }
    // let the last copies land before the block can exit
    if (lane == 0) {
      const int first = n - R > 0 ? n - R : 0;
      for (int m = first; m < n; ++m) mbar_wait_bounded(&full[m % R], (m / R) & 1, nullptr, p.err, kDrainLimitNs);
    }
    __syncwarp();
  } else if (warp == 5 || warp == 6) {
    // ------------------------------ MMA issuers ------------------------------
    // Lane 0 of warp 5 issues the score MMAs of every tile, lane 0 of warp 6 the
    // P V MMAs: a tile's P V goes out as soon as its P is written, never behind
    // the next tile's score MMAs. Each commit tracks the issuing thread's own
    // MMAs; the commit of a tile's P V to v_empty frees its V slot.
    if (lane == 0) {
      int n = 0;
      bool issued = false;
      PItem it;
      if (warp == 5) {
        const uint64_t qdesc = tc_desc(q_base, 16, 1024);  // built once; the MMAs add offsets
        // an item's Q tile: rows member x group + head, from a box of (M / group)
        // sequences x group heads of its kv head, one box per 64 columns
        const int qrows = p.group * (M / p.group);
        int q_loads = 0, q_landed = 0;  // Q copies issued, and waited for
        auto load_q = [&](const PItem& x) {
          ++q_loads;
          mbar_arrive_expect_tx(q_full, (uint32_t)(qrows * D * 2));
#pragma unroll
          for (int rg = 0; rg < NREG; ++rg)
            tma_load_3d(smem + rg * (M * 128), &qmap, rg * 64, x.kv * p.group, x.s0, q_full);
        };
        bool have = get(0, it);
        if (have) load_q(it);
        for (int k = 0; have; ++k) {
          if (!mbar_wait_sleep(q_full, k & 1, abort_flag, p.err, kWaitLimitNs)) break;
          ++q_landed;
          const int nt = num_tiles(it);
          bool stop = false;
          for (int i = 0; i < nt; ++i, ++n) {
            const int slot = n % RK, b = n & 1;
            if (!mbar_wait_sleep(&k_full[slot], (n / RK) & 1, abort_flag, p.err, kWaitLimitNs) ||
                !mbar_wait_sleep(&s_free[b], ((n >> 1) & 1) ^ 1, abort_flag, p.err, kWaitLimitNs)) {
              stop = true;
              break;
            }
            tc_fence_after();
            const uint64_t kdesc = tc_desc(k_base + slot * L.slot_bytes, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
              const uint64_t a = tc_desc_add(qdesc, (ks >> 2) * (M * 128) + (ks & 3) * 32);
              const uint64_t bd = tc_desc_add(kdesc, (ks >> 2) * REG_BYTES + (ks & 3) * 32);
              tc_mma(tbase + S_COL + b * NT, a, bd, ID_S, ks > 0);
            }
            tc_commit(&s_full[b]);
            issued = true;
          }
          if (stop) break;
          PItem nx;
          const bool have_next = get(k + 1, nx);
          if (have_next) {  // the next item's Q, once this item's score MMAs have read the tile
            tc_commit(q_free);
            if (!mbar_wait_sleep(q_free, k & 1, abort_flag, p.err, kWaitLimitNs)) break;
            load_q(nx);
          }
          have = have_next;
          it = nx;
        }
        if (q_loads > q_landed)  // a Q copy still in flight after an abort lands before the block exits
          mbar_wait_bounded(q_full, (q_loads - 1) & 1, nullptr, p.err, kDrainLimitNs);
      } else {
        for (int k = 0; get(k, it); ++k) {
          const int nt = num_tiles(it);
          bool stop = false;
          for (int i = 0; i < nt; ++i, ++n) {
            // the item's first tile overwrites O, once the softmax has read the last item's O
            const bool first = i == 0;
            const int pb = n & 1;
            if (!mbar_wait_sleep(&p_full[pb], (n >> 1) & 1, abort_flag, p.err, kWaitLimitNs) ||
                !mbar_wait_sleep(&v_full[n % RV], (n / RV) & 1, abort_flag, p.err, kWaitLimitNs) ||
                (first && k > 0 && !mbar_wait_sleep(o_free, (k - 1) & 1, abort_flag, p.err, kWaitLimitNs))) {
              stop = true;
              break;
            }
            tc_fence_after();
            const uint64_t vdesc = tc_desc(v_base + (n % RV) * L.slot_bytes, REG_BYTES, 1024);
            // P buffer pb: columns 16 ks .. 16 ks + 7 hold the hi weights of tokens
            // 16 ks .. 16 ks + 15, the next 8 columns their lo weights
#pragma unroll
            for (int ks = 0; ks < NT / 16; ++ks) {
              const uint64_t b = tc_desc_add(vdesc, ks * 2048);
#pragma unroll
              for (int part = 0; part < 2; ++part)
                tc_mma_tmem_a(tbase + O_COL, tbase + P_COL + pb * NT + ks * 16 + part * 8, b, ID_PV,
                              !(first && part == 0 && ks == 0));
            }
            tc_commit(&pv_done[pb]);
            tc_commit(&v_empty[n % RV]);
            issued = true;
          }
          if (stop) break;
        }
      }
      if (issued) {  // every MMA this thread issued has completed before the tensor memory is released
        uint64_t* done = warp == 5 ? fin : fin_pv;
        tc_commit(done);
        mbar_wait_bounded(done, 0, nullptr, p.err, kDrainLimitNs);
      }
    }
    __syncwarp();
  } else if (warp < 4) {
    // -------------------------------- softmax --------------------------------
    const float NEG_INF = -__int_as_float(0x7f800000);
    // The row this thread owns. An M = 128 accumulator keeps row 32 w + t in lane
    // 32 w + t: thread t of warp w takes that whole row. An M = 64 one keeps row
    // 16 w + t in lane 32 w + t (t < 16) and nothing in lanes 16-31, so threads t
    // and t + 16 share row 16 w + t (HALF): the 16x32bx2 loads give thread t its
    // columns 0-15 and thread t + 16 its columns 16-31 (of a tile's 32 scores; of
    // O, the first and second half of head_dim). The two halves exchange the row
    // max per tile and the sum at the end of an item.
    constexpr bool HALF = MR == 64;
    constexpr int CW = HALF ? NT / 2 : NT;  // score columns per thread
    const int half = HALF ? lane >> 4 : 0;
    const int row = HALF ? 16 * warp + (lane & 15) : 32 * warp + lane;
    const uint32_t lane_addr = tbase + ((uint32_t)(32 * warp) << 16);
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      const bool ok = mbar_wait_bounded(bar, parity, abort_flag, p.err, kWaitLimitNs);
      return __all_sync(0xffffffffu, ok);
    };
    int n = 0;
    PItem it, nx;
    bool have = get(0, it);
    for (int k = 0; have; ++k) {
      const bool have_next = get(k + 1, nx);
      const int rows = it.members * p.group;
      const int nt = num_tiles(it);
      float m_ref = NEG_INF, l = 0.f;
      bool stop = false;
      for (int i = 0; i < nt; ++i, ++n) {
        const int b = n & 1;
        const int kslot = n % RK;
        if (!wait_all(&s_full[b], (n >> 1) & 1) || !wait_all(&k_full[kslot], (n / RK) & 1)) {
          stop = true;
          break;
        }
        // the tile's jobs with a block in the pool (the producer zero-filled the
        // others); k_full[kslot] completed before S was computed and cannot move on
        // before these warps release the slot
        const unsigned ok = job_ok[kslot];
        tc_fence_after();
        uint32_t s[CW];
        if constexpr (HALF)
          tc_ld16x2<NT / 2>(lane_addr + S_COL + b * NT, s);
        else
          tc_ld32(lane_addr + S_COL + b * NT, s);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&s_free[b]);
          mbar_arrive(&k_empty[kslot]);  // the score MMAs are done with the K slot
        }
        // scores of this tile's real tokens (this thread's columns tok0 ..), in base-2 units
        const int nv = min(NT, it.t1 - (it.t0 + 2 * i * JT));
        const int tok0 = half * CW;
        float z[CW], tm[CW / 2];
        if (nv == NT && ok == 3u) {  // every tile but an item's ragged or faulty last one
#pragma unroll
          for (int t = 0; t < CW; ++t) z[t] = __uint_as_float(s[t]) * p.scale_log2;
        } else {
#pragma unroll
          for (int t = 0; t < CW; ++t) {
            const bool real = tok0 + t < nv && ((ok >> ((tok0 + t) / JT)) & 1u);
            z[t] = real ? __uint_as_float(s[t]) * p.scale_log2 : NEG_INF;
          }
        }
#pragma unroll
        for (int e = 0; e < CW / 2; ++e) tm[e] = fmaxf(z[e], z[e + CW / 2]);  // the row max as a tree
#pragma unroll
        for (int w = CW / 4; w > 0; w >>= 1)
#pragma unroll
          for (int e = 0; e < w; ++e) tm[e] = fmaxf(tm[e], tm[e + w]);
        float mx = tm[0];
        if constexpr (HALF) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));  // the other half of the row
        const bool move = mx > m_ref + kTcRescale || (m_ref == NEG_INF && mx > NEG_INF);
        const float m_new = move ? mx : m_ref;
        const float c = move ? exp2f(m_ref - m_new) : 1.f;
        const float msub = m_new == NEG_INF ? 0.f : m_new;
        l *= c;
        m_ref = m_new;
        // this thread's weights as hi + lo 16-bit parts (l: this thread's columns' sum)
        uint32_t hw[CW / 2], lw[CW / 2];
        float ls[4] = {0.f, 0.f, 0.f, 0.f};  // four partial sums: short dependency chains
#pragma unroll
        for (int e = 0; e < CW / 2; ++e) {
          const float w0 = ex2_ftz(z[2 * e] - msub), w1 = ex2_ftz(z[2 * e + 1] - msub);
          ls[e & 3] += w0 + w1;
          hw[e] = Mma<DT>::pack(w0, w1);
          float r0, r1;
          unpack2(hw[e], (DT*)nullptr, r0, r1);
          lw[e] = Mma<DT>::pack(w0 - r0, w1 - r1);
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        // P buffer pb is free once the P V of tile n - 2 has completed; O is current
        // (for a rescale) once that of tile n - 1 has
        const int pb = n & 1;
        if (n >= 2 && !wait_all(&pv_done[pb], ((n - 2) >> 1) & 1)) {
          stop = true;
          break;
        }
        if (i > 0 && __any_sync(0xffffffffu, move)) {
          if (!wait_all(&pv_done[pb ^ 1], ((n - 1) >> 1) & 1)) {
            stop = true;
            break;
          }
          tc_fence_after();
          if constexpr (HALF) {  // thread t: columns [0, D/2) of its row, thread t + 16: [D/2, D)
#pragma unroll 1
            for (int c0 = 0; c0 < D / 2; c0 += 16) {
              uint32_t o[16];
              tc_ld16x2<D / 2>(lane_addr + O_COL + c0, o);
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * c);
              tc_st16x2<D / 2>(lane_addr + O_COL + c0, o);
            }
          } else {
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t o[32];
              tc_ld32(lane_addr + O_COL + c0, o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * c);
              tc_st32(lane_addr + O_COL + c0, o);
            }
          }
        }
        // P into buffer pb: per 16 tokens, 8 columns of hi weights then 8 of lo (M = 64:
        // thread t the first 16 columns of its row, thread t + 16 the next 16)
        tc_fence_after();
        if constexpr (HALF) {
          uint32_t pw[16];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            pw[e] = hw[e];
            pw[8 + e] = lw[e];
          }
          tc_st16x2<16>(lane_addr + P_COL + pb * NT, pw);
        } else {
          uint32_t pw[32];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            pw[e] = hw[e];
            pw[8 + e] = lw[e];
            pw[16 + e] = hw[8 + e];
            pw[24 + e] = lw[8 + e];
          }
          tc_st32(lane_addr + P_COL + pb * NT, pw);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[pb]);
      }
      if (stop) break;
      // the item's last P V, then this thread's row of O: normalised partial, max, sum
      if (!wait_all(&pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1)) break;
      tc_fence_after();
      if constexpr (HALF) l += __shfl_xor_sync(0xffffffffu, l, 16);  // the row's two halves
      const bool write = row < rows;
      const long long wrow = ((long long)(it.s0 + row / p.group) * p.H + it.kv * p.group + row % p.group) *
                                 p.max_partitions + it.part;
      const float inv = l > 0.f ? p.v_scale / l : 0.f;
      if constexpr (HALF) {
#pragma unroll 1
        for (int c0 = 0; c0 < D / 2; c0 += 16) {
          uint32_t o[16];
          tc_ld16x2<D / 2>(lane_addr + O_COL + c0, o);
          if (write) {
            float4* dst = reinterpret_cast<float4*>(p.ws_o + wrow * D + half * (D / 2) + c0);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                   __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
          }
        }
      } else {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tc_ld32(lane_addr + O_COL + c0, o);
          if (write) {
            float4* dst = reinterpret_cast<float4*>(p.ws_o + wrow * D + c0);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                   __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
          }
        }
      }
      if (write && half == 0) {
        p.ws_m[wrow] = m_ref;
        p.ws_l[wrow] = l;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
      have = have_next;
      it = nx;
    }
  }

  // ---- teardown: every role has stopped; release the tensor memory ----------------
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(TCOLS) : "memory");

  // The suffix pass's schedule (sequence order and first own tokens), computed
  // once here instead of by every CTA of the suffix pass: by the CTA with the
  // fewest items (when the items do not divide evenly over the grid it has a
  // round to spare). Shared memory is free: every copy has landed.
  if (p.sfx_order != nullptr && !*abort_flag) {
    const int grid = (int)gridDim.x, rem = num_items % grid, last = num_items / grid;
    const int sorter = (rem == 0 || (last & 1) == 0) ? grid - 1 : 0;  // the serpentine's last round
    if ((int)blockIdx.x == sorter) {
      uint16_t* order = reinterpret_cast<uint16_t*>(smem + kSortScratchBytes);
      int* sstart = reinterpret_cast<int*>(smem + kSortScratchBytes + round_up(p.S * 2, 16));
      suffix_schedule(p, smem, order, sstart, threadIdx.x, kTcThreads);
      for (int s = threadIdx.x; s < p.S; s += kTcThreads) {
        p.sfx_order[s] = order[s];
        p.sfx_start[s] = sstart[s];
      }
    }
  }
}

}  // namespace pa
