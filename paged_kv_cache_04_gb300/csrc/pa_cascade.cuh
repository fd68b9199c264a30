// Shared-prefix (cascade) decode, prefix pass.
//
// Parallel samples of one prompt share the prompt's KV blocks through their
// block tables (CS349E Lecture 7 notes §5.1 and §5.3; reference-counted shared
// blocks). Attention over a context is the merge of attention over any split
// of it (CMU 15-779 Lecture 16 notes §3.3), so the context of every sample of
// a group can be cut into the shared prefix and the sample's own tokens: this
// kernel attends all of a group's query rows (members x query heads of one kv
// head) to the shared prefix in one pass, so each prefix block crosses HBM
// once per group instead of once per sample; the split kernel handles each
// sample's own tokens and the log-sum-exp reduce merges both.
//
// Work item: (group, kv head, partition of T prefix tokens). Per CTA, one
// producer warp streams the item's 16-token K/V jobs by TMA into a ring of R
// stages shared by the CTA; four consumer warps read every stage, each for its
// own n-tiles of 8 query rows (row = member * group + head), so their results
// never need merging: at the end of an item each warp writes its rows'
// normalised partials (and max, sum) to the workspace slot of the partition.
// The stage is released when all four consumer warps have read it (an
// mbarrier with four arrivals); every wait is time-bounded.
#pragma once

#include "pa_decode.cuh"

namespace pa {

constexpr int kCascadeConsumers = 4;
constexpr int kCascadeStages = 6;

struct CascadeLayout {
  unsigned stage_bytes, full_off, empty_off, ok_off, sched_off, misc_off, total;
};

__host__ __device__ inline CascadeLayout cascade_layout(int D, int esize, int num_groups) {
  CascadeLayout L;
  L.stage_bytes = 2u * kJobTokens * D * esize;
  unsigned off = kCascadeStages * L.stage_bytes;
  L.full_off = off;
  off += kCascadeStages * 8;
  L.empty_off = off;
  off += kCascadeStages * 8;
  L.ok_off = off;
  off = round_up(off + kCascadeStages, 16);
  L.sched_off = off;
  off += (num_groups + 1) * 4;
  off = round_up(off, 16);
  L.misc_off = off;
  off += 16;
  L.total = off + 1024;
  return L;
}

// NT: n-tiles of 8 query rows per consumer warp (rows per group <= 32 * NT).
template <typename DT, int D, int NT>
__global__ void __launch_bounds__((kCascadeConsumers + 1) * 32)
    cascade_prefix_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                          const DecodeParams p) {
  pdl_begin();
  constexpr int WC = kCascadeConsumers, R = kCascadeStages, JT = kJobTokens, E = (int)sizeof(DT);
  constexpr int TILE = JT * D * E;
  constexpr int NREG = D * E / 128;
  constexpr int BOX_X = 128 / E;
  static_assert(sizeof(DT) == 2 && D % 16 == 0, "cascade prefix pass: 16-bit caches");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const CascadeLayout L = cascade_layout(D, E, p.num_groups);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full_off);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty_off);
  volatile uint8_t* stage_ok = smem + L.ok_off;
  int* pstart = reinterpret_cast<int*>(smem + L.sched_off);  // first item of each group, [num_groups + 1]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc_off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], WC);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
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
  __syncthreads();
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

  if (warp == WC) {
    // ------------------------------- producer -------------------------------
    int n = 0;
    if (lane == 0) {
      PItem it;
      for (int k = 0; get(k, it) && !*abort_flag; ++k) {
        const int32_t* table = p.block_tables + (long long)it.s0 * p.max_blocks;
        for (int u = it.t0 / JT; u < (it.t1 + JT - 1) / JT; ++u, ++n) {
          const int stage = n % R;
          if (!mbar_wait_bounded(&empty[stage], ((n / R) & 1) ^ 1, abort_flag, p.err, kWaitLimitNs)) break;
          const int tok = u * JT, blk = tok >> p.block_shift;
          const long long phys = __ldg(table + blk);
          if (phys < 0 || phys >= p.num_blocks) {
            atomicOr(p.err, kErrBlockId);
            stage_ok[stage] = 0;
            mbar_arrive(&full[stage]);
            continue;
          }
          stage_ok[stage] = 1;
          uint8_t* kdst = smem + stage * L.stage_bytes;
          const int r0 = tok - (blk << p.block_shift);
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(&full[stage], 2 * TILE);
#pragma unroll
          for (int rg = 0; rg < NREG; ++rg) {
            tma_load_tile(kdst + rg * JT * 128, &kmap, p, rg * BOX_X, phys, it.kv, r0, &full[stage]);
            tma_load_tile(kdst + TILE + rg * JT * 128, &vmap, p, rg * BOX_X, phys, it.kv, r0, &full[stage]);
          }
        }
      }
      // let the last copies land before the block can exit
      const int first = n - R > 0 ? n - R : 0;
      for (int m = first; m < n; ++m) mbar_wait_bounded(&full[m % R], (m / R) & 1, nullptr, p.err, kDrainLimitNs);
    }
    __syncwarp();
    return;
  }

  // --------------------------------- consumers ---------------------------------
  const float NEG_INF = -__int_as_float(0x7f800000);
  const int g = lane >> 2, t4 = lane & 3;
  int n = 0;
  PItem it;
  for (int k = 0; get(k, it); ++k) {
    const int rows = it.members * p.group;
    uint32_t qf[NT][D / 16][2];
    bool active[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int nt = warp + WC * j;
      active[j] = nt * 8 < rows;
      const int r = nt * 8 + g;  // this lane's B-operand row
      const bool ok = r < rows;
      const DT* qr = reinterpret_cast<const DT*>(p.q) +
                     ((long long)(it.s0 + (ok ? r / p.group : 0)) * p.H + it.kv * p.group + (ok ? r % p.group : 0)) * D;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qf[j][ks][0] = ok ? __ldg(reinterpret_cast<const uint32_t*>(qr + ks * 16 + 2 * t4)) : 0u;
        qf[j][ks][1] = ok ? __ldg(reinterpret_cast<const uint32_t*>(qr + ks * 16 + 2 * t4 + 8)) : 0u;
      }
    }
    float o[NT][D / 16][4];
    float m0[NT], m1[NT], l0[NT], l1[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      m0[j] = m1[j] = NEG_INF;
      l0[j] = l1[j] = 0.f;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) o[j][mt][0] = o[j][mt][1] = o[j][mt][2] = o[j][mt][3] = 0.f;
    }
    for (int u = it.t0 / JT; u < (it.t1 + JT - 1) / JT; ++u, ++n) {
      const int stage = n % R;
      bool ok = mbar_wait_bounded(&full[stage], (n / R) & 1, abort_flag, p.err, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok) && stage_ok[stage];
      if (ok) {
        const uint32_t kt = smem_u32(smem + stage * L.stage_bytes), vt = kt + TILE;
        const int nv = min(JT, it.t1 - u * JT);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          if (!active[j]) continue;
          float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int ks = 0; ks < D / 16; ks += 2) {
            uint32_t a[4], b[4];
            ldsm_x4(a, kt + sw128_offset(lane & 15, ks * 2 + (lane >> 4), JT));
            ldsm_x4(b, kt + sw128_offset(lane & 15, ks * 2 + 2 + (lane >> 4), JT));
            Mma<DT>::run(sc, a, qf[j][ks][0], qf[j][ks][1]);
            Mma<DT>::run(sd, b, qf[j][ks + 1][0], qf[j][ks + 1][1]);
          }
          float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tok = g + ((e >> 1) << 3);
            const float z = tok < nv ? (sc[e] + sd[e]) * p.scale_log2 : NEG_INF;
            sc[e] = z;
            if (e & 1) mx1 = fmaxf(mx1, z); else mx0 = fmaxf(mx0, z);
          }
#pragma unroll
          for (int o2 = 4; o2 < 32; o2 <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
          }
          const float mn0 = fmaxf(m0[j], mx0), mn1 = fmaxf(m1[j], mx1);
          const float c0 = exp2f(m0[j] - mn0), c1 = exp2f(m1[j] - mn1);
          m0[j] = mn0;
          m1[j] = mn1;
          sc[0] = exp2f(sc[0] - mn0);
          sc[1] = exp2f(sc[1] - mn1);
          sc[2] = exp2f(sc[2] - mn0);
          sc[3] = exp2f(sc[3] - mn1);
          l0[j] = l0[j] * c0 + sc[0] + sc[2];
          l1[j] = l1[j] * c1 + sc[1] + sc[3];
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            o[j][mt][0] *= c0;
            o[j][mt][2] *= c0;
            o[j][mt][1] *= c1;
            o[j][mt][3] *= c1;
          }
          // P as hi + lo 16-bit parts (see the decode kernel)
          const uint32_t h01 = Mma<DT>::pack(sc[0], sc[1]), h23 = Mma<DT>::pack(sc[2], sc[3]);
          float r0, r1, r2, r3;
          unpack2(h01, (DT*)nullptr, r0, r1);
          unpack2(h23, (DT*)nullptr, r2, r3);
          const uint32_t b0 = movmatrix_trans(h01), b1 = movmatrix_trans(h23);
          const uint32_t e0 = movmatrix_trans(Mma<DT>::pack(sc[0] - r0, sc[1] - r1));
          const uint32_t e1 = movmatrix_trans(Mma<DT>::pack(sc[2] - r2, sc[3] - r3));
          const int vtok = ((lane >> 4) << 3) + (lane & 7);
          const int tlo = 2 * t4;
          const uint32_t mlo = (tlo < nv ? 0x0000ffffu : 0u) | (tlo + 1 < nv ? 0xffff0000u : 0u);
          const uint32_t mhi = (tlo + 8 < nv ? 0x0000ffffu : 0u) | (tlo + 9 < nv ? 0xffff0000u : 0u);
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            uint32_t a[4];
            ldsm_x4_trans(a, vt + sw128_offset(vtok, mt * 2 + ((lane >> 3) & 1), JT));
            if (nv < JT) {
              a[0] &= mlo;
              a[1] &= mlo;
              a[2] &= mhi;
              a[3] &= mhi;
            }
            Mma<DT>::run(o[j][mt], a, b0, b1);
            Mma<DT>::run(o[j][mt], a, e0, e1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
    // this warp's rows: partials to the workspace slot of the partition
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) {
        l0[j] += __shfl_xor_sync(0xffffffffu, l0[j], o2);
        l1[j] += __shfl_xor_sync(0xffffffffu, l1[j], o2);
      }
      if (!active[j]) continue;
      const int nt = warp + WC * j;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int r = nt * 8 + 2 * t4 + half;
        if (r >= rows) continue;
        const float l = half ? l1[j] : l0[j], m = half ? m1[j] : m0[j];
        const float inv = l > 0.f ? p.v_scale / l : 0.f;
        const long long wrow = ((long long)(it.s0 + r / p.group) * p.H + it.kv * p.group + r % p.group) *
                                   p.max_partitions + it.part;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          p.ws_o[wrow * D + mt * 16 + g] = o[j][mt][half] * inv;
          p.ws_o[wrow * D + mt * 16 + g + 8] = o[j][mt][2 + half] * inv;
        }
        if (g == 0) {
          p.ws_m[wrow] = m;
          p.ws_l[wrow] = l;
        }
      }
    }
  }
}

}  // namespace pa
