"""Shared-memory budgets of the decode kernel, computed on the host.

The kernel's shared-memory map (make_layout in csrc/pa_decode.cuh) is a plain
host/device function: this test compiles it into a small host program and
checks how many CTAs of each configuration fit one SM. GB300 gives an SM
228 KiB of shared memory and reserves 1 KiB of it per resident CTA. The
measured speeds depend on these counts (two CTAs per SM for 16-bit tensor-core
decode, three for MHA and E4M3), so a layout change that costs a CTA fails here
before it shows up as a slower benchmark. No GPU is needed.
"""
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SM_BYTES = 228 * 1024
RESERVED_PER_CTA = 1024

PROGRAM = r"""
#include <cstdio>
#include "pa_decode.cuh"
#include "pa_cascade_tc.cuh"
using namespace pa;
// Plain mode keeps the sort order of its own items only, sized as the launcher
// sizes it: 152 SMs, 8 kv heads (the MHA rows: 40, the OPT-13B shape).
template <typename C, typename QT, int D, int PATH>
SmemLayout layout_of(int group, int split, int S) {
  const int kv_heads = PATH == kPathVecMha ? 40 : 8;
  return make_layout(C::W, C::R, D, C::E, (int)sizeof(QT), group, PATH, split != 0, S, C::JPS, false,
                     split ? 0 : plain_order_cap(S, kv_heads, 152));
}
template <typename DT, typename QT, int D, int PATH>
void row(const char* name, int group, int split, int S) {
  const SmemLayout L = split ? layout_of<StageCfg<DT, D, PATH, kModeSplit>, QT, D, PATH>(group, 1, S)
                             : layout_of<StageCfg<DT, D, PATH, kModePlain>, QT, D, PATH>(group, 0, S);
  printf("%s %d %d %d %u\n", name, group, split, S, L.total);
}
// the shared-prefix suffix pass (split slot 2 in the key): no merge area, and
// each sequence's first own token beside the sort order
template <typename DT, typename QT, int D, int PATH>
void row_suffix(const char* name, int group, int S) {
  using C = StageCfg<DT, D, PATH, kModeSuffix>;
  const SmemLayout L = make_layout(C::W, C::R, D, C::E, (int)sizeof(QT), group, PATH, false, S, C::JPS, true);
  printf("%s %d 2 %d %u\n", name, group, S, L.total);
}
int main() {
  for (int S : {64, 256, 752, 2048})
    for (int sp : {0, 1})
      for (int g : {1, 4, 8}) {
        row<__nv_bfloat16, __nv_bfloat16, 128, kPathMma>("mma16_d128", g, sp, S);
        row<fp8e4m3, __nv_bfloat16, 128, kPathMma>("fp8_d128", g, sp, S);
        row<__nv_bfloat16, __nv_bfloat16, 256, kPathMma>("mma16_d256", g, sp, S);
        if (!sp) {  // plain decode at groups of 5-8: merged four heads per round
          row<__nv_bfloat16, __nv_bfloat16, 128, kPathMmaG8>("mma16g8_d128", g, sp, S);
          row<fp8e4m3, __nv_bfloat16, 128, kPathMmaG8>("fp8g8_d128", g, sp, S);
          row<__nv_bfloat16, __nv_bfloat16, 256, kPathMmaG8>("mma16g8_d256", g, sp, S);
        }
        // (16-bit MHA split decode takes the tensor cores: the mma16 split rows at group 1)
        if (!sp) row<__half, __half, 128, kPathVecMha>("mha_d128", 1, sp, S);
        row<__nv_bfloat16, __nv_bfloat16, 256, kPathVec>("vec_d256", 2, sp, S);
      }
  for (int S : {512, 1024, 2048}) {
    row_suffix<__nv_bfloat16, __nv_bfloat16, 128, kPathMma>("sfx_mma16_d128", 4, S);
    row_suffix<__nv_bfloat16, __nv_bfloat16, 64, kPathMma>("sfx_mma16_d64", 4, S);
    row_suffix<__half, __half, 128, kPathVecMha>("sfx_mha_d128", 1, S);
  }
  // the tcgen05 prefix pass of shared-prefix decode: (groups) in the group slot
  for (int D : {64, 128})
    for (int MR : {64, 128})
      for (int g : {32, 512, 2048})
        printf("tc_d%d_m%d %d 0 0 %u\n", D, MR, g, tc_layout(D, g, MR).total);
  // plain mode's per-CTA order capacity: (S, kv heads) in the group and S slots
  for (int S : {1, 2, 7, 64, 151, 152, 153, 256, 1000, 2048})
    for (int G : {1, 2, 8, 40, 152, 153, 512})
      printf("cap %d 0 %d %d\n", G, S, plain_order_cap(S, G, 152));
}
"""


@pytest.fixture(scope="module")
def totals(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("smem")
    src, exe = d / "layout.cu", d / "layout"
    src.write_text(PROGRAM)
    subprocess.run([nvcc, "-std=c++17", "--expt-relaxed-constexpr", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "paged_kv_cache_04_gb300", "csrc"),
                    str(src), "-o", str(exe)], check=True, capture_output=True, timeout=300)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=60).stdout
    res = {}
    for line in out.splitlines():
        if line.startswith("cap "):
            _, g, _, S, cap = line.split()
            res[("cap", int(g), int(S))] = int(cap)
            continue
        name, g, sp, S, total = line.split()
        res[(name, int(g), int(sp), int(S))] = int(total)
    return res


def ctas_per_sm(total):
    return SM_BYTES // (total + RESERVED_PER_CTA)


# (configuration, group, split, sequences) -> CTAs per SM the measured kernels run with
HOLDS = [
    (("mma16_d128", 4, 0, 256), 2),   # the Llama batch (plain decode)
    (("mma16_d128", 4, 0, 2048), 2),
    (("mma16_d128", 4, 1, 2048), 2),  # split decode
    (("mma16_d128", 8, 1, 2048), 2),  # 70B-shaped split decode (group 8)
    (("fp8_d128", 4, 0, 256), 3),     # E4M3 plain decode
    (("fp8_d128", 4, 0, 752), 3),
    (("fp8_d128", 4, 0, 2048), 3),    # (the order of its own items only, not the batch's)
    (("fp8_d128", 8, 1, 2048), 3),    # E4M3 split decode
    (("mha_d128", 1, 0, 2048), 3),    # OPT-13B-shaped MHA
    (("mma16_d128", 1, 1, 2048), 2),  # 16-bit MHA split decode (the tensor-core path at group 1)
    (("mma16_d256", 4, 0, 2048), 2),  # head_dim 256: one stage per warp, two CTAs
    (("mma16g8_d128", 8, 0, 256), 2),  # plain decode at group 8 (64 q / 8 kv heads): merge rounds
    (("mma16g8_d128", 8, 0, 2048), 2),
    (("fp8g8_d128", 8, 0, 256), 3),    # E4M3 plain decode at group 8
    (("mma16g8_d256", 8, 0, 2048), 2),
    (("vec_d256", 2, 0, 2048), 2),
    (("sfx_mma16_d128", 4, 2, 512), 2),   # shared-prefix suffix pass (the 64 x 8-sample batch)
    (("sfx_mma16_d128", 4, 2, 2048), 2),
    (("sfx_mha_d128", 1, 2, 1024), 3),   # (each sequence's first own token kept up to 1,024)
    (("sfx_mha_d128", 1, 2, 2048), 3),
    (("tc_d128_m64", 512, 0, 0), 2),   # tcgen05 prefix pass, 17-64 rows per group
    (("tc_d128_m64", 2048, 0, 0), 2),
    (("tc_d128_m128", 2048, 0, 0), 2),  # 65-128 rows per group
    (("tc_d64_m64", 2048, 0, 0), 2),    # (tensor memory caps this kernel at two CTAs per SM)
]

# (The tcgen05 prefix pass's group scan, 4 bytes per group, keeps two CTAs per
# SM up to about 4,000 groups; the cascade call takes at most 2,048.)


@pytest.mark.parametrize("key,want", HOLDS, ids=[f"{k[0]}-g{k[1]}-split{k[2]}-S{k[3]}" for k, _ in HOLDS])
def test_ctas_per_sm(totals, key, want):
    assert ctas_per_sm(totals[key]) >= want, f"{key}: {totals[key]} bytes"


def test_no_layout_exceeds_the_per_cta_limit(totals):
    over = {k: v for k, v in totals.items() if k[0] != "cap" and v > 227 * 1024}
    assert not over, over


def _serpentine_items(S, G, grid):
    """Items of each CTA under the kernel's deal (item k*grid + b for even k,
    k*grid + grid - 1 - b for odd k), counted by brute force."""
    i = np.arange(S * G)
    k, pos = i // grid, i % grid
    cta = np.where(k % 2 == 0, pos, grid - 1 - pos)
    return int(np.bincount(cta, minlength=grid).max())


def test_plain_order_capacity_covers_every_grid(totals):
    """The per-CTA order holds every item a CTA is dealt, for every grid the
    launcher can pick (152 SMs x 1-3 CTAs, capped at the item count), except
    past S entries, where the kernel takes the batch order instead."""
    caps = {k[1:]: v for k, v in totals.items() if k[0] == "cap"}
    assert caps
    for (G, S), cap in caps.items():
        assert 1 <= cap <= max(S, 1)
        for per_sm in (1, 2, 3):
            grid = min(152 * per_sm, S * G)
            need = _serpentine_items(S, G, grid)
            assert need == -(-(S * G) // grid)
            if cap < S or G <= 152:
                assert need <= cap, (S, G, grid, need, cap)
