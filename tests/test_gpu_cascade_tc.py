"""The tcgen05 prefix pass of pa_decode_cascade (groups of 17-128 query rows).

Groups of 5-16 samples x 4 query heads (or 3-8 x 8) take the M = 64 tile,
groups of 17-32 x 4 (or 9-16 x 8) the M = 128 tile, so the shared-prefix decode
runs its prefix pass on the fifth-generation tensor cores; groups of up to 16
rows take the mma.sync pass. Query groups of 3, 5, 6 and 7 heads leave the
tile's Q box short of M rows (group x (M / group)).
Each case is checked against the oracle (which sees the pool before any kernel
ran) and against plain pa_decode of the same batch: long prefixes (many tiles
and several items per CTA), a last partition of one 16-token job, both block
sizes, fp16 and bf16, NHD pools, head_dim 64, out-of-pool block ids in a shared
prefix, and a score range wide enough to move a row's reference max.
"""
import os
import sys

import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import gpu_harness as H  # noqa: E402
from paged_kv_cache_04_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


def _cascade(pa, wl, out_dtype=torch.float32, T=256):
    dev = wl.q.device
    gs_l, pl_l = wl.meta["group_starts"], wl.meta["prefix_lens"]
    gs = torch.tensor(gs_l, dtype=torch.int32, device=dev)
    pl = torch.tensor(pl_l, dtype=torch.int32, device=dev)
    gmax = max(b - a for a, b in zip(gs_l[:-1], gs_l[1:]))
    mpre, mctx = max(pl_l), wl.max_context
    # poisoned (0x7f bytes: finite, huge sums and maxima): every slot the reduce merges must be written
    ws = torch.full((pa.pa_decode_cascade_workspace_bytes(wl.S, wl.H, wl.d, mpre, mctx, T),), 0x7F, dtype=torch.uint8,
                     device=dev)
    out = torch.empty(wl.q.shape, dtype=out_dtype, device=dev)
    pa.pa_decode_cascade(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, gs, pl,
                         gmax, mpre, mctx, T, ws, layout=wl.layout)
    return out


def _writes(pa, wl):
    if wl.copy_pairs is not None and wl.copy_pairs.numel():
        pa.pa_copy_blocks([wl.k_cache], [wl.v_cache], wl.copy_pairs)
    pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping, layout=wl.layout)


CASES = [
    # (samples, H, G, d, B, dtype, prefix, layout, cow)
    (16, 32, 8, 128, 16, torch.bfloat16, 1040, "HND", False),  # last partition: one 16-token job
    (16, 32, 8, 128, 32, torch.bfloat16, 1100, "HND", True),
    (16, 32, 8, 128, 16, torch.float16, 1700, "NHD", True),
    (8, 64, 8, 128, 16, torch.bfloat16, 900, "HND", False),    # 8 samples x group 8
    (12, 32, 8, 128, 16, torch.bfloat16, 777, "HND", True),    # 48 rows: a partly filled tile
    (16, 32, 8, 64, 16, torch.bfloat16, 1300, "HND", False),   # head_dim 64
    (16, 16, 4, 64, 32, torch.float16, 1500, "NHD", False),
    (8, 32, 8, 128, 16, torch.bfloat16, 1100, "HND", True),    # 32 rows: the 64 x 8-sample batch's groups
    (5, 32, 8, 128, 16, torch.float16, 900, "NHD", False),     # 20 rows
    (17, 8, 8, 128, 16, torch.bfloat16, 700, "HND", False),    # MHA, 17 rows: the smallest M = 64 group
    (4, 32, 8, 128, 32, torch.bfloat16, 800, "HND", True),     # 16 rows: the mma.sync pass
    # M = 128 tiles
    (32, 32, 8, 128, 16, torch.bfloat16, 1040, "HND", True),   # 128 rows
    (16, 64, 8, 128, 32, torch.float16, 1300, "NHD", False),   # 16 samples x group 8
    (20, 32, 8, 128, 16, torch.bfloat16, 700, "HND", False),   # 80 rows: a partly filled tile
    (32, 32, 8, 64, 16, torch.float16, 900, "NHD", True),      # head_dim 64
    # MHA and group 2: the vector-path suffix passes, and row counts that are not multiples of 16
    (8, 8, 8, 128, 16, torch.float16, 600, "HND", True),       # MHA, 8 rows (mma.sync prefix pass)
    (40, 8, 8, 128, 16, torch.bfloat16, 700, "HND", False),    # MHA, 40 rows (M = 64)
    (100, 8, 8, 128, 32, torch.float16, 500, "NHD", True),     # MHA, 100 rows (M = 128)
    (20, 16, 8, 128, 16, torch.bfloat16, 800, "HND", False),   # group 2, 40 rows
    # groups that do not divide the tile: the Q box holds group x (M / group) rows
    (8, 24, 8, 128, 16, torch.bfloat16, 900, "HND", False),    # group 3, 24 rows: a 63-row box
    (30, 24, 8, 128, 16, torch.float16, 700, "NHD", True),     # group 3, 90 rows: a 126-row box (M = 128)
    (10, 48, 8, 128, 16, torch.bfloat16, 800, "HND", False),   # group 6, 60 rows: a 60-row box
    (7, 40, 8, 64, 16, torch.bfloat16, 600, "HND", True),      # group 5, 35 rows, head_dim 64
    (18, 56, 8, 128, 32, torch.float16, 700, "HND", False),    # group 7, 126 rows (M = 128)
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"s{c[0]}H{c[1]}G{c[2]}d{c[3]}B{c[4]}{str(c[5])[6:]}"
                                                      f"p{c[6]}{c[7]}{'cow' if c[8] else ''}")
def test_tc_prefix_matches_oracle(pa, cuda_device, case):
    samples, Hh, G, d, B, dt, prefix, layout, cow = case
    wl = workloads.shared_prefix(device=cuda_device, prompts=3, samples=samples, prefix=prefix, tail_hi=120,
                                 cow=cow, H=Hh, G=G, d=d, B=B, dtype=dt)
    if layout == "NHD":
        wl = workloads.to_nhd(wl)
    ref = H.Pristine(wl).decode()
    _writes(pa, wl)
    out = _cascade(pa, wl)
    H.check_close(out, ref, torch.float32, f"tc cascade {case}")
    plain = torch.empty(wl.q.shape, dtype=torch.float32, device=cuda_device)
    pa.pa_decode(plain, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                 layout=wl.layout)
    assert (out - plain).abs().max().item() <= 2e-3
    assert pa.pa_get_error() == 0


@pytest.mark.parametrize("samples", [16, 32], ids=["m64", "m128"])
def test_tc_prefix_rescales(pa, cuda_device, samples):
    """q scaled by 40: scores spread over tens of log2 units, so a row's reference
    max moves many times within an item (and the accumulator is rescaled)."""
    wl = workloads.shared_prefix(device=cuda_device, prompts=2, samples=samples, prefix=2000, tail_hi=50)
    wl.q.mul_(40.0)
    ref = H.Pristine(wl).decode()
    _writes(pa, wl)
    out = _cascade(pa, wl, T=1024)
    H.check_close(out, ref, torch.float32, "tc cascade rescale")
    assert pa.pa_get_error() == 0


def test_tc_prefix_bf16_output_and_full_size(pa, cuda_device):
    """The 32-prompt x 16-sample benchmark batch (prefix 2048, partitions of 512),
    bf16 output, sampled sequences against the oracle."""
    wl = workloads.shared_prefix(device=cuda_device, prompts=32, samples=16)
    seqs = H.sample_seqs(wl, 8)
    P = H.Pristine(wl, seqs)
    ref = P.decode()
    _writes(pa, wl)
    out = _cascade(pa, wl, out_dtype=torch.bfloat16, T=512)
    H.check_close(out[seqs], ref, torch.bfloat16, "tc cascade full")
    assert pa.pa_get_error() == 0


def test_tc_prefix_skips_out_of_pool_blocks(pa, cuda_device):
    """An out-of-pool id in a shared prefix is recorded, and its 16 tokens are left
    out of every member's attention (as pa_decode leaves them out)."""
    wl = workloads.shared_prefix(device=cuda_device, prompts=2, samples=16, prefix=640, tail_hi=30)
    _writes(pa, wl)
    wl.block_tables[0:16, 5] = wl.num_blocks + 7  # block 5 of prompt 0's shared prefix, in all its members
    out = _cascade(pa, wl)
    assert pa.pa_get_error() & 1
    plain = torch.empty(wl.q.shape, dtype=torch.float32, device=cuda_device)
    pa.pa_decode(plain, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    assert pa.pa_get_error() & 1  # (read and cleared)
    assert (out - plain).abs().max().item() <= 2e-3
