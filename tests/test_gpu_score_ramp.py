"""GPU parity on scores that climb (or fall) steadily along each sequence.

Each sequence's K rows get a component along a per-kv-head unit vector u that
grows linearly with the token's logical position, and every query points
mostly along u, so the base-2 scores rise by about `slope` per token on top of
a little noise. With a gentle slope a warp's running max trails the new
scores by a few units for several jobs and then jumps; with a steep one it
jumps on most jobs; with a falling ramp the first job holds the max for the
whole item. All three are the same softmax (online-softmax rule, Month 2 ·
PagedAttention §2.1 and CS349E Lecture 7 notes §4.2), compared with the
float64 oracle on the same pool.
"""
import math
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import gpu_harness as H  # noqa: E402
from oracle import fp8 as ofp8  # noqa: E402
from paged_kv_cache_04_gb300 import workloads  # noqa: E402

CTX = [1, 17, 300, 1000, 2500, 4100, 64, 777]
LOG2E = 1.4426950408889634
QN = 4.0  # length of the query's component along u


def _ramp(wl, slope, seed=11):
    """Add slope * t / (scale * log2 e * QN) * u[kv] to token t's K row, and make q QN u + noise / 4."""
    g = torch.Generator().manual_seed(seed)
    u = torch.randn((wl.G, wl.d), generator=g, dtype=torch.float64)
    u /= u.norm(dim=1, keepdim=True)
    dev = wl.k_cache.device
    grp = wl.H // wl.G
    q = wl.q.double() * 0.25 + QN * u.to(dev).repeat_interleave(grp, dim=0)[None]
    wl.q.copy_(q.to(wl.q.dtype))
    wl.k_cache.mul_(0.5)
    bt = wl.block_tables.cpu()
    ud = u.to(dev)
    for s, c in enumerate(wl.context_lens.cpu().tolist()):
        if c == 0:
            continue
        t = torch.arange(c)
        phys = bt[s, t // wl.B].long().to(dev)
        slot = (t % wl.B).to(dev)
        coef = (slope * t.double() / (wl.scale * LOG2E * QN)).to(dev)
        rows = wl.k_cache[phys, :, slot, :].double() + coef[:, None, None] * ud[None]
        wl.k_cache[phys, :, slot, :] = rows.to(wl.k_cache.dtype)


def _batch(dev, Hq, G, dtype):
    nb = sum(-(-c // 16) for c in CTX) + 7
    return workloads.batch_with_new_tokens("ramp", len(CTX), Hq, G, 128, 16, dtype, CTX, nb, dev,
                                           new_token=False)


SLOPES = [0.02, 0.1, -0.1]
SHAPES = [("gqa_bf16", 32, 8, torch.bfloat16), ("mha_fp16", 8, 8, torch.float16),
          ("g2_bf16", 8, 4, torch.bfloat16)]


@pytest.mark.gpu
@pytest.mark.parametrize("slope", SLOPES)
@pytest.mark.parametrize("name,Hq,G,dt", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("split", [False, True], ids=["plain", "split"])
def test_score_ramp_matches_oracle(pa, cuda_device, name, Hq, G, dt, slope, split):
    wl = _batch(cuda_device, Hq, G, dt)
    _ramp(wl, slope)
    ref = H.Pristine(wl).decode()
    out = H.gpu_step(pa, wl, out_dtype=torch.float32, split=split, partition=256)
    H.check_close(out, ref, torch.float32, f"ramp {name} slope={slope} split={split}")
    assert pa.pa_get_error() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("slope", SLOPES)
def test_score_ramp_fp8_matches_oracle(pa, cuda_device, slope):
    """The same ramps through an E4M3 pool (Llama shape, tensor-core path)."""
    base = _batch(cuda_device, 32, 8, torch.bfloat16)
    _ramp(base, slope)
    wl = workloads.to_fp8(base)
    ks, vs = wl.meta["k_scale"], wl.meta["v_scale"]
    ref = ofp8.decode(wl.q.cpu(), wl.k_cache.cpu().numpy(), wl.v_cache.cpu().numpy(), wl.block_tables.cpu(),
                      wl.context_lens.cpu(), wl.scale, ks, vs)
    out = torch.empty(wl.q.shape, dtype=torch.float32, device=cuda_device)
    pa.pa_decode_fp8(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, ks, vs)
    H.check_close(out, ref, torch.float32, f"ramp fp8 slope={slope}")
    assert pa.pa_get_error() == 0


def test_ramp_really_moves_the_max():
    """Host check of the construction (no GPU): the oracle's base-2 scores of the
    longest sequence rise by about `slope` per token, so the running max moves."""
    wl = _batch("cpu", 8, 8, torch.float32)
    _ramp(wl, 0.1)
    s = CTX.index(max(CTX))
    c = CTX[s]
    t = torch.arange(c)
    phys = wl.block_tables[s, t // wl.B].long()
    k = wl.k_cache[phys, 0, t % wl.B, :].double()
    z = (k @ wl.q[s, 0].double()) * wl.scale * LOG2E
    fit = np.polyfit(np.arange(c), z.numpy(), 1)[0]
    assert abs(fit - 0.1) < 0.01
