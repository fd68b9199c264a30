"""pa_decode_cascade (shared-prefix decode) against the oracle and against pa_decode."""
import os
import sys

import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import gpu_harness as H  # noqa: E402
from paged_kv_cache_04_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


def _cascade(pa, wl, group_starts, prefix_lens, out_dtype=None, T=512):
    dev = wl.q.device
    gs = torch.tensor(group_starts, dtype=torch.int32, device=dev)
    pl = torch.tensor(prefix_lens, dtype=torch.int32, device=dev)
    sizes = [b - a for a, b in zip(group_starts[:-1], group_starts[1:])]
    mpre, mctx = max(prefix_lens), wl.max_context
    # poisoned (0x7f bytes: finite, huge sums and maxima): every slot the reduce merges must be written
    ws = torch.full((pa.pa_decode_cascade_workspace_bytes(wl.S, wl.H, wl.d, mpre, mctx, T),), 0x7F, dtype=torch.uint8,
                     device=dev)
    out = torch.empty(wl.q.shape, dtype=out_dtype or wl.dtype, device=dev)
    pa.pa_decode_cascade(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, gs, pl,
                         max(sizes), mpre, mctx, T, ws)
    return out


def _writes(pa, wl):
    if wl.copy_pairs is not None and wl.copy_pairs.numel():
        pa.pa_copy_blocks([wl.k_cache], [wl.v_cache], wl.copy_pairs)
    pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping)


@pytest.mark.parametrize("cow", [False, True])
def test_cascade_matches_oracle_reduced(pa, cuda_device, cow):
    wl = workloads.shared_prefix(device=cuda_device, prompts=5, samples=8, prefix=1040, tail_hi=300, cow=cow)
    H.poison_free_slots(wl)
    ref = H.Pristine(wl).decode()
    _writes(pa, wl)
    out = _cascade(pa, wl, wl.meta["group_starts"], wl.meta["prefix_lens"], out_dtype=torch.float32, T=256)
    H.check_close(out, ref, torch.float32, f"cascade cow={cow}")
    plain = torch.empty_like(out)
    pa.pa_decode(plain, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    assert (plain - out).abs().max().item() <= 2e-4
    assert pa.pa_get_error() == 0


def test_cascade_full_size_sampled(pa, cuda_device):
    wl = workloads.shared_prefix(device=cuda_device, cow=True)
    seqs = [0, 3, 8, 200, 511]
    P = H.Pristine(wl, seqs)
    _writes(pa, wl)
    out = _cascade(pa, wl, wl.meta["group_starts"], wl.meta["prefix_lens"])
    H.check_close(out[seqs], P.decode(), torch.bfloat16, "cascade full")
    assert pa.pa_get_error() == 0


def test_cascade_degenerate_groupings(pa, cuda_device):
    """Singleton groups, a zero-length prefix, a prefix shorter than a block and
    group sizes that need two row tiles per warp (16 members x 4 heads)."""
    wl = workloads.shared_prefix(device=cuda_device, prompts=2, samples=16, prefix=100, tail_hi=40)
    ref = H.Pristine(wl).decode()
    _writes(pa, wl)
    k0, v0 = wl.k_cache.clone(), wl.v_cache.clone()
    out = _cascade(pa, wl, wl.meta["group_starts"], wl.meta["prefix_lens"], torch.float32, T=32)
    H.check_close(out, ref, torch.float32, "16 members")
    S = wl.S
    singles = list(range(S + 1))
    out1 = _cascade(pa, wl, singles, [0] * S, torch.float32, T=32)
    H.check_close(out1, ref, torch.float32, "singletons, no prefix")
    out2 = _cascade(pa, wl, [0, 16, 32], [7, 100], torch.float32, T=32)  # 7 rounds down to 0
    H.check_close(out2, ref, torch.float32, "short prefix")
    assert torch.equal(wl.k_cache, k0) and torch.equal(wl.v_cache, v0)
    assert pa.pa_get_error() == 0


def test_cascade_rejects_wide_groups(pa, cuda_device):
    wl = workloads.shared_prefix(device=cuda_device, prompts=1, samples=33, prefix=64, tail_hi=8)
    with pytest.raises(pa.PAError):
        _cascade(pa, wl, wl.meta["group_starts"], wl.meta["prefix_lens"])  # 33 x 4 rows > 128


@pytest.mark.parametrize("heads", [(32, 8), (8, 8)], ids=["gqa4", "mha"])
def test_cascade_batch_above_start_cache(pa, cuda_device, heads):
    """More than 1,024 sequences: the suffix pass finds each sequence's first own
    token by a search over the groups per item instead of its shared-memory copy."""
    Hh, G = heads
    prompts, samples = (65, 16) if Hh // G > 1 else (130, 8)
    wl = workloads.shared_prefix(device=cuda_device, prompts=prompts, samples=samples, prefix=160, tail_hi=64,
                                 H=Hh, G=G)
    assert wl.S > 1024
    ref = H.Pristine(wl).decode()
    _writes(pa, wl)
    out = _cascade(pa, wl, wl.meta["group_starts"], wl.meta["prefix_lens"], torch.float32, T=64)
    H.check_close(out, ref, torch.float32, f"cascade S={wl.S}")
    assert pa.pa_get_error() == 0
