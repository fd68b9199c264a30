"""FP8 (E4M3) KV cache on the GPU against the oracle: quantising cache write
bit-exact, attention (plain and split, tensor-core and vector paths) within the
attention tolerance."""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import gpu_harness as H  # noqa: E402
from oracle import fp8 as ofp8  # noqa: E402
from paged_kv_cache_04_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


def _fp8_step(pa, wl, out_dtype, split=False, T=512):
    ks, vs = wl.meta["k_scale"], wl.meta["v_scale"]
    if wl.slot_mapping is not None:
        pa.pa_reshape_and_cache_fp8(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping, ks, vs)
    out = torch.empty(wl.q.shape, dtype=out_dtype, device=wl.q.device)
    if split:
        mctx = wl.max_context
        ws = torch.empty(pa.pa_decode_split_workspace_bytes(wl.S, wl.H, wl.d, mctx, T), dtype=torch.uint8,
                         device=wl.q.device)
        pa.pa_decode_split_fp8(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                               ks, vs, mctx, T, ws)
    else:
        pa.pa_decode_fp8(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, ks, vs)
    return out


def _oracle(wl_host_k, wl_host_v, wl, seqs=None):
    """Oracle: quantising write of the new tokens, then scaled attention (host copies only)."""
    ks, vs = wl.meta["k_scale"], wl.meta["v_scale"]
    k, v = wl_host_k, wl_host_v
    if wl.slot_mapping is not None:
        k, v = ofp8.reshape_and_cache(wl.new_key.cpu(), wl.new_value.cpu(), k, v, wl.slot_mapping.cpu(), ks, vs)
    sel = slice(None) if seqs is None else seqs
    return ofp8.decode(wl.q.cpu()[sel], k, v, wl.block_tables.cpu()[sel], wl.context_lens.cpu()[sel],
                       wl.scale, ks, vs), k, v


SHAPES = [("llama", 32, 8, torch.bfloat16), ("mha", 16, 16, torch.float16), ("g2", 8, 4, torch.bfloat16),
          ("g3", 12, 4, torch.float16), ("g6", 48, 8, torch.bfloat16), ("g8", 64, 8, torch.float16)]


@pytest.mark.parametrize("name,Hq,G,qt", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("split", [False, True])
def test_fp8_decode_matches_oracle(pa, cuda_device, name, Hq, G, qt, split):
    ctx = [1, 15, 16, 17, 100, 513, 1500, 40]
    nb = sum(-(-c // 16) for c in ctx) + 9
    base = workloads.batch_with_new_tokens("f8", len(ctx), Hq, G, 128, 16, qt, ctx, nb, cuda_device)
    wl = workloads.to_fp8(base)
    # NaN codes in every free slot: masking must keep them out
    H.poison_free_slots(wl, value=0x7F)
    ref, kref, vref = _oracle(wl.k_cache.cpu().numpy(), wl.v_cache.cpu().numpy(), wl)
    out = _fp8_step(pa, wl, torch.float32, split=split, T=64)
    H.check_close(out, ref, torch.float32, f"fp8 {name} split={split}")
    assert np.array_equal(wl.k_cache.cpu().numpy(), kref) and np.array_equal(wl.v_cache.cpu().numpy(), vref)
    assert pa.pa_get_error() == 0


def test_fp8_full_size_llama_sampled(pa, cuda_device):
    """The benchmark batch with an E4M3 pool; sampled sequences against the oracle
    on a compacted copy of just their blocks (taken before any kernel ran)."""
    wl = workloads.to_fp8(workloads.llama8b(device=cuda_device))
    seqs = H.sample_seqs(wl, 8)
    P = H.Pristine(wl, seqs)
    ks, vs = wl.meta["k_scale"], wl.meta["v_scale"]
    k, v = ofp8.reshape_and_cache(P.new[0], P.new[1], P.k.numpy(), P.v.numpy(), P.new[2], ks, vs)
    ref = ofp8.decode(P.q, k, v, P.bt, P.ctx, wl.scale, ks, vs)
    out = _fp8_step(pa, wl, torch.bfloat16)
    H.check_close(out[seqs], ref, torch.bfloat16, "fp8 llama8b full")
    out32 = _fp8_step(pa, wl, torch.float32)
    assert torch.equal(out, out32.to(torch.bfloat16))
    assert pa.pa_get_error() == 0


def test_fp8_large_batch_every_sequence(pa, cuda_device):
    """2,048 sequences, the largest batch the kernel orders longest first, where
    E4M3 plain decode still runs three CTAs per SM (each CTA keeps the order of
    its own items only): every sequence against the oracle, the output filled
    with NaN first so that an item dealt to no CTA shows."""
    S = 2048
    ctx = [int(x) for x in torch.randint(1, 97, (S,), generator=torch.Generator().manual_seed(11))]
    nb = sum(-(-c // 16) for c in ctx) + 9
    wl = workloads.to_fp8(workloads.batch_with_new_tokens("f8big", S, 32, 8, 128, 16, torch.bfloat16, ctx, nb,
                                                          cuda_device))
    ref, _, _ = _oracle(wl.k_cache.cpu().numpy(), wl.v_cache.cpu().numpy(), wl)
    ks, vs = wl.meta["k_scale"], wl.meta["v_scale"]
    pa.pa_reshape_and_cache_fp8(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping, ks, vs)
    out = torch.full(wl.q.shape, float("nan"), dtype=torch.float32, device=cuda_device)
    pa.pa_decode_fp8(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, ks, vs)
    H.check_close(out, ref, torch.float32, "fp8 S=2048")
    assert pa.pa_get_error() == 0


def test_fp8_cache_write_bit_exact_all_dtypes(pa, cuda_device):
    g = torch.Generator(device=cuda_device).manual_seed(3)
    for dt in (torch.float32, torch.float16, torch.bfloat16):
        key = (torch.randn(50, 8, 128, device=cuda_device, generator=g) * 30).to(dt)  # some saturate
        val = torch.randn(50, 8, 128, device=cuda_device, generator=g).to(dt)
        key[0, 0, :4] = torch.tensor([float("nan"), 1e6, -1e6, 0.0])
        kc = torch.zeros(20, 8, 16, 128, dtype=torch.uint8, device=cuda_device)
        vc = torch.zeros_like(kc)
        slots = torch.randperm(320, device=cuda_device)[:50].to(torch.int64)
        slots[7] = -1
        pa.pa_reshape_and_cache_fp8(key, val, kc, vc, slots, 0.37, 0.011)
        rk, rv = ofp8.reshape_and_cache(key.cpu(), val.cpu(), np.zeros((20, 8, 16, 128), np.uint8),
                                        np.zeros((20, 8, 16, 128), np.uint8), slots.cpu(), 0.37, 0.011)
        assert np.array_equal(kc.cpu().numpy(), rk), dt
        assert np.array_equal(vc.cpu().numpy(), rv), dt
    assert pa.pa_get_error() == 0


def test_fp8_pools_copy_and_swap(pa, cuda_device):
    kc = torch.randint(0, 255, (30, 8, 16, 128), dtype=torch.uint8, device=cuda_device)
    vc = torch.randint(0, 255, (30, 8, 16, 128), dtype=torch.uint8, device=cuda_device)
    pairs = torch.tensor([[1, 20], [2, 21]], dtype=torch.int64, device=cuda_device)
    pa.pa_copy_blocks([kc], [vc], pairs)
    torch.cuda.synchronize()
    assert torch.equal(kc[20], kc[1]) and torch.equal(vc[21], vc[2])
    hk = torch.zeros(4, 8, 16, 128, dtype=torch.uint8).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    pa.pa_swap_blocks([hk], [hv], [kc], [vc], torch.tensor([[5, 3]], dtype=torch.int64, device=cuda_device))
    torch.cuda.synchronize()
    assert torch.equal(hk[3], kc[5].cpu()) and torch.equal(hv[3], vc[5].cpu())
