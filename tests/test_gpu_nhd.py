"""NHD pools ([num_blocks, B, G, d]) on the GPU.

Every entry point that reads or writes a pool takes the layout. Each case is
checked against the oracle (which reads the NHD pool by its own indexing).
Attention over an NHD pool must also be bit-identical to the same batch
stored HND: the kernels stage the same 16-token tiles either way.
"""
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

SHAPES = [
    # (H, G, d, B, dtype): vector MHA path, vector GQA path, tensor-core path, both block sizes and head dims
    (4, 4, 64, 16, torch.float32), (8, 8, 128, 16, torch.float16), (8, 4, 64, 32, torch.float16),
    (32, 8, 128, 16, torch.bfloat16), (16, 2, 128, 32, torch.bfloat16), (32, 4, 64, 16, torch.bfloat16),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"H{s[0]}G{s[1]}d{s[2]}B{s[3]}{str(s[4])[6:]}")
@pytest.mark.parametrize("split", [False, True])
def test_nhd_matches_oracle_and_hnd(pa, cuda_device, shape, split):
    Hh, G, d, B, dt = shape
    ctx = [0, 1, B - 1, B, B + 1, 3 * B, 7 * B + 5, 200, 333, 1000]
    nb = sum(-(-c // B) for c in ctx) + 13
    hnd = workloads.batch_with_new_tokens("nhd", len(ctx), Hh, G, d, B, dt, ctx, nb, cuda_device)
    H.poison_free_slots(hnd)
    nhd = workloads.to_nhd(hnd)
    ref = H.Pristine(nhd).decode()
    out = H.gpu_step(pa, nhd, out_dtype=torch.float32, split=split, partition=4 * B)
    H.check_close(out, ref, torch.float32, f"nhd {shape}")
    out_h = H.gpu_step(pa, hnd, out_dtype=torch.float32, split=split, partition=4 * B)
    assert torch.equal(out, out_h), "NHD and HND pools must give bit-identical results"
    # the cache writes landed in the same places, each in its own layout (free rows hold NaN)
    assert torch.equal(nhd.k_cache.transpose(1, 2).nan_to_num(7.0), hnd.k_cache.nan_to_num(7.0))
    assert torch.equal(nhd.v_cache.transpose(1, 2).nan_to_num(7.0), hnd.v_cache.nan_to_num(7.0))
    assert pa.pa_get_error() == 0


def _bits(t):
    """Bit patterns of a CUDA tensor, as the oracle's cache writes return them."""
    t = t.cpu()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.int32).numpy().view(np.uint32)


def test_nhd_cache_write_bit_exact(pa, cuda_device):
    """16-bit and FP8 cache writes into NHD pools against the oracle's writes."""
    from oracle import cache_ops
    g = torch.Generator(device=cuda_device).manual_seed(5)
    N, G, B, d, nb = 300, 8, 16, 128, 40
    slots = torch.randperm(nb * B, device=cuda_device, generator=g)[:N].to(torch.int64)
    slots[11] = -1
    for dt in (torch.float32, torch.float16, torch.bfloat16):
        key = torch.randn(N, G, d, device=cuda_device, generator=g).to(dt)
        val = torch.randn(N, G, d, device=cuda_device, generator=g).to(dt)
        kc = torch.zeros(nb, B, G, d, dtype=dt, device=cuda_device)
        vc = torch.zeros_like(kc)
        k0, v0 = kc.cpu(), vc.cpu()
        pa.pa_reshape_and_cache(key, val, kc, vc, slots, layout="NHD")
        rk, rv = cache_ops.reshape_and_cache(key.cpu(), val.cpu(), k0, v0, slots.cpu(), layout="NHD")
        assert np.array_equal(rk, _bits(kc)) and np.array_equal(rv, _bits(vc)), dt
        kq = torch.zeros(nb, B, G, d, dtype=torch.uint8, device=cuda_device)
        vq = torch.zeros_like(kq)
        pa.pa_reshape_and_cache_fp8(key, val, kq, vq, slots, 0.03, 0.02, layout="NHD")
        qk, qv = ofp8.reshape_and_cache(key.cpu(), val.cpu(), np.zeros((nb, B, G, d), np.uint8),
                                        np.zeros((nb, B, G, d), np.uint8), slots.cpu(), 0.03, 0.02, layout="NHD")
        assert np.array_equal(kq.cpu().numpy(), qk), dt
        assert np.array_equal(vq.cpu().numpy(), qv), dt
    assert pa.pa_get_error() == 0


@pytest.mark.parametrize("split", [False, True])
def test_nhd_fp8_decode(pa, cuda_device, split):
    ctx = [1, 15, 16, 17, 100, 513, 1500, 40]
    nb = sum(-(-c // 16) for c in ctx) + 9
    base = workloads.batch_with_new_tokens("f8", len(ctx), 32, 8, 128, 16, torch.bfloat16, ctx, nb, cuda_device)
    hnd = workloads.to_fp8(base)
    H.poison_free_slots(hnd, value=0x7F)
    nhd = workloads.to_nhd(hnd)
    ks, vs = hnd.meta["k_scale"], hnd.meta["v_scale"]
    k, v = ofp8.reshape_and_cache(nhd.new_key.cpu(), nhd.new_value.cpu(), nhd.k_cache.cpu().numpy(),
                                  nhd.v_cache.cpu().numpy(), nhd.slot_mapping.cpu(), ks, vs, layout="NHD")
    ref = ofp8.decode(nhd.q.cpu(), k, v, nhd.block_tables.cpu(), nhd.context_lens.cpu(), nhd.scale, ks, vs,
                      layout="NHD")
    outs = []
    for wl in (nhd, hnd):
        pa.pa_reshape_and_cache_fp8(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping, ks, vs,
                                    layout=wl.layout)
        out = torch.empty(wl.q.shape, dtype=torch.float32, device=cuda_device)
        if split:
            mctx = wl.max_context
            ws = torch.empty(pa.pa_decode_split_workspace_bytes(wl.S, wl.H, wl.d, mctx, 64), dtype=torch.uint8,
                             device=cuda_device)
            pa.pa_decode_split_fp8(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                                   ks, vs, mctx, 64, ws, layout=wl.layout)
        else:
            pa.pa_decode_fp8(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, ks, vs,
                             layout=wl.layout)
        outs.append(out)
    H.check_close(outs[0], ref, torch.float32, f"fp8 nhd split={split}")
    assert torch.equal(outs[0], outs[1])
    assert np.array_equal(nhd.k_cache.cpu().numpy(), k)
    assert pa.pa_get_error() == 0


def test_nhd_cascade(pa, cuda_device):
    hnd = workloads.shared_prefix(device=cuda_device, prompts=4, samples=8, prefix=700, tail_hi=200, cow=True)
    nhd = workloads.to_nhd(hnd)
    ref = H.Pristine(nhd).decode()
    outs = []
    for wl in (nhd, hnd):
        if wl.copy_pairs.numel():
            pa.pa_copy_blocks([wl.k_cache], [wl.v_cache], wl.copy_pairs)
        pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping,
                                layout=wl.layout)
        gs = torch.tensor(wl.meta["group_starts"], dtype=torch.int32, device=cuda_device)
        pl = torch.tensor(wl.meta["prefix_lens"], dtype=torch.int32, device=cuda_device)
        mpre, mctx = max(wl.meta["prefix_lens"]), wl.max_context
        ws = torch.empty(pa.pa_decode_cascade_workspace_bytes(wl.S, wl.H, wl.d, mpre, mctx, 256),
                         dtype=torch.uint8, device=cuda_device)
        out = torch.empty(wl.q.shape, dtype=torch.float32, device=cuda_device)
        pa.pa_decode_cascade(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, gs, pl,
                             8, mpre, mctx, 256, ws, layout=wl.layout)
        outs.append(out)
    H.check_close(outs[0], ref, torch.float32, "cascade nhd")
    assert torch.equal(outs[0], outs[1])
    assert pa.pa_get_error() == 0


def test_nhd_full_size_sampled(pa, cuda_device):
    """The benchmark batch stored NHD: sampled sequences against the oracle, and
    the whole output bit-identical to the HND pool's."""
    hnd = workloads.llama8b(device=cuda_device)
    nhd = workloads.to_nhd(hnd)
    seqs = H.sample_seqs(nhd, 8)
    P = H.Pristine(nhd, seqs)
    out = H.gpu_step(pa, nhd)
    H.check_close(out[seqs], P.decode(), torch.bfloat16, "llama8b nhd")
    out_h = H.gpu_step(pa, hnd)
    assert torch.equal(out, out_h)
    assert pa.pa_get_error() == 0
