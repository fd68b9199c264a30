"""Seeded random configurations of every attention entry point against the oracle.

Each case draws a cache type (fp32, fp16, bf16, E4M3), a pool layout (HND,
NHD), query / kv heads, head_dim, block size, plain or split decode with a
random partition size, an output type, and a batch of lengths that mixes empty,
one-token, exact-block and ragged contexts. Free pool rows are poisoned, so a
read past a context shows up as a non-finite output.
"""
import os
import random
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import gpu_harness as H  # noqa: E402
from oracle import fp8 as ofp8  # noqa: E402
from paged_kv_cache_04_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu
CASES = 48


def _case(i):
    r = random.Random(1000 + i)
    kind = r.choice(["f32", "f16", "bf16", "bf16", "fp8"])
    G = r.choice([1, 2, 4, 8])
    group = r.choice([1, 2, 3, 4, 5, 8]) if kind != "fp8" else r.choice([1, 2, 4, 8])
    d = 128 if kind == "fp8" else r.choice([64, 128])
    B = r.choice([16, 32])
    S = r.randint(1, 24)
    ctx = []
    for _ in range(S):
        c = r.choice([0, 1, B - 1, B, B + 1, r.randint(2, 300), r.randint(300, 2500)])
        ctx.append(c)
    split = r.random() < 0.5
    T = B * r.choice([1, 2, 4, 8, 32])
    layout = r.choice(["HND", "NHD"])
    out_f32 = r.random() < 0.5
    return kind, G, group, d, B, ctx, split, T, layout, out_f32


@pytest.mark.parametrize("i", range(CASES))
def test_fuzz(pa, cuda_device, i):
    kind, G, group, d, B, ctx, split, T, layout, out_f32 = _case(i)
    dt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "fp8": torch.bfloat16}[kind]
    H_ = G * group
    nb = sum(-(-c // B) for c in ctx) + 7
    wl = workloads.batch_with_new_tokens("fuzz", len(ctx), H_, G, d, B, dt, ctx, nb, cuda_device,
                                         new_token=False, rotate=i)
    what = f"case {i}: {kind} G={G} group={group} d={d} B={B} split={split} T={T} {layout} out_f32={out_f32}"
    out_dt = torch.float32 if out_f32 else dt
    if kind == "fp8":
        wl = workloads.to_fp8(wl)
        H.poison_free_slots(wl, value=0x7F)
        if layout == "NHD":
            wl = workloads.to_nhd(wl)
        ks, vs = wl.meta["k_scale"], wl.meta["v_scale"]
        ref = ofp8.decode(wl.q.cpu(), wl.k_cache.cpu().numpy(), wl.v_cache.cpu().numpy(), wl.block_tables.cpu(),
                          wl.context_lens.cpu(), wl.scale, ks, vs, layout=wl.layout)
        out = torch.empty(wl.q.shape, dtype=out_dt, device=cuda_device)
        if split:
            mctx = max(1, wl.max_context)
            ws = torch.empty(pa.pa_decode_split_workspace_bytes(wl.S, wl.H, d, mctx, T), dtype=torch.uint8,
                             device=cuda_device)
            pa.pa_decode_split_fp8(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                                   ks, vs, mctx, T, ws, layout=wl.layout)
        else:
            pa.pa_decode_fp8(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, ks, vs,
                             layout=wl.layout)
    else:
        H.poison_free_slots(wl)
        if layout == "NHD":
            wl = workloads.to_nhd(wl)
        ref = H.Pristine(wl).decode()
        out = H.gpu_step(pa, wl, out_dtype=out_dt, split=split, partition=T)
    H.check_close(out, ref, out_dt, what)
    zero = [s for s, c in enumerate(ctx) if c == 0]
    if zero:
        assert torch.equal(out[zero].float(), torch.zeros_like(out[zero].float())), what
    assert pa.pa_get_error() == 0, what


def _cascade_case(i):
    r = random.Random(5000 + i)
    return dict(prompts=r.randint(1, 6), samples=r.choice([1, 2, 3, 8, 16, 24, 32]),
                prefix=r.choice([0, 5, 16, 100, 700]),
                tail_hi=r.choice([1, 40, 300]), cow=r.random() < 0.5, T=16 * r.choice([1, 4, 32]),
                layout=r.choice(["HND", "NHD"]))


@pytest.mark.parametrize("i", range(20))
def test_fuzz_cascade(pa, cuda_device, i):
    c = _cascade_case(i)
    wl = workloads.shared_prefix(device=cuda_device, prompts=c["prompts"], samples=c["samples"], prefix=c["prefix"],
                                 tail_hi=c["tail_hi"], cow=c["cow"])
    if c["layout"] == "NHD":
        wl = workloads.to_nhd(wl)
    ref = H.Pristine(wl).decode()
    if wl.copy_pairs.numel():
        pa.pa_copy_blocks([wl.k_cache], [wl.v_cache], wl.copy_pairs)
    pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping, layout=wl.layout)
    gs = torch.tensor(wl.meta["group_starts"], dtype=torch.int32, device=cuda_device)
    pl = torch.tensor(wl.meta["prefix_lens"], dtype=torch.int32, device=cuda_device)
    mpre, mctx, T = max(wl.meta["prefix_lens"]), wl.max_context, c["T"]
    # poisoned (0x7f bytes: finite, huge sums and maxima): every slot the reduce merges must be written
    ws = torch.full((pa.pa_decode_cascade_workspace_bytes(wl.S, wl.H, wl.d, mpre, mctx, T),), 0x7F, dtype=torch.uint8,
                     device=cuda_device)
    out = torch.empty(wl.q.shape, dtype=torch.float32, device=cuda_device)
    pa.pa_decode_cascade(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, gs, pl,
                         c["samples"], mpre, mctx, T, ws, layout=wl.layout)
    H.check_close(out, ref, torch.float32, f"cascade case {i}: {c}")
    assert pa.pa_get_error() == 0


@pytest.mark.parametrize("i", range(12))
def test_fuzz_cache_writes_and_copies(pa, cuda_device, i):
    """Random shapes of the cache write (16-bit, fp32 and E4M3, both layouts) and
    of the block copy, bit-exact against the oracle."""
    from oracle import cache_ops
    r = random.Random(9000 + i)
    dt = r.choice([torch.float32, torch.float16, torch.bfloat16])
    G, d, B = r.choice([1, 2, 8]), r.choice([64, 80, 128, 256]), r.choice([8, 16, 32])
    nb = r.randint(4, 40)
    N = min(r.randint(1, 300), nb * B)
    layout = r.choice(["HND", "NHD"])
    shape = (nb, G, B, d) if layout == "HND" else (nb, B, G, d)
    g = torch.Generator().manual_seed(i)
    kc = torch.randn(shape, generator=g).to(dt)
    vc = torch.randn(shape, generator=g).to(dt)
    key = torch.randn((N, G, d), generator=g).to(dt)
    val = torch.randn((N, G, d), generator=g).to(dt)
    slots = torch.randperm(nb * B, generator=g)[:N]
    if N > 2:
        slots[N // 2] = -1  # padding token
    dk, dv = kc.to(cuda_device), vc.to(cuda_device)
    pa.pa_reshape_and_cache(key.to(cuda_device), val.to(cuda_device), dk, dv, slots.to(cuda_device), layout=layout)
    rk, rv = cache_ops.reshape_and_cache(key, val, kc, vc, slots, layout=layout)
    bits = (lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)) if dt != torch.float32 else \
        (lambda t: t.cpu().view(torch.int32).numpy().view(np.uint32))
    assert np.array_equal(bits(dk), rk) and np.array_equal(bits(dv), rv), (dt, G, d, B, layout)
    # block copies between distinct blocks
    perm = torch.randperm(nb, generator=g).tolist()
    P = r.randint(1, nb // 2)
    pairs = torch.tensor([[perm[j], perm[P + j]] for j in range(P)], dtype=torch.int64)
    pa.pa_copy_blocks([dk], [dv], pairs.to(cuda_device))
    ks, vs = cache_ops.copy_blocks([rk], [rv], pairs)
    assert np.array_equal(bits(dk), ks[0]) and np.array_equal(bits(dv), vs[0])
    if d % 16 == 0:  # E4M3 rows are written 16 codes at a time
        qk = torch.zeros(shape, dtype=torch.uint8, device=cuda_device)
        qv = torch.zeros(shape, dtype=torch.uint8, device=cuda_device)
        pa.pa_reshape_and_cache_fp8(key.to(cuda_device), val.to(cuda_device), qk, qv, slots.to(cuda_device), 0.05,
                                    0.02, layout=layout)
        ek, ev = ofp8.reshape_and_cache(key, val, np.zeros(tuple(shape), np.uint8), np.zeros(tuple(shape), np.uint8),
                                        slots, 0.05, 0.02, layout=layout)
        assert np.array_equal(qk.cpu().numpy(), ek) and np.array_equal(qv.cpu().numpy(), ev)
    assert pa.pa_get_error() == 0
