"""Beam search on the paged cache: forks, frees and copy-on-write over many steps.

The pages name beam search beside parallel sampling as a user of shared blocks
and copy-on-write (CS349E Lecture 7 notes §5.1-§5.3). Each step every live beam
appends one token (a beam whose last block is shared copies it first), then the
best half of the beams fork into two children each and the rest are freed. The
GPU runs each step's block copies and cache writes; the oracle runs the same
steps on host copies of the pools. The pools must stay bit-identical, and the
final beams' attention must match the oracle's.
"""
import os
import random
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import gpu_harness as H  # noqa: E402
import oracle  # noqa: E402
from paged_kv_cache_04_gb300.block_manager import BlockManager  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("prompt", [37, 48])  # a partial last prompt block, and a multiple of B
def test_beam_search_steps(pa, cuda_device, prompt):
    G, Hq, d, B, nb, beams, steps = 8, 32, 128, 16, 400, 4, 24
    dt = torch.bfloat16
    rng = random.Random(prompt)
    g = torch.Generator().manual_seed(prompt)
    k_pool = torch.randn((nb, G, B, d), generator=g).to(dt)
    v_pool = torch.randn((nb, G, B, d), generator=g).to(dt)
    kc, vc = k_pool.to(cuda_device), v_pool.to(cuda_device)
    host_k = k_pool.view(torch.int16).numpy().view(np.uint16).copy()
    host_v = v_pool.view(torch.int16).numpy().view(np.uint16).copy()

    bm = BlockManager(nb, B, free_order=torch.randperm(nb, generator=g).tolist())
    bm.add_sequence(0, prompt)
    # prompt tokens: written once, through the same kernels
    slots = torch.tensor([bm.slot_of(0, t) for t in range(prompt)], dtype=torch.int64)
    key = torch.randn((prompt, G, d), generator=g).to(dt)
    val = torch.randn((prompt, G, d), generator=g).to(dt)
    pa.pa_reshape_and_cache(key.to(cuda_device), val.to(cuda_device), kc, vc, slots.to(cuda_device))
    host_k, host_v = oracle.reshape_and_cache(key, val, host_k, host_v, slots)
    for j in range(1, beams):
        bm.fork(0, j)
    live, next_id, copies = list(range(beams)), beams, 0
    for _ in range(steps):
        pairs, new_slots = [], []
        for b in live:
            slot, pair = bm.append_slot(b)
            new_slots.append(slot)
            if pair is not None:
                pairs.append(pair)
        copies += len(pairs)
        key = torch.randn((len(live), G, d), generator=g).to(dt)
        val = torch.randn((len(live), G, d), generator=g).to(dt)
        sl = torch.tensor(new_slots, dtype=torch.int64)
        if pairs:
            pt = torch.tensor(pairs, dtype=torch.int64)
            pa.pa_copy_blocks([kc], [vc], pt.to(cuda_device))
            ks, vs = oracle.copy_blocks([host_k], [host_v], pt)
            host_k, host_v = ks[0], vs[0]
        pa.pa_reshape_and_cache(key.to(cuda_device), val.to(cuda_device), kc, vc, sl.to(cuda_device))
        host_k, host_v = oracle.reshape_and_cache(key, val, host_k, host_v, sl)
        # keep the better half (a seeded stand-in for beam scores), each forking into two
        order = sorted(live, key=lambda _: rng.random())
        keep, drop = order[:beams // 2], order[beams // 2:]
        for b in drop:
            bm.free_sequence(b)
        live = []
        for b in keep:
            bm.fork(b, next_id)
            live += [b, next_id]
            next_id += 1
    assert copies > 0
    torch.cuda.synchronize()
    assert np.array_equal(kc.cpu().view(torch.int16).numpy().view(np.uint16), host_k), "K pool differs"
    assert np.array_equal(vc.cpu().view(torch.int16).numpy().view(np.uint16), host_v), "V pool differs"

    # attention of the final beams over their shared-and-private blocks
    ctx = [bm.context_len(b) for b in live]
    width = max(len(bm.block_table(b)) for b in live)
    bt = torch.full((len(live), width), -1, dtype=torch.int32)
    for i, b in enumerate(live):
        tab = bm.block_table(b)
        bt[i, :len(tab)] = torch.tensor(tab, dtype=torch.int32)
    q = torch.randn((len(live), Hq, d), generator=g).to(dt)
    scale = d ** -0.5
    ref = oracle.decode(q, torch.from_numpy(host_k.view(np.int16)).view(dt),
                        torch.from_numpy(host_v.view(np.int16)).view(dt), bt, torch.tensor(ctx, dtype=torch.int32),
                        scale)
    out = torch.empty(q.shape, dtype=torch.float32, device=cuda_device)
    pa.pa_decode(out, q.to(cuda_device), kc, vc, bt.to(cuda_device), torch.tensor(ctx, dtype=torch.int32,
                                                                                     device=cuda_device), scale)
    H.check_close(out, ref, torch.float32, f"beam search prompt={prompt}")
    assert pa.pa_get_error() == 0
