"""Host logic pinned to the pages' worked examples (tests/golden/pages_worked_examples.json).

Covers the block manager (on-demand allocation, fork / append / free,
copy-on-write counts), the cache-write oracle, the per-token KV byte formula in
both the oracle and the benchmark's byte accounting, and the synthetic
workloads' structure.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_04_gb300 import roofline, workloads
from paged_kv_cache_04_gb300.block_manager import BlockManager, OutOfBlocks

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_worked_examples.json")))


@pytest.mark.parametrize("case", GOLD["kv_bytes_per_token"], ids=lambda c: c["model"])
def test_kv_bytes_per_token(case):
    args = (case["layers"], case["kv_heads"], case["head_dim"], case["dtype_bytes"])
    assert oracle.kv_bytes_per_token(*args) == case["bytes"]
    assert roofline.kv_bytes_per_token(*args) == case["bytes"]


def test_block_and_tile_bytes():
    b = GOLD["block_bytes_per_layer"]
    assert roofline.kv_block_bytes(b["block_size"], b["kv_heads"], b["head_dim"], b["dtype_bytes"]) == b["bytes"]
    t = GOLD["swap_tile_bytes"]
    assert roofline.kv_block_bytes(t["block_size"], t["kv_heads"], t["head_dim"], t["dtype_bytes"]) // 2 == t["bytes"]


def test_block_table_walkthrough():
    w = GOLD["block_table_walkthrough"]
    bm = BlockManager(8, w["block_size"], free_order=w["free_order"])
    bm.add_sequence(0, w["prompt_tokens"])
    assert bm.block_table(0) == w["block_table_after_prompt"]
    fills = [min(w["block_size"], w["prompt_tokens"] - i * w["block_size"]) for i in range(2)]
    assert fills == w["fill_after_prompt"]
    for _ in range(w["decode_tokens"]):
        bm.append_slot(0)
    assert bm.block_table(0) == w["block_table_after_decode"]
    assert [bm.slot_of(0, t) for t in range(bm.context_len(0))] == w["slots"]


def test_block_table_walkthrough_cache_write_and_read():
    """Writing the walk-through's tokens through their slots and reading them back in order."""
    w = GOLD["block_table_walkthrough"]
    B, n = w["block_size"], len(w["slots"])
    rng = np.random.default_rng(3)
    key = rng.standard_normal((n, 1, 2)).astype(np.float32)
    kc = np.zeros((8, 1, B, 2), np.float32)
    kb, _ = oracle.reshape_and_cache(key, key, kc, kc, np.array(w["slots"], np.int64))
    got = kb.view(np.float32)
    table = w["block_table_after_decode"]
    for t in range(n):
        assert np.array_equal(got[table[t // B], 0, t % B], key[t, 0])
    # untouched physical blocks stay zero
    for b in set(range(8)) - set(table):
        assert not got[b].any()


def test_parallel_sampling_exercise():
    e = GOLD["parallel_sampling_exercise"]
    B, n = e["block_size"], e["samples"]
    bm = BlockManager(100, B)
    bm.add_sequence(0, e["prompt"])
    for j in range(1, n):
        bm.fork(0, j)
    pairs = []
    for j in range(n):
        for _ in range(e["generated"]):
            _, pair = bm.append_slot(j)
            if pair:
                pairs.append(pair)
    assert len(pairs) == e["cow_copies"]
    assert 100 - bm.num_free() == e["blocks_shared"]
    unshared = BlockManager(100, B)
    for j in range(n):
        unshared.add_sequence(j, e["prompt"] + e["generated"])
    assert 100 - unshared.num_free() == e["blocks_unshared"]


def test_parallel_sampling_demo_and_n_minus_1():
    e = GOLD["parallel_sampling_demo"]
    for n in (2, 4, 8):
        bm = BlockManager(64, e["block_size"])
        bm.add_sequence(0, e["prompt"])
        table = bm.block_table(0)
        assert len(table) == e["full_blocks"] + 1
        assert e["prompt"] - e["full_blocks"] * e["block_size"] == e["last_block_fill"]
        for j in range(1, n):
            bm.fork(0, j)
        copies = sum(bm.append_slot(j)[1] is not None for j in range(n))
        assert copies == n - 1
        # the last writer kept the original block, the others point at fresh copies
        lasts = {bm.block_table(j)[-1] for j in range(n)}
        assert len(lasts) == n and table[-1] in lasts


def test_cow_multiple_of_block_size():
    e = GOLD["cow_multiple_of_block"]
    bm = BlockManager(64, e["block_size"])
    bm.add_sequence(0, e["prompt"])
    for j in range(1, e["samples"]):
        bm.fork(0, j)
    copies = sum(bm.append_slot(j)[1] is not None for j in range(e["samples"]))
    assert copies == e["cow_copies"]


def test_fragmentation_exercise():
    e = GOLD["fragmentation_exercise"]
    bm = BlockManager(100, e["block_size"])
    bm.add_sequence(0, e["length"])
    assert len(bm.block_table(0)) == e["blocks"]
    assert e["blocks"] * e["block_size"] - e["length"] == e["wasted_slots"]


def test_free_returns_blocks_at_refcount_zero():
    bm = BlockManager(16, 4)
    bm.add_sequence(0, 10)
    bm.fork(0, 1)
    used = 16 - bm.num_free()
    bm.free_sequence(0)
    assert 16 - bm.num_free() == used  # still held by the fork
    bm.free_sequence(1)
    assert bm.num_free() == 16
    with pytest.raises(OutOfBlocks):
        bm.add_sequence(2, 100)


def test_copy_blocks_oracle_semantics():
    """After the CoW copy the forked sample reads exactly the prompt's K/V."""
    rng = np.random.default_rng(5)
    nb, G, B, d = 12, 2, 4, 8
    kc = rng.standard_normal((nb, G, B, d)).astype(np.float32)
    vc = rng.standard_normal((nb, G, B, d)).astype(np.float32)
    pairs = np.array([[1, 7], [3, 9]], np.int64)
    ks, vs = oracle.copy_blocks([kc, kc * 2], [vc, vc * 2], pairs)
    for layer, f in enumerate((1, 2)):
        k = ks[layer].view(np.float32)
        for src, dst in pairs:
            assert np.array_equal(k[dst], kc[src] * f)
        untouched = [b for b in range(nb) if b not in pairs[:, 1]]
        assert np.array_equal(k[untouched], (kc * f)[untouched])


def test_reshape_and_cache_skips_padding():
    kc = np.zeros((2, 1, 4, 2), np.float32)
    key = np.ones((3, 1, 2), np.float32)
    kb, _ = oracle.reshape_and_cache(key, key, kc, kc, np.array([-1, 5, -1], np.int64))
    got = kb.view(np.float32)
    assert got.sum() == 2 and np.array_equal(got[1, 0, 1], [1, 1])


def test_workload_shapes_and_tables():
    wl = workloads.tiny()
    assert wl.context_lens.tolist() == [1, 17, 33, 100]
    assert wl.k_cache.shape == (64, 4, 16, 64) and wl.dtype == torch.float32
    used = wl.block_tables[wl.block_tables >= 0]
    assert used.numel() == sum(-(-c // 16) for c in [1, 17, 33, 100])
    assert torch.unique(used).numel() == used.numel()          # no block shared
    for s, c in enumerate(wl.context_lens.tolist()):
        nblk = -(-c // 16)
        assert (wl.block_tables[s, :nblk] >= 0).all() and (wl.block_tables[s, nblk:] == -1).all()


def test_workload_new_token_slots():
    wl = workloads.batch_with_new_tokens("t", 5, 4, 2, 16, 16, torch.bfloat16, [1, 16, 17, 40, 3],
                                         40, "cpu")
    assert wl.slot_mapping.numel() == 5
    for s in range(5):
        pos = int(wl.context_lens[s]) - 1
        want = int(wl.block_tables[s, pos // 16]) * 16 + pos % 16
        assert int(wl.slot_mapping[s]) == want


def test_shared_prefix_workload_cow_counts():
    lit = workloads.shared_prefix(prompts=3, samples=8, prefix=64, tail_hi=20)
    assert lit.meta["cow_copies"] == 0 and lit.copy_pairs.numel() == 0
    cow = workloads.shared_prefix(prompts=3, samples=8, prefix=64, tail_hi=20, cow=True)
    assert cow.meta["cow_copies"] == 3 * 7
    pairs = cow.copy_pairs
    assert torch.unique(pairs[:, 1]).numel() == pairs.shape[0]           # distinct destinations
    assert not set(pairs[:, 1].tolist()) & set(pairs[:, 0].tolist())     # no chains
    # every sample of a prompt shares the prompt's full blocks
    full = 64 // 16
    for p in range(3):
        rows = cow.block_tables[p * 8:(p + 1) * 8, :full]
        assert (rows == rows[0]).all()


def test_lognormal_context_shape():
    ctx = workloads.lognormal_lengths(20000, 390.0, 493.0, 1, 2048, workloads._gen(1)).double()
    assert ctx.min() >= 1 and ctx.max() <= 2048
    assert abs(ctx.median().item() - 390) < 15
    assert abs(ctx.mean().item() - 493) < 25  # truncation at 2048 trims the mean slightly
