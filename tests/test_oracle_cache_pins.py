"""Pins for the oracle's block-movement functions (``oracle/cache_ops.py``).

``swap_blocks`` and ``copy_blocks`` are the only checkers of the GPU swap and
copy-on-write kernels, so they are tied here to what the pages fix:

* hand-chosen (src, dst) pairs over two pools of different sizes, K and V
  different, several layers: every destination block named by a pair holds the
  source block, K from K and V from V, of its own layer; every other
  destination block is unchanged; the source pools are not written;
* the swap count of CS349E Lecture 7 notes, exercise 6 (OPT-13B, block size 32,
  a 1,024-token sequence: 40 layers x 2 x 32 blocks = 2,560 per-block copies of
  327,680 bytes, 59.2 ms out and 118.3 ms out and back at 10 us + 25 GB/s per
  copy), counted from the blocks the oracle changes;
* copy-on-write (CS349E §5.1): the copy leaves the source block readable and
  gives the writer an identical private block.

``test_cache_mutants_are_caught`` plants mistakes in a copy of the oracle's
source (on the CPU) and checks that this battery fails for each of them.
"""
import importlib.util
import os

import numpy as np
import pytest

import oracle
from oracle import cache_ops

CACHE_OPS_SRC = os.path.join(os.path.dirname(oracle.__file__), "cache_ops.py")


def _pools(rng, layers, nb, G=2, B=4, d=8, salt=0):
    """Per-layer K and V pools of uint16 patterns, distinct per (layer, K/V, block)."""
    ks, vs = [], []
    for layer in range(layers):
        k = rng.integers(0, 1 << 16, size=(nb, G, B, d), dtype=np.uint16)
        v = rng.integers(0, 1 << 16, size=(nb, G, B, d), dtype=np.uint16)
        # a tag in element 0 of each block keeps every block distinct from every other
        for b in range(nb):
            k[b, 0, 0, 0] = (salt * 7 + layer * 1000 + 2 * b) & 0xFFFF
            v[b, 0, 0, 0] = (salt * 7 + layer * 1000 + 2 * b + 1) & 0xFFFF
        ks.append(k)
        vs.append(v)
    return ks, vs


# hand-chosen pairs (src id in a 9-block pool, dst id in a 13-block pool); reversing
# any pair stays inside both pools, so a reversed copy is caught by value
SWAP_PAIRS = np.array([[0, 8], [5, 3], [8, 0], [2, 7], [7, 5]], np.int64)


def pin_swap_hand_pairs(mod):
    rng = np.random.default_rng(41)
    L = 3
    src_k, src_v = _pools(rng, L, 9, salt=1)
    dst_k, dst_v = _pools(rng, L, 13, salt=2)
    keep = [(a.copy(), b.copy()) for a, b in zip(src_k, src_v)]
    before = [(a.copy(), b.copy()) for a, b in zip(dst_k, dst_v)]
    out_k, out_v = mod.swap_blocks(dst_k, dst_v, src_k, src_v, SWAP_PAIRS)
    assert len(out_k) == L and len(out_v) == L
    written = set(SWAP_PAIRS[:, 1].tolist())
    for layer in range(L):
        ok, ov = np.asarray(out_k[layer]), np.asarray(out_v[layer])
        sk0, sv0 = keep[layer]
        for s, d in SWAP_PAIRS:
            assert np.array_equal(ok[d], sk0[s]), f"K block {d} of layer {layer} is not source block {s}"
            assert np.array_equal(ov[d], sv0[s]), f"V block {d} of layer {layer} is not source block {s}"
        for b in range(13):
            if b not in written:
                assert np.array_equal(ok[b], before[layer][0][b]) and np.array_equal(ov[b], before[layer][1][b])
        # the source pools are read, never written
        assert np.array_equal(src_k[layer], sk0) and np.array_equal(src_v[layer], sv0)
        # and the caller's destination arrays are left as they were (the oracle returns new ones)
        assert np.array_equal(dst_k[layer], before[layer][0]) and np.array_equal(dst_v[layer], before[layer][1])


def pin_swap_order_free_and_round_trip(mod):
    """Distinct destinations make the order of the pairs irrelevant; swapping a
    sequence's blocks out to a host pool and back into other free blocks returns
    its K/V bit for bit (CS349E §6.2: the blocks come back later, anywhere)."""
    rng = np.random.default_rng(42)
    gpu_k, gpu_v = _pools(rng, 2, 11, salt=3)
    host_k, host_v = _pools(rng, 2, 6, salt=4)
    out_pairs = np.array([[4, 0], [9, 1], [1, 2]], np.int64)        # gpu block -> host block
    a = mod.swap_blocks(host_k, host_v, gpu_k, gpu_v, out_pairs)
    b = mod.swap_blocks(host_k, host_v, gpu_k, gpu_v, out_pairs[::-1].copy())
    for x, y in zip(a[0] + a[1], b[0] + b[1]):
        assert np.array_equal(x, y)
    back_pairs = np.array([[0, 6], [1, 10], [2, 3]], np.int64)      # host block -> new gpu block
    rk, rv = mod.swap_blocks(gpu_k, gpu_v, a[0], a[1], back_pairs)
    for layer in range(2):
        for (g_src, h), (h2, g_dst) in zip(out_pairs, back_pairs):
            assert h == h2
            assert np.array_equal(np.asarray(rk[layer])[g_dst], gpu_k[layer][g_src])
            assert np.array_equal(np.asarray(rv[layer])[g_dst], gpu_v[layer][g_src])


def pin_swap_exercise6_count(mod):
    """CS349E Lecture 7 notes, exercise 6: a 1,024-token OPT-13B sequence in
    32-token blocks swaps as 40 layers x 2 x 32 blocks = 2,560 copies of
    327,680 bytes; at 10 us + bytes / 25 GB/s each that is 59.2 ms out and
    118.3 ms out and back.

    The count is taken from the oracle: every source block is distinct, the
    destination pool starts as a sentinel, and the blocks that changed are
    counted. The per-copy size is the byte size of one block of one layer's K at
    the exercise's shape, moved by the oracle and compared byte for byte."""
    layers, seq_tokens, B = 40, 1024, 32
    nblk = seq_tokens // B
    rng = np.random.default_rng(43)
    # the count does not depend on the block's payload: small blocks (G = 1, d = 8)
    src_k, src_v = _pools(rng, layers, nblk, G=1, B=B, d=8, salt=5)
    sentinel = [np.full((nblk + 4, 1, B, 8), 0xFFFF, np.uint16) for _ in range(layers)]
    pairs = np.stack([np.arange(nblk), rng.permutation(nblk + 4)[:nblk]], axis=1).astype(np.int64)
    out_k, out_v = mod.swap_blocks(sentinel, [s.copy() for s in sentinel], src_k, src_v, pairs)
    changed = 0
    for layer in range(layers):
        for pool in (out_k[layer], out_v[layer]):
            pool = np.asarray(pool)
            changed += sum(1 for b in range(nblk + 4) if not np.all(pool[b] == 0xFFFF))
    assert changed == 2560, changed
    # one copy at the exercise's shape: [40 kv heads][32 rows][128] fp16 of one layer's K
    big_src = [rng.integers(0, 1 << 16, size=(2, 40, B, 128), dtype=np.uint16)]
    big_dst = [np.zeros((2, 40, B, 128), np.uint16)]
    bk, _ = mod.swap_blocks(big_dst, [big_dst[0].copy()], big_src, [big_src[0].copy()],
                            np.array([[1, 0]], np.int64))
    moved = np.asarray(bk[0])[0]
    assert moved.nbytes == 327680 and np.array_equal(moved, big_src[0][1])
    t_out = changed * (10e-6 + moved.nbytes / 25e9)
    assert round(t_out * 1e3, 1) == 59.2 and round(2 * t_out * 1e3, 1) == 118.3


def pin_copy_blocks_k_and_v(mod):
    """Copy-on-write (CS349E §5.1): after the copy the writer's private block
    equals the shared one, K and V of every layer; the shared block and every
    block not named as a destination are unchanged."""
    rng = np.random.default_rng(44)
    L, nb = 3, 12
    ks, vs = _pools(rng, L, nb, salt=6)
    keep = [(a.copy(), b.copy()) for a, b in zip(ks, vs)]
    pairs = np.array([[1, 7], [3, 9], [10, 2]], np.int64)
    ok, ov = mod.copy_blocks(ks, vs, pairs)
    for layer in range(L):
        k0, v0 = keep[layer]
        k1, v1 = np.asarray(ok[layer]), np.asarray(ov[layer])
        for s, d in pairs:
            assert np.array_equal(k1[d], k0[s]) and np.array_equal(v1[d], v0[s])
        for b in range(nb):
            if b not in pairs[:, 1]:
                assert np.array_equal(k1[b], k0[b]) and np.array_equal(v1[b], v0[b])
        assert np.array_equal(ks[layer], k0) and np.array_equal(vs[layer], v0)


CACHE_PINS = [pin_swap_hand_pairs, pin_swap_order_free_and_round_trip, pin_swap_exercise6_count,
              pin_copy_blocks_k_and_v]


@pytest.mark.parametrize("pin", CACHE_PINS, ids=[p.__name__ for p in CACHE_PINS])
def test_cache_pin(pin):
    pin(cache_ops)


def test_swap_blocks_rejects_out_of_range_ids():
    rng = np.random.default_rng(45)
    sk, sv = _pools(rng, 1, 4)
    dk, dv = _pools(rng, 1, 3)
    for bad in ([[4, 0]], [[0, 3]], [[-1, 0]]):
        with pytest.raises(IndexError):
            cache_ops.swap_blocks(dk, dv, sk, sv, np.array(bad, np.int64))


# ---------------------------------------------------------------------------
# planted mistakes: each mutant of cache_ops.py must fail at least one pin
# ---------------------------------------------------------------------------
CACHE_MUTANTS = {
    # swap_blocks
    "swap_pairs_reversed": [("dks[layer][dst] = sk[src]\n            dvs[layer][dst] = sv[src]",
                             "dks[layer][src] = sk[dst]\n            dvs[layer][src] = sv[dst]")],
    "swap_kv_crossed": [("dvs[layer][dst] = sv[src]", "dvs[layer][dst] = sk[src]")],
    "swap_source_written": [
        ("sk, sv = _bits(src_k_caches[layer]), _bits(src_v_caches[layer])",
         "sk, sv = src_k_caches[layer], src_v_caches[layer]"),
        ("dvs[layer][dst] = sv[src]", "dvs[layer][dst] = sv[src]\n            sk[src] = 0"),
    ],
    "swap_layer_zero_only": [("_bits(src_k_caches[layer]), _bits(src_v_caches[layer])",
                              "_bits(src_k_caches[0]), _bits(src_v_caches[0])")],
    "swap_v_dropped": [("            dvs[layer][dst] = sv[src]\n", "")],
    # copy_blocks
    "copy_pairs_reversed": [("ks[layer][dst] = src_k[src]\n            vs[layer][dst] = src_v[src]",
                             "ks[layer][src] = src_k[dst]\n            vs[layer][src] = src_v[dst]")],
    "copy_kv_crossed": [("vs[layer][dst] = src_v[src]", "vs[layer][dst] = src_k[src]")],
}


def _load_variant(path, name):
    spec = importlib.util.spec_from_file_location(name, path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _run_cache_battery(mod):
    failed = []
    for pin in CACHE_PINS:
        try:
            pin(mod)
        except (AssertionError, IndexError, ValueError) as e:
            failed.append((pin.__name__, str(e)[:80]))
    return failed


@pytest.mark.parametrize("name", sorted(CACHE_MUTANTS))
def test_cache_mutants_are_caught(name, tmp_path):
    src = open(CACHE_OPS_SRC).read()
    for old, new in CACHE_MUTANTS[name]:
        assert src.count(old) == 1, f"mutation site for {name} not found once"
        src = src.replace(old, new)
    p = tmp_path / f"cache_ops_{name}.py"
    p.write_text(src)
    failed = _run_cache_battery(_load_variant(str(p), f"cache_ops_{name}"))
    assert failed, f"planted mistake {name} went unnoticed by every pin"


def test_unmutated_cache_battery_passes(tmp_path):
    p = tmp_path / "cache_ops_copy.py"
    p.write_text(open(CACHE_OPS_SRC).read())
    assert _run_cache_battery(_load_variant(str(p), "cache_ops_copy")) == []
