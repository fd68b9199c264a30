"""The native (C++) block manager: the pages' worked examples, the prefix-cache
behaviour the pages describe, and a differential test against the Python
manager (itself pinned to the pages) on random operation sequences."""
import json
import os
import random

import pytest

from paged_kv_cache_04_gb300 import _build
from paged_kv_cache_04_gb300.block_manager import BlockManager, NativeBlockManager, OutOfBlocks

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_worked_examples.json")))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.ensure_built()


def test_parallel_sampling_exercise():
    e = GOLD["parallel_sampling_exercise"]
    bm = NativeBlockManager(100, e["block_size"], prefix_caching=False)
    bm.add_sequence(0, list(range(e["prompt"])))
    for j in range(1, e["samples"]):
        bm.fork(0, j)
    copies = 0
    for j in range(e["samples"]):
        for t in range(e["generated"]):
            copies += bm.append_slot(j, 1000 + t)[1] is not None
    assert copies == e["cow_copies"]
    assert 100 - bm.num_free() == e["blocks_shared"]
    assert bm.stats()["copies"] == e["cow_copies"]


def test_cow_n_minus_1_and_multiple_of_block():
    for prompt, n, want in ((100, 8, 7), (GOLD["cow_multiple_of_block"]["prompt"], 4, 0)):
        bm = NativeBlockManager(64, 16, prefix_caching=False)
        bm.add_sequence(0, list(range(prompt)))
        for j in range(1, n):
            bm.fork(0, j)
        assert sum(bm.append_slot(j, 7)[1] is not None for j in range(n)) == want


def test_fragmentation_exercise():
    e = GOLD["fragmentation_exercise"]
    bm = NativeBlockManager(100, e["block_size"])
    bm.add_sequence(0, list(range(e["length"])))
    assert len(bm.block_table(0)) == e["blocks"]


def test_prefix_hit_survives_release():
    """A 16-token system prompt computed for request 1 is reused by request 2, even
    after request 1 finished (Month 2 · PagedAttention §7.1-§7.2)."""
    system = list(range(500, 516))
    bm = NativeBlockManager(32, 16)
    assert bm.add_sequence(1, system + [1, 2, 3, 4, 5]) == 0
    first = bm.block_table(1)[0]
    bm.free_sequence(1)
    assert bm.stats()["evictable"] == 1
    assert bm.add_sequence(2, system + [9, 8, 7, 6, 5, 4]) == 16
    assert bm.block_table(2)[0] == first
    assert bm.stats()["hits"] == 1


def test_only_block_aligned_prefixes_match():
    """Prompts that diverge at token 17 share exactly the first block (§7.5)."""
    base = list(range(40))
    bm = NativeBlockManager(32, 16)
    bm.add_sequence(1, base)
    other = base[:16] + [999] + base[17:]
    assert bm.add_sequence(2, other) == 16
    t1, t2 = bm.block_table(1), bm.block_table(2)
    assert t1[0] == t2[0] and t1[1] != t2[1]


def test_chain_hash_needs_the_whole_prefix():
    """The same block contents after a different first block is not a hit."""
    a, b, shared = list(range(16)), list(range(100, 116)), list(range(200, 216))
    bm = NativeBlockManager(32, 16)
    bm.add_sequence(1, a + shared)
    assert bm.add_sequence(2, b + shared) == 0


def test_blocks_filled_by_decode_become_cacheable():
    bm = NativeBlockManager(32, 4)
    bm.add_sequence(1, [1, 2])
    for t in (3, 4, 5, 6, 7, 8):
        bm.append_slot(1, t)
    assert bm.add_sequence(2, [1, 2, 3, 4, 5, 6, 7, 8, 9]) == 8


def test_lru_eviction_order():
    """Released cached blocks are evicted least recently released first; a freed
    sequence releases its tail first, so its head survives longest."""
    B = 4
    bm = NativeBlockManager(6, B)
    bm.add_sequence(1, list(range(12)))       # blocks for 3 full blocks
    bm.add_sequence(2, list(range(50, 62)))   # 3 more: pool full
    t1 = bm.block_table(1)
    bm.free_sequence(1)                       # released tail first: t1[2], t1[1], t1[0]
    bm.free_sequence(2)
    assert bm.num_free() == 6 and bm.stats()["evictable"] == 6
    bm.add_sequence(3, list(range(90, 94)))   # needs one new block: evicts t1[2] (oldest)
    assert bm.block_table(3) == [t1[2]]
    assert bm.stats()["evictions"] == 1
    assert bm.add_sequence(4, list(range(12))) == 8  # blocks 0 and 1 of sequence 1 still cached


def test_out_of_blocks_changes_nothing():
    bm = NativeBlockManager(4, 4)
    bm.add_sequence(1, list(range(12)))
    with pytest.raises(OutOfBlocks):
        bm.add_sequence(2, list(range(100, 110)))
    assert bm.num_free() == 1 and bm.context_len(2) == -1
    bm.add_sequence(3, list(range(200, 204)))
    with pytest.raises(OutOfBlocks):
        bm.append_slot(3, 1)


def test_invalid_calls():
    bm = NativeBlockManager(8, 4)
    with pytest.raises(ValueError):
        bm.fork(5, 6)
    bm.add_sequence(1, [1])
    with pytest.raises(ValueError):
        bm.add_sequence(1, [2])
    with pytest.raises(KeyError):
        bm.block_table(99)


def _same_structure(py, nat, live):
    """Live block ids correspond one to one (the managers may number blocks differently)."""
    fwd, back = {}, {}
    for s in live:
        a, b = py.block_table(s), nat.block_table(s)
        assert len(a) == len(b)
        for x, y in zip(a, b):
            assert fwd.setdefault(y, x) == x and back.setdefault(x, y) == y
    return fwd


@pytest.mark.parametrize("seed", range(6))
def test_matches_python_manager_without_caching(seed):
    """Random add / fork / append / free: the same tables up to block numbering,
    the same slot offsets and the same copy-on-write events as the Python
    manager (the native one releases a sequence's blocks tail first)."""
    rng = random.Random(seed)
    nb, B = 120, rng.choice([1, 4, 16])
    py, nat = BlockManager(nb, B), NativeBlockManager(nb, B, prefix_caching=False)
    live, next_id = [], 0
    for _ in range(400):
        op = rng.random()
        try:
            if op < 0.2 or not live:
                n = rng.randint(0, 40)
                if -(-n // B) > py.num_free():
                    continue
                py.add_sequence(next_id, n)
                nat.add_sequence(next_id, [0] * n)
                live.append(next_id)
                next_id += 1
            elif op < 0.35:
                parent = rng.choice(live)
                py.fork(parent, next_id)
                nat.fork(parent, next_id)
                live.append(next_id)
                next_id += 1
            elif op < 0.85:
                s = rng.choice(live)
                if py.num_free() == 0:
                    continue
                (ps, pp), (ns, np_) = py.append_slot(s), nat.append_slot(s, 0)
                assert ps % B == ns % B and (pp is None) == (np_ is None)
                fwd = _same_structure(py, nat, live)
                assert fwd[ns // B] == ps // B
                if pp is not None:
                    assert fwd[np_[1]] == pp[1]
            else:
                s = live.pop(rng.randrange(len(live)))
                py.free_sequence(s)
                nat.free_sequence(s)
        except OutOfBlocks:
            continue
        _same_structure(py, nat, live)
        assert py.num_free() == nat.num_free()
        for s in live:
            assert py.context_len(s) == nat.context_len(s)


def test_chain_hash_demo():
    """The pages' block-size-4 demo: a shared system prompt and start give three
    equal block hashes and a different fourth; one changed system-prompt token
    changes that block's hash and every later one."""
    e = GOLD["chain_hash_demo"]
    B, n = e["block_size"], e["shared_blocks"]
    system, start = [11, 12, 13, 14, 15, 16], [21, 22, 23, 24, 25, 26]
    a = system + start + [31, 32, 33, 34]   # 16 tokens: four full blocks
    b = system + start + [41, 42, 43, 44]   # differs only in the fourth block
    bm = NativeBlockManager(64, B)
    assert bm.add_sequence(0, a) == 0
    assert bm.add_sequence(1, b) == n * B
    assert bm.block_table(1)[:n] == bm.block_table(0)[:n]
    assert bm.block_table(1)[n] != bm.block_table(0)[n]
    c = list(b)
    c[5] = 99                               # a system-prompt token in the second block
    assert bm.add_sequence(2, c) == 1 * B   # only the first block still matches
    d = list(b)
    d[0] = 99                               # ... in the first block: nothing matches
    assert bm.add_sequence(3, d) == 0


def test_block_aligned_prefix_only():
    """Prompts that first differ at token 17 share exactly the first 16-token block."""
    e = GOLD["block_aligned_prefix"]
    B = e["block_size"]
    k = e["first_differing_token"] - 1       # 0-based index of the first different token
    a = list(range(100, 140))
    b = a[:k] + [999] + a[k + 1:]
    bm = NativeBlockManager(64, B)
    bm.add_sequence(0, a)
    assert bm.add_sequence(1, b) == e["shared_tokens"]
