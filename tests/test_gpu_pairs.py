"""The copy and swap kernels check their pair list for races on the device.

All pairs of one call are copied in parallel, so a destination written twice,
or a block that one pair writes while another reads it, would give whatever
the race leaves. Copy-on-write gives every writer its own block (CS349E
Lecture 7 notes §5.1), so a well-formed list never has such pairs; the kernels
skip the ones that do (in every layer, K and V) and set PA_DEVERR_PAIR_ALIAS,
and copy the rest bit for bit (checked against the oracle on the pairs that
remain).
"""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import oracle  # noqa: E402

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _pools(n, nb, dev, seed, pinned=False):
    g = torch.Generator().manual_seed(seed)
    out = []
    for _ in range(n):
        t = torch.randn(nb, 4, 16, 64, generator=g).to(torch.bfloat16)
        out.append(t.pin_memory() if pinned else t.to(dev))
    return out


def _copy_and_compare(pa, dev, pairs, good, expect_alias):
    L, nb = 3, 40
    ks, vs = _pools(L, nb, dev, 1), _pools(L, nb, dev, 2)
    rk, rv = oracle.copy_blocks(ks, vs, np.array(good, np.int64).reshape(-1, 2))
    pa.pa_get_error()
    pa.pa_copy_blocks(ks, vs, torch.tensor(pairs, dtype=torch.int64, device=dev))
    bits = pa.pa_get_error()
    assert bool(bits & pa.PA_DEVERR_PAIR_ALIAS) == expect_alias, bits
    assert not bits & ~pa.PA_DEVERR_PAIR_ALIAS, bits
    for layer in range(L):
        assert np.array_equal(_bits(ks[layer]), rk[layer]) and np.array_equal(_bits(vs[layer]), rv[layer])


@pytest.mark.parametrize("case", ["chain", "dup_dst", "dst_is_src", "self", "clean"])
def test_copy_blocks_skips_racing_pairs(pa, cuda_device, case):
    valid = [[30, 31], [32, 33]]  # copied in every case
    racing = {
        "chain": [[1, 2], [2, 3]],            # pair 0 writes what pair 1 reads
        "dup_dst": [[4, 9], [5, 9]],          # two writers of block 9
        "dst_is_src": [[6, 7], [8, 6]],       # pair 1 writes pair 0's source
        "self": [[10, 10]],                   # a block copied onto itself
        "clean": [],
    }[case]
    pairs = racing + valid
    _copy_and_compare(pa, cuda_device, pairs, valid, expect_alias=bool(racing))


def test_copy_blocks_alias_and_out_of_range_together(pa, cuda_device):
    """An out-of-range pair is reported as such and races with nothing: the pair
    sharing its (invalid) destination id is copied."""
    L, nb = 2, 20
    ks, vs = _pools(L, nb, cuda_device, 3), _pools(L, nb, cuda_device, 4)
    pairs = [[1, nb + 3], [2, 5], [3, 5], [7, 8]]
    rk, rv = oracle.copy_blocks(ks, vs, np.array([[7, 8]], np.int64))
    pa.pa_get_error()
    pa.pa_copy_blocks(ks, vs, torch.tensor(pairs, dtype=torch.int64, device=cuda_device))
    bits = pa.pa_get_error()
    assert bits & pa.PA_DEVERR_PAIR and bits & pa.PA_DEVERR_PAIR_ALIAS
    for layer in range(L):
        assert np.array_equal(_bits(ks[layer]), rk[layer]) and np.array_equal(_bits(vs[layer]), rv[layer])


def test_swap_duplicate_destination_is_skipped(pa, cuda_device):
    """Two pools: a source id equal to a destination id is fine (they name
    different memory); a destination written twice is not."""
    L = 2
    dk, dv = _pools(L, 12, cuda_device, 5), _pools(L, 12, cuda_device, 6)
    hk, hv = _pools(L, 8, cuda_device, 7, pinned=True), _pools(L, 8, cuda_device, 8, pinned=True)
    good = [[3, 3], [4, 0]]
    pairs = [[1, 6], [2, 6]] + good
    rk, rv = oracle.swap_blocks(hk, hv, dk, dv, np.array(good, np.int64))
    pa.pa_get_error()
    pa.pa_swap_blocks(hk, hv, dk, dv, torch.tensor(pairs, dtype=torch.int64, device=cuda_device))
    bits = pa.pa_get_error()
    assert bits == pa.PA_DEVERR_PAIR_ALIAS, bits
    for layer in range(L):
        assert np.array_equal(_bits(hk[layer]), rk[layer]) and np.array_equal(_bits(hv[layer]), rv[layer])


def test_swap_within_one_pool_uses_the_copy_rule(pa, cuda_device):
    """Source and destination pools that are the same memory: a destination that
    is another pair's source races and is skipped."""
    L = 2
    ks, vs = _pools(L, 16, cuda_device, 9), _pools(L, 16, cuda_device, 10)
    good = [[12, 13]]
    pairs = [[1, 2], [2, 3]] + good
    rk, rv = oracle.copy_blocks(ks, vs, np.array(good, np.int64))
    pa.pa_get_error()
    pa.pa_swap_blocks(ks, vs, ks, vs, torch.tensor(pairs, dtype=torch.int64, device=cuda_device))
    assert pa.pa_get_error() == pa.PA_DEVERR_PAIR_ALIAS
    for layer in range(L):
        assert np.array_equal(_bits(ks[layer]), rk[layer]) and np.array_equal(_bits(vs[layer]), rv[layer])


def test_debug_check_reports_the_alias(pa, cuda_device):
    ks, vs = _pools(1, 8, cuda_device, 11), _pools(1, 8, cuda_device, 12)
    pa.pa_get_error()
    assert pa.pa_debug_check() == pa.PA_OK
    pa.pa_copy_blocks(ks, vs, torch.tensor([[0, 1], [1, 2]], dtype=torch.int64, device=cuda_device))
    assert pa.pa_debug_check() == pa.PA_ERR_OUT_OF_RANGE
    assert pa.pa_debug_check() == pa.PA_OK  # the word was cleared
