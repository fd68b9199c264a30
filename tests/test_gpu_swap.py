"""pa_swap_blocks: blocks moved between a device pool and a pinned host pool, bit-exact."""
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
        t = torch.randn(nb, 8, 16, 128, generator=g).to(torch.bfloat16)
        out.append(t.pin_memory() if pinned else t.to(dev))
    return out


def test_swap_out_and_back_in(pa, cuda_device):
    L, nb_dev, nb_host = 4, 300, 120
    dk, dv = _pools(L, nb_dev, cuda_device, 1), _pools(L, nb_dev, cuda_device, 2)
    hk, hv = _pools(L, nb_host, cuda_device, 3, pinned=True), _pools(L, nb_host, cuda_device, 4, pinned=True)
    g = torch.Generator().manual_seed(5)
    src = torch.randperm(nb_dev, generator=g)[:77]
    dst = torch.randperm(nb_host, generator=g)[:77]
    out_pairs = torch.stack([src, dst], 1).to(torch.int64).to(cuda_device)
    rk, rv = oracle.swap_blocks(hk, hv, dk, dv, out_pairs)
    pa.pa_swap_blocks(hk, hv, dk, dv, out_pairs)          # device -> host
    torch.cuda.synchronize()
    for layer in range(L):
        assert np.array_equal(_bits(hk[layer]), rk[layer]) and np.array_equal(_bits(hv[layer]), rv[layer])
    # back in, to different device blocks, with the pairs in pinned host memory
    back = torch.randperm(nb_dev, generator=g)[:77]
    in_pairs = torch.stack([dst, back], 1).to(torch.int64).pin_memory()
    rk2, rv2 = oracle.swap_blocks(dk, dv, hk, hv, in_pairs)
    pa.pa_swap_blocks(dk, dv, hk, hv, in_pairs)           # host -> device
    torch.cuda.synchronize()
    for layer in range(L):
        assert np.array_equal(_bits(dk[layer]), rk2[layer]) and np.array_equal(_bits(dv[layer]), rv2[layer])
    assert pa.pa_get_error() == 0


def test_swap_many_layers_device_to_device(pa, cuda_device):
    L = 40  # more layers than one launch carries
    a, b = _pools(L, 20, cuda_device, 6), _pools(L, 20, cuda_device, 7)
    c, d = _pools(L, 30, cuda_device, 8), _pools(L, 30, cuda_device, 9)
    pairs = torch.tensor([[0, 29], [19, 0], [5, 5]], dtype=torch.int64, device=cuda_device)
    rk, rv = oracle.swap_blocks(c, d, a, b, pairs)
    pa.pa_swap_blocks(c, d, a, b, pairs)
    torch.cuda.synchronize()
    for layer in range(L):
        assert np.array_equal(_bits(c[layer]), rk[layer]) and np.array_equal(_bits(d[layer]), rv[layer])


def test_swap_rejects_out_of_range_ids(pa, cuda_device):
    a, b = _pools(1, 10, cuda_device, 10), _pools(1, 10, cuda_device, 11)
    c, d = _pools(1, 4, cuda_device, 12), _pools(1, 4, cuda_device, 13)
    before = c[0].clone()
    pa.pa_get_error()
    pairs = torch.tensor([[9, 4], [10, 0]], dtype=torch.int64, device=cuda_device)  # dst 4 and src 10 invalid
    pa.pa_swap_blocks(c, d, a, b, pairs)
    assert pa.pa_get_error() & pa.PA_DEVERR_PAIR
    assert torch.equal(c[0], before)
