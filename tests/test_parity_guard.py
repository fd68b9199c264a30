"""The GPU parity tests' regression guard is tight enough to catch a real loss of precision.

The spec bound (2e-3 max abs error on the fp32 result) is loose next to what
the kernels reach (~1e-6): a kernel that rounded the softmax weights to one
16-bit part before P V (dropping the lo part of its hi + lo split) would still
pass it. ``gpu_harness.check_close`` therefore also asserts a guard of 1e-4 on
the error beyond the output rounding. Here that mistake is planted in a plain
CPU restatement of attention (float64, the weights rounded to bf16 before they
multiply V, the normaliser left exact) on the tiny and Llama-shaped inputs: the
spec bound accepts it, the guard rejects it. The unplanted restatement matches
the oracle to 1e-12, so the difference is the planted rounding alone.
"""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import gpu_harness as H  # noqa: E402
import oracle  # noqa: E402
from paged_kv_cache_04_gb300 import workloads  # noqa: E402


def _attention(wl, weights_bf16):
    """softmax(scale q K^T) V per (sequence, head) from the gathered blocks, float64;
    with weights_bf16 each weight is rounded to bf16 before it multiplies V."""
    q = wl.q.double().numpy()
    kc, vc = wl.k_cache.double().numpy(), wl.v_cache.double().numpy()
    bt, ctx = wl.block_tables.numpy(), wl.context_lens.numpy()
    B, group = wl.B, wl.H // wl.G
    out = np.zeros(q.shape)
    for s in range(wl.S):
        c = int(ctx[s])
        n = -(-c // B)
        K = kc[bt[s, :n]].transpose(0, 2, 1, 3).reshape(n * B, wl.G, wl.d)[:c]
        V = vc[bt[s, :n]].transpose(0, 2, 1, 3).reshape(n * B, wl.G, wl.d)[:c]
        for h in range(wl.H):
            z = K[:, h // group] @ q[s, h] * wl.scale
            w = np.exp(z - z.max())
            total = w.sum()
            if weights_bf16:
                w = torch.tensor(w, dtype=torch.float32).to(torch.bfloat16).double().numpy()
            out[s, h] = w @ V[:, h // group] / total
    return out


@pytest.mark.parametrize("name", ["tiny", "llama8b_6seqs"])
def test_guard_catches_weights_without_their_lo_part(name):
    wl = workloads.tiny() if name == "tiny" else workloads.llama8b(S=6, num_blocks=1500, new_token=False)
    ref = oracle.decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    exact = _attention(wl, weights_bf16=False)
    assert np.abs(exact - ref).max() < 1e-12
    planted = torch.from_numpy(_attention(wl, weights_bf16=True)).float()
    err = H.check_close(planted, ref, torch.float32, "planted", guard=False)  # the spec bound accepts it
    assert H.GUARD < err < H.TOL
    with pytest.raises(AssertionError, match="guard"):
        H.check_close(planted, ref, torch.float32, "planted")
