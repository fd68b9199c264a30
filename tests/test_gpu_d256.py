"""head_dim 256 on the GPU: every decode path against the oracle.

A 16-token job of a 256-wide head is 16 KiB (16-bit) or 32 KiB (fp32), so the
kernels run one stage per warp; MHA keeps q in shared memory. The shapes cover
the vector path (group 1 and 2, as in Gemma-style models), the tensor-core path
(group 4 and 8) and fp32, both block sizes, ragged contexts (empty, one token,
a partial last block, several partitions), plain and split decode, HND and NHD.
"""
import os
import sys

import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import gpu_harness as H  # noqa: E402
from paged_kv_cache_04_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu

SHAPES = [
    # (H, G, B, dtype)
    (16, 16, 16, torch.bfloat16),   # MHA
    (16, 8, 16, torch.bfloat16),    # group 2
    (16, 8, 32, torch.float16),
    (32, 8, 16, torch.bfloat16),    # group 4: tensor cores
    (16, 2, 32, torch.float16),     # group 8: tensor cores
    (4, 4, 16, torch.float32),      # fp32 MHA
    (8, 2, 16, torch.float32),      # fp32 group 4 (vector path)
]
CTX = [0, 1, 15, 16, 17, 31, 33, 100, 257, 700, 1500, 2049]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"H{s[0]}G{s[1]}B{s[2]}{str(s[3])[6:]}")
@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("out_f32", [True, False])
def test_d256_matches_oracle(pa, cuda_device, shape, split, out_f32):
    Hh, G, B, dt = shape
    ctx = CTX
    nb = sum(-(-c // B) for c in ctx) + 11
    wl = workloads.batch_with_new_tokens(f"d256-{Hh}-{G}-{B}", len(ctx), Hh, G, 256, B, dt, ctx, nb, cuda_device)
    H.poison_free_slots(wl)
    ref = H.Pristine(wl).decode()
    odt = torch.float32 if out_f32 else dt
    out = H.gpu_step(pa, wl, out_dtype=odt, split=split, partition=8 * B)
    H.check_close(out, ref, odt, f"d256 {shape} split={split}")
    assert pa.pa_get_error() == 0


@pytest.mark.parametrize("shape", [(16, 8, 16, torch.bfloat16), (32, 8, 16, torch.bfloat16)],
                         ids=["group2", "group4"])
def test_d256_nhd_bit_identical(pa, cuda_device, shape):
    Hh, G, B, dt = shape
    ctx = [3, 16, 40, 600, 1111]
    nb = sum(-(-c // B) for c in ctx) + 5
    hnd = workloads.batch_with_new_tokens("d256nhd", len(ctx), Hh, G, 256, B, dt, ctx, nb, cuda_device)
    H.poison_free_slots(hnd)
    nhd = workloads.to_nhd(hnd)
    ref = H.Pristine(nhd).decode()
    for split in (False, True):
        a = H.gpu_step(pa, nhd, out_dtype=torch.float32, split=split, partition=256)
        b = H.gpu_step(pa, hnd, out_dtype=torch.float32, split=split, partition=256)
        H.check_close(a, ref, torch.float32, f"d256 nhd split={split}")
        assert torch.equal(a, b)
    assert pa.pa_get_error() == 0


def test_d256_full_size_sampled(pa, cuda_device):
    """The head_dim-256 benchmark batch (256 sequences, 16 q / 8 kv heads, contexts
    U[512, 4096]): sampled sequences against the oracle, plain and split."""
    wl = workloads.gemma_d256(device=cuda_device)
    seqs = H.sample_seqs(wl, 6)
    P = H.Pristine(wl, seqs)
    ref = P.decode()
    out = H.gpu_step(pa, wl)
    H.check_close(out[seqs], ref, torch.bfloat16, "d256 full")
    out_s = H.gpu_step(pa, wl, split=True, partition=512)
    H.check_close(out_s[seqs], ref, torch.bfloat16, "d256 full split")
    assert pa.pa_get_error() == 0


def test_d256_rejected_where_unsupported(pa, cuda_device):
    """E4M3 caches and the shared-prefix decode stop at head_dim 128."""
    wl = workloads.batch_with_new_tokens("d256r", 2, 16, 8, 256, 16, torch.bfloat16, [5, 20], 4, cuda_device)
    q8 = workloads.to_fp8(wl)
    out = torch.empty(wl.q.shape, dtype=torch.float32, device=cuda_device)
    with pytest.raises(RuntimeError, match="unsupported"):
        pa.pa_decode_fp8(out, q8.q, q8.k_cache, q8.v_cache, q8.block_tables, q8.context_lens, q8.scale,
                         q8.meta["k_scale"], q8.meta["v_scale"])
