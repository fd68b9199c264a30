"""pa_decode_split_static: the split decode for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run attention (a plugin whose
host framework owns every device allocation, a serving loop that must stay out
of the allocator once running). For them the library keeps the split path's
partition results in a scratch array of its own instead of a caller workspace.
These tests call that entry point through the C ABI and compare it with
pa_decode_split (caller workspace) on two calls in a row with different inputs,
so the second call runs on a scratch array still holding the first call's
results. This file is collected last on purpose.
"""
import os
import sys

import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import gpu_harness as H  # noqa: E402
from paged_kv_cache_04_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


def _reference(pa, wl, T, out_dtype):
    out = torch.empty(wl.q.shape, dtype=out_dtype, device=wl.q.device)
    ws = torch.empty(pa.pa_decode_split_workspace_bytes(wl.S, wl.H, wl.d, wl.max_context, T),
                     dtype=torch.uint8, device=wl.q.device)
    pa.pa_decode_split(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                       wl.max_context, T, ws)
    return out


def _static(pa, wl, T, out_dtype):
    out = torch.empty(wl.q.shape, dtype=out_dtype, device=wl.q.device)
    pa.pa_decode_split_static(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                              wl.max_context, T)
    return out


def test_static_scratch_matches_workspace_two_calls(pa, cuda_device):
    T = 512
    first = workloads.long70b(device=cuda_device, S=4, lo=9000, hi=20000, new_token=False)
    second = workloads.llama8b(device=cuda_device, S=24, num_blocks=7000, new_token=False)
    for wl, out_dtype in ((first, torch.bfloat16), (second, torch.float32)):
        need = pa.pa_decode_split_workspace_bytes(wl.S, wl.H, wl.d, wl.max_context, T)
        assert 0 < need <= pa.PA_STATIC_SCRATCH_BYTES
        ref = _reference(pa, wl, T, out_dtype)
        got = _static(pa, wl, T, out_dtype)
        torch.cuda.synchronize()
        H.check_close(got, ref.double().cpu().numpy(), out_dtype, f"static scratch vs workspace ({wl.name})")
    assert pa.pa_get_error() == 0


def test_static_scratch_rejects_oversize_requests(pa, cuda_device):
    wl = workloads.llama8b(device=cuda_device, S=4, num_blocks=1200, new_token=False)
    # 4 x 32 heads x 128 dims with 1,024 partitions needs ~66 MB, more than the array
    huge_ctx = 1024 * 512
    assert pa.pa_decode_split_workspace_bytes(wl.S, wl.H, wl.d, huge_ctx, 512) > pa.PA_STATIC_SCRATCH_BYTES
    out = torch.full(wl.q.shape, 7.0, dtype=wl.q.dtype, device=cuda_device)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_split_static(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                                  wl.scale, huge_ctx, 512)
    assert e.value.status == 2  # PA_ERR_UNSUPPORTED, and nothing was launched:
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())


def test_static_call_allocates_no_device_memory(pa, cuda_device):
    """After a first call (which may load the library's device code and commit
    the array), a further call changes neither torch's allocator count nor the
    device's free memory."""
    T = 512
    wl = workloads.long70b(device=cuda_device, S=4, lo=9000, hi=20000, new_token=False)
    out = torch.empty(wl.q.shape, dtype=torch.float32, device=cuda_device)
    args = (out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, wl.max_context, T)
    pa.pa_decode_split_static(*args)
    torch.cuda.synchronize()
    ref = out.clone()
    alloc0 = torch.cuda.memory_allocated(cuda_device)
    free0, _ = torch.cuda.mem_get_info(cuda_device)
    pa.pa_decode_split_static(*args)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated(cuda_device) == alloc0
    free1, _ = torch.cuda.mem_get_info(cuda_device)
    assert free1 == free0, (free0, free1)
    assert torch.equal(out, ref)  # the same inputs give the same bits
