"""The bounded waits on the GPU: a wait that nothing completes runs out, is
reported in the error word, pulls the CTA's other warp out through the abort
flag, and leaves the CUDA context usable for the next call."""
import os
import sys
import time

import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import gpu_harness as H  # noqa: E402
from paged_kv_cache_04_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ms", [2, 20])
def test_wait_runs_out_and_is_reported(pa, cuda_device, limit_ms):
    assert pa.pa_get_error() == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pa.pa_check_wait_limit(limit_ms * 1_000_000)
    bits = pa.pa_get_error()  # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert bits == pa.PA_DEVERR_TIMEOUT
    # warp 0 gave up after the limit; warp 1 (50 x the limit) followed it through
    # the abort flag instead of running out its own limit
    assert limit_ms * 1e-3 <= elapsed < 10 * limit_ms * 1e-3 + 0.05


def test_context_usable_after_a_timeout(pa, cuda_device):
    pa.pa_check_wait_limit(5_000_000)
    assert pa.pa_get_error() == pa.PA_DEVERR_TIMEOUT
    wl = workloads.tiny(device=cuda_device)
    ref = H.Pristine(wl).decode()
    out = H.gpu_step(pa, wl, out_dtype=torch.float32)
    H.check_close(out, ref, torch.float32, "decode after a timeout")
    assert pa.pa_get_error() == 0
