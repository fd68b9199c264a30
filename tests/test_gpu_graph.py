"""A decode step captured in a CUDA graph replays to the same bits as the
eager calls. Every kernel of the library is launched with programmatic
dependent launch, so capture turns the stream order into programmatic edges;
the replay must still see each kernel's writes before the next one reads."""
import os
import sys

import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import gpu_harness as H  # noqa: E402
from paged_kv_cache_04_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


def _step(pa, wl, out, ws, T):
    pa.pa_copy_blocks([wl.k_cache], [wl.v_cache], wl.copy_pairs)
    pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping)
    pa.pa_decode_split(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                       wl.meta["mctx"], T, ws)


def test_graph_replay_matches_eager(pa, cuda_device):
    T = 128
    eager = workloads.shared_prefix(device=cuda_device, prompts=4, samples=8, prefix=300, tail_hi=200, cow=True)
    graph = workloads.shared_prefix(device=cuda_device, prompts=4, samples=8, prefix=300, tail_hi=200, cow=True)
    for wl in (eager, graph):
        wl.meta["mctx"] = wl.max_context
    ref = H.Pristine(eager).decode()
    ws_bytes = pa.pa_decode_split_workspace_bytes(eager.S, eager.H, eager.d, eager.meta["mctx"], T)
    out_e = torch.empty(eager.q.shape, dtype=torch.float32, device=cuda_device)
    ws_e = torch.empty(ws_bytes, dtype=torch.uint8, device=cuda_device)
    _step(pa, eager, out_e, ws_e, T)
    torch.cuda.synchronize()

    out_g = torch.full(graph.q.shape, float("nan"), dtype=torch.float32, device=cuda_device)
    ws_g = torch.empty(ws_bytes, dtype=torch.uint8, device=cuda_device)
    pa.pa_get_error()  # first call on the device happens before capture
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            _step(pa, graph, out_g, ws_g, T)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.isnan(out_g).all(), "capture must not run the kernels"
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g, out_e)
    assert torch.equal(graph.k_cache, eager.k_cache) and torch.equal(graph.v_cache, eager.v_cache)
    H.check_close(out_g, ref, torch.float32, "graph replay")
    # replaying again (the copies and writes are idempotent) gives the same bits
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g, out_e)
    assert pa.pa_get_error() == 0


@pytest.mark.parametrize("samples", [8, 16], ids=["mma_sync_prefix", "tcgen05_prefix"])
def test_graph_replay_cascade(pa, cuda_device, samples):
    """Shared-prefix decode (prefix pass, suffix pass, reduce) captured after one
    eager call: the replay gives the eager bits, on both prefix passes."""
    T = 256

    def make():
        return workloads.shared_prefix(device=cuda_device, prompts=3, samples=samples, prefix=900, tail_hi=150,
                                       cow=True)

    eager, graph = make(), make()
    ref = H.Pristine(eager).decode()
    gs = torch.tensor(eager.meta["group_starts"], dtype=torch.int32, device=cuda_device)
    pl = torch.tensor(eager.meta["prefix_lens"], dtype=torch.int32, device=cuda_device)
    pmax, mctx = max(eager.meta["prefix_lens"]), eager.max_context
    ws_bytes = pa.pa_decode_cascade_workspace_bytes(eager.S, eager.H, eager.d, pmax, mctx, T)

    def step(wl, out, ws):
        pa.pa_copy_blocks([wl.k_cache], [wl.v_cache], wl.copy_pairs)
        pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping)
        pa.pa_decode_cascade(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, gs,
                             pl, samples, pmax, mctx, T, ws)

    out_e = torch.empty(eager.q.shape, dtype=torch.float32, device=cuda_device)
    step(eager, out_e, torch.empty(ws_bytes, dtype=torch.uint8, device=cuda_device))
    torch.cuda.synchronize()
    out_g = torch.full(graph.q.shape, float("nan"), dtype=torch.float32, device=cuda_device)
    ws_g = torch.empty(ws_bytes, dtype=torch.uint8, device=cuda_device)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step(graph, out_g, ws_g)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.isnan(out_g).all(), "capture must not run the kernels"
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_g, out_e)
    H.check_close(out_g, ref, torch.float32, f"graph cascade {samples}")
    assert pa.pa_get_error() == 0
