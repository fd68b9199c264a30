"""GPU parity: every call of the C ABI against the CPU oracle on the same seeded inputs.

Small cases are compared element by element in full; the full-size workloads
(in the launch configuration the benchmark times) on a sample of sequences the
oracle recomputes one by one. Cache writes and copies must be bit-exact;
attention within 2e-3 (fp32 output) or 2e-3 plus half an output ulp (16-bit
output), and the 16-bit output must equal the rounding of the fp32 output.
"""
import sys
import os

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import gpu_harness as H  # noqa: E402
import oracle  # noqa: E402
from paged_kv_cache_04_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu
LOG2E = 1.4426950408889634


def _no_device_errors(pa):
    assert pa.pa_get_error() == 0


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------
def test_tiny_fp32_full(pa, cuda_device):
    wl = workloads.tiny(device=cuda_device)
    ref = H.Pristine(wl).decode()
    out = H.gpu_step(pa, wl)
    err = H.check_close(out, ref, torch.float32, "tiny")
    assert err < 1e-5  # fp32 data, fp32 accumulation: far inside the bound
    _no_device_errors(pa)


def test_tiny_one_token_context_returns_v(pa, cuda_device):
    wl = workloads.tiny(device=cuda_device)
    out = H.gpu_step(pa, wl)
    b0 = int(wl.block_tables[0, 0])
    for h in range(4):  # MHA: head h reads kv head h; context of one token
        assert torch.equal(out[0, h].cpu(), wl.v_cache[b0, h, 0].cpu())


@pytest.mark.parametrize("out_f32", [False, True])
def test_opt13b_fp16_mha_full(pa, cuda_device, out_f32):
    wl = workloads.opt13b(device=cuda_device)
    H.poison_free_slots(wl)
    ref = H.Pristine(wl).decode()
    out = H.gpu_step(pa, wl, out_dtype=torch.float32 if out_f32 else None)
    H.check_close(out, ref, torch.float32 if out_f32 else torch.float16, "opt13b")
    _no_device_errors(pa)


def test_llama8b_reduced_full(pa, cuda_device):
    """Llama-3.1-8B GQA shape, 48 sequences, every output element checked, NaN in free slots."""
    wl = workloads.llama8b(device=cuda_device, S=48, num_blocks=12_000)
    H.poison_free_slots(wl)
    P = H.Pristine(wl)
    ref = P.decode()
    k0, v0 = wl.k_cache.clone(), wl.v_cache.clone()
    out32 = H.gpu_step(pa, wl, out_dtype=torch.float32)
    H.check_close(out32, ref, torch.float32, "llama8b/48 fp32 out")
    # the same step again from the same cache, with bf16 output
    wl.k_cache.copy_(k0)
    wl.v_cache.copy_(v0)
    out16 = H.gpu_step(pa, wl)
    H.check_close(out16, ref, torch.bfloat16, "llama8b/48 bf16 out")
    assert torch.equal(out16, out32.to(torch.bfloat16)), "bf16 output must be RNE of the fp32 result"
    _no_device_errors(pa)


def test_llama8b_full_size_sampled(pa, cuda_device):
    """The benchmark's workload (256 sequences, 100k-block pool), sampled sequences checked."""
    wl = workloads.llama8b(device=cuda_device)
    seqs = H.sample_seqs(wl, 12)
    P = H.Pristine(wl, seqs)
    out = H.gpu_step(pa, wl)
    ref = P.decode()
    H.check_close(out[seqs], ref, torch.bfloat16, "llama8b full")
    assert torch.isfinite(out.float()).all()
    _no_device_errors(pa)


def test_llama70b_short_full_size_sampled(pa, cuda_device):
    """Plain decode at group 8 (64 q / 8 kv heads) on the benchmark's lengths and
    pool, sampled sequences checked, with bf16 and fp32 output."""
    wl = workloads.llama70b_short(device=cuda_device)
    seqs = H.sample_seqs(wl, 12)
    P = H.Pristine(wl, seqs)
    out = H.gpu_step(pa, wl)
    ref = P.decode()
    H.check_close(out[seqs], ref, torch.bfloat16, "llama70b_short full")
    o32 = torch.empty(wl.q.shape, dtype=torch.float32, device=cuda_device)
    pa.pa_decode(o32, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    H.check_close(o32[seqs], ref, torch.float32, "llama70b_short full, fp32 out")
    assert torch.equal(out, o32.to(torch.bfloat16)), "bf16 output must be the RNE of the fp32 output"
    _no_device_errors(pa)


def test_llama8b_full_size_cache_write_bit_exact(pa, cuda_device):
    wl = workloads.llama8b(device=cuda_device)
    k0, v0 = wl.k_cache.clone(), wl.v_cache.clone()
    pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping)
    torch.cuda.synchronize()
    blocks = torch.unique(wl.slot_mapping // wl.B)
    touched = torch.zeros(wl.num_blocks, dtype=torch.bool, device=cuda_device)
    touched[blocks] = True
    assert torch.equal(wl.k_cache[~touched], k0[~touched])
    assert torch.equal(wl.v_cache[~touched], v0[~touched])
    # touched blocks: oracle on host copies of the pristine blocks
    remap = {int(b): i for i, b in enumerate(blocks.tolist())}
    slots = torch.tensor([remap[int(s) // wl.B] * wl.B + int(s) % wl.B for s in wl.slot_mapping.tolist()])
    kb, vb = oracle.reshape_and_cache(wl.new_key.cpu(), wl.new_value.cpu(), k0[blocks].cpu(),
                                      v0[blocks].cpu(), slots)
    got_k = wl.k_cache[blocks].cpu().view(torch.int16).numpy().view(np.uint16)
    got_v = wl.v_cache[blocks].cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got_k, kb) and np.array_equal(got_v, vb)
    _no_device_errors(pa)


@pytest.mark.parametrize("cow", [False, True])
def test_shared_prefix_reduced_full(pa, cuda_device, cow):
    wl = workloads.shared_prefix(device=cuda_device, prompts=6, samples=8, prefix=2048, tail_hi=512, cow=cow)
    assert wl.meta["cow_copies"] == (6 * 7 if cow else 0)
    H.poison_free_slots(wl)
    P = H.Pristine(wl)
    k_ref, v_ref = P.caches_after_writes()
    ref = P.decode()
    out = H.gpu_step(pa, wl)
    H.check_close(out, ref, torch.bfloat16, f"shared cow={cow}")
    # caches after copy_blocks + reshape_and_cache are bit-exact (all blocks in use)
    idx = torch.tensor(sorted({int(b) for b in wl.block_tables.flatten().tolist() if b >= 0}
                              | {int(b) for b in wl.copy_pairs[:, 0].tolist()}), device=cuda_device)
    assert torch.equal(wl.k_cache.index_select(0, idx).cpu().view(torch.int16), k_ref.view(torch.int16))
    assert torch.equal(wl.v_cache.index_select(0, idx).cpu().view(torch.int16), v_ref.view(torch.int16))
    _no_device_errors(pa)


def test_shared_prefix_full_size_sampled(pa, cuda_device):
    wl = workloads.shared_prefix(device=cuda_device, cow=True)
    assert wl.meta["cow_copies"] == 448
    seqs = [0, 1, 7, 8, 100, 511]
    P = H.Pristine(wl, seqs)
    out = H.gpu_step(pa, wl)
    ref = P.decode()
    H.check_close(out[seqs], ref, torch.bfloat16, "shared full")
    _no_device_errors(pa)


@pytest.mark.parametrize("B", [16, 32])
def test_long70b_split_reduced_full(pa, cuda_device, B):
    wl = workloads.long70b(device=cuda_device, S=3, B=B, lo=4000, hi=9000)
    H.poison_free_slots(wl)
    P = H.Pristine(wl)
    ref = P.decode()
    k0, v0 = wl.k_cache.clone(), wl.v_cache.clone()
    out = H.gpu_step(pa, wl, split=True)
    H.check_close(out, ref, torch.bfloat16, f"long70b split B={B}")
    wl.k_cache.copy_(k0)
    wl.v_cache.copy_(v0)
    out1 = H.gpu_step(pa, wl, out_dtype=torch.float32)
    H.check_close(out1, ref, torch.float32, f"long70b unsplit B={B}")
    _no_device_errors(pa)


@pytest.mark.parametrize("B", [16, 32])
def test_long70b_full_size_sampled(pa, cuda_device, B):
    wl = workloads.long70b(device=cuda_device, B=B)
    seqs = H.sample_seqs(wl, 4)  # the shortest and the longest context and two more
    P = H.Pristine(wl, seqs)
    out = H.gpu_step(pa, wl, split=True)
    ref = P.decode()
    H.check_close(out[seqs], ref, torch.bfloat16, f"long70b full B={B}")
    assert torch.isfinite(out.float()).all()
    _no_device_errors(pa)


# ---------------------------------------------------------------------------
# the split path's partition results against the oracle's per-partition statistics
# ---------------------------------------------------------------------------
def test_split_partials_match_oracle(pa, cuda_device):
    wl = workloads.long70b(device=cuda_device, S=2, lo=1000, hi=2000, partition_tokens=256)
    P = H.Pristine(wl)
    T = 256
    mctx = wl.max_context
    nbytes = pa.pa_decode_split_workspace_bytes(wl.S, wl.H, wl.d, mctx, T)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=cuda_device)
    H.gpu_step(pa, wl, split=True, partition=T, workspace=ws)
    torch.cuda.synchronize()
    Pn = -(-mctx // T)
    rows = wl.S * wl.H * Pn
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    o = ws[:rows * wl.d * 4].view(torch.float32).view(wl.S, wl.H, Pn, wl.d).cpu().numpy()
    m = ws[al(rows * wl.d * 4):al(rows * wl.d * 4) + rows * 4].view(torch.float32).view(wl.S, wl.H, Pn).cpu().numpy()
    off = al(rows * wl.d * 4) + al(rows * 4)
    l = ws[off:off + rows * 4].view(torch.float32).view(wl.S, wl.H, Pn).cpu().numpy()
    ro, rm, rl = P.partitions(T)
    for s in range(wl.S):
        n = -(-int(wl.context_lens[s]) // T)
        assert np.abs(o[s, :, :n] - ro[s, :, :n]).max() <= H.TOL
        assert np.abs(m[s, :, :n] / LOG2E - rm[s, :, :n]).max() <= 1e-4
        assert np.allclose(l[s, :, :n], rl[s, :, :n], rtol=1e-4, atol=1e-4)


def test_split_equals_unsplit_many_partitions(pa, cuda_device):
    wl = workloads.llama8b(device=cuda_device, S=16, num_blocks=6000)
    k0, v0 = wl.k_cache.clone(), wl.v_cache.clone()
    a = H.gpu_step(pa, wl, out_dtype=torch.float32)
    for T in (16, 64, 512, 4096):
        wl.k_cache.copy_(k0)
        wl.v_cache.copy_(v0)
        b = H.gpu_step(pa, wl, out_dtype=torch.float32, split=True, partition=T)
        # same mathematics, different fp32 grouping of the softmax merge
        assert (a - b).abs().max().item() <= 2e-4, f"partition {T}"


# ---------------------------------------------------------------------------
# shapes and paths: head_dim, block size, group, dtype
# ---------------------------------------------------------------------------
SHAPES = [
    # (H, G, d, B, dtype)
    (4, 4, 64, 16, torch.float32), (8, 4, 128, 32, torch.float32), (8, 1, 64, 16, torch.float32),
    (8, 8, 128, 16, torch.float16), (8, 4, 64, 32, torch.float16), (12, 4, 128, 16, torch.float16),
    (16, 4, 128, 16, torch.bfloat16), (32, 4, 64, 16, torch.bfloat16), (16, 2, 128, 32, torch.bfloat16),
    (40, 5, 128, 16, torch.bfloat16), (64, 8, 128, 32, torch.bfloat16), (6, 2, 64, 32, torch.bfloat16),
    # groups of 5-7 and group 8 at head_dim 64: plain decode merges them in two rounds of four heads
    (20, 4, 64, 16, torch.float16), (24, 4, 128, 32, torch.bfloat16), (28, 4, 128, 16, torch.float16),
    (16, 2, 64, 32, torch.bfloat16),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"H{s[0]}G{s[1]}d{s[2]}B{s[3]}{str(s[4])[6:]}")
@pytest.mark.parametrize("split", [False, True])
def test_shape_sweep(pa, cuda_device, shape, split):
    Hh, G, d, B, dt = shape
    ctx = [0, 1, B - 1, B, B + 1, 3 * B, 7 * B + 5, 200, 333, 1000]
    nb = sum(-(-c // B) for c in ctx) + 13
    wl = workloads.batch_with_new_tokens("sweep", len(ctx), Hh, G, d, B, dt, ctx, nb, cuda_device)
    H.poison_free_slots(wl)
    ref = H.Pristine(wl).decode()
    out = H.gpu_step(pa, wl, out_dtype=torch.float32, split=split, partition=4 * B)
    H.check_close(out, ref, torch.float32, f"sweep {shape}")
    assert torch.equal(out[0], torch.zeros_like(out[0])), "empty context must give zeros"
    _no_device_errors(pa)


# ---------------------------------------------------------------------------
# edge cases and device-side range checks
# ---------------------------------------------------------------------------
def test_padding_slots_are_skipped(pa, cuda_device):
    wl = workloads.llama8b(device=cuda_device, S=8, num_blocks=2200)
    k0 = wl.k_cache.clone()
    slots = wl.slot_mapping.clone()
    slots[::2] = -1
    pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, slots)
    torch.cuda.synchronize()
    for t in range(8):
        s = int(wl.slot_mapping[t])
        got = wl.k_cache[s // 16, :, s % 16]
        want = k0[s // 16, :, s % 16] if t % 2 == 0 else wl.new_key[t]
        assert torch.equal(got, want)
    _no_device_errors(pa)


def test_out_of_range_values_are_skipped_and_reported(pa, cuda_device):
    wl = workloads.llama8b(device=cuda_device, S=4, num_blocks=1100)
    pa.pa_get_error()
    bt = wl.block_tables.clone()
    bt[1, 0] = wl.num_blocks + 5
    bt[2, 1] = -7
    out = torch.empty_like(wl.q)
    pa.pa_decode(out, wl.q, wl.k_cache, wl.v_cache, bt, wl.context_lens, wl.scale)
    assert pa.pa_get_error() & pa.PA_DEVERR_BLOCK_ID
    assert pa.pa_get_error() == 0  # cleared by the read
    slots = wl.slot_mapping.clone()
    slots[0] = wl.num_blocks * wl.B
    pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, slots)
    assert pa.pa_get_error() & pa.PA_DEVERR_SLOT
    ctx = wl.context_lens.clone()
    ctx[3] = wl.max_blocks * wl.B + 100
    pa.pa_decode(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, ctx, wl.scale)
    assert pa.pa_get_error() & pa.PA_DEVERR_CONTEXT
    pairs = torch.tensor([[0, 1], [wl.num_blocks, 2]], dtype=torch.int64, device=cuda_device)
    pa.pa_copy_blocks([wl.k_cache], [wl.v_cache], pairs)
    assert pa.pa_get_error() & pa.PA_DEVERR_PAIR
    # the context is still usable afterwards
    out2 = H.gpu_step(pa, workloads.tiny(device=cuda_device))
    assert torch.isfinite(out2).all()


def test_copy_blocks_multi_layer_bit_exact(pa, cuda_device):
    L, nb, G, B, d = 3, 64, 8, 16, 128
    g = torch.Generator(device=cuda_device).manual_seed(0)
    ks = [torch.randn(nb, G, B, d, device=cuda_device, generator=g).to(torch.bfloat16) for _ in range(L)]
    vs = [torch.randn(nb, G, B, d, device=cuda_device, generator=g).to(torch.bfloat16) for _ in range(L)]
    pairs = torch.tensor([[3, 40], [5, 41], [3, 42], [60, 0]], dtype=torch.int64, device=cuda_device)
    rk, rv = oracle.copy_blocks([k.cpu() for k in ks], [v.cpu() for v in vs], pairs.cpu())
    pa.pa_copy_blocks(ks, vs, pairs)
    torch.cuda.synchronize()
    for layer in range(L):
        assert np.array_equal(ks[layer].cpu().view(torch.int16).numpy().view(np.uint16), rk[layer])
        assert np.array_equal(vs[layer].cpu().view(torch.int16).numpy().view(np.uint16), rv[layer])
    _no_device_errors(pa)


def test_deterministic(pa, cuda_device):
    wl = workloads.llama8b(device=cuda_device, S=64, num_blocks=15_000, new_token=False)
    a = H.gpu_step(pa, wl)
    b = H.gpu_step(pa, wl)
    assert torch.equal(a, b)


def test_non_default_stream(pa, cuda_device):
    wl = workloads.llama8b(device=cuda_device, S=16, num_blocks=4000, new_token=False)
    ref = H.gpu_step(pa, wl)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = H.gpu_step(pa, wl, stream=s)
    s.synchronize()
    assert torch.equal(out, ref)


@pytest.mark.parametrize("S", [2048, 2500])
def test_large_batches(pa, cuda_device, S):
    """2048 sequences (the largest batch the kernel orders longest first) and 2500
    (above it: batch order); results must not depend on the order. At 2048 the
    tensor-core case checks every sequence: each CTA keeps the order of its own
    items only, so an item dealt to no CTA would leave its rows unwritten (NaN)."""
    ctx = [int(x) for x in torch.randint(1, 200, (S,), generator=torch.Generator().manual_seed(3))]
    nb = sum(-(-c // 16) for c in ctx) + 10
    for Hh, G in ((8, 2), (32, 8)):  # vector path and tensor-core path
        wl = workloads.batch_with_new_tokens("big", S, Hh, G, 64, 16, torch.bfloat16, ctx, nb, cuda_device,
                                             new_token=False)
        seqs = list(range(S)) if S == 2048 and Hh == 32 else H.sample_seqs(wl, 40)
        ref = H.Pristine(wl, seqs).decode()
        out = H.gpu_step(pa, wl, out_dtype=torch.float32)
        H.check_close(out[seqs], ref, torch.float32, f"S={S} H={Hh} G={G}")
    _no_device_errors(pa)


@pytest.mark.parametrize("G", [200, 512])
def test_many_kv_heads(pa, cuda_device, G):
    """More kv heads than SMs: each CTA keeps the sort order of its own items, at
    most S entries. With 200 heads that still holds every CTA's items (sorted);
    with 512 a CTA is dealt more items than that and the kernel runs the batch
    in batch order. Every sequence against the oracle."""
    S = 64
    ctx = [int(x) for x in torch.randint(1, 120, (S,), generator=torch.Generator().manual_seed(5))]
    nb = sum(-(-c // 16) for c in ctx) + 4
    wl = workloads.batch_with_new_tokens("heads", S, G, G, 64, 16, torch.float16, ctx, nb, cuda_device)
    ref = H.Pristine(wl).decode()
    out = H.gpu_step(pa, wl, out_dtype=torch.float32)
    H.check_close(out, ref, torch.float32, f"G={G}")
    _no_device_errors(pa)


def test_all_contexts_empty(pa, cuda_device):
    """A batch in which no sequence has a token yet: every output row is zero, plain and split."""
    wl = workloads.batch_with_new_tokens("empty", 6, 32, 8, 128, 16, torch.bfloat16, [0] * 6, 8, cuda_device,
                                         new_token=False)
    for split in (False, True):
        out = H.gpu_step(pa, wl, out_dtype=torch.float32, split=split, partition=64)
        assert torch.equal(out, torch.zeros_like(out))
    _no_device_errors(pa)


def test_one_long_sequence_plain(pa, cuda_device):
    """A single 64K-token sequence through the single-pass kernel (8 work items for
    the whole GPU): long items, a last block of one token."""
    ctx = [65537]
    nb = -(-ctx[0] // 16) + 5
    wl = workloads.batch_with_new_tokens("long1", 1, 32, 8, 128, 16, torch.bfloat16, ctx, nb, cuda_device)
    ref = H.Pristine(wl).decode()
    out = H.gpu_step(pa, wl, out_dtype=torch.float32)
    H.check_close(out, ref, torch.float32, "one 64K sequence")
    _no_device_errors(pa)


def test_mha_split_at_the_batch_limit(pa, cuda_device):
    """MHA split decode at 2,048 sequences, the largest batch split mode takes
    (the tensor-core path at group 1, its per-sequence schedule in shared
    memory): every sequence against the oracle, several partitions each, the
    output filled with NaN first."""
    S = 2048
    ctx = [int(x) for x in torch.randint(1, 160, (S,), generator=torch.Generator().manual_seed(9))]
    nb = sum(-(-c // 16) for c in ctx) + 4
    wl = workloads.batch_with_new_tokens("mha_split", S, 8, 8, 128, 16, torch.float16, ctx, nb, cuda_device)
    ref = H.Pristine(wl).decode()
    out = H.gpu_step(pa, wl, out_dtype=torch.float32, split=True, partition=32)
    H.check_close(out, ref, torch.float32, "MHA split S=2048")
    _no_device_errors(pa)


def test_split_rejects_batches_above_its_limit(pa, cuda_device):
    S = 2049
    wl = workloads.batch_with_new_tokens("wide", S, 8, 8, 64, 16, torch.bfloat16, [3] * S, S + 2, cuda_device,
                                         new_token=False)
    with pytest.raises(pa.PAError):
        H.gpu_step(pa, wl, split=True, partition=64)
