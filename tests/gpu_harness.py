"""Shared helpers for the GPU parity tests: run a step through the C ABI, and
run the same step through the CPU oracle on inputs that never pass through the
CUDA path (the oracle sees the pool as it was drawn, before any kernel ran).
"""
import numpy as np
import torch

import oracle

TOL = 2e-3  # max abs error of the fp32 result, bf16/fp16 inputs with fp32 accumulation
# Regression guard, far inside TOL: the kernels accumulate in fp32 and carry the
# softmax weights as hi + lo 16-bit parts, which keeps their error near 1e-6 on
# these inputs. A loss of precision that TOL would still accept (weights rounded
# to one 16-bit part, a 16-bit accumulator) lands between 1e-4 and 2e-3 and
# fails here.
GUARD = 1e-4


def half_ulp(x, dtype):
    """Half a unit in the last place of ``dtype`` at |x| (numpy float64 array)."""
    ax = np.maximum(np.abs(x), 1e-30)
    e = np.floor(np.log2(ax))
    if dtype == torch.bfloat16:
        return np.exp2(np.maximum(e, -126) - 8)
    if dtype == torch.float16:
        return np.exp2(np.maximum(e, -14) - 11)
    return np.exp2(np.maximum(e, -126) - 24)


def check_close(gpu, ref, dtype, what="", guard=True):
    """fp32 output: |gpu - ref| <= 2e-3; 16-bit output: plus half an ulp of the output type.
    With ``guard`` the error beyond the output rounding must also stay within GUARD."""
    g = gpu.detach().float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    rounding = half_ulp(ref, dtype) if dtype in (torch.bfloat16, torch.float16) else 0.0
    bad = err > TOL + rounding
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside tolerance, "
                           f"max err {err.max():.3e}")
    if guard:
        excess = float(np.max(err - rounding)) if err.size else 0.0
        assert excess <= GUARD, f"{what}: error {excess:.3e} beyond the output rounding exceeds the guard {GUARD:.0e}"
    return float(err.max())


def gpu_step(pa, wl, out_dtype=None, split=False, partition=None, workspace=None, stream=None):
    """copy_blocks -> reshape_and_cache -> decode on the GPU, in place on wl's caches."""
    if wl.copy_pairs is not None and wl.copy_pairs.numel():
        pa.pa_copy_blocks([wl.k_cache], [wl.v_cache], wl.copy_pairs, stream=stream)
    if wl.slot_mapping is not None:
        pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping,
                                stream=stream, layout=wl.layout)
    # NaN in every output row first: a row that no kernel wrote fails check_close
    out = torch.full(wl.q.shape, float("nan"), dtype=out_dtype or wl.dtype, device=wl.q.device)
    if split:
        T = partition or wl.partition_tokens or 512
        mctx = wl.max_context
        if workspace is None:
            nbytes = pa.pa_decode_split_workspace_bytes(wl.S, wl.H, wl.d, mctx, T)
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=wl.q.device)
        pa.pa_decode_split(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                           mctx, T, workspace, stream=stream, layout=wl.layout)
    else:
        pa.pa_decode(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                     stream=stream, layout=wl.layout)
    return out


class Pristine:
    """Host copies of a workload's inputs taken before any kernel touched them."""

    def __init__(self, wl, seqs=None):
        S = wl.S
        self.seqs = list(range(S)) if seqs is None else list(seqs)
        B = wl.B
        bt = wl.block_tables.cpu()
        ctx = wl.context_lens.cpu()
        used = set()
        for s in self.seqs:
            n = -(-int(ctx[s]) // B)
            used.update(int(b) for b in bt[s, :n].tolist())
        pairs = None
        if wl.copy_pairs is not None and wl.copy_pairs.numel():
            pairs = wl.copy_pairs.cpu()
            keep = [i for i in range(pairs.shape[0]) if int(pairs[i, 1]) in used]
            pairs = pairs[keep]
            used.update(int(b) for b in pairs[:, 0].tolist())
        blocks = sorted(used)
        remap = {b: i for i, b in enumerate(blocks)}
        idx = torch.tensor(blocks, dtype=torch.long, device=wl.k_cache.device)
        self.k = wl.k_cache.index_select(0, idx).cpu()
        self.v = wl.v_cache.index_select(0, idx).cpu()
        self.nb = len(blocks)
        self.q = wl.q.cpu()[self.seqs]
        width = bt.shape[1]
        nbt = torch.full((len(self.seqs), width), -1, dtype=torch.int32)
        for i, s in enumerate(self.seqs):
            n = -(-int(ctx[s]) // B)
            nbt[i, :n] = torch.tensor([remap[int(b)] for b in bt[s, :n].tolist()], dtype=torch.int32)
        self.bt = nbt
        self.ctx = ctx[self.seqs].clone()
        self.pairs = None if pairs is None else torch.tensor(
            [[remap[int(a)], remap[int(b)]] for a, b in pairs.tolist()], dtype=torch.int64).view(-1, 2)
        self.new = None
        if wl.slot_mapping is not None:
            slots = wl.slot_mapping.cpu()
            keep, nslots = [], []
            for t, sl in enumerate(slots.tolist()):
                if sl >= 0 and sl // B in remap:
                    keep.append(t)
                    nslots.append(remap[sl // B] * B + sl % B)
            kt = torch.tensor(keep, dtype=torch.long)
            self.new = (wl.new_key.cpu()[kt], wl.new_value.cpu()[kt], torch.tensor(nslots, dtype=torch.int64))
        self.B, self.scale, self.dtype, self.layout = B, wl.scale, wl.dtype, wl.layout

    def caches_after_writes(self):
        """Oracle: CoW copies, then new-token writes, on the host copies (bit patterns)."""
        k, v = self.k, self.v
        if self.pairs is not None and self.pairs.numel():
            ks, vs = oracle.copy_blocks([k], [v], self.pairs)
            k, v = _from_bits(ks[0], self.dtype), _from_bits(vs[0], self.dtype)
        if self.new is not None:
            kb, vb = oracle.reshape_and_cache(self.new[0], self.new[1], k, v, self.new[2], layout=self.layout)
            k, v = _from_bits(kb, self.dtype), _from_bits(vb, self.dtype)
        return k, v

    def decode(self, num_threads=0):
        k, v = self.caches_after_writes()
        return oracle.decode(self.q, k, v, self.bt, self.ctx, self.scale, num_threads=num_threads,
                             layout=self.layout)

    def partitions(self, T):
        k, v = self.caches_after_writes()
        return oracle.partitions(self.q, k, v, self.bt, self.ctx, self.scale, T, layout=self.layout)


def _from_bits(bits, dtype):
    a = np.ascontiguousarray(bits)
    if dtype == torch.float32:
        return torch.from_numpy(a.view(np.float32))
    return torch.from_numpy(a.view(np.int16)).view(dtype)


def poison_free_slots(wl, value=float("nan")):
    """Fill every pool row that no sequence's context covers with ``value``."""
    B = wl.B
    bt = wl.block_tables.cpu()
    ctx = wl.context_lens.cpu()
    live = torch.zeros(wl.num_blocks, B, dtype=torch.bool)
    for s in range(wl.S):
        c = int(ctx[s])
        n = -(-c // B)
        if n == 0:
            continue
        live[bt[s, :n].long()] = True
        tail = c - (n - 1) * B
        live[int(bt[s, n - 1]), tail:] = False
    shape = (wl.num_blocks, 1, B, 1) if wl.layout == "HND" else (wl.num_blocks, B, 1, 1)
    mask = (~live).to(wl.k_cache.device).view(*shape)
    wl.k_cache.masked_fill_(mask, value)
    wl.v_cache.masked_fill_(mask, value)


def sample_seqs(wl, n, seed=7):
    """The longest and shortest sequences plus a seeded random sample."""
    ctx = wl.context_lens.cpu()
    order = torch.argsort(ctx)
    pick = {int(order[0]), int(order[-1])}
    g = torch.Generator().manual_seed(seed)
    for i in torch.randperm(wl.S, generator=g).tolist():
        if len(pick) >= n:
            break
        pick.add(i)
    return sorted(pick)

