"""Oracle for the cache-maintenance writes: plain element copies on host arrays.

Test infrastructure: see the header of ``oracle/__init__.py``.

The pages name three fused GPU operations around paged attention (CS349E
Lecture 7 notes, §4.3 "代价：间接寻址"): writing each new token's K/V into its
block slot, attention that reads through the block table, and the batched
copy of the blocks that copy-on-write must duplicate. The two writes are
plain data movement, so their oracle is that movement written out, one token
row or one block at a time, on raw bit patterns (bit-exact by construction).
"""
import numpy as np


def _bits(x):
    """Host numpy view of a tensor/array with the same bytes (16-bit floats as uint16)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            t = x.detach().to("cpu").contiguous()
            if t.element_size() == 2:
                return t.view(torch.int16).numpy().view(np.uint16).copy()
            if t.element_size() == 4 and t.is_floating_point():
                return t.view(torch.int32).numpy().view(np.uint32).copy()
            return t.numpy().copy()
    except ImportError:  # pragma: no cover
        pass
    a = np.array(x, copy=True)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype == np.float32:
        return a.view(np.uint32)
    return a


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, layout="HND"):
    """Return new (k_cache, v_cache) bit arrays after writing every new token.

    key, value: [N, G, d]; caches: [num_blocks, G, B, d] (HND) or
    [num_blocks, B, G, d] (NHD; Month 2 · PagedAttention §5.2 names both).
    For token t with slot = slot_mapping[t] >= 0: block = slot // B, row = slot % B,
    and cache[block, h, row, :] = key[t, h, :] for every kv head h (CS349E
    Lecture 7 notes §4.1: a slot is a position inside a physical block; CMU
    15-779 Lecture 16 notes §3.3: new tokens fill the last block's free rows).
    A negative slot means "no write" (a padding token).
    """
    kb, vb = _bits(key), _bits(value)
    kc, vc = _bits(k_cache), _bits(v_cache)
    slots = np.asarray(_bits(slot_mapping), dtype=np.int64)
    if layout not in ("HND", "NHD"):
        raise ValueError(f"unknown layout {layout!r}")
    nhd = layout == "NHD"
    if nhd:
        nb, B, G, d = kc.shape
    else:
        nb, G, B, d = kc.shape
    N = kb.shape[0]
    if kb.shape != (N, G, d) or vb.shape != kb.shape or slots.shape != (N,) or vc.shape != kc.shape:
        raise ValueError("shape mismatch")
    for t in range(N):
        slot = int(slots[t])
        if slot < 0:
            continue
        block, row = divmod(slot, B)
        if block >= nb:
            raise IndexError(f"slot {slot} outside a pool of {nb} blocks of {B}")
        for h in range(G):
            if nhd:
                kc[block, row, h, :] = kb[t, h, :]
                vc[block, row, h, :] = vb[t, h, :]
            else:
                kc[block, h, row, :] = kb[t, h, :]
                vc[block, h, row, :] = vb[t, h, :]
    return kc, vc


def copy_blocks(k_caches, v_caches, block_pairs):
    """Return new per-layer (k, v) bit arrays after the copy-on-write block copies.

    For every pair (src, dst) and every layer: cache[dst] = cache[src], all kv
    heads and rows (CS349E Lecture 7 notes §5.1: a sample writing into a shared
    block first gets its own copy; §4.3: the pending copies go in one batch).
    The pairs must not chain (no dst is also a src), so their order is irrelevant.
    """
    pairs = np.asarray(_bits(block_pairs), dtype=np.int64).reshape(-1, 2)
    ks = [_bits(k) for k in k_caches]
    vs = [_bits(v) for v in v_caches]
    for layer in range(len(ks)):
        src_k, src_v = ks[layer].copy(), vs[layer].copy()
        nb = ks[layer].shape[0]
        for src, dst in pairs:
            if not (0 <= src < nb and 0 <= dst < nb):
                raise IndexError(f"pair ({src}, {dst}) outside a pool of {nb} blocks")
            ks[layer][dst] = src_k[src]
            vs[layer][dst] = src_v[src]
    return ks, vs


def swap_blocks(dst_k_caches, dst_v_caches, src_k_caches, src_v_caches, block_pairs):
    """Return new per-layer destination (k, v) bit arrays after moving blocks between pools.

    For every pair (src, dst) and layer: dst_pool[dst] = src_pool[src], K and V
    (CS349E Lecture 7 notes §6.2: a preempted sequence's blocks are copied to
    CPU memory and later back). The source pools are not modified.
    """
    pairs = np.asarray(_bits(block_pairs), dtype=np.int64).reshape(-1, 2)
    dks = [_bits(k) for k in dst_k_caches]
    dvs = [_bits(v) for v in dst_v_caches]
    for layer in range(len(dks)):
        sk, sv = _bits(src_k_caches[layer]), _bits(src_v_caches[layer])
        for src, dst in pairs:
            if not (0 <= src < sk.shape[0] and 0 <= dst < dks[layer].shape[0]):
                raise IndexError(f"pair ({src}, {dst}) outside its pool")
            dks[layer][dst] = sk[src]
            dvs[layer][dst] = sv[src]
    return dks, dvs


def kv_bytes_per_token(num_layers, num_kv_heads, head_dim, dtype_bytes):
    """KV-cache bytes one token occupies: 2 (K and V) x layers x kv heads x head dim x bytes.

    Month 2 · PagedAttention (infra learning path) §2.1; CS349E Lecture 7 notes §1.
    """
    return 2 * num_layers * num_kv_heads * head_dim * dtype_bytes
