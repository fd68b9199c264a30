"""Algorithmic byte counts for the kernels' roofline (bytes that must cross HBM).

The per-token KV size is 2 (K and V) x layers x kv heads x head dim x element
bytes (Month 2 · PagedAttention, infra learning path, §2.1); one physical block
of one layer holds block_size tokens of it (same page, §5.2).
"""
from __future__ import annotations


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, dtype_bytes: int) -> int:
    return 2 * num_layers * num_kv_heads * head_dim * dtype_bytes


def kv_block_bytes(block_size: int, num_kv_heads: int, head_dim: int, dtype_bytes: int) -> int:
    """K plus V of one physical block of one layer."""
    return block_size * kv_bytes_per_token(1, num_kv_heads, head_dim, dtype_bytes)


def decode_bytes(context_lens, H, G, d, dtype_bytes, out_bytes=None) -> int:
    """Decode attention: the K/V of every attended token, plus q in and out.

    Block-table and context-length reads (4 B per entry) are left out: they are
    below 0.01% of the total at every shape used here.
    """
    out_bytes = dtype_bytes if out_bytes is None else out_bytes
    tokens = int(sum(int(c) for c in context_lens))
    S = len(context_lens)
    return (tokens * kv_bytes_per_token(1, G, d, dtype_bytes)
            + S * H * d * dtype_bytes + S * H * d * out_bytes)


def reshape_and_cache_bytes(num_tokens, G, d, dtype_bytes) -> int:
    """New K and V rows read once and written once, plus the 8-byte slot per token."""
    return 2 * 2 * num_tokens * G * d * dtype_bytes + 8 * num_tokens


def copy_blocks_bytes(num_pairs, num_layers, block_size, G, d, dtype_bytes) -> int:
    """Each pair reads and writes one K and one V block per layer."""
    return 2 * num_pairs * num_layers * kv_block_bytes(block_size, G, d, dtype_bytes)


def split_workspace_bytes(S, H, d, num_partitions) -> int:
    """fp32 partial outputs plus the (max, sum) pair, written by pass 1 and read by the reduce."""
    return S * H * num_partitions * (d + 2) * 4
