"""GB300 paged KV-cache library: Python binding of the C ABI in ``include/pa.h``.

The functions below carry the C entry points' names and only marshal
arguments (shapes, dtypes, data pointers, the current CUDA stream); every step
of the computation runs in the CUDA kernels of ``libpa.so``. There is no CPU
fallback: if the library is missing or cannot load, every call raises.

Tensors are ``torch`` CUDA tensors in the layouts the header documents:

* ``q``, ``out``                 ``[num_seqs, num_heads, head_dim]``
* ``k_cache``, ``v_cache``       ``[num_blocks, num_kv_heads, block_size, head_dim]`` (``layout="HND"``,
  the default) or ``[num_blocks, block_size, num_kv_heads, head_dim]`` (``layout="NHD"``)
* ``block_tables``               int32 ``[num_seqs, max_blocks_per_seq]``
* ``context_lens``               int32 ``[num_seqs]``
* ``key``, ``value``             ``[num_tokens, num_kv_heads, head_dim]``
* ``slot_mapping``               int64 ``[num_tokens]``
* ``block_pairs``                int64 ``[num_pairs, 2]``
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "PAError", "library", "library_path", "pa_reshape_and_cache", "pa_decode", "pa_decode_split",
    "pa_decode_split_workspace_bytes", "pa_decode_split_static", "pa_copy_blocks", "pa_swap_blocks",
    "pa_reshape_and_cache_fp8", "pa_decode_fp8", "pa_decode_split_fp8", "pa_decode_cascade",
    "pa_decode_cascade_workspace_bytes", "pa_get_error", "pa_check_wait_limit",
    "pa_version", "PA_STATIC_SCRATCH_BYTES", "PA_LAYOUT_HND", "PA_LAYOUT_NHD",
    "PA_DEVERR_BLOCK_ID", "PA_DEVERR_SLOT", "PA_DEVERR_CONTEXT", "PA_DEVERR_PAIR", "PA_DEVERR_TIMEOUT",
    "PA_DEVERR_PAIR_ALIAS", "pa_debug_check", "pa_status_str",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libpa.so")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_OUT_OF_RANGE, PA_ERR_CUDA = range(5)
PA_F32, PA_F16, PA_BF16, PA_FP8_E4M3 = 0, 1, 2, 3
PA_LAYOUT_HND, PA_LAYOUT_NHD = 0, 1
PA_DEVERR_BLOCK_ID, PA_DEVERR_SLOT, PA_DEVERR_CONTEXT, PA_DEVERR_PAIR, PA_DEVERR_TIMEOUT = 1, 2, 4, 8, 16
PA_DEVERR_PAIR_ALIAS = 32

_lib = None


class PAError(RuntimeError):
    def __init__(self, func, status, detail=""):
        names = {1: "invalid argument", 2: "unsupported configuration", 3: "device-side value out of range",
                 4: "CUDA error"}
        super().__init__(f"{func}: {names.get(status, status)}{(' (' + detail + ')') if detail else ''}")
        self.status = status


def library():
    """Load ``libpa.so`` (raises if it is absent: build it with ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise PAError("load", PA_ERR_CUDA, f"{library_path} not built")
    lib = ctypes.CDLL(library_path)
    P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.pa_reshape_and_cache.argtypes = [P, P, P, P, P, I, I, I, I, I, I64, I, P]
    lib.pa_decode.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I64, F, I, I, P]
    lib.pa_decode_split_workspace_bytes.argtypes = [I, I, I, I, I]
    lib.pa_decode_split_workspace_bytes.restype = SZ
    lib.pa_decode_split.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I64, F, I, I, I, I, P, SZ, P]
    lib.pa_decode_split_static.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I64, F, I, I, I, I, P]
    lib.pa_copy_blocks.argtypes = [P, P, I, P, I, I, I, I, I64, I, P]
    lib.pa_swap_blocks.argtypes = [P, P, P, P, I, P, I, I, I, I, I64, I64, I, P]
    lib.pa_reshape_and_cache_fp8.argtypes = [P, P, P, P, P, I, I, I, I, I, I64, I, F, F, P]
    lib.pa_decode_fp8.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I64, F, F, F, I, I, P]
    lib.pa_decode_split_fp8.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I64, F, F, F, I, I, I, I, P, SZ, P]
    lib.pa_decode_cascade_workspace_bytes.argtypes = [I, I, I, I, I, I]
    lib.pa_decode_cascade_workspace_bytes.restype = SZ
    lib.pa_decode_cascade.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I64, F, I, I, P, P, I, I, I, I, I, P,
                                      SZ, P]
    lib.pa_get_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), P]
    lib.pa_check_wait_limit.argtypes = [ctypes.c_uint64, P]
    lib.pa_status_string.argtypes = [I]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_status_str.argtypes = [I]
    lib.pa_status_str.restype = ctypes.c_char_p
    lib.pa_debug_check.argtypes = [P]
    lib.pa_static_scratch_bytes.argtypes = []
    lib.pa_static_scratch_bytes.restype = SZ
    lib.pa_version.argtypes = []
    lib.pa_bm_create.argtypes = [I64, I, I]
    lib.pa_bm_create.restype = P
    lib.pa_bm_destroy.argtypes = [P]
    lib.pa_bm_destroy.restype = None
    lib.pa_bm_add_sequence.argtypes = [P, I64, P, ctypes.c_int32, P]
    lib.pa_bm_fork.argtypes = [P, I64, I64]
    lib.pa_bm_append.argtypes = [P, I64, ctypes.c_int32, P, P, P]
    lib.pa_bm_free.argtypes = [P, I64]
    for f in ("pa_bm_add_sequence", "pa_bm_fork", "pa_bm_append", "pa_bm_free"):
        getattr(lib, f).restype = I
    lib.pa_bm_block_table.argtypes = [P, I64, P, ctypes.c_int32]
    lib.pa_bm_block_table.restype = ctypes.c_int32
    lib.pa_bm_context_len.argtypes = [P, I64]
    lib.pa_bm_context_len.restype = I64
    lib.pa_bm_num_free.argtypes = [P]
    lib.pa_bm_num_free.restype = I64
    lib.pa_bm_stats.argtypes = [P, P]
    lib.pa_bm_stats.restype = None
    for f in ("pa_reshape_and_cache", "pa_decode", "pa_decode_split", "pa_decode_split_static",
              "pa_copy_blocks", "pa_swap_blocks", "pa_reshape_and_cache_fp8", "pa_decode_fp8",
              "pa_decode_split_fp8", "pa_decode_cascade", "pa_get_error", "pa_debug_check", "pa_check_wait_limit",
              "pa_version"):
        getattr(lib, f).restype = I
    _lib = lib
    return lib


def __getattr__(name):
    # PA_STATIC_SCRATCH_BYTES is read from the library, so it cannot drift from the C macro
    if name == "PA_STATIC_SCRATCH_BYTES":
        return int(library().pa_static_scratch_bytes())
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")


def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    codes = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16, torch.uint8: PA_FP8_E4M3,
             torch.float8_e4m3fn: PA_FP8_E4M3}
    if t.dtype not in codes:
        raise PAError("dtype", PA_ERR_UNSUPPORTED, str(t.dtype))
    return codes[t.dtype]


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(cond, func, what):
    if not cond:
        raise PAError(func, PA_ERR_INVALID_ARG, what)


def _dev(func, *ts):
    for t in ts:
        _need(t.is_cuda and t.is_contiguous(), func, "tensors must be contiguous CUDA tensors")


def _check(func, status):
    if status != PA_OK:
        raise PAError(func, status)


def _pool(func, cache, layout):
    """(layout code, num_blocks, num_kv_heads, block_size, head_dim) of a pool tensor."""
    _need(layout in ("HND", "NHD"), func, "layout must be 'HND' or 'NHD'")
    _need(cache.dim() == 4, func, "pools are 4-D")
    nb, a, b, d = cache.shape
    return (PA_LAYOUT_HND, nb, a, b, d) if layout == "HND" else (PA_LAYOUT_NHD, nb, b, a, d)


def pa_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, stream=None, layout="HND"):
    """Write each new token's K/V into ``k_cache`` / ``v_cache`` at its slot (negative slot: skip)."""
    f = "pa_reshape_and_cache"
    torch = _torch()
    _dev(f, key, value, k_cache, v_cache, slot_mapping)
    _need(slot_mapping.dtype == torch.int64, f, "slot_mapping must be int64")
    _need(key.dtype == value.dtype == k_cache.dtype == v_cache.dtype, f, "dtype mismatch")
    N, G, d = key.shape
    lc, nb, G2, B, d2 = _pool(f, k_cache, layout)
    _need(value.shape == key.shape and v_cache.shape == k_cache.shape and G2 == G and d2 == d, f, "shapes")
    _need(slot_mapping.shape == (N,), f, "slot_mapping shape")
    _check(f, library().pa_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                             _ptr(slot_mapping), N, G, d, B, lc, nb, _dtype_code(key),
                                             _stream(stream)))


def _decode_args(f, out, q, k_cache, v_cache, block_tables, context_lens, layout):
    torch = _torch()
    _dev(f, out, q, k_cache, v_cache, block_tables, context_lens)
    _need(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32, f,
          "block_tables and context_lens must be int32")
    _need(q.dtype == k_cache.dtype == v_cache.dtype, f, "q / cache dtype mismatch")
    S, H, d = q.shape
    lc, nb, G, B, d2 = _pool(f, k_cache, layout)
    _need(v_cache.shape == k_cache.shape and d2 == d and out.shape == q.shape, f, "shapes")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == S and context_lens.shape == (S,), f,
          "table shapes")
    return S, H, G, d, B, lc, nb, int(block_tables.shape[1])


def pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale, stream=None, layout="HND"):
    """``out[s, h] = softmax(scale * q[s, h] K_s^T) V_s`` over each sequence's paged context."""
    f = "pa_decode"
    S, H, G, d, B, lc, nb, maxb = _decode_args(f, out, q, k_cache, v_cache, block_tables, context_lens, layout)
    _check(f, library().pa_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                  maxb, _ptr(context_lens), S, H, G, d, B, lc, nb, float(scale),
                                  _dtype_code(q), _dtype_code(out), _stream(stream)))


def pa_decode_split_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, partition_tokens):
    return int(library().pa_decode_split_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len,
                                                         partition_tokens))


def pa_decode_split(out, q, k_cache, v_cache, block_tables, context_lens, scale, max_context_len,
                    partition_tokens, workspace, stream=None, layout="HND"):
    """Partitioned decode (per-partition softmax, then a log-sum-exp reduce) into ``out``.

    ``workspace`` is a CUDA tensor of at least ``pa_decode_split_workspace_bytes(...)`` bytes.
    """
    f = "pa_decode_split"
    S, H, G, d, B, lc, nb, maxb = _decode_args(f, out, q, k_cache, v_cache, block_tables, context_lens, layout)
    _dev(f, workspace)
    nbytes = workspace.numel() * workspace.element_size()
    _check(f, library().pa_decode_split(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                        maxb, _ptr(context_lens), S, H, G, d, B, lc, nb, float(scale),
                                        _dtype_code(q), _dtype_code(out), int(max_context_len),
                                        int(partition_tokens), _ptr(workspace), nbytes, _stream(stream)))


def pa_decode_split_static(out, q, k_cache, v_cache, block_tables, context_lens, scale, max_context_len,
                           partition_tokens, stream=None, layout="HND"):
    """``pa_decode_split`` for callers that cannot allocate: no workspace argument.

    The partition results go to a scratch array inside the library
    (``PA_STATIC_SCRATCH_BYTES`` per GPU, held until exit), so nothing is
    allocated per call. Requests whose workspace would exceed that size raise
    (status "unsupported"). All calls share the one array: calls that overlap
    on the GPU race. The first call on a device looks up the array's address;
    make it before any stream capture.
    """
    f = "pa_decode_split_static"
    S, H, G, d, B, lc, nb, maxb = _decode_args(f, out, q, k_cache, v_cache, block_tables, context_lens, layout)
    _check(f, library().pa_decode_split_static(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                               _ptr(block_tables), maxb, _ptr(context_lens), S, H, G, d, B,
                                               lc, nb, float(scale), _dtype_code(q), _dtype_code(out),
                                               int(max_context_len), int(partition_tokens), _stream(stream)))


def pa_decode_cascade_workspace_bytes(num_seqs, num_heads, head_dim, max_prefix_len, max_context_len,
                                      partition_tokens):
    return int(library().pa_decode_cascade_workspace_bytes(num_seqs, num_heads, head_dim, max_prefix_len,
                                                           max_context_len, partition_tokens))


def pa_decode_cascade(out, q, k_cache, v_cache, block_tables, context_lens, scale, group_starts, prefix_lens,
                      max_group_size, max_prefix_len, max_context_len, partition_tokens, workspace, stream=None,
                      layout="HND"):
    """Decode for batches whose sequences share prompt prefixes (same result as ``pa_decode``).

    ``group_starts`` (int32 [G+1]) and ``prefix_lens`` (int32 [G]) are CUDA
    tensors: sequences ``group_starts[g] .. group_starts[g+1]-1`` share their
    first ``prefix_lens[g]`` tokens through the same physical blocks.
    """
    f = "pa_decode_cascade"
    torch = _torch()
    S, H, G, d, B, lc, nb, maxb = _decode_args(f, out, q, k_cache, v_cache, block_tables, context_lens, layout)
    _dev(f, workspace, group_starts, prefix_lens)
    _need(group_starts.dtype == torch.int32 and prefix_lens.dtype == torch.int32, f, "group arrays must be int32")
    ng = int(prefix_lens.numel())
    _need(group_starts.numel() == ng + 1, f, "group_starts must have num_groups + 1 entries")
    nbytes = workspace.numel() * workspace.element_size()
    _check(f, library().pa_decode_cascade(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                          maxb, _ptr(context_lens), S, H, G, d, B, lc, nb, float(scale), _dtype_code(q),
                                          _dtype_code(out), _ptr(group_starts), _ptr(prefix_lens), ng,
                                          int(max_group_size), int(max_prefix_len), int(max_context_len),
                                          int(partition_tokens), _ptr(workspace), nbytes, _stream(stream)))


def pa_copy_blocks(k_caches, v_caches, block_pairs, stream=None):
    """For every (src, dst) pair and layer: ``cache[dst] = cache[src]`` for K and V."""
    f = "pa_copy_blocks"
    torch = _torch()
    k_caches, v_caches = list(k_caches), list(v_caches)
    _need(len(k_caches) == len(v_caches) and k_caches, f, "one K and one V pool per layer")
    _dev(f, block_pairs, *k_caches, *v_caches)
    _need(block_pairs.dtype == torch.int64 and block_pairs.dim() == 2 and block_pairs.shape[1] == 2, f,
          "block_pairs must be int64 [P, 2]")
    shape, dt = k_caches[0].shape, k_caches[0].dtype
    for t in k_caches + v_caches:
        _need(t.shape == shape and t.dtype == dt, f, "all pools must share shape and dtype")
    nb, G, B, d = shape
    L = len(k_caches)
    karr = (ctypes.c_void_p * L)(*[t.data_ptr() for t in k_caches])
    varr = (ctypes.c_void_p * L)(*[t.data_ptr() for t in v_caches])
    _check(f, library().pa_copy_blocks(karr, varr, L, _ptr(block_pairs), int(block_pairs.shape[0]), G, d, B,
                                       nb, _dtype_code(k_caches[0]), _stream(stream)))


def pa_swap_blocks(dst_k_caches, dst_v_caches, src_k_caches, src_v_caches, block_pairs, stream=None):
    """For every (src, dst) pair and layer: ``dst[dst] = src[src]`` for K and V, in one launch.

    Pools may be CUDA tensors or pinned CPU tensors (``pin_memory()``), which
    the kernel reaches directly; ``block_pairs`` (int64 [P, 2]) likewise.
    """
    f = "pa_swap_blocks"
    torch = _torch()
    dk, dv, sk, sv = list(dst_k_caches), list(dst_v_caches), list(src_k_caches), list(src_v_caches)
    L = len(dk)
    _need(L > 0 and len(dv) == L and len(sk) == L and len(sv) == L, f, "one K and one V pool per layer")
    for t in dk + dv + sk + sv + [block_pairs]:
        _need(t.is_contiguous() and (t.is_cuda or t.is_pinned()), f, "tensors must be CUDA or pinned host memory")
    _need(block_pairs.dtype == torch.int64 and block_pairs.dim() == 2 and block_pairs.shape[1] == 2, f,
          "block_pairs must be int64 [P, 2]")
    dshape, sshape, dt = dk[0].shape, sk[0].shape, dk[0].dtype
    for t in dk + dv:
        _need(t.shape == dshape and t.dtype == dt, f, "destination pools must share shape and dtype")
    for t in sk + sv:
        _need(t.shape == sshape and t.dtype == dt, f, "source pools must share shape and dtype")
    _need(dshape[1:] == sshape[1:], f, "pools must share the block shape")
    _, G, B, d = dshape
    arr = lambda ts: (ctypes.c_void_p * L)(*[t.data_ptr() for t in ts])  # noqa: E731
    _check(f, library().pa_swap_blocks(arr(dk), arr(dv), arr(sk), arr(sv), L, _ptr(block_pairs),
                                       int(block_pairs.shape[0]), G, d, B, dshape[0], sshape[0], _dtype_code(dk[0]),
                                       _stream(stream)))


def _is_code_tensor(t):
    torch = _torch()
    return t.dtype in (torch.uint8, torch.float8_e4m3fn)


def pa_reshape_and_cache_fp8(key, value, k_cache, v_cache, slot_mapping, k_scale, v_scale, stream=None,
                             layout="HND"):
    """Quantise each new token's K/V to E4M3 (x / scale, round to nearest even, saturating) into its slot.

    ``k_cache`` / ``v_cache`` are uint8 (or float8_e4m3fn) CUDA tensors in ``layout``.
    """
    f = "pa_reshape_and_cache_fp8"
    torch = _torch()
    _dev(f, key, value, k_cache, v_cache, slot_mapping)
    _need(slot_mapping.dtype == torch.int64, f, "slot_mapping must be int64")
    _need(key.dtype == value.dtype and _is_code_tensor(k_cache) and _is_code_tensor(v_cache), f, "dtypes")
    N, G, d = key.shape
    lc, nb, G2, B, d2 = _pool(f, k_cache, layout)
    _need(value.shape == key.shape and v_cache.shape == k_cache.shape and G2 == G and d2 == d, f, "shapes")
    _need(slot_mapping.shape == (N,), f, "slot_mapping shape")
    _check(f, library().pa_reshape_and_cache_fp8(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                                 _ptr(slot_mapping), N, G, d, B, lc, nb, _dtype_code(key),
                                                 float(k_scale), float(v_scale), _stream(stream)))


def _decode_args_fp8(f, out, q, k_cache, v_cache, block_tables, context_lens, layout):
    torch = _torch()
    _dev(f, out, q, k_cache, v_cache, block_tables, context_lens)
    _need(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32, f,
          "block_tables and context_lens must be int32")
    _need(_is_code_tensor(k_cache) and _is_code_tensor(v_cache), f, "caches must hold E4M3 codes")
    S, H, d = q.shape
    lc, nb, G, B, d2 = _pool(f, k_cache, layout)
    _need(v_cache.shape == k_cache.shape and d2 == d and out.shape == q.shape, f, "shapes")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == S and context_lens.shape == (S,), f,
          "table shapes")
    return S, H, G, d, B, lc, nb, int(block_tables.shape[1])


def pa_decode_fp8(out, q, k_cache, v_cache, block_tables, context_lens, scale, k_scale, v_scale, stream=None,
                  layout="HND"):
    """Decode attention over an E4M3 cache: softmax(scale q . k_scale K) (v_scale V)."""
    f = "pa_decode_fp8"
    S, H, G, d, B, lc, nb, maxb = _decode_args_fp8(f, out, q, k_cache, v_cache, block_tables, context_lens, layout)
    _check(f, library().pa_decode_fp8(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), maxb,
                                      _ptr(context_lens), S, H, G, d, B, lc, nb, float(scale), float(k_scale),
                                      float(v_scale), _dtype_code(q), _dtype_code(out), _stream(stream)))


def pa_decode_split_fp8(out, q, k_cache, v_cache, block_tables, context_lens, scale, k_scale, v_scale,
                        max_context_len, partition_tokens, workspace, stream=None, layout="HND"):
    """Partitioned decode over an E4M3 cache (workspace as for ``pa_decode_split``)."""
    f = "pa_decode_split_fp8"
    S, H, G, d, B, lc, nb, maxb = _decode_args_fp8(f, out, q, k_cache, v_cache, block_tables, context_lens, layout)
    _dev(f, workspace)
    nbytes = workspace.numel() * workspace.element_size()
    _check(f, library().pa_decode_split_fp8(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                            maxb, _ptr(context_lens), S, H, G, d, B, lc, nb, float(scale),
                                            float(k_scale), float(v_scale), _dtype_code(q), _dtype_code(out),
                                            int(max_context_len), int(partition_tokens), _ptr(workspace), nbytes,
                                            _stream(stream)))


def pa_get_error(stream=None) -> int:
    """Read and clear the device error word (``PA_DEVERR_*`` bits); synchronises the stream."""
    bits = ctypes.c_uint32(0)
    st = library().pa_get_error(ctypes.byref(bits), _stream(stream))
    if st not in (PA_OK, PA_ERR_OUT_OF_RANGE):
        raise PAError("pa_get_error", st)
    return int(bits.value)


def pa_debug_check(stream=None) -> int:
    """Wait for the stream, read and clear the device error word; the status
    (``PA_OK`` or ``PA_ERR_OUT_OF_RANGE`` = 3) is returned, other statuses raise."""
    st = library().pa_debug_check(_stream(stream))
    if st not in (PA_OK, PA_ERR_OUT_OF_RANGE):
        raise PAError("pa_debug_check", st)
    return int(st)


def pa_status_str(status) -> str:
    """The library's name for a status code."""
    return library().pa_status_str(int(status)).decode()


def pa_check_wait_limit(limit_ns, stream=None):
    """Diagnostic: one warp's mbarrier wait runs out after ``limit_ns`` and a second
    warp, whose limit is 50 times longer, follows it out through the abort flag;
    ``PA_DEVERR_TIMEOUT`` is then set in the error word (read it with ``pa_get_error``)."""
    _check("pa_check_wait_limit", library().pa_check_wait_limit(int(limit_ns), _stream(stream)))


def pa_version() -> int:
    return int(library().pa_version())
