"""ctypes front of the float64 C oracle (``pa_oracle.c``).

Test infrastructure: see the header of ``oracle/__init__.py``.
Arrays may be numpy arrays or torch tensors (copied to host memory first);
16-bit values are handed to C as their raw bit patterns and decoded there.
"""
import ctypes

import numpy as np

from .build import LIB, build, ensure_built

_F32, _F16, _BF16 = 0, 1, 2
_lib = None


def _load(path=None):
    global _lib
    if path is not None:
        lib = ctypes.CDLL(path)
    else:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(ensure_built())
    P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.pa_oracle_decode.argtypes = [P, P, P, P, I, P, I, P, I, I, I, I, I, I64, D, I]
    lib.pa_oracle_decode.restype = I
    lib.pa_oracle_partitions.argtypes = [P, P, P, P, P, P, I, P, I, P, I, I, I, I, I, I64, D, I, I, I]
    lib.pa_oracle_partitions.restype = I
    lib.pa_oracle_merge.argtypes = [P, P, P, P, I64, I, I]
    lib.pa_oracle_merge.restype = None
    lib.pa_oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.pa_oracle_f16_to_f64.restype = D
    lib.pa_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.pa_oracle_bf16_to_f64.restype = D
    lib.pa_oracle_max_threads.restype = I
    if path is None:
        _lib = lib
    return lib


def load_variant(src_path, out_path):
    """Compile and load another copy of the C source (used by the mutation tests)."""
    build(src_path, out_path)
    return _load(out_path)


def _host(x, name):
    """Contiguous host numpy array + dtype code; 16-bit floats as uint16 bit patterns."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        t = x.detach().to("cpu").contiguous()
        if t.dtype == torch.float32:
            return t.numpy(), _F32
        if t.dtype == torch.float16:
            return t.view(torch.int16).numpy().view(np.uint16), _F16
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16), _BF16
        if t.dtype in (torch.int32, torch.int64, torch.float64):
            return t.numpy(), None
        raise TypeError(f"{name}: unsupported dtype {t.dtype}")
    a = np.ascontiguousarray(x)
    if a.dtype == np.float32:
        return a, _F32
    if a.dtype == np.float16:
        return a.view(np.uint16), _F16
    return a, None


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _hnd(a, layout):
    """The pool as [num_blocks][G][B][d]. Month 2 · PagedAttention §5.2 names two
    pool layouts: HND [blocks][heads][tokens][d] and NHD [blocks][tokens][heads][d];
    NHD element [b][r][h] is HND element [b][h][r], so an NHD pool is its HND
    form with axes 1 and 2 exchanged."""
    if layout == "HND":
        return a
    if layout != "NHD":
        raise ValueError(f"unknown layout {layout!r}")
    return np.ascontiguousarray(a.transpose(0, 2, 1, 3))


def _common(q, k_cache, v_cache, block_tables, context_lens, layout="HND"):
    qa, dq = _host(q, "q")
    ka, dk = _host(k_cache, "k_cache")
    va, dv = _host(v_cache, "v_cache")
    ka, va = _hnd(ka, layout), _hnd(va, layout)
    if not (dq == dk == dv) or dq is None:
        raise TypeError("q, k_cache and v_cache must share one float dtype")
    bt = np.ascontiguousarray(_host(block_tables, "block_tables")[0], dtype=np.int32)
    cl = np.ascontiguousarray(_host(context_lens, "context_lens")[0], dtype=np.int32)
    S, H, d = qa.shape
    nb, G, B, d2 = ka.shape
    if d2 != d or va.shape != ka.shape or bt.shape[0] != S or cl.shape != (S,):
        raise ValueError("shape mismatch")
    return qa, ka, va, dq, bt, cl, S, H, G, d, B, nb


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, num_threads=0, lib=None, layout="HND"):
    """float64 ``out[S, H, d]`` = softmax(scale * q K^T) V over each sequence's paged context."""
    lib = lib or _load()
    qa, ka, va, dt, bt, cl, S, H, G, d, B, nb = _common(q, k_cache, v_cache, block_tables, context_lens, layout)
    out = np.zeros((S, H, d), dtype=np.float64)
    rc = lib.pa_oracle_decode(_ptr(out), _ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(bt), bt.shape[1],
                              _ptr(cl), S, H, G, d, B, nb, float(scale), int(num_threads))
    if rc:
        raise ValueError(f"oracle decode rejected its inputs (code {rc})")
    return out


def partitions(q, k_cache, v_cache, block_tables, context_lens, scale, T, P=None,
               num_threads=0, lib=None, layout="HND"):
    """Per-partition ``(o[S,H,P,d], m[S,H,P], l[S,H,P])`` for partitions of T tokens."""
    lib = lib or _load()
    qa, ka, va, dt, bt, cl, S, H, G, d, B, nb = _common(q, k_cache, v_cache, block_tables, context_lens, layout)
    if P is None:
        P = max(1, -(-int(cl.max(initial=0)) // T))
    o = np.zeros((S, H, P, d), dtype=np.float64)
    m = np.zeros((S, H, P), dtype=np.float64)
    l = np.zeros((S, H, P), dtype=np.float64)
    rc = lib.pa_oracle_partitions(_ptr(o), _ptr(m), _ptr(l), _ptr(qa), _ptr(ka), _ptr(va), dt,
                                  _ptr(bt), bt.shape[1], _ptr(cl), S, H, G, d, B, nb,
                                  float(scale), int(T), int(P), int(num_threads))
    if rc:
        raise ValueError(f"oracle partitions rejected its inputs (code {rc})")
    return o, m, l


def merge(o, m, l, lib=None):
    """Merge per-partition results ``o[..., P, d]``, ``m[..., P]``, ``l[..., P]``."""
    lib = lib or _load()
    o = np.ascontiguousarray(o, dtype=np.float64)
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    P, d = o.shape[-2], o.shape[-1]
    lead = o.shape[:-2]
    R = int(np.prod(lead)) if lead else 1
    out = np.zeros(lead + (d,), dtype=np.float64)
    lib.pa_oracle_merge(_ptr(out), _ptr(o), _ptr(m), _ptr(l), R, P, d)
    return out


def f16_bits_to_f64(bits, lib=None):
    lib = lib or _load()
    return np.array([lib.pa_oracle_f16_to_f64(int(b)) for b in np.asarray(bits).ravel()])


def bf16_bits_to_f64(bits, lib=None):
    lib = lib or _load()
    return np.array([lib.pa_oracle_bf16_to_f64(int(b)) for b in np.asarray(bits).ravel()])


def max_threads():
    return int(_load().pa_oracle_max_threads())


__all__ = ["decode", "partitions", "merge", "f16_bits_to_f64", "bf16_bits_to_f64",
           "max_threads", "load_variant", "LIB"]
