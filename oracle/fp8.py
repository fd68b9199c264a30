"""FP8 (E4M3) KV-cache oracle: the code format written out from its definition.

Test infrastructure: see the header of ``oracle/__init__.py``.

KV-cache quantisation is one of the ways the pages list to make KV smaller
(CS349E Lecture 7 notes, §10 and §11: 8-bit and lower KV formats). Reading
taken here: a cache element is an E4M3 code c with one fp32 scale per tensor
(one for K, one for V), value = decode(c) * scale.

E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0
gives subnormals m/8 * 2^-6; the all-ones code S.1111.111 is NaN; there are no
infinities; the largest finite magnitude is 1.75 * 2^8 = 448.
Encoding rounds to nearest, ties to even, on that grid; finite values beyond
448 in magnitude saturate to +-448; NaN stays NaN.
"""
import numpy as np

from .attention import decode as _decode

MAX_E4M3 = 448.0


def _np(x):
    """Host numpy copy (torch tensors are moved to the CPU and 16-bit floats upcast exactly)."""
    if hasattr(x, "detach"):
        t = x.detach().cpu()
        if t.is_floating_point() and t.element_size() == 2:
            t = t.float()
        return t.numpy()
    return np.asarray(x)


def e4m3_decode(codes):
    """float64 values of E4M3 codes (uint8 array)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = m / 8.0 * 2.0 ** -6
    norm = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    v = np.where(e == 0, sub, norm)
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return sign * v


def e4m3_encode(x):
    """E4M3 codes (uint8) of float32 values: RNE on the E4M3 grid, saturating at +-448."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    nan = np.isnan(x)
    neg = np.signbit(x)
    a = np.minimum(np.abs(np.where(nan, 0.0, x)), MAX_E4M3)
    # binade of a; below 2^-6 the spacing is the subnormal one, 2^-9
    with np.errstate(divide="ignore"):
        e = np.where(a >= 2.0 ** -6, np.floor(np.log2(np.where(a > 0, a, 1.0))), -6.0)
    step = np.exp2(e - 3.0)
    q = np.rint(a / step) * step          # np.rint rounds half to even
    q = np.minimum(q, MAX_E4M3)
    # bit fields of q
    with np.errstate(divide="ignore"):
        qe = np.where(q >= 2.0 ** -6, np.floor(np.log2(np.where(q > 0, q, 1.0))), -7.0)
    E = np.where(q >= 2.0 ** -6, qe + 7.0, 0.0)
    M = np.where(q >= 2.0 ** -6, (q / np.exp2(qe) - 1.0) * 8.0, q / 2.0 ** -9)
    code = (E.astype(np.int64) << 3) | np.rint(M).astype(np.int64)
    code = np.where(nan, 0x7F, code)
    code = code | np.where(neg, 0x80, 0)
    return code.astype(np.uint8)


def quantize(x, scale):
    """Codes of x / scale, the division done in float32 (the quotient the kernel rounds)."""
    q = np.asarray(x, dtype=np.float32) / np.float32(scale)
    return e4m3_encode(q)


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, k_scale, v_scale, layout="HND"):
    """New (k_cache, v_cache) code arrays after quantising and writing every new token.

    key, value: float arrays [N, G, d] (their exact values); caches: uint8 codes
    [num_blocks, G, B, d] (HND) or [num_blocks, B, G, d] (NHD). Token t with
    slot >= 0 lands in block slot // B, row slot % B, as in the unquantised
    cache write.
    """
    kq = quantize(_np(key), k_scale)
    vq = quantize(_np(value), v_scale)
    kc = np.array(_np(k_cache), dtype=np.uint8, copy=True)
    vc = np.array(_np(v_cache), dtype=np.uint8, copy=True)
    slots = np.asarray(_np(slot_mapping), dtype=np.int64)
    if layout not in ("HND", "NHD"):
        raise ValueError(f"unknown layout {layout!r}")
    nhd = layout == "NHD"
    B = kc.shape[1] if nhd else kc.shape[2]
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        b, r = divmod(int(slot), B)
        if nhd:
            kc[b, r, :, :] = kq[t]
            vc[b, r, :, :] = vq[t]
        else:
            kc[b, :, r, :] = kq[t]
            vc[b, :, r, :] = vq[t]
    return kc, vc


def decode(q, k_codes, v_codes, block_tables, context_lens, scale, k_scale, v_scale, num_threads=0,
           layout="HND"):
    """float64 attention over an E4M3 cache with per-tensor scales.

    softmax(scale * q . (k_scale * K)) (v_scale * V): the scales are constants,
    so this is the unscaled-code attention with score scale scale * k_scale and
    the result multiplied by v_scale (E4M3 codes are exact in float32).
    """
    kf = e4m3_decode(_np(k_codes)).astype(np.float32)
    vf = e4m3_decode(_np(v_codes)).astype(np.float32)
    qf = _np(q).astype(np.float32)
    out = _decode(qf, kf, vf, block_tables, context_lens, float(scale) * float(k_scale),
                  num_threads=num_threads, layout=layout)
    return out * float(v_scale)
