"""Pins for the E4M3 oracle: torch's own float8_e4m3fn type, the format's closed
forms (largest value, subnormal step, ties to even, saturation), and the scaled
attention against torch's float64 SDPA on the dequantised values."""
import numpy as np
import pytest
import torch

from oracle import fp8
from test_oracle_pins import paged_from_contiguous, sdpa_reference


def test_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    got = fp8.e4m3_decode(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_closed_forms():
    assert fp8.e4m3_decode(np.array([0x7E]))[0] == 448.0
    assert fp8.e4m3_decode(np.array([0x01]))[0] == 2.0 ** -9
    assert fp8.e4m3_decode(np.array([0x08]))[0] == 2.0 ** -6
    assert fp8.e4m3_decode(np.array([0x38]))[0] == 1.0
    assert np.isnan(fp8.e4m3_decode(np.array([0x7F, 0xFF]))).all()
    # saturation and NaN
    assert list(fp8.e4m3_encode([470.0, 1000.0, -500.0, 448.0, np.inf])) == [0x7E, 0x7E, 0xFE, 0x7E, 0x7E]
    assert fp8.e4m3_encode([np.nan])[0] & 0x7F == 0x7F
    # ties go to the even code: 1 + 1/16 lies between 1 (0x38) and 1.125 (0x39)
    assert fp8.e4m3_encode([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10])[:].tolist() == [0x38, 0x3A, 0x00, 0x02]


def test_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = fp8.e4m3_decode(codes).astype(np.float32)
    back = fp8.e4m3_encode(vals)
    zero = vals == 0
    assert np.array_equal(back[~zero], codes[~zero])
    assert set(back[zero].tolist()) <= {0x00, 0x80}


def test_encode_matches_torch_in_range():
    g = torch.Generator().manual_seed(0)
    x = torch.cat([torch.randn(200000, generator=g) * s for s in (0.003, 0.05, 1.0, 30.0, 200.0)])
    x = x[x.abs() < 464]
    mids = (fp8.e4m3_decode(np.arange(0, 126)) + fp8.e4m3_decode(np.arange(1, 127))) / 2  # exact ties
    x = torch.cat([x, torch.from_numpy(mids).float(), -torch.from_numpy(mids).float()])
    got = fp8.e4m3_encode(x.numpy())
    want = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


def test_quantize_divides_in_float32():
    x = np.array([1.0, 3.0, 100.0], np.float32)
    s = np.float32(0.1)
    assert np.array_equal(fp8.quantize(x, s), fp8.e4m3_encode(x / s))


@pytest.mark.parametrize("H,G", [(4, 4), (8, 2), (8, 1)])
def test_scaled_attention_matches_sdpa(H, G):
    rng = np.random.default_rng(21)
    ctxs = [1, 9, 40, 100]
    d, ks, vs = 32, 0.37, 1.9
    Kc = [rng.integers(0, 256, (c, G, d)).astype(np.uint8) for c in ctxs]
    Vc = [rng.integers(0, 256, (c, G, d)).astype(np.uint8) for c in ctxs]
    for arr in Kc + Vc:
        arr[(arr & 0x7F) == 0x7F] = 0x11  # no NaN codes in data
    q = rng.standard_normal((len(ctxs), H, d)).astype(np.float32)
    Kf = [fp8.e4m3_decode(k).astype(np.float32) for k in Kc]
    Vf = [fp8.e4m3_decode(v).astype(np.float32) for v in Vc]
    kc, vc, bt = paged_from_contiguous([k.astype(np.float32) for k in Kc], [v.astype(np.float32) for v in Vc],
                                       16, rng, fill=0)
    out = fp8.decode(q, kc.astype(np.uint8), vc.astype(np.uint8), bt, np.array(ctxs, np.int32), 0.2, ks, vs)
    for s in range(len(ctxs)):
        ref = sdpa_reference(q[s], (Kf[s].astype(np.float64) * ks), (Vf[s].astype(np.float64) * vs), 0.2)
        assert np.abs(out[s] - ref).max() <= 1e-9


def test_fp8_cache_write():
    rng = np.random.default_rng(22)
    key = rng.standard_normal((3, 2, 16)).astype(np.float32)
    val = rng.standard_normal((3, 2, 16)).astype(np.float32)
    kc = np.zeros((4, 2, 16, 16), np.uint8)
    k2, v2 = fp8.reshape_and_cache(key, val, kc, kc, np.array([5, -1, 63]), 0.5, 2.0)
    assert np.array_equal(k2[0, :, 5, :], fp8.quantize(key[0], 0.5))
    assert np.array_equal(v2[3, :, 15, :], fp8.quantize(val[2], 2.0))
    assert k2[1:3].sum() == 0 and (k2[0, :, :5] == 0).all()
