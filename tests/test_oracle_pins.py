"""Pins for the CPU oracle: it is checked against things other than itself.

* library routines: torch's float64 scaled_dot_product_attention on the
  contiguous K/V (paging must not change the result: CS349E Lecture 7 notes
  §4.2, CMU 15-779 Lecture 16 notes §3.3), numpy's and torch's own 16-bit float
  decoders;
* closed forms: one token returns its V row exactly; equal scores (q = 0)
  return the mean of V; V = 1 returns 1 (the weights sum to one);
* brute force at 50 significant digits (mpmath) on the tiny workload;
* the merge rule: merging per-partition results gives the unsplit result.

``test_mutants_are_caught`` plants mistakes in copies of the C source (on the
CPU) and checks that this battery fails for every one of them.
"""
import os
import re
import shutil

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oatt
from paged_kv_cache_04_gb300 import workloads

ORACLE_SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")


# ---------------------------------------------------------------------------
# helpers (test-side): scatter a contiguous K/V into a shuffled block pool
# ---------------------------------------------------------------------------
def paged_from_contiguous(Ks, Vs, B, rng, extra_blocks=3, fill=np.nan, layout="HND"):
    """Ks, Vs: lists of float32 arrays [ctx, G, d]. Returns (k_cache, v_cache, block_tables).

    layout "HND" gives pools [nb, G, B, d]; "NHD" gives [nb, B, G, d].
    """
    G, d = Ks[0].shape[1], Ks[0].shape[2]
    nblk = [-(-K.shape[0] // B) for K in Ks]
    nb = sum(nblk) + extra_blocks
    perm = rng.permutation(nb)
    shape = (nb, G, B, d) if layout == "HND" else (nb, B, G, d)
    k_cache = np.full(shape, fill, dtype=np.float32)
    v_cache = np.full(shape, fill, dtype=np.float32)
    width = max(1, max(nblk))
    bt = np.full((len(Ks), width), -1, dtype=np.int32)
    nxt = 0
    for s, (K, V) in enumerate(zip(Ks, Vs)):
        for j in range(nblk[s]):
            phys = int(perm[nxt])
            nxt += 1
            bt[s, j] = phys
            for r in range(B):
                t = j * B + r
                if t < K.shape[0]:
                    for h in range(G):
                        idx = (phys, h, r) if layout == "HND" else (phys, r, h)
                        k_cache[idx] = K[t, h, :]
                        v_cache[idx] = V[t, h, :]
    return k_cache, v_cache, bt


def sdpa_reference(q, K, V, scale):
    """torch float64 SDPA of one sequence; q [H, d], K/V [ctx, G, d] (contiguous)."""
    H, G = q.shape[0], K.shape[1]
    if K.shape[0] == 0:
        return np.zeros_like(q, dtype=np.float64)
    qt = torch.from_numpy(q.astype(np.float64)).view(1, H, 1, -1)
    Kt = torch.from_numpy(K.astype(np.float64)).permute(1, 0, 2).repeat_interleave(H // G, 0)
    Vt = torch.from_numpy(V.astype(np.float64)).permute(1, 0, 2).repeat_interleave(H // G, 0)
    out = torch.nn.functional.scaled_dot_product_attention(qt, Kt.unsqueeze(0), Vt.unsqueeze(0),
                                                           scale=scale)
    return out.view(H, -1).numpy()


def random_case(rng, ctxs, H, G, d):
    Ks = [rng.standard_normal((c, G, d)).astype(np.float32) for c in ctxs]
    Vs = [rng.standard_normal((c, G, d)).astype(np.float32) for c in ctxs]
    q = rng.standard_normal((len(ctxs), H, d)).astype(np.float32)
    return q, Ks, Vs


# ---------------------------------------------------------------------------
# the pin battery (each takes the oracle library to check)
# ---------------------------------------------------------------------------
def pin_paged_equals_contiguous(lib):
    rng = np.random.default_rng(11)
    ctxs = [1, 5, 16, 17, 40, 64, 100]
    for H, G in ((4, 4), (8, 2), (8, 1)):
        q, Ks, Vs = random_case(rng, ctxs, H, G, 32)
        scale = 0.37
        for B in (1, 4, 16, 64):
            kc, vc, bt = paged_from_contiguous(Ks, Vs, B, rng)
            out = oatt.decode(q, kc, vc, bt, np.array(ctxs, np.int32), scale, lib=lib)
            for s in range(len(ctxs)):
                ref = sdpa_reference(q[s], Ks[s], Vs[s], scale)
                err = np.abs(out[s] - ref).max()
                assert err <= 1e-12, f"paged != contiguous (H={H} G={G} B={B} s={s}): {err}"


def pin_nhd_paged_equals_contiguous(lib):
    """NHD pools (Month 2 · PagedAttention §5.2) give the contiguous result too,
    for the plain and the partitioned oracle; G != B and G == B both occur."""
    rng = np.random.default_rng(19)
    ctxs = [1, 4, 9, 33, 70]
    for H, G, B in ((8, 2, 4), (4, 4, 4), (8, 8, 16)):
        q, Ks, Vs = random_case(rng, ctxs, H, G, 16)
        kc, vc, bt = paged_from_contiguous(Ks, Vs, B, rng, layout="NHD")
        cl = np.array(ctxs, np.int32)
        out = oatt.decode(q, kc, vc, bt, cl, 0.41, lib=lib, layout="NHD")
        o, m, l = oatt.partitions(q, kc, vc, bt, cl, 0.41, 2 * B, lib=lib, layout="NHD")
        merged = oatt.merge(o, m, l, lib=lib)
        for s in range(len(ctxs)):
            ref = sdpa_reference(q[s], Ks[s], Vs[s], 0.41)
            assert np.abs(out[s] - ref).max() <= 1e-12, f"NHD paged != contiguous (G={G} B={B} s={s})"
            assert np.abs(merged[s] - ref).max() <= 1e-12, f"NHD partitions != contiguous (G={G} B={B})"


def pin_head_dim_256(lib):
    """head_dim 256 (HND and NHD, plain and partitioned) gives the contiguous SDPA
    result: nothing in the oracle depends on the width of a head."""
    rng = np.random.default_rng(23)
    ctxs = [1, 17, 50]
    for layout in ("HND", "NHD"):
        for H, G, B in ((4, 2, 16), (2, 2, 32)):
            q, Ks, Vs = random_case(rng, ctxs, H, G, 256)
            kc, vc, bt = paged_from_contiguous(Ks, Vs, B, rng, layout=layout)
            cl = np.array(ctxs, np.int32)
            out = oatt.decode(q, kc, vc, bt, cl, 0.0625, lib=lib, layout=layout)
            merged = oatt.merge(*oatt.partitions(q, kc, vc, bt, cl, 0.0625, B, lib=lib, layout=layout), lib=lib)
            for s in range(len(ctxs)):
                ref = sdpa_reference(q[s], Ks[s], Vs[s], 0.0625)
                assert np.abs(out[s] - ref).max() <= 1e-12, f"d=256 {layout} paged != contiguous"
                assert np.abs(merged[s] - ref).max() <= 1e-12, f"d=256 {layout} partitions != contiguous"


def pin_one_token_is_v(lib):
    rng = np.random.default_rng(12)
    q, Ks, Vs = random_case(rng, [1, 1, 1], 4, 2, 16)
    kc, vc, bt = paged_from_contiguous(Ks, Vs, 16, rng)
    out = oatt.decode(q, kc, vc, bt, np.ones(3, np.int32), 2.5, lib=lib)
    for s in range(3):
        want = np.repeat(Vs[s][0].astype(np.float64), 2, axis=0)  # heads 2g, 2g+1 read kv g
        assert np.array_equal(out[s], want), "one-token context must return V exactly"


def pin_equal_scores_give_mean(lib):
    rng = np.random.default_rng(13)
    _, Ks, Vs = random_case(rng, [7, 33], 4, 4, 16)
    q = np.zeros((2, 4, 16), np.float32)
    kc, vc, bt = paged_from_contiguous(Ks, Vs, 4, rng)
    out = oatt.decode(q, kc, vc, bt, np.array([7, 33], np.int32), 1.0, lib=lib)
    for s in range(2):
        want = Vs[s].astype(np.float64).mean(axis=0)
        assert np.abs(out[s] - want).max() <= 1e-14, "q = 0 must average V"


def pin_weights_sum_to_one(lib):
    rng = np.random.default_rng(14)
    q, Ks, _ = random_case(rng, [3, 50, 129], 4, 4, 16)
    Vs = [np.ones_like(K) for K in Ks]
    kc, vc, bt = paged_from_contiguous(Ks, Vs, 16, rng)
    out = oatt.decode(q * 3, kc, vc, bt, np.array([3, 50, 129], np.int32), 1.0, lib=lib)
    assert np.abs(out - 1.0).max() <= 1e-15, "softmax weights must sum to one"


def pin_brute_force_tiny(lib):
    """Configuration 'tiny' (fp32, B 16, contexts {1,17,33,100}) against mpmath at 50 digits."""
    mpmath = pytest.importorskip("mpmath")
    wl = workloads.tiny()
    out = oatt.decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                      lib=lib)
    q = wl.q.double().numpy()
    kc, vc = wl.k_cache.double().numpy(), wl.v_cache.double().numpy()
    bt = wl.block_tables.numpy()
    mpmath.mp.dps = 50
    for s, h in ((0, 1), (1, 0), (2, 3), (3, 2)):
        ctx = int(wl.context_lens[s])
        kv = h // (wl.H // wl.G)
        rows = [(bt[s, t // wl.B], t % wl.B) for t in range(ctx)]
        z = [mpmath.mpf(wl.scale) * mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(b))
                                                for a, b in zip(q[s, h], kc[p, kv, r]))
             for p, r in rows]
        zmax = max(z)
        w = [mpmath.exp(x - zmax) for x in z]
        tot = mpmath.fsum(w)
        for i in range(wl.d):
            ref = mpmath.fsum(wi * mpmath.mpf(float(vc[p, kv, r, i])) for wi, (p, r) in zip(w, rows)) / tot
            assert abs(out[s, h, i] - float(ref)) <= 1e-14, f"brute force mismatch s={s} h={h} i={i}"


def pin_decoders(lib):
    bits = np.arange(65536, dtype=np.uint16)
    got = oatt.f16_bits_to_f64(bits, lib=lib)
    want = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok]), "fp16 decode differs from numpy"
    got = oatt.bf16_bits_to_f64(bits, lib=lib)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok]), "bf16 decode differs from torch"


def pin_16bit_paths_match_upcast(lib):
    """bf16 / fp16 inputs: the oracle equals SDPA on the exactly upcast values."""
    rng = np.random.default_rng(15)
    for dt in (torch.float16, torch.bfloat16):
        q, Ks, Vs = random_case(rng, [9, 31], 8, 2, 32)
        Ks = [torch.from_numpy(K).to(dt).float().numpy() for K in Ks]
        Vs = [torch.from_numpy(V).to(dt).float().numpy() for V in Vs]
        q = torch.from_numpy(q).to(dt).float().numpy()
        kc, vc, bt = paged_from_contiguous(Ks, Vs, 16, rng, fill=0.0)
        out = oatt.decode(torch.from_numpy(q).to(dt), torch.from_numpy(kc).to(dt),
                          torch.from_numpy(vc).to(dt), bt, np.array([9, 31], np.int32), 0.2, lib=lib)
        for s in range(2):
            ref = sdpa_reference(q[s], Ks[s], Vs[s], 0.2)
            assert np.abs(out[s] - ref).max() <= 1e-12, f"{dt} path mismatch"


def pin_partitions_merge_to_decode(lib):
    rng = np.random.default_rng(16)
    ctxs = [0, 1, 15, 16, 100, 257]
    q, Ks, Vs = random_case(rng, ctxs, 8, 4, 32)
    kc, vc, bt = paged_from_contiguous(Ks, Vs, 16, rng)
    cl = np.array(ctxs, np.int32)
    full = oatt.decode(q, kc, vc, bt, cl, 0.3, lib=lib)
    for T in (16, 32, 48, 512):
        o, m, l = oatt.partitions(q, kc, vc, bt, cl, 0.3, T, lib=lib)
        merged = oatt.merge(o, m, l, lib=lib)
        assert np.abs(merged - full).max() <= 1e-12, f"merge of T={T} partitions != unsplit"
    # one partition covering everything is the unsplit result with its own stats
    o, m, l = oatt.partitions(q, kc, vc, bt, cl, 0.3, 512, lib=lib)
    assert np.array_equal(o[:, :, 0], full)
    for s, c in enumerate(ctxs):
        if c == 0:
            assert np.all(l[s] == 0) and np.all(np.isneginf(m[s]))
            continue
        K = Ks[s].astype(np.float64)
        for h in range(8):
            z = 0.3 * K[:, h // 2, :] @ q[s, h].astype(np.float64)
            assert abs(m[s, h, 0] - z.max()) <= 1e-13
            assert abs(l[s, h, 0] - np.exp(z - z.max()).sum()) <= 1e-12 * c


def pin_empty_context_is_zero(lib):
    rng = np.random.default_rng(17)
    q, Ks, Vs = random_case(rng, [0, 3], 4, 4, 16)
    kc, vc, bt = paged_from_contiguous(Ks, Vs, 16, rng)
    out = oatt.decode(q, kc, vc, bt, np.array([0, 3], np.int32), 1.0, lib=lib)
    assert np.array_equal(out[0], np.zeros_like(out[0]))


PINS = [pin_paged_equals_contiguous, pin_nhd_paged_equals_contiguous, pin_head_dim_256, pin_one_token_is_v,
        pin_equal_scores_give_mean, pin_weights_sum_to_one, pin_brute_force_tiny, pin_decoders, pin_16bit_paths_match_upcast,
        pin_partitions_merge_to_decode, pin_empty_context_is_zero]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(oatt._load())


# ---------------------------------------------------------------------------
# planted mistakes: every mutant of the C source must fail at least one pin
# ---------------------------------------------------------------------------
MUTANTS = {
    "gqa_mapping_modulo": ("h / group,", "h % G,"),
    "row_reversed": ("+ (t % B)) * (int64_t)d", "+ (B - 1 - t % B)) * (int64_t)d"),
    "nhd_layout": ("((phys * G + kv) * B + (t % B))", "((phys * B + (t % B)) * G + kv)"),
    "scale_dropped": ("z[j] = scale * acc;", "z[j] = acc;"),
    "exp_sign": ("z[j] = exp(z[j] - m);", "z[j] = exp(m - z[j]);"),
    "v_reads_k": ("load(v_cache, row[j] + i, dtype)", "load(k_cache, row[j] + i, dtype)"),
    "floor_block_count": ("block_tables + (int64_t)s * max_blocks, 0, ctx,",
                          "block_tables + (int64_t)s * max_blocks, 0, ctx / B * B,"),
    "no_normalise": ("o[i] /= l;", "o[i] /= 1.0;"),
    "f16_exponent": ("e - 25);", "e - 24);"),
    "bf16_hidden_bit": ("(double)(128 + f)", "(double)(f)"),
    "merge_weight_sign": ("exp(m[r * P + p] - M)", "exp(M - m[r * P + p])"),
    "max_skipped": ("if (z[j] > m)\n            m = z[j];", "if (0)\n            m = z[j];"),
    "q_row_swapped": ("load(q, q_row * d + i, dtype)", "load(q, (q_row ^ 1) * d + i, dtype)"),
}


def _run_battery(lib):
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError) as e:
            failed.append((pin.__name__, str(e)[:80]))
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants_are_caught(name, tmp_path):
    src = open(ORACLE_SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    p = tmp_path / f"mut_{name}.c"
    p.write_text(mutated)
    lib = oatt.load_variant(str(p), str(tmp_path / f"mut_{name}.so"))
    failed = _run_battery(lib)
    assert failed, f"planted mistake {name} went unnoticed by every pin"


def test_unmutated_battery_passes(tmp_path):
    p = tmp_path / "copy.c"
    shutil.copy(ORACLE_SRC, p)
    lib = oatt.load_variant(str(p), str(tmp_path / "copy.so"))
    assert _run_battery(lib) == []


def test_dropped_nhd_transpose_is_caught(monkeypatch):
    """Planted mistake in the oracle's layout handling: reading an NHD pool as if
    it were HND must fail the NHD pin."""
    monkeypatch.setattr(oatt, "_hnd", lambda a, layout: a)
    with pytest.raises((AssertionError, ValueError)):
        pin_nhd_paged_equals_contiguous(oatt._load())


def test_nhd_cache_write_places_rows():
    """NHD cache write: token t lands at [slot // B, slot % B, h, :]; the HND
    write of the same tokens holds the same rows with axes 1 and 2 exchanged."""
    from oracle import cache_ops
    rng = np.random.default_rng(20)
    N, G, B, d, nb = 7, 3, 4, 8, 5
    key = rng.standard_normal((N, G, d)).astype(np.float32)
    val = rng.standard_normal((N, G, d)).astype(np.float32)
    slots = np.array([0, 5, 19, -1, 7, 12, 3], np.int64)
    zh = np.zeros((nb, G, B, d), np.float32)
    zn = np.zeros((nb, B, G, d), np.float32)
    kh, vh = cache_ops.reshape_and_cache(key, val, zh, zh, slots)
    kn, vn = cache_ops.reshape_and_cache(key, val, zn, zn, slots, layout="NHD")
    for t, sl in enumerate(slots):
        if sl < 0:
            continue
        b, r = divmod(int(sl), B)
        assert np.array_equal(kn[b, r].view(np.float32), key[t])
        assert np.array_equal(vn[b, r].view(np.float32), val[t])
    assert np.array_equal(kn, kh.transpose(0, 2, 1, 3)) and np.array_equal(vn, vh.transpose(0, 2, 1, 3))
    assert np.count_nonzero(kn.view(np.float32)) == 6 * G * d


def test_oracle_rejects_out_of_range_block():
    rng = np.random.default_rng(18)
    q, Ks, Vs = random_case(rng, [20], 4, 4, 16)
    kc, vc, bt = paged_from_contiguous(Ks, Vs, 16, rng)
    bt[0, 1] = kc.shape[0]
    with pytest.raises(ValueError):
        oracle.decode(q, kc, vc, bt, np.array([20], np.int32), 1.0)


def test_header_says_test_infrastructure():
    for f in ("__init__.py", "attention.py", "cache_ops.py", "build.py", "pa_oracle.c"):
        text = open(os.path.join(os.path.dirname(ORACLE_SRC), f)).read()
        assert re.search(r"test infrastructure", text, re.I), f

