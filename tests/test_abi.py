"""The C-ABI library loads without a GPU and exports every entry point the headers declare."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(pa_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


@pytest.fixture(scope="module")
def lib_path():
    from paged_kv_cache_04_gb300 import _build
    return _build.ensure_built()


def test_header_declares_the_calls():
    names = declared_functions()
    for must in ("pa_reshape_and_cache", "pa_decode", "pa_decode_split", "pa_decode_split_workspace_bytes",
                 "pa_copy_blocks", "pa_get_error"):
        assert must in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_host_only_calls(lib_path):
    import paged_kv_cache_04_gb300 as pa
    lib = pa.library()
    assert pa.pa_version() >= 100
    assert lib.pa_status_string(0) == b"ok"
    # workspace size: S=8, H=64, d=128, max ctx 131072, partitions of 512 -> P = 256
    P = 256
    rows = 8 * 64 * P
    want = ((rows * 128 * 4 + 255) // 256) * 256 + 2 * (((rows * 4) + 255) // 256) * 256
    assert pa.pa_decode_split_workspace_bytes(8, 64, 128, 131072, 512) == want
    assert pa.pa_decode_split_workspace_bytes(8, 64, 128, -1, 512) == 0


def test_invalid_arguments_rejected_before_any_launch(lib_path):
    """Argument checks run on the host; these calls never reach a kernel."""
    import paged_kv_cache_04_gb300 as pa
    lib = pa.library()
    null = ctypes.c_void_p(0)
    # H % G != 0
    assert lib.pa_decode(null, null, null, null, null, 1, null, 1, 6, 4, 128, 16, 0, 10, 1.0, 2, 2, null) == 1
    # num_seqs == 0 is a no-op
    assert lib.pa_decode(null, null, null, null, null, 1, null, 0, 8, 8, 128, 16, 0, 10, 1.0, 2, 2, null) == 0
    # null pointers
    assert lib.pa_decode(null, null, null, null, null, 1, null, 2, 8, 8, 128, 16, 0, 10, 1.0, 2, 2, null) == 1
    # misaligned pointers are rejected before the shape checks launch anything
    odd = ctypes.c_void_p(0x1008)
    assert lib.pa_decode(odd, odd, odd, odd, odd, 1, odd, 2, 8, 8, 128, 16, 0, 10, 1.0, 2, 2, null) == 1
    # unsupported head_dim / block size / group
    al = ctypes.c_void_p(0x10000)
    assert lib.pa_decode(al, al, al, al, al, 1, al, 2, 8, 8, 96, 16, 0, 10, 1.0, 2, 2, null) == 2
    assert lib.pa_decode(al, al, al, al, al, 1, al, 2, 8, 8, 128, 8, 0, 10, 1.0, 2, 2, null) == 2
    assert lib.pa_decode(al, al, al, al, al, 1, al, 2, 32, 2, 128, 16, 0, 10, 1.0, 2, 2, null) == 2
    assert lib.pa_decode(al, al, al, al, al, 1, al, 2, 8, 8, 512, 16, 0, 10, 1.0, 2, 2, null) == 2
    # head_dim 256 is served by pa_decode / pa_decode_split, not by the E4M3 calls or the cascade
    assert lib.pa_decode_fp8(al, al, al, al, al, 1, al, 2, 8, 8, 256, 16, 0, 10, 1.0, 1.0, 1.0, 2, 2, null) == 2
    assert lib.pa_decode_cascade(al, al, al, al, al, 4, al, 2, 8, 8, 256, 16, 0, 10, 1.0, 2, 2, al, al, 1, 2, 32,
                                 64, 32, al, 1 << 30, null) == 2
    # out dtype must be the cache dtype or fp32
    assert lib.pa_decode(al, al, al, al, al, 1, al, 2, 8, 8, 128, 16, 0, 10, 1.0, 2, 1, null) == 2
    # split: partition not a multiple of the block size; workspace too small
    assert lib.pa_decode_split(al, al, al, al, al, 1, al, 2, 8, 8, 128, 16, 0, 10, 1.0, 2, 2, 100, 24, al, 1 << 20,
                               null) == 1
    assert lib.pa_decode_split(al, al, al, al, al, 1, al, 2, 8, 8, 128, 16, 0, 10, 1.0, 2, 2, 100, 32, al, 16,
                               null) == 1
    # reshape_and_cache: zero tokens is a no-op; misaligned slot mapping rejected
    assert lib.pa_reshape_and_cache(null, null, null, null, null, 0, 8, 128, 16, 0, 10, 2, null) == 0
    assert lib.pa_reshape_and_cache(al, al, al, al, ctypes.c_void_p(0x10004), 4, 8, 128, 16, 0, 10, 2, null) == 1
    # pools whose rows (num_blocks x kv heads x block size) overflow the 32-bit TMA row coordinate
    assert lib.pa_decode(al, al, al, al, al, 1, al, 2, 8, 8, 128, 16, 0, 1 << 28, 1.0, 2, 2, null) == 2
    # a pool layout other than HND (0) and NHD (1) is rejected, even with nothing to do
    assert lib.pa_decode(null, null, null, null, null, 1, null, 0, 8, 8, 128, 16, 2, 10, 1.0, 2, 2, null) == 1
    assert lib.pa_reshape_and_cache(null, null, null, null, null, 0, 8, 128, 16, 7, 10, 2, null) == 1
    assert lib.pa_reshape_and_cache_fp8(null, null, null, null, null, 0, 8, 128, 16, -1, 10, 2, 1.0, 1.0,
                                        null) == 1
    # copy_blocks: no pairs is a no-op
    arr = (ctypes.c_void_p * 1)(0x10000)
    assert lib.pa_copy_blocks(arr, arr, 1, al, 0, 8, 128, 16, 10, 2, null) == 0
    assert lib.pa_copy_blocks(arr, arr, 1, null, 3, 8, 128, 16, 10, 2, null) == 1
    # the bounded-wait diagnostic takes limits of 1 us to 100 ms only
    assert lib.pa_check_wait_limit(0, null) == 1
    assert lib.pa_check_wait_limit(999, null) == 1
    assert lib.pa_check_wait_limit(100_000_001, null) == 1


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import paged_kv_cache_04_gb300 as pa
    monkeypatch.setattr(pa, "_lib", None)
    monkeypatch.setattr(pa, "library_path", str(tmp_path / "missing.so"))
    with pytest.raises(pa.PAError):
        pa.library()


def test_survey_boundary_names(lib_path):
    """The boundary's names for the status string and the error-word check:
    pa_status_str is pa_status_string under another name; pa_debug_check is
    declared and exported."""
    import paged_kv_cache_04_gb300 as pa
    lib = pa.library()
    names = declared_functions()
    assert "pa_status_str" in names and "pa_debug_check" in names
    for st in range(-1, 7):
        assert lib.pa_status_str(st) == lib.pa_status_string(st)
    assert pa.pa_status_str(0) == "ok"


def test_static_scratch_size_matches_header(lib_path):
    """The binding reads the scratch size from the library; the header's macro agrees."""
    import paged_kv_cache_04_gb300 as pa
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    m = re.search(r"#define\s+PA_STATIC_SCRATCH_BYTES\s+\((\d+)u\s*\*\s*(\d+)u\s*\*\s*(\d+)u\)", text)
    assert m, "macro not found"
    macro = int(m.group(1)) * int(m.group(2)) * int(m.group(3))
    assert pa.PA_STATIC_SCRATCH_BYTES == macro == int(pa.library().pa_static_scratch_bytes())


def test_static_split_rejects_bad_arguments_like_the_workspace_call(lib_path):
    """pa_decode_split_static runs pa_decode_split's argument checks first, so a
    bad call gets the same status from both, even when it is also too large for
    the scratch array (these calls return before any CUDA call)."""
    import paged_kv_cache_04_gb300 as pa
    lib = pa.library()
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: the calls fail on the host
    huge = 1 << 20  # max_context_len far beyond the scratch array
    cases = [
        # null q/out with sequences
        (null, null, 8, 64, 8, 128, 16, huge, 512),
        # partition not a multiple of the block size
        (fake, fake, 8, 64, 8, 128, 16, huge, 500),
        # more sequences than split mode takes
        (fake, fake, 4096, 64, 8, 128, 16, huge, 512),
        # unsupported head_dim
        (fake, fake, 8, 64, 8, 96, 16, huge, 512),
        # negative max_context_len
        (fake, fake, 8, 64, 8, 128, 16, -1, 512),
    ]
    for out, q, S, H, G, d, B, mctx, T in cases:
        a = lib.pa_decode_split(out, q, fake, fake, fake, 64, fake, S, H, G, d, B, 0, 1000, 1.0, 2, 2, mctx, T,
                                fake, 1 << 40, null)
        b = lib.pa_decode_split_static(out, q, fake, fake, fake, 64, fake, S, H, G, d, B, 0, 1000, 1.0, 2, 2,
                                       mctx, T, null)
        assert a == b != 0, (S, d, mctx, T, a, b)
    # a valid call that is only too large: UNSUPPORTED from the static call alone
    assert lib.pa_decode_split_static(fake, fake, fake, fake, fake, 1 << 16, fake, 8, 64, 8, 128, 16, 0, 1 << 20,
                                      1.0, 2, 2, huge, 512, null) == 2
