"""The library driven from C alone (tests/c_abi/pa_c_example.c): only
include/pa.h and the CUDA runtime. The program's cache contents and outputs are
checked here against the oracle."""
import os
import shutil
import subprocess
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import oracle  # noqa: E402

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def test_c_program_matches_oracle(pa, tmp_path):
    lib_dir = os.path.dirname(pa.library_path)
    pa.library()  # builds and loads libpa.so
    cuda = _cuda_home()
    exe = tmp_path / "pa_c_example"
    cc = ["gcc", "-O2", "-std=c11", "-Wall", "-Werror", os.path.join(ROOT, "tests", "c_abi", "pa_c_example.c"),
          "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"), "-o", str(exe),
          "-L", lib_dir, "-lpa", "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
          f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    r = subprocess.run(cc, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    dump = tmp_path / "out.bin"
    r = subprocess.run([str(exe), str(dump)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    raw = dump.read_bytes()
    S, Hq, G, D, B, NB, width = np.frombuffer(raw, np.int32, 7)
    off = 28
    scale = float(np.frombuffer(raw, np.float32, 1, off)[0])
    off += 4

    def take(dtype, n, shape):
        nonlocal off
        a = np.frombuffer(raw, dtype, n, off).reshape(shape)
        off += a.nbytes
        return a
    ntok, npairs, nprompt = np.frombuffer(raw, np.int32, 3, off)
    off += 12
    slots = take(np.int64, ntok, (ntok,))
    pairs = take(np.int64, 2 * npairs, (npairs, 2))
    key = take(np.float32, ntok * G * D, (ntok, G, D))
    val = take(np.float32, ntok * G * D, (ntok, G, D))
    k0 = take(np.float32, NB * G * B * D, (NB, G, B, D))
    v0 = take(np.float32, NB * G * B * D, (NB, G, B, D))
    ctx = take(np.int32, S, (S,))
    bt = take(np.int32, S * width, (S, width))
    q = take(np.float32, S * Hq * D, (S, Hq, D))
    k = take(np.float32, NB * G * B * D, (NB, G, B, D))
    v = take(np.float32, NB * G * B * D, (NB, G, B, D))
    out = take(np.float32, S * Hq * D, (S, Hq, D))
    out_split = take(np.float32, S * Hq * D, (S, Hq, D))
    assert off == len(raw)
    # the oracle's version of the step: prompt writes, copy-on-write copies, the samples' writes
    kb, vb = oracle.reshape_and_cache(key[:nprompt], val[:nprompt], k0, v0, slots[:nprompt])
    ks, vs = oracle.copy_blocks([kb], [vb], pairs)
    kb, vb = oracle.reshape_and_cache(key[nprompt:], val[nprompt:], ks[0], vs[0], slots[nprompt:])
    assert np.array_equal(kb, k.view(np.uint32)) and np.array_equal(vb, v.view(np.uint32)), "cache writes differ"
    assert npairs > 0
    ref = oracle.decode(q, k, v, bt, ctx, scale)
    assert np.abs(out - ref).max() <= 2e-3
    assert np.abs(out_split - ref).max() <= 2e-3
    assert "copy-on-write pairs" in r.stdout
