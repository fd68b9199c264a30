"""Register budgets of the decode kernels, from the compiler's own report.

An SM has 65,536 registers, handed out per thread in steps of 8. Shared memory
lets two 128-thread CTAs of the 16-bit tensor-core decode kernel share an SM
and three of the MHA and E4M3 kernels; this test compiles the decode units with
`-Xptxas -v` (as the build does, for sm_103a) and checks that their register
counts allow the same number, and that these kernels do not spill. A change
that pushes, say, the MHA kernel past 168 registers would otherwise cost it a
CTA per SM without any other sign. No GPU is needed (about half a minute).
"""
import os
import re
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_cache_04_gb300", "csrc")
UNITS = ["pa_decode_bf16.cu", "pa_decode_f16.cu", "pa_decode_fp8.cu", "pa_decode_g8.cu"]
THREADS = 128
SM_REGS = 65536


def _compile(nvcc, unit, out_dir):
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
                        "-Xptxas", "-v", "-c", os.path.join(CSRC, unit), "-o", os.path.join(out_dir, unit + ".o")],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stderr


@pytest.fixture(scope="module")
def kernels(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    cxxfilt = shutil.which("c++filt")
    if not os.path.exists(nvcc) or cxxfilt is None:
        pytest.skip("nvcc or c++filt not found")
    d = str(tmp_path_factory.mktemp("regs"))
    with ThreadPoolExecutor(len(UNITS)) as ex:
        logs = list(ex.map(lambda u: _compile(nvcc, u, d), UNITS))
    found = {}
    for log in logs:
        name = spill = None
        for line in log.splitlines():
            m = re.search(r"Compiling entry function '(\S+)'", line)
            if m:
                name = subprocess.run([cxxfilt, m.group(1)], capture_output=True, text=True).stdout.strip()
                spill = None
                continue
            m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
            if m:
                spill = int(m.group(1)) + int(m.group(2))
            m = re.search(r"Used (\d+) registers", line)
            if m and name and "paged_decode_kernel" in name:
                args = re.search(r"paged_decode_kernel<([^>]*)>", name).group(1).split(",")
                dt, qt, ot = (a.strip() for a in args[:3])
                D, path, mode = int(args[3]), int(args[4]), int(args[5])
                found[(dt, qt, ot, D, path, mode)] = (int(m.group(1)), spill or 0)
                name = None
    return found


PATH_MHA, PATH_MMA, PATH_MMA_G8 = 1, 2, 3


def expected_ctas(dt, D, path):
    """CTAs per SM that shared memory allows the measured head_dim-128 kernels."""
    if D != 128:
        return None
    if path in (PATH_MMA, PATH_MMA_G8):
        return 3 if "fp8" in dt else 2
    if path == PATH_MHA and dt != "float":
        return 3
    return None


def test_the_measured_kernels_were_found(kernels):
    keys = {(k[0], k[3], k[4], k[5]) for k in kernels}
    for want in [("__nv_bfloat16", 128, PATH_MMA, 0), ("__nv_bfloat16", 128, PATH_MMA, 1),
                 ("__half", 128, PATH_MHA, 0), ("pa::fp8e4m3", 128, PATH_MMA, 0), ("pa::fp8e4m3", 128, PATH_MMA, 1),
                 ("__nv_bfloat16", 128, PATH_MMA_G8, 0), ("pa::fp8e4m3", 128, PATH_MMA_G8, 0)]:
        assert want in keys, (want, sorted(keys)[:8])


def test_registers_allow_the_shared_memory_occupancy(kernels):
    bad = {}
    for (dt, qt, ot, D, path, mode), (regs, spill) in kernels.items():
        n = expected_ctas(dt, D, path)
        if n is None:
            continue
        per_thread = -(-regs // 8) * 8
        if per_thread * THREADS * n > SM_REGS:
            bad[(dt, qt, ot, D, path, mode)] = (regs, n)
    assert not bad, f"register count below the CTAs per SM that shared memory allows: {bad}"


def test_measured_kernels_do_not_spill(kernels):
    spills = {k: v[1] for k, v in kernels.items() if expected_ctas(k[0], k[3], k[4]) is not None and v[1]}
    assert not spills, spills
