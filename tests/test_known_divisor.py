"""The quantising append divides bf16 values by a per-head scale with a reciprocal computed
once and one fused multiply-add correction instead of a full division per element. This checks,
on the CPU and for every case, that the result is the IEEE quotient the quantiser's definition
("KV cache and PagedAttention", section 7; fp32(x / s), then the code) asks for: all 128 bf16
significands against all 2^23 fp32 significands of the scale (``known_divisor_check.c``)."""
import os
import platform
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def _flags():
    flags = ["-O2", "-std=c11", "-ffp-contract=off"]
    if platform.machine() in ("x86_64", "AMD64"):
        try:
            with open("/proc/cpuinfo") as f:
                if " fma " in f.read():
                    flags.append("-mfma")  # hardware fused multiply-add for fmaf
        except OSError:
            pass
    return flags


def test_reciprocal_and_one_correction_equal_ieee_division(tmp_path):
    if not shutil.which("gcc"):
        pytest.skip("no C compiler")
    exe = str(tmp_path / "known_divisor_check")
    src = os.path.join(HERE, "known_divisor_check.c")
    try:
        subprocess.run(["gcc"] + _flags() + ["-fopenmp", src, "-o", exe, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(["gcc"] + _flags() + [src, "-o", exe, "-lm"], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=600).stdout
    n, wrong, wrong_uncorrected, zero_signs = (int(v) for v in out.split())
    assert n == 128 * 2 ** 23
    assert wrong == 0
    assert zero_signs == 0  # +0 / s = +0 and -0 / s = -0
    assert wrong_uncorrected > n // 10  # without the correction the check does fail
