"""Exhaustive GPU check of the NVFP4 encode helpers (hardware E2M1/E4M3 converters, corrected
division) against encoders written from the format definitions: tests/cuda/nvfp4_convert_check.cu,
compiled for sm_103a and run as its own program."""
import os
import re
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_encode_helpers_match_the_definitions_on_every_input(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "nvfp4_convert_check")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "bit_kv_cache_03_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "cuda", "nvfp4_convert_check.cu"), "-o", exe],
                   check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=300).stdout
    counts = dict(re.findall(r"^(\w+) mismatches (\d+)", out, flags=re.M))
    assert len(counts) == 11, out
    assert all(v == "0" for v in counts.values()), out
