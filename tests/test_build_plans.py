"""Compile-time layouts of every tensor-core kernel build, checked on the host
(no GPU): shared memory within the 227 KB a CTA may opt into, tensor memory
within 512 columns, at least two stages, at most 16 warps (so that the
128-register budget per thread holds), and the 32-row build taking the 16-row
build's zero-point method, which keeps rows bitwise equal between them."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MAX_DYN_SMEM = 227 * 1024


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("plans") / "plan_check")
    subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I" + os.path.join(ROOT, "include"),
                    "-I" + os.path.join(ROOT, "weight_only_bit_wq_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "plan_check.cu"), "-o", exe],
                   check=True, capture_output=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    rows = {}
    for line in out.split("\n"):
        if line.strip():
            b, g, nc, st, smem, z, na, nd, tend, thr = map(int, line.split())
            rows[(b, g, nc)] = dict(stages=st, smem=smem, z=z, na=na, nd=nd, tmem_end=tend,
                                    threads=thr)
    return rows


def test_every_build_is_listed(plans):
    assert len(plans) == 18


def test_resources_fit(plans):
    for key, p in plans.items():
        assert p["smem"] <= MAX_DYN_SMEM, key
        assert p["tmem_end"] <= 512, key
        assert p["stages"] >= 2, key
        assert 1 <= p["na"] <= 3 and 1 <= p["nd"] <= 2, key
        assert p["threads"] <= 16 * 32, key


def test_wide_build_keeps_the_zero_point_method(plans):
    for (b, g, nc), p in plans.items():
        if nc == 32:
            assert p["z"] == plans[(b, g, 16)]["z"], (b, g)


def test_headline_format_plan(plans):
    # 4-bit, group 128, 16 rows: four stages, three A slots, two accumulator
    # slots, zero point on the tensor core
    p = plans[(4, 128, 16)]
    assert (p["stages"], p["na"], p["nd"], p["z"]) == (4, 3, 2, 1)
