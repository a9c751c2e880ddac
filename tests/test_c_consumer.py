"""The C ABI from plain C: tests/c_abi/consumer.c includes only
include/tr_fused_norm.h and the CUDA runtime's C header, links libtrfn.so,
and runs the tiled kernel on a seeded batch; its output is checked against
the oracle.  The CPU test compiles and links it (C99), the GPU test runs it."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import image_preprocessing_gb300 as trfn

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None or not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime_api.h")):
        pytest.skip("no C compiler or CUDA headers")
    exe = os.path.join(tmp, "consumer")
    libdir = os.path.dirname(trfn.LIB_PATH)
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), os.path.join(HERE, "c_abi", "consumer.c"), "-o", exe,
           trfn.LIB_PATH, "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + libdir, "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_consumer_compiles_and_links(tmp_path):
    assert os.path.exists(_build(str(tmp_path)))


@pytest.mark.gpu
def test_c_consumer_matches_the_oracle(tmp_path):
    exe = _build(str(tmp_path))
    r = subprocess.run([exe, str(tmp_path)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    N, H, W, C = 8, 32, 48, 3
    src = np.fromfile(tmp_path / "src.u8", np.uint8).reshape(N, H, W, C)
    rec = np.fromfile(tmp_path / "rec.i32", np.int32).reshape(N, 5)
    got = np.fromfile(tmp_path / "out.f16", np.uint16).reshape(N, H, W, C)
    mean, std, _ = trfn.tr_norm_preset("IMAGENET")
    ref = oracle.fused_norm(src, np.asarray(mean, np.float32), np.asarray(std, np.float32), rec,
                            out_dtype=oracle.OUT_F16)

    def ordered(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)

    assert int(np.max(np.abs(ordered(got) - ordered(ref)))) <= 1
    assert np.array_equal(got[ref == 0], ref[ref == 0])
    assert rec[:, 0].min() >= 0 and rec[:, 0].max() <= 1
