"""The host record that decides whether a launch may overlap the kernel
before it (TR_LAUNCH_OVERLAP_PREVIOUS is dropped when the launch's workspace
is the one this library's previous launch on that stream used, or when the
stream's entry may have been replaced): tests/c_abi/stream_guard_test.cpp
drives image_preprocessing_gb300/csrc/stream_guard.h directly, with a table
smaller than the library's to reach replacement, and from eight threads."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_stream_guard_host_logic(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = str(tmp_path / "stream_guard_test")
    cmd = [cxx, "-std=c++17", "-O2", "-Wall", "-Wextra", "-Werror", "-pthread",
           "-I", os.path.join(ROOT, "image_preprocessing_gb300", "csrc"),
           os.path.join(HERE, "c_abi", "stream_guard_test.cpp"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "all checks passed" in r.stdout
