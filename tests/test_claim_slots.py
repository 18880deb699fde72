"""The host rule that gives each streaming launch its unit-claim word
(gated_group_rmsnorm_gb300/csrc/ggrn_slots.h), built into a small C++ program
with the host compiler and run on the CPU: a word is never given to a launch
while another stream's launch on it is still running, so two launches never
claim from one word at once."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_claim_slot_rule(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path / "slots_test")
    r = subprocess.run([cxx, "-O1", "-std=c++17", "-Wall", "-Werror", "-I",
                        os.path.join(ROOT, "gated_group_rmsnorm_gb300", "csrc"),
                        os.path.join(ROOT, "tests", "c", "ggrn_slots_test.cpp"), "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "failures 0" in r.stdout
