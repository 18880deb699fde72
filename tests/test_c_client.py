"""The C ABI from a plain C program (tests/c/ggrn_c_client.c), no Python in
the process: built with the host C compiler against include/ggrn.h and
libggrn.so.  Without a GPU it checks the argument statuses; on a GPU it runs
ggrn_forward and ggrn_forward_host on inputs from the seeded generator, and
the output is compared with the oracle."""
import glob
import os
import shutil
import subprocess

import pytest
import torch

import ggrn_inputs
import gated_group_rmsnorm_gb300 as g
from gated_group_rmsnorm_gb300 import binding, build
from tests import gpu_util
from tests.tolerance import assert_parity

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "ggrn_c_client.c")


def _cuda_home():
    return os.path.dirname(os.path.dirname(os.path.realpath(build.nvcc())))


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    lib = build.build()
    cuda = _cuda_home()
    cands = [os.path.join(cuda, "lib64"), os.path.join(cuda, "lib")]
    cands += sorted(glob.glob(os.path.join(cuda, "targets", "*", "lib")))
    libdirs = [os.path.dirname(lib)] + [d for d in cands
                                        if os.path.exists(os.path.join(d, "libcudart.so"))][:1]
    exe = str(tmp_path_factory.mktemp("cclient") / "ggrn_c_client")
    cmd = [cc, "-O2", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), SRC, "-o", exe]
    cmd += [f"-L{d}" for d in libdirs] + ["-lggrn", "-lcudart"]
    cmd += [f"-Wl,-rpath,{d}" for d in libdirs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def _lines(out):
    return dict(line.split(" ", 1) for line in out.strip().splitlines())


def test_c_client_argument_statuses(client):
    r = subprocess.run([client, "validate"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    got = _lines(r.stdout)
    assert int(got["version"]) >= 100
    assert int(got["null_y"]) == binding.ERR_NULL
    assert int(got["shape"]) == binding.ERR_SHAPE
    assert int(got["dtype"]) == binding.ERR_DTYPE
    assert int(got["overlap"]) == binding.ERR_OVERLAP
    assert int(got["rows0"]) == binding.OK
    assert int(got["host_null_ws"]) == binding.ERR_NULL
    assert got["status_string_1"] == g.status_string(1)


def _bytes(t):
    if t.dtype in (torch.bfloat16, torch.float16):
        t = t.view(torch.int16)
    return t.contiguous().numpy().tobytes()


@pytest.mark.gpu
@pytest.mark.parametrize("name,rows", [("mamba2_prefill", 67), ("gdn_onnx", 45),
                                       ("wide_single_group", 33)])
def test_c_client_matches_oracle(client, tmp_path, name, rows):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = ggrn_inputs.WORKLOADS[name].with_rows(rows)
    host = ggrn_inputs.make_inputs(wl, seed=rows)
    src, dst = tmp_path / "in.bin", tmp_path / "out.bin"
    src.write_bytes(_bytes(host.y) + _bytes(host.gate) + _bytes(host.w))
    r = subprocess.run([client, "run", str(src), str(dst), str(rows), str(wl.width),
                        str(wl.group_size), str(binding.DTYPE_CODE[wl.dtype]), str(wl.mode),
                        repr(wl.eps)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, (r.stdout, r.stderr)
    got = _lines(r.stdout)
    assert int(got["forward"]) == binding.OK and int(got["forward_host"]) == binding.OK
    assert got["fault"] == "0"
    for path in (dst, tmp_path / "out.bin.host"):   # ggrn_forward, ggrn_forward_host
        raw = torch.frombuffer(bytearray(path.read_bytes()),
                               dtype=torch.int16 if wl.dtype != torch.float32 else torch.float32)
        out = raw.view(wl.dtype).reshape(rows, wl.width)
        res = gpu_util.compare(out, host, wl.group_size, wl.eps, wl.mode)
        assert res["ok"], (path.name, res)


@pytest.mark.gpu
@pytest.mark.parametrize("rows", [1531, 65536])
def test_c_client_strided_views(client, tmp_path, rows):
    """The strided workload's packed in-proj layout from C: the two strided
    views through ggrn_forward, the packed matrix through
    ggrn_forward_inproj, and pinned host memory (read in place) through
    ggrn_forward_host, every row against the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = ggrn_inputs.WORKLOADS["strided_odd_span"].with_rows(rows)
    host = ggrn_inputs.make_inputs(wl, seed=rows)
    src, dst = tmp_path / "in.bin", tmp_path / "out.bin"
    src.write_bytes(_bytes(host.packed) + _bytes(host.w))
    r = subprocess.run([client, "packed", str(src), str(dst), str(rows), str(wl.width),
                        str(wl.group_size), str(binding.DTYPE_CODE[wl.dtype]), str(wl.mode),
                        repr(wl.eps), str(wl.packed_width), str(wl.width)],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, (r.stdout, r.stderr)
    got = _lines(r.stdout)
    for k in ("forward", "forward_inproj", "forward_host"):
        assert int(got[k]) == binding.OK, (k, got)
    assert got["fault"] == "0"
    for suffix in ("", ".inproj", ".host"):
        raw = torch.frombuffer(bytearray((tmp_path / ("out.bin" + suffix)).read_bytes()),
                               dtype=torch.int16)
        out = raw.view(wl.dtype).reshape(rows, wl.width)
        res = gpu_util.compare_all_rows(out, host, wl.group_size, wl.eps, wl.mode)
        assert_parity(res, "c client " + (suffix or "forward"))
