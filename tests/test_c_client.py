"""The C ABI from a plain C program (tests/c/abi_client.c), built with the
system C compiler against include/ew.h and linked to libew.so."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import memory_bound_elementwise_gb300 as ew
import oracle
from memory_bound_elementwise_gb300 import inputs
from tests.gpu_util import assert_bits_equal

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_client.c")

pytestmark = pytest.mark.skipif(not os.path.exists(ew.LIB_PATH), reason="libew.so not built")


def _cuda_lib_dirs():
    """Library folders of the CUDA toolkit, on x86_64 and on Arm (sbsa) hosts."""
    import glob
    roots = [os.environ.get("CUDA_HOME"), "/usr/local/cuda"]
    nv = shutil.which("nvcc")
    if nv:
        roots.append(os.path.dirname(os.path.dirname(os.path.realpath(nv))))
    dirs = []
    for r in roots:
        if r:
            dirs += [os.path.join(r, "lib64")] + sorted(glob.glob(os.path.join(r, "targets", "*", "lib")))
    return dirs


def _cudart_link_args():
    """Link arguments for the CUDA runtime calls the client makes itself: the
    toolkit's static runtime (present wherever nvcc is), else the shared one."""
    for d in _cuda_lib_dirs():
        if os.path.exists(os.path.join(d, "libcudart_static.a")):
            return [os.path.join(d, "libcudart_static.a"), "-lpthread", "-ldl", "-lrt"]
    for d in _cuda_lib_dirs():
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return ["-L", d, "-lcudart", "-Wl,-rpath," + d]
    return None


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    out = str(tmp_path_factory.mktemp("cabi") / "abi_client")
    libdir = os.path.dirname(ew.LIB_PATH)
    cudart = _cudart_link_args()
    if cudart is None:
        pytest.skip("no CUDA runtime library to link the client against")
    # the library file is libew.so: link it by path so no -l lookup rules apply
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1", SRC, "-I", os.path.join(ROOT, "include"),
           ew.LIB_PATH, "-Wl,-rpath," + libdir] + cudart
    subprocess.run(cmd + ["-o", out], check=True)
    return out


def test_c_client_host_checks(client):
    r = subprocess.run([client, "host"], stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    assert r.returncode == 0, r.stdout
    assert "host ok" in r.stdout


@pytest.mark.gpu
def test_c_client_on_the_gpu(client, tmp_path):
    n = 1_000_003
    a = inputs.normal(n, 9100)
    b = inputs.normal(n, 9101)
    pa, pb = tmp_path / "a.bin", tmp_path / "b.bin"
    a.tofile(pa)
    b.tofile(pb)
    outs = [tmp_path / ("%s.bin" % k) for k in ("add", "relu", "add_relu")]
    r = subprocess.run([client, "gpu", str(pa), str(pb)] + [str(o) for o in outs],
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    assert r.returncode == 0, r.stdout
    got = [np.fromfile(o, dtype=np.float32) for o in outs]
    assert_bits_equal(got[0], oracle.add("f32", a, b), "f32", True, "C client add")
    assert_bits_equal(got[1], oracle.relu("f32", a), "f32", False, "C client relu")
    assert_bits_equal(got[2], oracle.relu("f32", oracle.add("f32", a, b)), "f32", True, "C client add_relu")
