"""The C ABI from plain C: tests/c/kvq_c_client.c is compiled with gcc against
include/kvq.h and the in-tree libkvq.so, and run (no Python or torch in the client)."""

import os
import shutil
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import certified_quantized_kv_gb300 as kvq  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_client(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libdir = os.path.dirname(kvq.LIB_PATH)
    exe = str(tmp_path / "kvq_c_client")
    cmd = [cc, "-O2", "-std=c11", os.path.join(ROOT, "tests", "c", "kvq_c_client.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           "-L", libdir, "-l:libkvq.so", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           "-Wl,-rpath," + libdir + ":" + os.path.join(cuda, "lib64"), "-lm", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c client ok" in r.stdout
