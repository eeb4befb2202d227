"""The library from C alone: tests/c/gdn_c_abi_test.c is compiled with gcc against
include/liblinattn.h, the built liblinattn.so and the CUDA runtime (plus the fp64 oracle, test
infrastructure), and run.  It checks gdn_fwd against the oracle, gdn_fwd_host bitwise against
gdn_fwd, and synchronous argument errors; exit status 0 means every check passed."""
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_through_the_abi():
    from gated_delta_rule_29_gb300 import _build
    lib = _build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    out_dir = os.path.join(ROOT, "tests", "_build")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "gdn_c_abi_test")
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-O2", "-std=c11", "-o", exe, os.path.join(ROOT, "tests", "c", "gdn_c_abi_test.c"),
           os.path.join(ROOT, "oracle", "gdn_oracle.c"), "-I" + os.path.join(ROOT, "include"),
           "-I" + os.path.join(cuda, "include"), lib, "-Wl,-rpath," + libdir,
           "-L" + os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64"),
           "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    print(res.stdout)
    assert res.returncode == 0, res.stdout + res.stderr
