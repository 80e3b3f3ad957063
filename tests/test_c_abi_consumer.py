"""The C ABI is usable from plain C: tests/c_abi_consumer.c includes the public
header (and the CUDA runtime's, for cudaMalloc), is compiled by gcc as C11 and
linked against the built libw4a16.so, then run: status strings, set-up and
validation everywhere; with a GPU also a closed-form GEMV through plain
cudaMalloc'ed buffers (the GPU test below runs it there)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_program_links_and_runs():
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    import __graft_entry__
    __graft_entry__.build()
    import bit_weight_only_w4a16_gb300 as w4
    libdir = os.path.dirname(w4.LIB_PATH)
    out_dir = os.path.join(ROOT, "_build")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "c_abi_consumer")
    cuda_lib = next((d for d in ("/usr/local/cuda/lib64", "/usr/local/cuda/targets/sbsa-linux/lib",
                                 "/usr/local/cuda/targets/x86_64-linux/lib") if os.path.isdir(d)), None)
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", "/usr/local/cuda/include", os.path.join(ROOT, "tests", "c_abi_consumer.c"), "-o", exe,
           "-L", libdir, "-lw4a16", "-Wl,-rpath," + libdir]
    if cuda_lib:
        cmd += ["-L", cuda_lib, "-lcudart", "-Wl,-rpath-link," + cuda_lib, "-Wl,-rpath," + cuda_lib]
    subprocess.check_call(cmd)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert "c consumer ok" in r.stdout


@pytest.mark.gpu
def test_plain_c_program_runs_a_gemv_on_the_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    test_plain_c_program_links_and_runs()
