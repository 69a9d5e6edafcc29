"""include/vc.h from plain C99: compile, link against libvcoll.so, run the
host-only entry points (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_header_compiles_and_links_from_c(tmp_path):
    from collective_communication_algorithms_virtual_gb300 import build

    lib = build.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "abi_smoke"
    libdir = os.path.dirname(lib)
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-pedantic", os.path.join(ROOT, "tests", "c", "abi_smoke.c"),
                    "-I", os.path.join(ROOT, "include"), "-L", libdir, "-l:libvcoll.so",
                    f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stdout, out.stderr)
    assert out.stdout.startswith("ok")


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _build_c_program(tmp_path, name, cuda=False):
    from collective_communication_algorithms_virtual_gb300 import build

    lib = build.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / name
    libdir = os.path.dirname(lib)
    # vc.h alone is pedantic C99; CUDA's runtime header needs C11 (anonymous unions)
    std = ["-std=c11"] if cuda else ["-std=c99", "-pedantic"]
    cmd = [cc, *std, "-Wall", "-Werror", os.path.join(ROOT, "tests", "c", name + ".c"),
           "-I", os.path.join(ROOT, "include"), "-L", libdir, "-l:libvcoll.so", f"-Wl,-rpath,{libdir}"]
    if cuda:
        home = _cuda_home()
        cudalib = os.path.join(home, "lib64")
        cmd += ["-I", os.path.join(home, "include"), "-L", cudalib, "-lcudart", f"-Wl,-rpath,{cudalib}"]
    subprocess.run(cmd + ["-o", str(exe)], check=True)
    return exe


def test_c_program_compiles_against_cuda_runtime(tmp_path):
    """The device-work C program builds here (no GPU needed to compile)."""
    assert _build_c_program(tmp_path, "abi_allreduce", cuda=True).exists()


@pytest.mark.gpu
def test_allreduce_and_broadcast_driven_from_c(tmp_path):
    """A C program allocates rank buffers with the CUDA runtime and runs
    vc_allreduce (Ring, RHD, DBT, fused, AUTO) and vc_broadcast through the
    header, checking every element it copies back."""
    exe = _build_c_program(tmp_path, "abi_allreduce", cuda=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, (out.returncode, out.stdout, out.stderr)
    assert out.stdout.startswith("ok")
