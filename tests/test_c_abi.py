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
