"""The C ABI from plain C: tests/c_abi_client.c compiles as C11 against include/nvfp4.h
(-Wall -Wextra -Werror), links against the library and runs its host-side checks (no GPU)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_client_builds_links_and_runs(tmp_path):
    import __graft_entry__
    lib = __graft_entry__.build_library()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "c_abi_client")
    libdir = os.path.dirname(lib)
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi_client.c"), "-o", exe, "-L", libdir, "-lnvfp4_gb300",
                    f"-Wl,-rpath,{libdir}"], check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok 0", r.stdout + r.stderr
