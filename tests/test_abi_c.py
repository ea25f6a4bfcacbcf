"""The boundary from plain C: include/oasis.h compiles as strict C99 and a C
program linked against liboasis.so gets the documented answers (no GPU work:
version string, argument validation, workspace size)."""
import os
import shutil
import subprocess

import pytest

from sparse_decode_attention_oasis_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_from_c.c")


@pytest.fixture(scope="module")
def c_program(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    build.build()
    libdir = os.path.dirname(binding.LIB_PATH)
    exe = str(tmp_path_factory.mktemp("abi_c") / "abi_from_c")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           SRC, "-o", exe, os.path.join(libdir, os.path.basename(binding.LIB_PATH)), f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_gets_the_documented_answers(c_program):
    r = subprocess.run([c_program], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    out = dict(line.split(" ", 1) for line in r.stdout.strip().splitlines())
    assert out["version"].startswith("oasis-gb300")
    assert int(out["score_null"]) == 1        # OASIS_ERR_INVALID: NULL device pointers
    assert int(out["score_d64"]) == 4         # OASIS_ERR_UNSUPPORTED: head dim 64
    assert int(out["topk_group"]) == 1        # OASIS_ERR_INVALID: Hq not a multiple of Hkv
    assert int(out["shape_null"]) == 1        # OASIS_ERR_INVALID: no shape
    shape = binding.Shape.of(B=2, Hq=32, Hkv=8, nb_max=256, n_la=4, Kb=32, P=32)
    assert int(out["workspace"]) == binding.oasis_attn_workspace_bytes(shape) > 0
    assert int(out["workspace_bad"]) == 0
