"""The header is plain C: a C11 program includes it, links libqmm.so and
checks the host-side contract (sizes, statuses) without a GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c11_consumer_compiles_links_and_runs(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    from quantized_weight_gguf_gb300 import build_lib
    lib = build_lib.build()
    exe = str(tmp_path / "abi_consumer")
    src = os.path.join(ROOT, "tests", "c", "abi_consumer.c")
    cmd = [gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), src,
           "-o", exe, "-L", os.path.dirname(lib), "-lqmm",
           "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")   # host-side checks only
    r = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "all checks passed" in r.stdout
