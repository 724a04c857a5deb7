"""The ABI from plain C: tests/c/abi_check.c is compiled with the host C
compiler against include/zero.h, linked with libzero.so, the oracle library
and the CUDA runtime, and run as its own process (no Python or torch in it).

"host" mode (CPU suite): plan and memory-model answers agree with the oracle,
bad arguments are rejected without a launch.  "gpu" mode: device buffers from
cudaMalloc, zero_init_shards + two zero_step calls on 4 virtual ranks, the
gathered bf16 buffer bit-identical to the oracle and the fp32 masters within
1e-6 relative.  "amp" mode: the mixed-precision step from C, fused and as
bucket reductions (last bucket first) plus zero_step_amp_reduced, the two
bit-identical and both matching the oracle's mixed-precision step.
"offload" mode: zero_offload_step with malloc'd host state and cudaHostAlloc'd
shards, in ragged chunks on 3 host threads, against the oracle; pageable
gradient shards are refused without a launch.
"""
import glob
import os
import shutil
import subprocess

import pytest

import oracle
from zero_sharded_optimizer_flatten_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_check.c")


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    zlib = _build.build()
    olib = oracle.build()
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(_build.nvcc())))
    cudalib = os.path.join(cuda, "lib64")
    if not os.path.exists(os.path.join(cudalib, "libcudart.so")):
        cudalib = next(iter(glob.glob(os.path.join(cuda, "targets", "*", "lib"))), cudalib)
    out = str(tmp_path_factory.mktemp("abi") / "abi_check")
    libdirs = [os.path.dirname(zlib), os.path.dirname(olib), cudalib]
    cmd = [cc, "-O2", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), SRC, "-o", out]
    for d in libdirs:
        cmd += ["-L", d, f"-Wl,-rpath,{d}"]
    cmd += ["-lzero", "-loracle", "-lcudart", "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _run(program, mode):
    r = subprocess.run([program, mode], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    return r.stdout


def test_c_program_host_checks(program):
    assert "host ok" in _run(program, "host")


@pytest.mark.gpu
def test_c_program_steps_match_oracle(program):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    assert "gpu ok" in _run(program, "gpu")


@pytest.mark.gpu
def test_c_program_mixed_precision_paths_match_oracle(program):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    assert "amp ok" in _run(program, "amp")


@pytest.mark.gpu
def test_c_program_offload_step_matches_oracle(program):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    assert "offload ok" in _run(program, "offload")
