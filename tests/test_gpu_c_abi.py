"""The C ABI from plain C: `tests/c_abi_program.c` is compiled with the host C compiler
against `include/qgemv.h`, linked with `libqgemv.so`, the CUDA runtime and the oracle's own
library, and run once per format.  It allocates its device buffers with cudaMalloc, calls
qgemv_run on a stream of its own, compares every output with the oracle within the GEMV
tolerance (|y - y_ref| <= 2e-3 * sum|x w| + 1e-5), and checks that invalid arguments are
refused with the documented status (null x, N = 0, a ragged K, a misaligned x)."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from quantized_weight_dequant_gb300 import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    from quantized_weight_dequant_gb300.build import build_library
    libdir = os.path.dirname(build_library())
    odir = os.path.dirname(oracle.build())
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path_factory.mktemp("c_abi") / "c_abi_program")
    cmd = [cc, "-O2", "-std=c11", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_abi_program.c"), "-o", exe,
           "-L", libdir, "-lqgemv", "-L", odir, "-loracle", "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           f"-Wl,-rpath,{libdir}:{odir}:{os.path.join(cuda, 'lib64')}"]
    p = subprocess.run(cmd, capture_output=True, text=True)
    assert p.returncode == 0, p.stderr
    return exe


@pytest.mark.parametrize("fmt,N,K", [(synth.Q4_K, 1000, 4096), (synth.NVFP4, 513, 2048), (synth.TQ1_0, 300, 4096),
                                     (synth.Q5_K, 129, 2048), (synth.Q6_K, 77, 4096), (synth.Q8_0, 250, 1024)])
def test_c_program_matches_the_oracle(program, tmp_path, fmt, N, K):
    seed = 31 + N + fmt
    W = synth.make_weights(fmt, N, K, seed)
    x = synth.make_x(fmt, K, seed)
    wpath, xpath = str(tmp_path / "w.bin"), str(tmp_path / "x.bin")
    np.ascontiguousarray(W, dtype=np.uint8).tofile(wpath)
    np.ascontiguousarray(x, dtype=np.uint16).tofile(xpath)
    p = subprocess.run([program, str(fmt), str(N), str(K), wpath, xpath], capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stdout + p.stderr
    assert p.stdout.startswith("ok"), p.stdout
