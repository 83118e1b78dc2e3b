"""The library called from a plain C program (GPU): tests/c_abi/ce_from_c.c,
compiled with gcc against include/gbce.h, libgbce.so and the CUDA runtime (no
Python or torch in the process), runs softmax_fwd and ce_fwd_bwd on inputs from
a file; its outputs are compared with the oracle on the same inputs."""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import workloads
from cross_entropy_loss_ce_gb300 import build as gbuild
from gpu_util import oracle_ce, require_gpu
from parity import check_grad, check_loss, check_softmax

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "ce_from_c.c")


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    require_gpu()
    lib = gbuild.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    out = str(tmp_path_factory.mktemp("c_abi") / "ce_from_c")
    libdir, cudalib = os.path.dirname(lib), os.path.join(cuda, "lib64")
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Werror", SRC, "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), "-L", libdir, "-lgbce", "-L", cudalib, "-lcudart",
           f"-Wl,-rpath,{libdir}:{cudalib}", "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return out


def run(exe, tmp_path, x: torch.Tensor, t: torch.Tensor):
    M, V = x.shape
    inp, outp = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        f.write(np.array([M, V], dtype=np.int64).tobytes())
        f.write(x.numpy().astype(np.float32).tobytes())
        f.write(t.numpy().astype(np.int64).tobytes())
    r = subprocess.run([exe, str(inp), str(outp)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    raw = open(outp, "rb").read()
    loss = np.frombuffer(raw[:4], np.float32)[0]
    status = np.frombuffer(raw[4:12], np.int32)
    n = M * V
    grad = np.frombuffer(raw[12:12 + 4 * n], np.float32).reshape(M, V)
    soft = np.frombuffer(raw[12 + 4 * n:12 + 8 * n], np.float32).reshape(M, V)
    return float(loss), status, torch.from_numpy(grad.copy()), torch.from_numpy(soft.copy())


@pytest.mark.parametrize("M,V", [(64, 1000), (32, 8000), (6, 100003)])  # warp, resident, ring
def test_c_program_matches_the_oracle(exe, tmp_path, M, V):
    w = workloads.CE_WORKLOADS["ce_f32_64x1000"]
    x, t = workloads.make_ce_inputs(w.with_rows(M), "cpu") if V == w.V else (None, None)
    if x is None:
        g = torch.Generator().manual_seed(V)
        x = torch.randn((M, V), generator=g) * 2
        t = torch.randint(0, V, (M,), generator=g)
        t[1] = workloads.IGNORE_INDEX
    loss, status, grad, soft = run(exe, tmp_path, x, t)
    assert list(status) == [0, 0]
    ref = oracle_ce(x, t)
    check_grad(grad, ref["grad"], ref["n"], torch.float32, f"C program gradient {M}x{V}")
    check_loss(loss, oracle.ce_mean(ref["row_loss"], ref["n"]), torch.float32, "C program loss")
    check_softmax(soft, oracle.softmax_fwd(oracle.host_array(x)), torch.float32,
                  f"C program softmax {M}x{V}")
