"""The library called from a plain C program (GPU): tests/c_abi/ce_from_c.c,
compiled with gcc against include/gbce.h, libgbce.so and the CUDA runtime (no
Python or torch in the process), runs softmax_fwd, softmax_bwd_ex (in place,
with a status word of its own),
ce_fwd_bwd, ce_fwd_bwd_ex (reduction none, per-row scale, row losses) and
gbce_plan on inputs from a file; its outputs are compared with the oracle on
the same inputs."""
import os
import subprocess

import numpy as np
import pytest
import torch

import cross_entropy_loss_ce_gb300 as gbce
import oracle
import workloads
from cross_entropy_loss_ce_gb300 import build as gbuild
from gpu_util import oracle_ce, require_gpu
from parity import check_grad, check_grad_factor, check_loss, check_softmax, check_softmax_bwd

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


def run(exe, tmp_path, x: torch.Tensor, t: torch.Tensor, dy: torch.Tensor, scale: np.ndarray):
    M, V = x.shape
    inp, outp = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        f.write(np.array([M, V], dtype=np.int64).tobytes())
        f.write(x.numpy().astype(np.float32).tobytes())
        f.write(t.numpy().astype(np.int64).tobytes())
        f.write(dy.numpy().astype(np.float32).tobytes())
        f.write(scale.astype(np.float32).tobytes())
    r = subprocess.run([exe, str(inp), str(outp)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    raw = open(outp, "rb").read()
    n = M * V
    out = dict(loss=float(np.frombuffer(raw[:4], np.float32)[0]),
               status=list(np.frombuffer(raw[4:16], np.int32)))
    off = 16
    for key in ("grad", "soft", "dx", "grad_none"):
        out[key] = torch.from_numpy(np.frombuffer(raw[off:off + 4 * n], np.float32).reshape(M, V).copy())
        off += 4 * n
    out["row_loss"] = np.frombuffer(raw[off:off + 4 * M], np.float32).astype(np.float64)
    off += 4 * M
    out["ctas"] = int(np.frombuffer(raw[off:off + 4], np.int32)[0])
    out["plan"] = raw[off + 4:off + 36].split(b"\0")[0].decode()
    assert off + 36 == len(raw)
    return out


@pytest.mark.parametrize("M,V", [(64, 1000), (32, 8000), (6, 100003), (200, 20001)])
def test_c_program_matches_the_oracle(exe, tmp_path, M, V):
    """Warp, resident, the ring split across a cluster (a small batch) and the
    ring on one CTA (200 rows): the mean CE, the CE with reduction none and a
    per-row gradient scale, the softmax forward and its backward in place."""
    w = workloads.CE_WORKLOADS["ce_f32_64x1000"]
    x, t = workloads.make_ce_inputs(w.with_rows(M), "cpu") if V == w.V else (None, None)
    g = torch.Generator().manual_seed(V + M)
    if x is None:
        x = torch.randn((M, V), generator=g) * 2
        t = torch.randint(0, V, (M,), generator=g)
        t[1] = workloads.IGNORE_INDEX
    dy = torch.randn((M, V), generator=g)
    scale = np.random.default_rng(M).standard_normal(M).astype(np.float32)
    out = run(exe, tmp_path, x, t, dy, scale)
    assert out["status"] == [0, 0, 0]  # calls, device flags, the call's status word
    assert (out["plan"], out["ctas"]) == gbce.plan("ce", M, V, torch.float32)
    ref = oracle_ce(x, t)
    what = f"C program {M}x{V}"
    check_grad(out["grad"], ref["grad"], ref["n"], torch.float32, what + " gradient",
               targets=t.numpy())
    check_loss(out["loss"], oracle.ce_mean(ref["row_loss"], ref["n"]), torch.float32, what + " loss")
    y_ref = oracle.softmax_fwd(oracle.host_array(x))
    check_softmax(out["soft"], y_ref, torch.float32, what + " softmax")
    dx_ref = oracle.softmax_bwd(oracle.host_array(out["soft"]), oracle.host_array(dy))
    check_softmax_bwd(out["dx"], dx_ref, out["soft"], dy, torch.float32, what + " softmax backward")
    g_none, rl_none = oracle.ce_rows_ex(oracle.host_array(x), t.numpy(), V, ref["n"],
                                        workloads.IGNORE_INDEX, "none", scale.astype(np.float64))
    check_grad_factor(out["grad_none"], g_none, scale.astype(np.float64), torch.float32,
                      what + " reduction none", targets=t.numpy())
    assert np.allclose(out["row_loss"], rl_none, rtol=1e-5, atol=1e-6), what + " row losses"
