"""ce_fwd_bwd_noalloc, the allocation-free form of the fused cross-entropy.

Some callers cannot let a library allocate device memory while they run: a
process whose caching allocator already holds the device's memory, a serving
runtime that forbids allocation after start-up to keep a fixed budget, or a
driver without stream-ordered memory pools.  The allocation-free entry point
keeps its temporary storage in a fixed static device array instead.

These tests call it through the C ABI (ctypes on libgbce.so) twice in a row,
on different shapes and dtypes, and require results bit-identical to the
regular ce_fwd_bwd entry point on the same inputs (both run the same kernels
with the same launch plan and a fixed-order mean), and check one shape
against the oracle directly.  A fresh process calls it through the Python
wrapper before anything else and checks that the library's scratch pool was
never created.  The file is named to be collected last.
"""
import ctypes
import math
import os
import subprocess
import sys

import pytest
import torch

import cross_entropy_loss_ce_gb300 as gbce
import oracle
import workloads
from gpu_util import oracle_ce, require_gpu
from parity import check_grad, check_loss

pytestmark = pytest.mark.gpu
II = workloads.IGNORE_INDEX
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def noalloc_fn():
    fn = gbce.load_library().ce_fwd_bwd_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def call_noalloc(fn, x, t, loss):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(x.data_ptr(), x.stride(0), t.data_ptr(), loss.data_ptr(), x.shape[0], x.shape[1],
              II, gbce.DTYPES[x.dtype], stream)


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32)


def test_noalloc_matches_ce_fwd_bwd_on_two_calls_in_a_row():
    require_gpu()
    fn = noalloc_fn()
    # first a larger bf16 batch, then a smaller fp32 one: the second call runs
    # on the static storage the first one left behind
    for name, M in (("ce_bf16_16384x128256", 96), ("ce_f32_64x1000", 64)):
        w = workloads.CE_WORKLOADS[name].with_rows(M)
        x, t = workloads.make_ce_inputs(w, "cuda")
        ref = x.clone()
        ref_loss = gbce.ce_fwd_bwd(ref, t, II)
        got = x.clone()
        loss = torch.empty((), dtype=torch.float32, device="cuda")
        assert call_noalloc(fn, got, t, loss) == gbce.OK
        assert gbce.last_error() == gbce.OK
        assert torch.equal(bits(got), bits(ref)), f"{name}: gradient bits differ"
        assert torch.equal(bits(loss.reshape(1)), bits(ref_loss.reshape(1))), \
            f"{name}: loss bits differ"


def test_noalloc_matches_the_oracle():
    require_gpu()
    fn = noalloc_fn()
    w = workloads.CE_WORKLOADS["ce_bf16_8192x32000"].with_rows(96)
    x, t = workloads.make_ce_inputs(w, "cpu")
    ref = oracle_ce(x, t)
    xd, td = x.cuda(), t.cuda()
    loss = torch.empty((), dtype=torch.float32, device="cuda")
    assert call_noalloc(fn, xd, td, loss) == gbce.OK
    assert gbce.last_error() == gbce.OK
    check_grad(xd, ref["grad"], ref["n"], w.dtype, "noalloc gradient")
    check_loss(float(loss.item()), oracle.ce_mean(ref["row_loss"], ref["n"]), w.dtype)


def test_noalloc_all_ignored_batch_after_a_normal_one():
    """A batch whose targets are all ignore_index, right after a normal batch
    left its count and row losses in the static storage: n = 0, a NaN loss
    and all-zero gradient rows, not the previous call's numbers."""
    require_gpu()
    fn = noalloc_fn()
    for V in (1000, 32000, 128256):  # warp, resident and ring row kernels
        w = workloads.CE_WORKLOADS["ce_bf16_16384x128256"].with_rows(64)
        x, t = workloads.make_ce_inputs(w, "cuda")
        x = x[:, :V].contiguous()
        t = t % V
        loss = torch.empty((), dtype=torch.float32, device="cuda")
        assert call_noalloc(fn, x, t, loss) == gbce.OK
        assert math.isfinite(float(loss.item()))
        x2 = torch.randn((64, V), device="cuda").to(torch.bfloat16)
        t2 = torch.full((64,), II, dtype=torch.int64, device="cuda")
        assert call_noalloc(fn, x2, t2, loss) == gbce.OK
        assert gbce.last_error() == gbce.OK
        assert math.isnan(float(loss.item())), f"V={V}: all-ignored batch gave {loss.item()}"
        assert bool((x2 == 0).all())


def test_noalloc_rejects_more_rows_than_its_storage():
    require_gpu()
    fn = noalloc_fn()
    M, V = 65537, 8
    x = torch.zeros((M, V), dtype=torch.float32, device="cuda")
    t = torch.zeros((M,), dtype=torch.int64, device="cuda")
    loss = torch.full((), 3.0, dtype=torch.float32, device="cuda")
    assert call_noalloc(fn, x, t, loss) == gbce.ERR_SIZE
    torch.cuda.synchronize()
    assert float(loss.item()) == 3.0 and bool((x == 0).all())  # nothing was launched


FRESH_PROCESS = r"""
import ctypes, sys
import torch
sys.path.insert(0, sys.argv[1])
import cross_entropy_loss_ce_gb300 as gbce
import workloads

def pool_bytes():
    fn = gbce.load_library().gbce_pool_reserved
    fn.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_uint64)]
    fn.restype = ctypes.c_int
    v = ctypes.c_uint64(12345)
    assert fn(torch.cuda.current_device(), ctypes.byref(v)) == gbce.OK
    return v.value

w = workloads.CE_WORKLOADS["ce_bf16_16384x128256"].with_rows(64)
x, t = workloads.make_ce_inputs(w, "cuda")
loss = torch.empty((), dtype=torch.float32, device="cuda")
ref = x.clone()
assert pool_bytes() == 0
for _ in range(2):
    gbce.ce_fwd_bwd_noalloc(x, t, -100, loss)
torch.cuda.synchronize()
assert gbce.last_error() == gbce.OK
assert pool_bytes() == 0, "the allocation-free call created the scratch pool"
gbce.ce_fwd_bwd(ref, t, -100)
torch.cuda.synchronize()
assert pool_bytes() > 0, "the pool query does not see the regular call's pool"
print("no pool")
"""


def test_noalloc_creates_no_pool_in_a_fresh_process():
    """Through the Python wrapper, first in a new process: after two calls the
    library's stream-ordered scratch pool does not exist; the regular call then
    creates it (so the query would have seen it)."""
    require_gpu()
    r = subprocess.run([sys.executable, "-c", FRESH_PROCESS, ROOT], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "no pool" in r.stdout, r.stdout + r.stderr
