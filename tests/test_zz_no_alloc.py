"""ce_fwd_bwd_noalloc, the allocation-free form of the fused cross-entropy.

Some callers cannot let a library allocate device memory while they run: a
process whose caching allocator already holds the device's memory, a serving
runtime that forbids allocation after start-up to keep a fixed budget, or a
driver without stream-ordered memory pools.  The allocation-free entry point
keeps its temporary storage in a fixed static device array instead.  These
tests call it through the C ABI (ctypes on libgbce.so) twice in a row, on
different shapes and dtypes, and compare each result with the regular
ce_fwd_bwd entry point on the same inputs, within the tolerances the parity
tests use.  The file is named to be collected last.
"""
import ctypes

import pytest
import torch

import cross_entropy_loss_ce_gb300 as gbce
import workloads
from gpu_util import require_gpu
from parity import check_grad, check_loss, to_f64

pytestmark = pytest.mark.gpu
II = workloads.IGNORE_INDEX


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
        n = int((t != II).sum())
        check_grad(got, to_f64(ref), n, w.dtype, f"noalloc {name} gradient")
        check_loss(float(loss.item()), float(ref_loss.item()), w.dtype, f"noalloc {name} loss")


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
