"""The bounded waits of the staged row kernels, made to run out on purpose (GPU).

gbce_test_failure_path makes CTA 0 of each staged row-kernel launch leave out
one of its bulk copies.  Nothing will ever complete that copy's barrier phase,
so the waits for it end by their own limit (the production 2 s): a wait on a
signal that nothing sends, which the kernel turns into an error status.
Nothing here faults or hangs the GPU: every wait gives up after 2 s, and
before a CTA exits it waits (within a fixed budget) only for the copies it did
issue.  Each failing call takes a few seconds.

Each test checks that the call returns, that gbce_last_error reports
GBCE_ERR_TIMEOUT, that the reduced loss is NaN, that nothing outside the rows'
[0, V) columns was written, that every row the failing CTA finished (finite
row loss, or written softmax row) matches the oracle, that rows it had not
started are untouched, and that the same call with no copy left out is
correct.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import cross_entropy_loss_ce_gb300 as gbce
import oracle
import workloads
from gpu_util import host, oracle_ce, require_gpu
from parity import check_grad, check_loss, check_softmax, check_softmax_bwd

pytestmark = pytest.mark.gpu
II = workloads.IGNORE_INDEX
CANARY = 64
FILL = 123.0


def _set(drop: int):
    fn = gbce.load_library().gbce_test_failure_path
    fn.argtypes = [ctypes.c_int64]
    fn.restype = ctypes.c_int
    torch.cuda.synchronize()
    assert fn(drop) == gbce.OK


@pytest.fixture
def failure_path():
    """Yields the setter; restores the default (no copy left out) after the test."""
    require_gpu()
    assert gbce.last_error() == gbce.OK
    yield _set
    _set(-1)
    gbce.last_error()


def guarded(x: torch.Tensor):
    """(buffer, [M, V] view): x on the GPU with rows padded to a 16-byte multiple
    and CANARY guard elements before the first and after the last row."""
    M, V = x.shape
    per16 = 16 // x.element_size()
    stride = (V + 1 + per16 - 1) // per16 * per16
    buf = torch.full((CANARY + M * stride + CANARY,), FILL, dtype=x.dtype, device="cuda")
    view = buf[CANARY: CANARY + (M - 1) * stride + V].as_strided((M, V), (stride, 1))
    view.copy_(x.cuda())
    return buf, view


def outside_untouched(buf: torch.Tensor, view: torch.Tensor) -> bool:
    M, V = view.shape
    stride = view.stride(0)
    out = buf.cpu().float()
    keep = torch.ones_like(out, dtype=torch.bool)
    for r in range(M):
        keep[CANARY + r * stride: CANARY + r * stride + V] = False
    return bool(torch.all(out[keep] == FILL))


# (workload, rows, copy left out, that copy is in the first read of its row)
CE_CASES = [
    # ring, 256 KB rows read twice in 8 copies each: a copy of the first read,
    # then one of the second read (its row is then partly written)
    ("ce_bf16_16384x128256", 600, 3, True),
    ("ce_bf16_16384x128256", 600, 10, False),
    # resident kernel: a 64 KB row staged in 8 copies (more rows than SMs:
    # smaller batches of such rows take the ring)
    ("ce_bf16_8192x32000", 200, 2, True),
    # ring split across a cluster of 4 CTAs (the rank-0 CTA of cluster 0 fails;
    # its peers see the failure in the exchange and write nothing either)
    ("ce_f32_4096x250007", 40, 1, True),
    # a small batch: 4 rows in one wave, each split across a cluster of 8 or
    # more CTAs; CTA 0 holds the first slice of row 0 in a single copy
    ("ce_bf16_16384x128256", 4, 0, True),
]


@pytest.mark.parametrize("name,rows,drop,first_read", CE_CASES,
                         ids=[f"{c[0]}-copy{c[2]}" for c in CE_CASES])
def test_ce_wait_that_runs_out(failure_path, name, rows, drop, first_read):
    w = workloads.CE_WORKLOADS[name].with_rows(rows)
    x, t = workloads.make_ce_inputs(w, "cpu")
    if t[0] == II:  # CTA 0 starts on row 0: make it a live row, so it issues copies
        t[0] = 0
    ref = oracle_ce(x, t)
    buf, view = guarded(x)
    td = t.cuda()
    failure_path(drop)
    loss, row_loss = gbce.ce_fwd_bwd_ex(view, td, II, "mean", want_row_loss=True)
    assert gbce.last_error() == gbce.ERR_TIMEOUT
    assert math.isnan(float(loss.item()))
    assert outside_untouched(buf, view), "wrote outside [0, V) of a row"
    rl = row_loss.cpu().numpy().astype(np.float64)
    failed = np.isnan(rl)
    assert failed.any() and not failed.all()
    done = np.flatnonzero(~failed)
    got = view.cpu()
    check_grad(got[done], ref["grad"][done], ref["n"], w.dtype, f"{name}: finished rows")
    assert np.allclose(rl[done], ref["row_loss"][done], rtol=1e-5 if w.dtype == torch.float32
                       else 1e-3, atol=2.0 ** -22)
    changed = [r for r in np.flatnonzero(failed) if not torch.equal(got[r], x[r])]
    # a row that failed in its first read was never written; a failure in the
    # second read leaves only that one row partly written
    assert len(changed) == (0 if first_read else 1), changed

    failure_path(-1)
    view.copy_(x.cuda())
    loss = gbce.ce_fwd_bwd(view, td, II)
    assert gbce.last_error() == gbce.OK
    check_grad(view, ref["grad"], ref["n"], w.dtype, f"{name}: after the defaults came back")
    check_loss(float(loss.item()), oracle.ce_mean(ref["row_loss"], ref["n"]), w.dtype)
    assert outside_untouched(buf, view)


# (N, rows, copy left out): ring with held 64 KB rows, resident 16 KB rows,
# and a small batch of 500 KB rows, each split across a cluster
SOFTMAX_FWD_CASES = [(16384, 400, 0), (16384, 400, 5), (4096, 64, 1), (128256, 3, 0)]


@pytest.mark.parametrize("N,rows,drop", SOFTMAX_FWD_CASES)
def test_softmax_fwd_wait_that_runs_out(failure_path, N, rows, drop):
    x, _, _ = workloads.make_softmax_inputs(rows, N)
    ref = oracle.softmax_fwd(host(x))
    xd = x.cuda()
    ybuf, y = guarded(torch.full_like(x, FILL))
    failure_path(drop)
    gbce.softmax_fwd(xd, y)
    assert gbce.last_error() == gbce.ERR_TIMEOUT
    assert outside_untouched(ybuf, y)
    got = y.cpu()
    unwritten = (got == FILL).all(dim=1).numpy()
    assert unwritten.any() and not unwritten.all()
    done = np.flatnonzero(~unwritten)
    check_softmax(got[done], ref[done], torch.float32, f"N={N}: finished rows")

    failure_path(-1)
    gbce.softmax_fwd(xd, y)
    assert gbce.last_error() == gbce.OK
    check_softmax(y, ref, torch.float32, f"N={N}: after the defaults came back")


# (N, rows, copy left out): ring streaming two 64 KB operands, resident 2 x 16 KB
SOFTMAX_BWD_CASES = [(16384, 400, 2), (4096, 64, 0)]


@pytest.mark.parametrize("N,rows,drop", SOFTMAX_BWD_CASES)
def test_softmax_bwd_wait_that_runs_out(failure_path, N, rows, drop):
    _, yv, dy = workloads.make_softmax_inputs(rows, N)
    ref = oracle.softmax_bwd(host(yv), host(dy))
    yd, dyd = yv.cuda(), dy.cuda()
    dxbuf, dx = guarded(torch.full_like(dy, FILL))
    failure_path(drop)
    gbce.softmax_bwd(yd, dyd, dx)
    assert gbce.last_error() == gbce.ERR_TIMEOUT
    assert outside_untouched(dxbuf, dx)
    got = dx.cpu()
    unwritten = (got == FILL).all(dim=1).numpy()
    assert unwritten.any() and not unwritten.all()
    done = np.flatnonzero(~unwritten)
    check_softmax_bwd(got[done], ref[done], yv[done], dy[done], torch.float32,
                      f"N={N}: finished rows")

    failure_path(-1)
    gbce.softmax_bwd(yd, dyd, dx)
    assert gbce.last_error() == gbce.OK
    check_softmax_bwd(dx, ref, yv, dy, torch.float32, f"N={N}: after the defaults came back")


def test_defaults_after_the_failure_tests():
    """After the failure tests, a 2048-row launch of the benchmark's workload
    runs with every copy issued and is right."""
    require_gpu()
    w = workloads.CE_WORKLOADS["ce_bf16_16384x128256"].with_rows(2048)
    xd, td = workloads.make_ce_inputs(w, "cuda")
    x_host, t_host = xd.cpu(), td.cpu()
    rows = np.array([0, 1, 151, 152, 1000, 2047])
    ref = oracle_ce(x_host, t_host, rows=rows)
    loss = gbce.ce_fwd_bwd(xd, td, II)
    assert gbce.last_error() == gbce.OK
    assert math.isfinite(float(loss.item()))
    check_grad(xd[torch.as_tensor(rows, device="cuda")], ref["grad"], ref["n"], w.dtype)


def test_status_words_tell_concurrent_calls_apart(failure_path):
    """softmax_fwd_ex / softmax_bwd_ex: with a copy left out, the staged calls
    (a ring forward, a resident backward) set bit 0 of their own status words
    while a warp-kernel call (no bulk copies) on another stream, running at the
    same time, leaves its word at 0; the device flag reports the timeout for
    the device.  With every copy issued again, a staged call's word stays 0."""
    xa, _, _ = workloads.make_softmax_inputs(400, 16384)      # ring, held 64 KB rows
    _, yb, dyb = workloads.make_softmax_inputs(64, 4096)      # resident backward
    xc, _, _ = workloads.make_softmax_inputs(64, 1000)        # warp kernel
    words = torch.zeros(4, dtype=torch.int32, device="cuda")
    sa, sb, sc = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    xad, ybd, dybd, xcd = xa.cuda(), yb.cuda(), dyb.cuda(), xc.cuda()
    torch.cuda.synchronize()
    failure_path(0)
    gbce.softmax_fwd_ex(xad, status=words[0:1], stream=sa)
    gbce.softmax_bwd_ex(ybd, dybd, status=words[1:2], stream=sb)
    yc = gbce.softmax_fwd_ex(xcd, status=words[2:3], stream=sc)
    torch.cuda.synchronize()
    assert words.tolist() == [1, 1, 0, 0]
    assert gbce.last_error() == gbce.ERR_TIMEOUT
    check_softmax(yc, oracle.softmax_fwd(host(xc)), torch.float32, "the unaffected call")

    failure_path(-1)
    words.zero_()
    ya = gbce.softmax_fwd_ex(xad, status=words[0:1])
    dx = gbce.softmax_bwd_ex(ybd, dybd, status=words[1:2])
    torch.cuda.synchronize()
    assert words.tolist() == [0, 0, 0, 0]
    assert gbce.last_error() == gbce.OK
    check_softmax(ya, oracle.softmax_fwd(host(xa)), torch.float32, "after the defaults came back")
    check_softmax_bwd(dx, oracle.softmax_bwd(host(yb), host(dyb)), yb, dyb, torch.float32,
                      "backward after the defaults came back")
