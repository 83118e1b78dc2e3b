"""Seeded random shapes against the oracle (GPU).

A fixed generator draws each case: the call (fused CE, softmax forward or
backward), the dtype, the row count M (1 to 400, so both the small-batch and
the large-batch plans occur), the row length (1 to 400000 columns, log-uniform,
so every kernel family and cluster size from 1 to 16 occurs), a padded row
stride, a base offset off the 16-byte grid, ignored rows and targets at the
row ends, and for the softmax out-of-place outputs at the input's phase or at
another one (the streaming fallback).  Every output element is compared with
the oracle at the stated tolerances, and nothing outside the rows may change.
"""
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
DTYPES = [torch.float32, torch.bfloat16, torch.float16]
ELEMS = {torch.float32: 4, torch.bfloat16: 2, torch.float16: 2}
MAX_ELEMENTS = 6_000_000  # per case: keeps the oracle to a fraction of a second
CANARY = 64
FILL = 77.0


def draw_cases(n=72, seed=20261203):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        op = ("ce", "softmax_fwd", "softmax_bwd")[i % 3]
        dtype = DTYPES[int(rng.integers(3))]
        cols = int(np.exp(rng.uniform(0.0, np.log(400000.0))))
        M = int(np.exp(rng.uniform(0.0, np.log(400.0))))
        M = max(1, min(M, MAX_ELEMENTS // max(cols, 1)))
        pad = int(rng.integers(0, 40)) if rng.random() < 0.5 else 0
        off = int(rng.integers(0, 8)) if rng.random() < 0.6 else 0
        other_phase = op != "ce" and rng.random() < 0.2
        cases.append(dict(op=op, dtype=dtype, M=M, cols=cols, pad=pad, off=off,
                          other_phase=other_phase, seed=int(rng.integers(1 << 30))))
    return cases


CASES = draw_cases()


def case_id(c):
    return (f"{c['op']}-{str(c['dtype']).split('.')[-1]}-{c['M']}x{c['cols']}"
            f"-pad{c['pad']}-off{c['off']}" + ("-phase" if c["other_phase"] else ""))


def guarded(x: torch.Tensor, off: int, pad: int, fill: float = FILL):
    """(device buffer, [M, cols] device view holding x, first row start, stride):
    rows at stride cols + pad, the first `off` elements past the buffer's
    16-byte-aligned start plus a canary, canaries after the last row."""
    M, cols = x.shape
    stride = cols + pad
    start = CANARY + off
    buf = torch.full((start + (M - 1) * stride + cols + CANARY,), fill, dtype=x.dtype)
    buf[start: start + (M - 1) * stride + cols].as_strided((M, cols), (stride, 1)).copy_(x)
    bd = buf.cuda()
    view = bd[start: start + (M - 1) * stride + cols].as_strided((M, cols), (stride, 1))
    return bd, view, start, stride


def outside_untouched(bd, start, stride, M, cols, fill=FILL):
    out = bd.cpu().float()
    mask = torch.ones_like(out, dtype=torch.bool)
    for r in range(M):
        mask[start + r * stride: start + r * stride + cols] = False
    return bool(torch.all(out[mask] == fill))


@pytest.mark.parametrize("c", CASES, ids=[case_id(c) for c in CASES])
def test_random_shape(c):
    require_gpu()
    op, dtype, M, cols, pad, off = c["op"], c["dtype"], c["M"], c["cols"], c["pad"], c["off"]
    g = torch.Generator().manual_seed(c["seed"])
    plan = gbce.plan(op, M, cols, dtype, same_phase=not c["other_phase"])
    what = f"{case_id(c)}, plan {plan}"
    if op == "ce":
        scale = float((1.0, 3.0, 10.0)[c["seed"] % 3])
        x = (torch.randn((M, cols), generator=g) * scale).to(dtype)
        t = torch.randint(0, cols, (M,), generator=g)
        t[torch.rand((M,), generator=g) < 0.1] = II
        t[0] = cols - 1                  # the last column: the tail of the last slice
        if M > 1:
            t[M - 1] = 0                 # the first column: the head of the first slice
        ref = oracle_ce(x, t)
        bd, view, start, stride = guarded(x, off, pad)
        loss = gbce.ce_fwd_bwd(view, t.cuda(), II)
        assert gbce.last_error() == gbce.OK, what
        check_grad(view, ref["grad"], ref["n"], dtype, what, targets=t.numpy())
        check_loss(float(loss.item()), oracle.ce_mean(ref["row_loss"], ref["n"]), dtype, what)
        assert outside_untouched(bd, start, stride, M, cols), what
        return
    # an output at the input's 16-byte phase, or one element further on (another phase)
    off_out = (off + 1) % 8 if c["other_phase"] else off
    if op == "softmax_fwd":
        x = (torch.randn((M, cols), generator=g) * 4).to(dtype)
        ref = oracle.softmax_fwd(host(x))
        _, xd, _, _ = guarded(x, off, pad)
        yb, yd, ystart, ystride = guarded(torch.zeros_like(x), off_out, pad)
        gbce.softmax_fwd(xd, yd)
        assert gbce.last_error() == gbce.OK, what
        check_softmax(yd, ref, dtype, what)
        assert outside_untouched(yb, ystart, ystride, M, cols), what
        gbce.softmax_fwd(xd, xd)  # in place
        assert gbce.last_error() == gbce.OK, what
        check_softmax(xd, ref, dtype, what + " in place")
        return
    e = torch.rand((M, cols), generator=g) + 0.01
    y = (e / e.sum(1, keepdim=True)).to(dtype)
    dy = torch.randn((M, cols), generator=g).to(dtype)
    ref = oracle.softmax_bwd(host(y), host(dy))
    _, ydev, _, _ = guarded(y, off, pad)
    _, dydev, _, _ = guarded(dy, off, pad)
    xb, dx, xstart, xstride = guarded(torch.zeros_like(y), off_out, pad)
    gbce.softmax_bwd(ydev, dydev, dx)
    assert gbce.last_error() == gbce.OK, what
    check_softmax_bwd(dx, ref, y, dy, dtype, what)
    assert outside_untouched(xb, xstart, xstride, M, cols), what
    gbce.softmax_bwd(ydev, dydev, dydev)  # in place over dy
    assert gbce.last_error() == gbce.OK, what
    check_softmax_bwd(dydev, ref, y, dy, dtype, what + " in place")


def test_random_cases_reach_every_plan():
    """The drawn cases cover every kernel family, small and large batches, and
    clusters (checked on the host plan of each case)."""
    require_gpu()
    names, clustered, small, large = set(), 0, 0, 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for c in CASES:
        name, C = gbce.plan(c["op"], c["M"], c["cols"], c["dtype"], same_phase=not c["other_phase"])
        names.add(name)
        clustered += C > 1
        small += c["M"] <= sms
        large += c["M"] > sms
    assert names == {"rows_warp_kernel", "rows_resident_kernel", "rows_ring_kernel",
                     "rows_streaming_kernel"}, names
    assert clustered >= 5 and small >= 10 and large >= 5, (clustered, small, large)
