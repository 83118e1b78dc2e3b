"""Small batches (GPU): at most one row per SM, rows that stage more than 32 KB.

Such a batch takes the ring, each row of 64 KB or more split across the
largest cluster of which all M rows fit on the device at once (16 KB slices at
least), so the cluster sizes here run from 1 to 16, with slices shorter than
one ring slot and, for odd row lengths, heads and tails.  Every output element is
checked against the oracle; the plans themselves are checked against the rule.
"""
import pytest
import torch

import cross_entropy_loss_ce_gb300 as gbce
import oracle
import workloads
from gpu_util import host, oracle_ce, require_gpu
from parity import check_grad, check_loss, check_softmax, check_softmax_bwd

pytestmark = pytest.mark.gpu
II = workloads.IGNORE_INDEX
ESIZE = {torch.float32: 4, torch.bfloat16: 2, torch.float16: 2}


def sm_count() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


def check_plan(op, M, cols, dtype):
    """The small-batch rule: the ring; rows under 64 KB per operand on one CTA,
    longer ones on at most 16 CTAs with slices of at least 16 KB."""
    name, C = gbce.plan(op, M, cols, dtype)
    row = cols * ESIZE[dtype]
    assert name == "rows_ring_kernel", (op, M, cols, name)
    assert 1 <= C <= (1 if row < 65536 else min(16, row // 16384)), (op, M, cols, C)
    return C


def ce_inputs(M, V, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn((M, V), generator=g) * 3).to(dtype)
    t = torch.randint(0, V, (M,), generator=g)
    if M >= 3:
        t[1] = II
        t[2] = V - 1  # the last column: the tail of the last CTA's slice
    if M >= 4:
        t[3] = (V // 2) & ~7  # near a slice boundary for an even split
    return x, t


CE_CASES = [
    (128256, torch.bfloat16, [1, 2, 7, 8, 9, 16, 24, 33, 64, 100, 152]),
    (250007, torch.float32, [1, 3, 8, 16, 36, 37]),   # odd rows: heads and tails
    (32000, torch.bfloat16, [1, 2, 5, 64, 152]),       # 64 KB: resident for large batches
    (20001, torch.bfloat16, [1, 6]),                   # 40 KB, odd: the ring on one CTA
    (130001, torch.float16, [1, 4]),
]


@pytest.mark.parametrize("V,dtype,M", [(V, d, M) for V, d, ms in CE_CASES for M in ms],
                         ids=lambda v: str(v))
def test_ce_small_batch_every_element(V, dtype, M):
    require_gpu()
    if M > sm_count():
        pytest.skip("more rows than SMs: the large-batch plan")
    C = check_plan("ce", M, V, dtype)
    x, t = ce_inputs(M, V, dtype, seed=V + M)
    ref = oracle_ce(x, t)
    xd, td = x.cuda(), t.cuda()
    loss = gbce.ce_fwd_bwd(xd, td, II)
    assert gbce.last_error() == gbce.OK
    what = f"CE {M}x{V} {dtype}, {C} CTAs per row"
    check_grad(xd, ref["grad"], ref["n"], dtype, what)
    check_loss(float(loss.item()), oracle.ce_mean(ref["row_loss"], ref["n"]), dtype, what)


def test_small_batch_plans_follow_the_rule():
    """One row of a large vocabulary takes a large cluster; the cluster shrinks
    as the batch grows; one row per SM takes one CTA per row; one more row
    goes back to the large-batch plan (the resident kernel for 64 KB rows)."""
    require_gpu()
    S = sm_count()
    c = [gbce.plan("ce", M, 128256, torch.bfloat16)[1] for M in (1, 8, 16, 32, 64, S)]
    assert c[0] >= 8 and c[-1] == 1, c
    assert all(a >= b for a, b in zip(c, c[1:])), c
    assert gbce.plan("ce", S, 32000, torch.bfloat16) == ("rows_ring_kernel", 1)
    assert gbce.plan("ce", 1, 32000, torch.bfloat16) == ("rows_ring_kernel", 1)  # 64000 B
    assert gbce.plan("ce", S + 1, 32000, torch.bfloat16)[0] == "rows_resident_kernel"
    assert gbce.plan("ce", 1, 16384, torch.bfloat16)[0] == "rows_resident_kernel"  # 32 KB
    assert gbce.plan("ce", 1, 2048, torch.float32)[0] == "rows_warp_kernel"
    # the fp32 large-vocabulary rows keep at least the cluster the L2 bound asks for
    assert gbce.plan("ce", 64, 250007, torch.float32)[1] >= \
        gbce.plan("ce", 4096, 250007, torch.float32)[1]


SOFTMAX_CASES = [
    (128256, torch.float32, [1, 3, 16, 40]),
    (32000, torch.float32, [1, 8, 152]),
    (100003, torch.bfloat16, [1, 5]),
    (6000, torch.float32, [1, 20]),   # backward stages 48 KB: the ring with one CTA
]


@pytest.mark.parametrize("N,dtype,M", [(N, d, M) for N, d, ms in SOFTMAX_CASES for M in ms],
                         ids=lambda v: str(v))
def test_softmax_small_batch_every_element(N, dtype, M):
    require_gpu()
    if M > sm_count():
        pytest.skip("more rows than SMs: the large-batch plan")
    g = torch.Generator().manual_seed(N + M)
    x = (torch.randn((M, N), generator=g) * 3).to(dtype)
    e = torch.rand((M, N), generator=g) + 0.01
    y = (e / e.sum(1, keepdim=True)).to(dtype)
    dy = torch.randn((M, N), generator=g).to(dtype)
    if N * ESIZE[dtype] > 32 * 1024:  # the forward stages one operand
        check_plan("softmax_fwd", M, N, dtype)
    check_plan("softmax_bwd", M, N, dtype)
    yo = gbce.softmax_fwd(x.cuda())
    dx = gbce.softmax_bwd(y.cuda(), dy.cuda())
    assert gbce.last_error() == gbce.OK
    check_softmax(yo, oracle.softmax_fwd(host(x)), dtype, f"softmax {M}x{N} {dtype}")
    check_softmax_bwd(dx, oracle.softmax_bwd(host(y), host(dy)), y, dy, dtype,
                      f"softmax backward {M}x{N} {dtype}")


@pytest.mark.parametrize("M", [1, 5, 40])
def test_ce_host_small_batch(M):
    """The host-buffer call launches its rows in up to eight pieces, each with
    the plan of the device call for all M rows (one row per piece for M <= 8)."""
    require_gpu()
    V = 128256
    x, t = ce_inputs(M, V, torch.bfloat16, seed=M)
    ref = oracle_ce(x, t)
    grad, loss = gbce.ce_fwd_bwd_host(x.pin_memory(), t.pin_memory(), II)
    torch.cuda.synchronize()
    assert gbce.last_error() == gbce.OK
    xd = x.cuda()
    loss_d = gbce.ce_fwd_bwd(xd, t.cuda(), II)
    assert torch.equal(grad, xd) and float(loss.item()) == float(loss_d.item())  # same kernel
    check_grad(grad, ref["grad"], ref["n"], torch.bfloat16, f"host CE {M}x{V}")
    check_loss(float(loss.item()), oracle.ce_mean(ref["row_loss"], ref["n"]), torch.bfloat16,
               f"host CE loss {M}x{V}")


def test_small_batch_in_a_cuda_graph():
    """A captured small-batch call replays with new inputs."""
    require_gpu()
    M, V = 4, 128256
    x1, t1 = ce_inputs(M, V, torch.bfloat16, seed=101)
    x2, t2 = ce_inputs(M, V, torch.bfloat16, seed=102)
    xd, td = x1.cuda(), t1.cuda()
    loss = torch.empty((), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gbce.ce_fwd_bwd(xd, td, II, loss)  # plans and configures outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    xd.copy_(x1.cuda())
    with torch.cuda.graph(graph):
        gbce.ce_fwd_bwd(xd, td, II, loss)
    for x, t in ((x1, t1), (x2, t2)):
        xd.copy_(x.cuda())
        td.copy_(t.cuda())
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle_ce(x, t)
        check_grad(xd, ref["grad"], ref["n"], torch.bfloat16, "graph replay")
        check_loss(float(loss.item()), oracle.ce_mean(ref["row_loss"], ref["n"]),
                   torch.bfloat16, "graph replay loss")
    assert gbce.last_error() == gbce.OK


def guarded_copy(x: torch.Tensor, off: int, pad: int, fill: float = 123.0):
    """(device buffer, [M, V] device view of it holding x): rows at a padded
    stride, the first one `off` elements past a 16-byte boundary, canaries
    around them."""
    M, V = x.shape
    stride, canary = V + pad, 64
    buf = torch.full((canary + M * stride + canary,), fill, dtype=x.dtype)
    view = buf[canary + off: canary + off + (M - 1) * stride + V].as_strided((M, V), (stride, 1))
    view.copy_(x)
    bd = buf.cuda()
    vd = bd[canary + off: canary + off + (M - 1) * stride + V].as_strided((M, V), (stride, 1))
    return bd, vd, canary + off, stride


def untouched_outside(bd, start, stride, M, V, fill=123.0):
    out = bd.cpu().float()
    mask = torch.ones_like(out, dtype=torch.bool)
    for r in range(M):
        mask[start + r * stride: start + r * stride + V] = False
    return bool(torch.all(out[mask] == fill))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=str)
@pytest.mark.parametrize("V", [20001, 40000, 65537, 100003])
def test_ce_one_row_more_than_sms(dtype, V):
    """One row more than the device has SMs: the large-batch plans (the
    resident kernel, the ring on one CTA per row, for 100003 fp32 a cluster of
    two), on rows whose start is off the 16-byte grid (heads and tails) at a
    padded stride; every element against the oracle, nothing written outside
    the rows."""
    require_gpu()
    M = sm_count() + 1
    g = torch.Generator().manual_seed(V)
    x = (torch.randn((M, V), generator=g) * 3).to(dtype)
    t = torch.randint(0, V, (M,), generator=g)
    t[1] = II
    t[2] = V - 1
    ref = oracle_ce(x, t)
    bd, vd, start, stride = guarded_copy(x, off=3, pad=13)
    loss = gbce.ce_fwd_bwd(vd, t.cuda(), II)
    assert gbce.last_error() == gbce.OK
    what = f"CE {M}x{V} {dtype}, {gbce.plan('ce', M, V, dtype, same_phase=True)}"
    check_grad(vd, ref["grad"], ref["n"], dtype, what)
    check_loss(float(loss.item()), oracle.ce_mean(ref["row_loss"], ref["n"]), dtype, what)
    assert untouched_outside(bd, start, stride, M, V), "wrote outside [0, V) of a row"


@pytest.mark.parametrize("N", [6001, 12001, 16387, 100003])
def test_softmax_one_row_more_than_sms(N):
    """The softmax forward and backward (fp32) on one row more than SMs, rows
    off the 16-byte grid: the large-batch plans of both directions."""
    require_gpu()
    M = sm_count() + 1
    g = torch.Generator().manual_seed(N)
    x = torch.randn((M, N), generator=g) * 3
    e = torch.rand((M, N), generator=g) + 0.01
    y = e / e.sum(1, keepdim=True)
    dy = torch.randn((M, N), generator=g)
    _, xd, _, _ = guarded_copy(x, off=1, pad=3)
    yb, yd, ystart, ystride = guarded_copy(torch.zeros_like(x), off=1, pad=3, fill=0.0)
    _, ysd, _, _ = guarded_copy(y, off=2, pad=6)
    _, dyd, _, _ = guarded_copy(dy, off=2, pad=6)
    _, dx, _, _ = guarded_copy(torch.zeros_like(x), off=2, pad=6, fill=0.0)  # y's phase
    gbce.softmax_fwd(xd, yd)
    gbce.softmax_bwd(ysd, dyd, dx)
    assert gbce.last_error() == gbce.OK
    check_softmax(yd, oracle.softmax_fwd(host(x)), torch.float32, f"softmax {M}x{N}")
    check_softmax_bwd(dx, oracle.softmax_bwd(host(y), host(dy)), y, dy, torch.float32,
                      f"softmax backward {M}x{N}")
    assert untouched_outside(yb, ystart, ystride, M, N, fill=0.0)
