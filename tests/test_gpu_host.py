"""ce_fwd_bwd_host: the fused cross-entropy from host buffers (chunked copies
overlapped with the row kernels) against the device call and the oracle (GPU)."""
import dataclasses
import math

import pytest
import torch

import cross_entropy_loss_ce_gb300 as gbce
import oracle
import workloads
from gpu_util import oracle_ce, require_gpu
from parity import check_grad, check_loss

pytestmark = pytest.mark.gpu


def device_reference(x_host, t_host, ignore_index=-100):
    xd = x_host.cuda()
    loss = gbce.ce_fwd_bwd(xd, t_host.cuda(), ignore_index)
    return xd, float(loss.item())


@pytest.mark.parametrize("name,rows", [("ce_f32_64x1000", 64), ("ce_bf16_8192x32000", 1001),
                                       ("ce_bf16_16384x128256", 37),
                                       ("ce_f32_4096x250007", 9)])
def test_host_call_equals_device_call(name, rows):
    """Same kernels per row and the same ordered mean: bit-identical results."""
    require_gpu()
    w = workloads.CE_WORKLOADS[name].with_rows(rows)
    x, t = workloads.make_ce_inputs(w, "cpu")
    ref_g, ref_l = device_reference(x, t)
    grad, loss = gbce.ce_fwd_bwd_host(x.pin_memory(), t.pin_memory())
    torch.cuda.synchronize()
    assert gbce.last_error() == gbce.OK
    assert torch.equal(grad, ref_g)
    assert float(loss.item()) == ref_l or (math.isnan(ref_l) and math.isnan(float(loss.item())))
    if rows <= 64:
        o = oracle_ce(x, t)
        check_grad(grad, o["grad"], o["n"], w.dtype, f"{name} host gradient")
        check_loss(float(loss.item()), oracle.ce_mean(o["row_loss"], o["n"]), w.dtype,
                   f"{name} host loss")


def test_host_call_full_size():
    require_gpu()
    w = workloads.CE_WORKLOADS["ce_bf16_16384x128256"]
    xd0, td = workloads.make_ce_inputs(w, "cuda")
    x_host, t_host = xd0.cpu().pin_memory(), td.cpu().pin_memory()
    ref = xd0.clone()
    ref_l = float(gbce.ce_fwd_bwd(ref, td).item())
    grad = torch.empty_like(xd0)
    _, loss = gbce.ce_fwd_bwd_host(x_host, t_host, grad=grad)
    torch.cuda.synchronize()
    assert gbce.last_error() == gbce.OK
    assert torch.equal(grad, ref) and float(loss.item()) == ref_l


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16], ids=str)
def test_host_call_strides_pageable_and_side_stream(dtype):
    """Padded host and device strides, pageable host memory, a non-default stream."""
    require_gpu()
    M, V = 13, 3001
    g = torch.Generator().manual_seed(5)
    xh = torch.full((M, V + 5), 9.0).to(dtype)
    xh[:, :V] = (torch.randn((M, V), generator=g) * 3).to(dtype)
    t = torch.randint(0, V, (M,), generator=g)
    t[4] = -100
    x = xh[:, :V]
    # the reference in the same device layout: a row's 16-byte phase decides
    # which elements take scalar accesses, hence the fp32 summation order
    rbuf = torch.full((M, V + 11), 5.0, dtype=dtype, device="cuda")
    ref_g = rbuf[:, :V]
    ref_g.copy_(x)
    ref_l = float(gbce.ce_fwd_bwd(ref_g, t.cuda()).item())
    gbuf = torch.full((M, V + 11), 5.0, dtype=dtype, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        grad, loss = gbce.ce_fwd_bwd_host(x, t, grad=gbuf[:, :V], stream=s)
    s.synchronize()
    assert gbce.last_error() == gbce.OK
    assert torch.equal(grad, ref_g) and float(loss.item()) == ref_l
    assert bool((gbuf[:, V:] == 5.0).all()), "written beyond the row"


def test_host_call_edge_cases():
    require_gpu()
    # M = 0: NaN mean, nothing else
    x = torch.empty((0, 10))
    _, loss = gbce.ce_fwd_bwd_host(x, torch.empty((0,), dtype=torch.int64))
    torch.cuda.synchronize()
    assert math.isnan(float(loss.item()))
    # M = 1, all ignored, and a bad target
    x = torch.randn((1, 10))
    grad, loss = gbce.ce_fwd_bwd_host(x, torch.tensor([-100]))
    torch.cuda.synchronize()
    assert math.isnan(float(loss.item())) and bool((grad == 0).all())
    x = torch.randn((3, 10))
    grad, loss = gbce.ce_fwd_bwd_host(x, torch.tensor([1, 10, 2]))
    assert gbce.last_error() == gbce.ERR_BAD_TARGET
    assert torch.equal(grad[1].cpu(), x[1]), "the bad row keeps its logits"
    assert math.isnan(float(loss.item()))


def test_host_call_in_a_cuda_graph():
    """Captured once (copy stream forked and joined by events), replayed with
    new host data in the same pinned buffers."""
    require_gpu()
    w = workloads.CE_WORKLOADS["ce_bf16_8192x32000"].with_rows(512)
    x, t = workloads.make_ce_inputs(w, "cpu")
    xp, tp = x.pin_memory(), t.pin_memory()
    grad = torch.empty(x.shape, dtype=x.dtype, device="cuda")
    loss_h = torch.empty((), dtype=torch.float32).pin_memory()
    gbce.ce_fwd_bwd_host(xp, tp, grad=grad, loss_host=loss_h)  # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            gbce.ce_fwd_bwd_host(xp, tp, grad=grad, loss_host=loss_h, stream=s)
    x2, t2 = workloads.make_ce_inputs(dataclasses.replace(w, seed=11), "cpu")
    xp.copy_(x2)
    tp.copy_(t2)
    graph.replay()
    torch.cuda.synchronize()
    ref_g, ref_l = device_reference(x2, t2)
    assert torch.equal(grad, ref_g) and float(loss_h.item()) == ref_l
