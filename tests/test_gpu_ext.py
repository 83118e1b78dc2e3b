"""Reductions, the folded grad_output, per-row losses, fp16, scale_rows and the
autograd wrapper, against the double-precision oracle (GPU)."""
import math

import numpy as np
import pytest
import torch

import cross_entropy_loss_ce_gb300 as gbce
import oracle
import workloads
from gpu_util import require_gpu
from parity import (check_grad_factor, check_loss, check_softmax, check_softmax_bwd, to_f64,
                    ulp_distance_16)

pytestmark = pytest.mark.gpu
II = workloads.IGNORE_INDEX
DTYPES = [torch.float32, torch.bfloat16, torch.float16]


def _inputs(M, V, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn((M, V), generator=g) * 2).to(dtype)
    t = torch.randint(0, V, (M,), generator=g)
    t[::5] = II
    return x, t


def _k_rows(reduction, n, scale, M):
    if reduction == "none":
        return np.asarray(scale if scale is not None else np.ones(M), dtype=np.float64)
    s = 1.0 if scale is None else float(scale)
    return np.full(M, s / n if reduction == "mean" else s)


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
# 24 rows: warp, resident, the ring on one CTA (bf16) or a cluster of 4 (fp32), a cluster
@pytest.mark.parametrize("V", [1000, 8000, 20000, 131072])
@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("scaled", [False, True])
def test_ce_ex_matches_oracle(dtype, V, reduction, scaled):
    require_gpu()
    M = 24
    x, t = _inputs(M, V, dtype, V + 7)
    n, _ = oracle.ce_count(t.numpy(), V)
    rng = np.random.default_rng(V)
    scale = None
    if scaled:
        scale = rng.standard_normal(M).astype(np.float32) if reduction == "none" else 2.5
    ref_grad, ref_rl = oracle.ce_rows_ex(oracle.host_array(x), t.numpy(), V, n, II, reduction,
                                         None if scale is None else np.asarray(scale, np.float64))
    xd = x.cuda()
    gs = None
    if scale is not None:
        gs = torch.as_tensor(np.atleast_1d(scale), dtype=torch.float32, device="cuda")
    loss, rl = gbce.ce_fwd_bwd_ex(xd, t.cuda(), II, reduction, gs, want_row_loss=True)
    assert gbce.last_error() == gbce.OK
    check_grad_factor(xd, ref_grad, _k_rows(reduction, n, scale, M), dtype,
                      f"{reduction} V={V} {dtype}")
    if dtype != torch.float32:  # the folded scale keeps it to one rounding
        assert ulp_distance_16(xd, ref_grad, dtype).max() <= 1
    got_rl = to_f64(rl)
    rel = 1e-5 if dtype == torch.float32 else 1e-3
    assert np.allclose(got_rl, ref_rl, rtol=rel, atol=1e-6), "row losses"
    if reduction == "mean":
        check_loss(float(loss.item()), oracle.ce_mean(ref_rl, n), dtype)
    elif reduction == "sum":
        check_loss(float(loss.item()), oracle.ce_sum(ref_rl), dtype)
    else:
        assert loss is None


def test_ce_ex_empty_batches():
    require_gpu()
    x = torch.empty((0, 10), device="cuda")
    t = torch.empty((0,), dtype=torch.int64, device="cuda")
    loss, _ = gbce.ce_fwd_bwd_ex(x, t, reduction="sum")
    assert float(loss.item()) == 0.0
    loss, _ = gbce.ce_fwd_bwd_ex(x, t, reduction="mean")
    assert math.isnan(float(loss.item()))
    loss, rl = gbce.ce_fwd_bwd_ex(x, t, reduction="none")
    assert loss is None and rl.shape == (0,)
    # every row ignored: sum 0, gradient 0
    x = torch.randn((4, 300), device="cuda")
    t = torch.full((4,), II, dtype=torch.int64, device="cuda")
    loss, rl = gbce.ce_fwd_bwd_ex(x, t, reduction="sum", want_row_loss=True)
    assert float(loss.item()) == 0.0 and bool((x == 0).all()) and bool((rl == 0).all())


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("N", [7, 1000, 4099, 65537])
def test_scale_rows_matches_torch(dtype, N):
    require_gpu()
    g = torch.Generator().manual_seed(N)
    M = 6
    base = torch.randn((M, N + 3), generator=g).to(dtype).cuda()
    x = base[:, 1:N + 1]  # padded rows, misaligned start
    pad_l, pad_r = base[:, 0].clone(), base[:, N + 1:].clone()
    ref = (x.float() * 0.37).to(dtype)
    gbce.scale_rows(x, 0.37)
    assert torch.equal(x.view(torch.int16), ref.view(torch.int16))
    w = torch.randn(M, generator=g).cuda()
    ref = (x.float() * w[:, None]).to(dtype)
    gbce.scale_rows(x, w)
    assert torch.equal(x.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(base[:, 0], pad_l) and torch.equal(base[:, N + 1:], pad_r)  # padding kept
    before = base.clone()
    gbce.scale_rows(x, 1.0)  # a device-side no-op
    assert torch.equal(base.view(torch.int16), before.view(torch.int16))


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_autograd_wrapper(dtype, reduction):
    require_gpu()
    M, V = 16, 5000
    x, t = _inputs(M, V, dtype, 99)
    n, _ = oracle.ce_count(t.numpy(), V)
    rng = np.random.default_rng(3)
    go = rng.standard_normal(M) if reduction == "none" else np.array(1.7)
    ref_grad, ref_rl = oracle.ce_rows_ex(oracle.host_array(x), t.numpy(), V, n, II, reduction,
                                         np.atleast_1d(go).astype(np.float64))
    # a leaf, copied by the wrapper (inplace=False), so x keeps its values
    xd = x.cuda().requires_grad_(True)
    out = gbce.cross_entropy(xd, t.cuda(), reduction=reduction, inplace=False)
    out.backward(torch.as_tensor(go, dtype=torch.float32, device="cuda"))
    assert torch.equal(xd.detach().cpu().view(torch.int16), x.view(torch.int16))
    resc = np.broadcast_to(np.atleast_1d(go), (M,))
    check_grad_factor(xd.grad, ref_grad, _k_rows(reduction, n, go, M), dtype, "autograd grad",
                      rescaled_by=resc)
    # in place on a non-leaf: the gradient flows back through the product
    xl = x.cuda().requires_grad_(True)
    y = xl * 1.0
    out2 = gbce.CrossEntropyLoss(reduction=reduction)(y, t.cuda())
    out2.backward(torch.as_tensor(go, dtype=torch.float32, device="cuda"))
    check_grad_factor(xl.grad, ref_grad, _k_rows(reduction, n, go, M), dtype, "in-place grad",
                      rescaled_by=resc)
    if reduction == "none":
        assert np.allclose(to_f64(out), ref_rl, rtol=1e-3, atol=1e-6)
    else:
        refl = oracle.ce_mean(ref_rl, n) if reduction == "mean" else oracle.ce_sum(ref_rl)
        check_loss(float(out.item()), refl, dtype)


@pytest.mark.parametrize("N", [256, 1024, 16384])
def test_softmax_fp16(N):
    require_gpu()
    x, y, dy = workloads.make_softmax_inputs(32, N, torch.float16)
    ref_y = oracle.softmax_fwd(oracle.host_array(x))
    ref_dx = oracle.softmax_bwd(oracle.host_array(y), oracle.host_array(dy))
    check_softmax(gbce.softmax_fwd(x.cuda()), ref_y, torch.float16, f"fp16 softmax N={N}")
    check_softmax_bwd(gbce.softmax_bwd(y.cuda(), dy.cuda()), ref_dx, y, dy, torch.float16,
                      f"fp16 softmax bwd N={N}")


@pytest.mark.parametrize("reduction", ["mean", "none"])
def test_autograd_under_torch_compile(reduction):
    """The autograd form inside torch.compile: dynamo breaks the graph at the
    library call (a foreign function) and runs it eagerly, in place, so the
    loss and gradients match the eager run."""
    require_gpu()
    torch.manual_seed(3)
    M, H, V = 256, 256, 32000
    head = torch.nn.Linear(H, V, bias=False).cuda().to(torch.bfloat16)
    loss_fn = gbce.CrossEntropyLoss(reduction=reduction)
    h = torch.randn(M, H, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    t = torch.randint(0, V, (M,), device="cuda")
    t[::9] = II
    w_out = torch.randn(M, device="cuda") if reduction == "none" else None

    def step(h, t):
        loss = loss_fn(head(h), t)
        return (loss * w_out).sum() if reduction == "none" else loss

    results = []
    for f in (step, torch.compile(step)):
        head.weight.grad, h.grad = None, None
        loss = f(h, t)
        loss.backward()
        torch.cuda.synchronize()
        results.append((loss.detach().float(), h.grad.float(), head.weight.grad.float()))
    assert gbce.last_error() == gbce.OK
    (le, he, we), (lc, hc, wc) = results
    assert torch.allclose(lc, le, rtol=1e-3, atol=1e-5), (lc, le)
    for got, ref in ((hc, he), (wc, we)):
        assert torch.allclose(got, ref, rtol=2e-2, atol=2e-2 * ref.abs().max().item())
