"""CUDA fused cross-entropy against the double-precision oracle (GPU)."""
import math

import numpy as np
import pytest
import torch

import cross_entropy_loss_ce_gb300 as gbce
import oracle
import workloads
from gpu_util import host, oracle_ce, require_gpu
from parity import check_grad, check_loss, to_f64, ulp_distance_16

pytestmark = pytest.mark.gpu
II = workloads.IGNORE_INDEX

# Reduced row counts that the oracle finishes in well under a second, full V.
REDUCED = {"ce_f32_64x1000": 64, "ce_bf16_8192x32000": 96, "ce_bf16_16384x128256": 48,
           "ce_f32_4096x250007": 32}


def run_ce(x_dev, t_dev):
    loss = gbce.ce_fwd_bwd(x_dev, t_dev, II)
    status = gbce.last_error()
    return float(loss.item()), status


@pytest.mark.parametrize("name", list(workloads.CE_WORKLOADS))
def test_ce_reduced_rows_all_elements(name):
    """Every gradient element and the loss, at full V, on a reduced row count."""
    require_gpu()
    w = workloads.CE_WORKLOADS[name].with_rows(REDUCED[name])
    x, t = workloads.make_ce_inputs(w, "cpu")
    ref = oracle_ce(x, t)
    ref_loss = oracle.ce_mean(ref["row_loss"], ref["n"])
    xd, td = x.cuda(), t.cuda()
    loss, status = run_ce(xd, td)
    assert status == gbce.OK
    check_grad(xd, ref["grad"], ref["n"], w.dtype, f"{name} gradient")
    check_loss(loss, ref_loss, w.dtype, f"{name} loss")
    if w.dtype != torch.float32:
        # fp32 arithmetic then one rounding: at most one bf16 step from the
        # correctly rounded value (off by one only next to a rounding midpoint)
        ulps = ulp_distance_16(xd, ref["grad"], w.dtype)
        assert ulps.max() <= 1, f"{name}: {int((ulps > 1).sum())} elements > 1 ulp"


@pytest.mark.parametrize("name", [n for n in workloads.CE_WORKLOADS if n != "ce_f32_64x1000"])
def test_ce_full_size_sampled_rows(name):
    """The full workload in the benchmark's launch configuration: the loss over
    all rows from the oracle, the gradient on sampled rows (ignored rows among them)."""
    require_gpu()
    w = workloads.CE_WORKLOADS[name]
    xd, td = workloads.make_ce_inputs(w, "cuda")
    x_host = xd.cpu()
    t_host = td.cpu()
    rng = np.random.default_rng(123)
    ignored = np.flatnonzero(t_host.numpy() == II)
    rows = np.unique(np.concatenate([[0, w.M - 1], rng.choice(w.M, 24, replace=False),
                                     ignored[:4]]))
    ref = oracle_ce(x_host, t_host, want_grad=False)
    ref_loss = oracle.ce_mean(ref["row_loss"], ref["n"])
    ref_rows = oracle_ce(x_host, t_host, rows=rows)
    loss, status = run_ce(xd, td)
    assert status == gbce.OK
    check_loss(loss, ref_loss, w.dtype, f"{name} loss")
    got = xd[torch.as_tensor(rows, device="cuda")]
    check_grad(got, ref_rows["grad"], ref["n"], w.dtype, f"{name} sampled gradient rows")
    del xd


def test_ce_deterministic():
    require_gpu()
    w = workloads.CE_WORKLOADS["ce_bf16_8192x32000"].with_rows(512)
    x, t = workloads.make_ce_inputs(w, "cuda")
    a, b = x.clone(), x.clone()
    la = gbce.ce_fwd_bwd(a, t, II)
    lb = gbce.ce_fwd_bwd(b, t, II)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert la.item() == lb.item() or (math.isnan(la.item()) and math.isnan(lb.item()))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16], ids=str)
@pytest.mark.parametrize("V", [1, 2, 3, 7, 8, 9, 33, 1000, 4099, 20000, 40000, 65537, 262147, 1000003])
def test_ce_shapes_padded_and_misaligned(dtype, V):
    """Ragged V (cluster sizes 1..16 and the streaming fallback), a padded row
    stride whose padding must stay untouched, and a base pointer off the
    16-byte grid, with canaries before and after the logits."""
    require_gpu()
    M = 6 if V < 500000 else 3
    g = torch.Generator().manual_seed(V)
    x = (torch.randn((M, V), generator=g) * 3).to(dtype)
    t = torch.randint(0, V, (M,), generator=g)
    t[1] = II
    ref = oracle_ce(x, t)
    ref_loss = oracle.ce_mean(ref["row_loss"], ref["n"])
    for off, pad in ((0, 0), (1, 5), (3, 13)):
        stride = V + pad
        canary = 64
        buf = torch.full((canary + M * stride + canary,), 123.0, dtype=dtype)
        view = buf[canary + off: canary + off + (M - 1) * stride + V].as_strided((M, V), (stride, 1))
        view.copy_(x)
        bd = buf.cuda()
        vd = bd[canary + off: canary + off + (M - 1) * stride + V].as_strided((M, V), (stride, 1))
        loss, status = run_ce(vd, t.cuda())
        assert status == gbce.OK
        check_grad(vd, ref["grad"], ref["n"], dtype, f"V={V} off={off} pad={pad}")
        check_loss(loss, ref_loss, dtype)
        # nothing outside the V columns of each row changed
        out = bd.cpu().float()
        mask = torch.ones_like(out, dtype=torch.bool)
        for r in range(M):
            s = canary + off + r * stride
            mask[s: s + V] = False
        assert torch.all(out[mask] == 123.0), "wrote outside [0, V) of a row"


def test_ce_empty_and_all_ignored():
    require_gpu()
    x = torch.empty((0, 10), device="cuda")
    t = torch.empty((0,), dtype=torch.int64, device="cuda")
    loss, status = run_ce(x, t)
    assert math.isnan(loss) and status == gbce.OK
    # every row ignored: n = 0, NaN loss, every gradient row zero, no reads needed
    x = torch.randn((3, 1000), device="cuda")
    t = torch.full((3,), II, dtype=torch.int64, device="cuda")
    loss, status = run_ce(x, t)
    assert math.isnan(loss) and status == gbce.OK
    assert torch.all(x == 0)


def test_ce_all_ignored_rows_of_the_large_vocabulary_workload():
    """Two rows of the V=250007 fp32 workload with every target ignored."""
    require_gpu()
    w = workloads.CE_WORKLOADS["ce_f32_4096x250007"].with_rows(2)
    x, _ = workloads.make_ce_inputs(w, "cpu")
    t = torch.full((2,), II, dtype=torch.int64)
    ref = oracle_ce(x, t)
    xd = x.cuda()
    loss, status = run_ce(xd, t.cuda())
    assert math.isnan(loss) and math.isnan(oracle.ce_mean(ref["row_loss"], ref["n"]))
    assert status == gbce.OK
    assert np.array_equal(to_f64(xd), ref["grad"])


def test_ce_bad_target_is_flagged():
    require_gpu()
    x = torch.randn((4, 300), device="cuda")
    x0 = x.clone()
    t = torch.tensor([5, 300, II, -7], dtype=torch.int64, device="cuda")
    loss, status = run_ce(x, t)
    assert status == gbce.ERR_BAD_TARGET
    assert math.isnan(loss)
    assert torch.equal(x[1], x0[1]) and torch.equal(x[3], x0[3])  # bad rows untouched
    assert torch.all(x[2] == 0)
    assert gbce.last_error() == gbce.OK  # the flag was cleared


def test_ce_single_row_and_spike():
    require_gpu()
    V = 128256
    x = torch.randn((1, V)) * 4
    x[0, 17] += 20
    for tgt in (17, 5):
        t = torch.tensor([tgt])
        xb = x.to(torch.bfloat16)
        ref = oracle_ce(xb, t)
        xd = xb.cuda()
        loss, status = run_ce(xd, t.cuda())
        assert status == gbce.OK
        check_grad(xd, ref["grad"], 1, torch.bfloat16)
        check_loss(loss, float(ref["row_loss"][0]), torch.bfloat16)


def test_every_regime_is_exercised():
    """The shapes above reach every row-kernel family on this device,
    including the ring split across a cluster."""
    require_gpu()
    M = 4096  # a batch that fills the device
    assert gbce.plan("ce", M, 1000, torch.float32)[0] == "rows_warp_kernel"
    assert gbce.plan("ce", M, 4099, torch.float32)[0] == "rows_resident_kernel"
    assert gbce.plan("ce", M, 65537, torch.bfloat16) == ("rows_ring_kernel", 1)
    name, c = gbce.plan("ce", M, 262147, torch.float32)
    assert name == "rows_ring_kernel" and c >= 2
    name, c = gbce.plan("ce", M, 1000003, torch.float32)
    assert name == "rows_ring_kernel" and c >= 8
    name, c = gbce.plan("ce", M, 250007, torch.float32)  # the large-vocabulary fp32 workload
    assert name == "rows_ring_kernel" and c >= 2
    assert gbce.plan("softmax_fwd", M, 1000, torch.float32, same_phase=False)[0] == \
        "rows_streaming_kernel"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=str)
def test_ignore_index_is_a_class_id(dtype):
    """ignore_index may be any int64: here class 0 itself, and 5."""
    require_gpu()
    for ii in (0, 5):
        g = torch.Generator().manual_seed(ii)
        x = torch.randn((40, 777), generator=g).to(dtype)
        t = torch.randint(0, 8, (40,), generator=g)
        ref = oracle_ce(x, t, ignore_index=ii)
        assert ref["n"] < 40
        xd = x.cuda()
        loss = gbce.ce_fwd_bwd(xd, t.cuda(), ii)
        assert gbce.last_error() == gbce.OK
        check_grad(xd, ref["grad"], ref["n"], dtype, f"ignore_index={ii}")
        check_loss(float(loss.item()), oracle.ce_mean(ref["row_loss"], ref["n"]), dtype)
        assert bool((xd[t.cuda() == ii] == 0).all())


def test_other_negative_ignore_index():
    """With ignore_index = -1, a -100 target is out of range: flagged, its row kept."""
    require_gpu()
    x = torch.randn((6, 300))
    t = torch.tensor([3, -1, -100, 299, -1, 0])
    ref = oracle_ce(x, t, ignore_index=-1)
    assert ref["bad"] == 1 and ref["n"] == 4
    xd = x.cuda()
    loss = gbce.ce_fwd_bwd(xd, t.cuda(), -1)
    assert gbce.last_error() == gbce.ERR_BAD_TARGET
    assert math.isnan(float(loss.item()))
    assert torch.equal(xd[2].cpu(), x[2])
    keep = [0, 1, 3, 4, 5]
    check_grad(xd[keep], ref["grad"][keep], ref["n"], torch.float32, "ignore_index=-1")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16], ids=str)
# 6 rows: warp, resident, the ring on one CTA (unaligned fp32 rows of 48 KB), the ring on a
# cluster (unaligned rows; a small batch), the ring on a cluster
@pytest.mark.parametrize("V", [1000, 8000, 12001, 100003, 262147])
@pytest.mark.parametrize("offset", [50.0, -150.0, 150.0, 1e4, -1e4, 1e6, -1e6])
def test_ce_large_logits(dtype, V, offset):
    """Logits far from zero, row maxima up to 2e6 in magnitude (2e4 for fp16,
    whose range ends at 65504), in every kernel regime, within the same
    tolerances as logits near zero: exp(x - m) is formed from the difference
    x - m, whose rounding follows |x - m| and not |m|, and the row loss from
    m - x_y.  Rows with different offsets, one of them ignored."""
    require_gpu()
    if dtype == torch.float16 and abs(offset) > 1e4:
        pytest.skip("beyond the fp16 range")
    M = 6
    g = torch.Generator().manual_seed(V)
    x = torch.randn((M, V), generator=g) * 4
    x += torch.tensor([offset, -offset, 0.5 * offset, offset, 2 * offset, -0.25 * offset])[:, None]
    t = torch.randint(0, V, (M,), generator=g)
    t[3] = II
    xh = x.to(dtype)
    ref = oracle_ce(xh, t)
    xd = xh.cuda()
    loss, status = run_ce(xd, t.cuda())
    assert status == gbce.OK
    check_grad(xd, ref["grad"], ref["n"], dtype, f"V={V} offset={offset}")
    check_loss(loss, oracle.ce_mean(ref["row_loss"], ref["n"]), dtype, f"V={V} offset={offset}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16], ids=str)
@pytest.mark.parametrize("V", [1000, 8000, 32000, 128256, 250007])
@pytest.mark.parametrize("M", [6, 200])
def test_ce_masked_logits(dtype, V, M):
    """-inf logits (never at the target) take no probability in every regime:
    rows with a short finite prefix, a -inf first half, a random -inf half,
    one finite entry (p_y = 1: loss 0, gradient 0 up to one rounding), and
    only the last entry finite; the gradient is exactly 0 at every -inf."""
    require_gpu()
    if M * V > 30_000_000:
        pytest.skip("large batch of long rows: covered by the 6-row case")
    g = torch.Generator().manual_seed(V + M)
    x = torch.randn((M, V), generator=g) * 3
    t = torch.empty((M,), dtype=torch.int64)
    ninf = float("-inf")
    for r in range(M):
        kind = r % 6
        if kind == 0:
            x[r, min(5, V):] = ninf
            t[r] = int(torch.randint(0, min(5, V), (1,), generator=g))
        elif kind == 1:
            x[r, : V // 2] = ninf
            t[r] = V // 2 + int(torch.randint(0, V - V // 2, (1,), generator=g))
        elif kind == 2:
            x[r, torch.rand(V, generator=g) < 0.5] = ninf
            t[r] = int(torch.randint(0, V, (1,), generator=g))
            x[r, t[r]] = 0.5
        elif kind == 3:
            t[r] = int(torch.randint(0, V, (1,), generator=g))
            v = float(x[r, t[r]])
            x[r] = ninf
            x[r, t[r]] = v
        elif kind == 4:
            t[r] = II if r == 4 else int(torch.randint(0, V, (1,), generator=g))
        else:
            x[r, : V - 1] = ninf
            t[r] = V - 1
    x = x.to(dtype)
    ref = oracle_ce(x, t)
    xd = x.cuda()
    loss, status = run_ce(xd, t.cuda())
    assert status == gbce.OK
    what = f"masked CE {M}x{V} {dtype}, plan {gbce.plan('ce', M, V, dtype)}"
    check_grad(xd, ref["grad"], ref["n"], dtype, what, targets=t.numpy())
    check_loss(loss, oracle.ce_mean(ref["row_loss"], ref["n"]), dtype, what)
    assert bool(torch.all(xd.cpu()[torch.isinf(x)] == 0)), "a -inf logit got a gradient"
