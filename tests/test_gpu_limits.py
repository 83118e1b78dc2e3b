"""The largest shapes the library accepts (GPU): M = 2^27 - 1 rows and
V = 2^31 - 1 columns.

Row and vector indices inside the kernels are 32-bit where the host limits
allow it; these calls put them at their largest values.  The gradient of a
row follows from its loss alone: with l = m + ln Z - x_y, p_i = exp(x_i - m) / Z
= exp(x_i - x_y - l), so sampled elements are checked against the oracle's
double-precision row loss where the oracle's full gradient would not fit in
host memory.
"""
import numpy as np
import pytest
import torch

import cross_entropy_loss_ce_gb300 as gbce
import oracle
import workloads
from gpu_util import require_gpu
from parity import check_grad, check_grad_factor, check_loss, check_softmax

pytestmark = pytest.mark.gpu
II = workloads.IGNORE_INDEX
MAX_ROWS = 2 ** 27 - 1
MAX_COLS = 2 ** 31 - 1


def test_ce_most_rows():
    """M = 2^27 - 1 rows of 3 fp32 logits (the warp kernel, 16.8 million CTAs);
    every 97th row ignored.  The loss over all rows against the oracle, and the
    gradient of sampled rows, the last ones included."""
    require_gpu()
    M, V = MAX_ROWS, 3
    g = torch.Generator(device="cuda").manual_seed(11)
    x = torch.randn((M, V), generator=g, device="cuda") * 2
    t = torch.randint(0, V, (M,), generator=g, device="cuda")
    t[::97] = II
    xh, th = x.cpu(), t.cpu().numpy()
    loss = gbce.ce_fwd_bwd(x, t, II)
    assert gbce.last_error() == gbce.OK
    xa = oracle.host_array(xh)
    n, bad = oracle.ce_count(th, V)
    assert bad == 0 and n == M - (M + 96) // 97
    _, row_loss = oracle.ce_rows(xa, th, V, n, want_grad=False)
    check_loss(float(loss.item()), oracle.ce_mean(row_loss, n), torch.float32, "loss over 2^27 - 1 rows")
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 1, 97, M // 2, M - 3, M - 2, M - 1],
                                     rng.choice(M, 200, replace=False)]))
    ref, _ = oracle.ce_rows(xa, th, V, n, rows=rows)
    got = x[torch.as_tensor(rows, device="cuda")]
    check_grad(got, ref, n, torch.float32, "sampled rows of 2^27 - 1")


def test_ce_most_columns():
    """One row of V = 2^31 - 1 bf16 logits: the ring split across a cluster of
    16 CTAs, each slice 2^24 16-byte vectors.  The loss against the oracle and
    sampled gradient elements (both ends of the row, the target, the slice
    boundaries) against exp(x_i - x_y - l) from the oracle's loss."""
    require_gpu()
    V = MAX_COLS
    name, C = gbce.plan("ce", 1, V, torch.bfloat16)
    assert name == "rows_ring_kernel" and C == 16
    g = torch.Generator(device="cuda").manual_seed(12)
    x = torch.randn((1, V), generator=g, device="cuda", dtype=torch.bfloat16)
    y = V - 5
    x[0, y] += 8  # keep p_y away from 0 so the target element is not all rounding
    t = torch.tensor([y], dtype=torch.int64, device="cuda")
    xh = x.cpu()
    loss = gbce.ce_fwd_bwd(x, t, II)
    assert gbce.last_error() == gbce.OK
    _, row_loss = oracle.ce_rows(oracle.host_array(xh), np.array([y]), V, 1, want_grad=False)
    ell = float(row_loss[0])
    check_loss(float(loss.item()), ell, torch.bfloat16, "loss of a 2^31 - 1 column row")
    per = -(-(V // 8) // C) * 8  # elements per CTA slice (the row starts on 16 bytes)
    rng = np.random.default_rng(6)
    cols = np.unique(np.concatenate([[0, 1, 7, 8, V - 9, V - 8, V - 2, V - 1, y, y - 1, y + 1],
                                     [k * per + d for k in range(1, C) for d in (-1, 0)],
                                     rng.choice(V, 4000, replace=False)]))
    xs = xh[0, torch.as_tensor(cols)].double().numpy()
    p = np.exp(xs - float(xh[0, y].double()) - ell)
    ref = p - (cols == y)
    got = x[0, torch.as_tensor(cols, device="cuda")].reshape(1, -1)
    check_grad_factor(got, ref.reshape(1, -1), np.ones(1), torch.bfloat16,
                      "sampled elements of a 2^31 - 1 column row")


def test_softmax_fwd_most_columns():
    """Softmax forward of one bf16 row of N = 2^31 - 1 (the ring split across a
    cluster of 16 CTAs): sampled outputs against exp(x_i - lse), where
    lse = l + x_t is taken from the oracle's cross-entropy loss l of the same
    row for some column t."""
    require_gpu()
    N = MAX_COLS
    name, C = gbce.plan("softmax_fwd", 1, N, torch.bfloat16)
    assert name == "rows_ring_kernel" and C == 16
    g = torch.Generator(device="cuda").manual_seed(13)
    x = torch.randn((1, N), generator=g, device="cuda", dtype=torch.bfloat16)
    yv = gbce.softmax_fwd(x)
    assert gbce.last_error() == gbce.OK
    xh = x.cpu()
    del x
    t = 12345
    _, row_loss = oracle.ce_rows(oracle.host_array(xh), np.array([t]), N, 1, want_grad=False)
    lse = float(row_loss[0]) + float(xh[0, t].double())
    per = -(-(N // 8) // C) * 8
    rng = np.random.default_rng(7)
    cols = np.unique(np.concatenate([[0, 1, 7, 8, N - 9, N - 8, N - 2, N - 1],
                                     [k * per + d for k in range(1, C) for d in (-1, 0)],
                                     rng.choice(N, 4000, replace=False)]))
    ref = np.exp(xh[0, torch.as_tensor(cols)].double().numpy() - lse)
    got = yv[0, torch.as_tensor(cols, device="cuda")].reshape(1, -1)
    check_softmax(got, ref.reshape(1, -1), torch.bfloat16, "softmax of a 2^31 - 1 column row")
