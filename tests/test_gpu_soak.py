"""Soak (GPU): many calls of every entry point, on two streams at once.

A seeded sequence of calls (the fused CE and its reductions, both softmax
directions, the block-sparse backward), over shapes that reach every kernel
family and plan (small batches on clusters, the ring, resident and warp
kernels), runs twice: each call is made on two streams at the same time with
the same inputs and separate outputs.  Every pair must be bit-identical and
equal to the same call made afterwards on one stream (the kernels are
deterministic, so any race in scratch, ordering or the cluster exchange
shows up as a difference), and no error flag may be raised.  Parity with the
oracle is checked elsewhere.
"""
import numpy as np
import pytest
import torch

import cross_entropy_loss_ce_gb300 as gbce
import workloads
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu
II = workloads.IGNORE_INDEX
DTYPES = [torch.float32, torch.bfloat16, torch.float16]


def draw_calls(n=60, seed=7):
    rng = np.random.default_rng(seed)
    calls = []
    for i in range(n):
        op = ("ce", "ce_sum", "ce_none", "fwd", "bwd", "bsr")[i % 6]
        dtype = DTYPES[int(rng.integers(3))]
        cols = int(np.exp(rng.uniform(np.log(3.0), np.log(300000.0))))
        M = int(np.exp(rng.uniform(0.0, np.log(300.0))))
        M = max(1, min(M, 3_000_000 // cols))
        calls.append((op, dtype, M, cols, int(rng.integers(1 << 30))))
    return calls


def make_inputs(op, dtype, M, cols, seed):
    g = torch.Generator().manual_seed(seed)
    if op == "bsr":
        w = workloads.BSR_WORKLOADS["bsr_f32_causal_2x16x4096_b32"].with_sizes(Z=2, H=2, S=512)
        y, dy, lut, meta = workloads.make_bsr_inputs(w, device="cuda")
        return (y, dy, lut, meta)
    x = (torch.randn((M, cols), generator=g) * 3).to(dtype).cuda()
    t = torch.randint(0, cols, (M,), generator=g)
    t[torch.rand((M,), generator=g) < 0.1] = II
    e = torch.rand((M, cols), generator=g) + 0.01
    y = (e / e.sum(1, keepdim=True)).to(dtype).cuda()
    dy = torch.randn((M, cols), generator=g).to(dtype).cuda()
    return (x, t.cuda(), y, dy)


def run(op, inputs):
    """The call's outputs (new tensors; inputs are not modified)."""
    if op == "bsr":
        y, dy, lut, meta = inputs
        return (gbce.softmax_bwd_bsr(y, dy, lut, meta["n_block_rows"], meta["nblocks"],
                                     meta["block"], meta["sizemax"], 0.5, dx=torch.empty_like(dy)),)
    x, t, y, dy = inputs
    if op == "fwd":
        return (gbce.softmax_fwd(x),)
    if op == "bwd":
        return (gbce.softmax_bwd(y, dy),)
    g = x.clone()
    if op == "ce":
        return g, gbce.ce_fwd_bwd(g, t, II)
    loss, rl = gbce.ce_fwd_bwd_ex(g, t, II, "sum" if op == "ce_sum" else "none",
                                  want_row_loss=True)
    return (g, rl) if loss is None else (g, loss, rl)


def bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def same(a, b):
    return len(a) == len(b) and all(torch.equal(bits(u), bits(v)) for u, v in zip(a, b))


def test_soak_two_streams_deterministic():
    require_gpu()
    calls = draw_calls()
    data = [make_inputs(op, dt, M, cols, seed) for op, dt, M, cols, seed in calls]
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    assert gbce.last_error() == gbce.OK
    for _ in range(2):
        outs = []
        for (op, *_), inputs in zip(calls, data):
            sa.wait_stream(torch.cuda.current_stream())
            sb.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(sa):
                oa = run(op, inputs)
            with torch.cuda.stream(sb):
                ob = run(op, inputs)
            outs.append((oa, ob))
        torch.cuda.synchronize()
        assert gbce.last_error() == gbce.OK
        for (op, dt, M, cols, _), inputs, (oa, ob) in zip(calls, data, outs):
            ref = run(op, inputs)
            torch.cuda.synchronize()
            what = f"{op} {dt} {M}x{cols}"
            assert same(oa, ob), f"{what}: the two streams differ"
            assert same(oa, ref), f"{what}: differs from the serial call"
    assert gbce.last_error() == gbce.OK
