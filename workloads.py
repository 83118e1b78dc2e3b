"""Seeded synthetic inputs for the fused cross-entropy and the row softmax.

This module only draws random numbers and lays them out in memory.  It holds
none of the method's arithmetic (no max, exp, sum or softmax); both the CUDA
path and the double-precision oracle are fed the very tensors it returns, so
the stored values are the ground truth for a comparison.

Each generator takes a ``device``: on ``"cpu"`` it draws with torch's CPU
generator, on ``"cuda"`` with the CUDA generator (used for the multi-GB
workloads).  The two devices give different streams for the same seed; a test
always generates once and hands the same stored values to both sides.

Workloads (shapes, value distributions, ignore fractions and seeds):

  ce_f32_64x1000        fp32, M=64,    V=1000,   x ~ N(0,1),   10% rows ignored, seed 0
  softmax_f32_4096xN    fp32, M=4096,  N in {256,1024,4096,16384}, x, dy ~ N(0,1), seed 1
  ce_bf16_8192x32000    bf16, M=8192,  V=32000,  x ~ N(0,2^2), 5% rows ignored,  seed 2
  ce_bf16_16384x128256  bf16, M=16384, V=128256, x ~ N(0,4^2) plus +20 at one uniform
                        column per row, 2% rows ignored, seed 3
  ce_f32_4096x250007    fp32, M=4096,  V=250007, x ~ N(0,1) with 1% of entries -inf
                        (never at the target), 3% rows ignored, seed 4

"x% rows ignored" means exactly round(x% * M) rows, picked by a seeded
permutation, get target = ignore_index (-100); every other target is uniform
in [0, V).
"""
from dataclasses import dataclass, replace
from typing import Optional

import torch

IGNORE_INDEX = -100


@dataclass(frozen=True)
class CEWorkload:
    name: str
    M: int
    V: int
    dtype: torch.dtype
    std: float
    ignore_frac: float
    seed: int
    spike: float = 0.0        # added at one uniform column per row
    neginf_frac: float = 0.0  # fraction of entries set to -inf (never the target)

    def with_rows(self, M: int) -> "CEWorkload":
        return replace(self, M=M)


CE_WORKLOADS = {
    w.name: w for w in [
        CEWorkload("ce_f32_64x1000", 64, 1000, torch.float32, 1.0, 0.10, 0),
        CEWorkload("ce_bf16_8192x32000", 8192, 32000, torch.bfloat16, 2.0, 0.05, 2),
        CEWorkload("ce_bf16_16384x128256", 16384, 128256, torch.bfloat16, 4.0, 0.02, 3,
                   spike=20.0),
        CEWorkload("ce_f32_4096x250007", 4096, 250007, torch.float32, 1.0, 0.03, 4,
                   neginf_frac=0.01),
    ]
}

SOFTMAX_M = 4096
SOFTMAX_NS = (256, 1024, 4096, 16384)
SOFTMAX_SEED = 1


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _place(x: torch.Tensor, stride: Optional[int], fill: float) -> torch.Tensor:
    """Return x laid out with row stride ``stride`` (>= its width) as a [M, width] view."""
    M, V = x.shape
    if stride is None or stride == V:
        return x.contiguous()
    assert stride > V
    buf = torch.full((M, stride), fill, dtype=x.dtype, device=x.device)
    buf[:, :V] = x
    return buf[:, :V]


def make_ce_inputs(w: CEWorkload, device="cpu", stride: Optional[int] = None,
                   pad_fill: float = 7.0):
    """(logits [M, V] view with row stride ``stride``, targets int64 [M]).

    Draw order: logits ~ N(0, std^2) in fp32; the spike column per row; the
    targets; the -inf mask (cleared at each target); the ignored rows; then a
    round-to-nearest-even cast to the workload dtype.
    """
    g = _gen(device, w.seed)
    M, V = w.M, w.V
    x = torch.randn((M, V), generator=g, device=device, dtype=torch.float32)
    if w.std != 1.0:
        x.mul_(w.std)
    rows = torch.arange(M, device=device)
    if w.spike:
        cols = torch.randint(0, V, (M,), generator=g, device=device)
        x[rows, cols] += w.spike
    targets = torch.randint(0, V, (M,), generator=g, device=device, dtype=torch.int64)
    if w.neginf_frac:
        mask = torch.rand((M, V), generator=g, device=device) < w.neginf_frac
        mask[rows, targets] = False
        x.masked_fill_(mask, float("-inf"))
        del mask
    k = int(round(w.ignore_frac * M))
    if k:
        perm = torch.randperm(M, generator=g, device=device)
        targets[perm[:k]] = IGNORE_INDEX
    x = x.to(w.dtype)
    return _place(x, stride, pad_fill), targets


def make_softmax_inputs(M: int, N: int, dtype=torch.float32, seed: int = SOFTMAX_SEED,
                        device="cpu", x_stride: Optional[int] = None,
                        dy_stride: Optional[int] = None, pad_fill: float = 7.0):
    """(x, y, dy), each [M, N].

    x and dy ~ N(0, 1).  y is an independent point on the probability simplex
    (normalised Exp(1) draws, i.e. a flat Dirichlet sample per row), so the
    backward pass can be checked without feeding it any output of the code
    under test.
    """
    g = _gen(device, seed)
    x = torch.randn((M, N), generator=g, device=device, dtype=torch.float32)
    dy = torch.randn((M, N), generator=g, device=device, dtype=torch.float32)
    e = torch.empty((M, N), device=device, dtype=torch.float32).exponential_(generator=g)
    y = e / e.sum(dim=1, keepdim=True)
    return (_place(x.to(dtype), x_stride, pad_fill), _place(y.to(dtype), None, pad_fill),
            _place(dy.to(dtype), dy_stride, pad_fill))
