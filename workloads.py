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

Block-sparse softmax backward workloads (the attention-style layouts the
block-sparse kernel's look-up table describes: Z batch items, H heads, an
S x S matrix per head cut into block x block tiles):

  bsr_f32_causal_2x16x4096_b32   fp32, Z=2, H=16, S=4096, block 32, causal layout
                                 (block-row i holds blocks 0..i), seed 5
  bsr_bf16_random_4x8x8192_b64   bf16, Z=4, H=8, S=8192, block 64, the diagonal
                                 block plus each other block with probability 0.1,
                                 entries of a block-row in random order, seed 6

y is Exp(1) divided by the number of stored elements of its row (so rows sum
to about 1, like a softmax output) and dy ~ N(0, 1).
"""
from dataclasses import dataclass, replace
from typing import Optional

import numpy as np

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


# ---------------------------------------------------------------------------
# block-sparse layouts and their look-up table

@dataclass(frozen=True)
class BsrWorkload:
    name: str
    Z: int            # batch items
    H: int            # heads
    S: int            # rows (and columns) of each head's matrix
    block: int
    dtype: torch.dtype
    layout: str       # "causal" or "random"
    density: float    # "random": probability of each off-diagonal block
    seed: int
    shuffle: bool = False   # entries of each block-row in a seeded random order
    diagonal: bool = True   # "random": always keep the diagonal block

    def with_sizes(self, **kw) -> "BsrWorkload":
        return replace(self, **kw)


BSR_WORKLOADS = {
    w.name: w for w in [
        BsrWorkload("bsr_f32_causal_2x16x4096_b32", 2, 16, 4096, 32, torch.float32, "causal",
                    0.0, 5),
        BsrWorkload("bsr_bf16_random_4x8x8192_b64", 4, 8, 8192, 64, torch.bfloat16, "random",
                    0.1, 6, shuffle=True),
    ]
}


def make_bsr_layout(w: BsrWorkload) -> np.ndarray:
    """Boolean [H, S/block, S/block]: which blocks are stored."""
    nb = w.S // w.block
    assert nb * w.block == w.S
    if w.layout == "causal":
        one = np.tril(np.ones((nb, nb), dtype=bool))
        return np.broadcast_to(one, (w.H, nb, nb)).copy()
    assert w.layout == "random"
    rng = np.random.Generator(np.random.PCG64(w.seed))
    lay = rng.random((w.H, nb, nb)) < w.density
    if w.diagonal:
        lay[:, np.arange(nb), np.arange(nb)] = True
    return lay


def make_bsr_lut(layout: np.ndarray, shuffle_seed: Optional[int] = None):
    """(lut int32, n_block_rows, nblocks, sizemax, block_row_of_block int64).

    Blocks are numbered in (head, block-row, block-column) order.  The table
    starts with one (size, offset) pair per block-row (head-major); each
    stored block then has a 4-int entry (block id, head, block-row,
    block-column) at offset + 4 * k.  With a seed, the entries of each
    block-row are put in a random order.
    """
    H, nb, _ = layout.shape
    nbr = H * nb
    h, r, c = np.nonzero(layout)                 # (h, r, c) in row-major order
    nblocks = h.size
    sizes = layout.reshape(nbr, nb).sum(axis=1).astype(np.int64)
    starts = np.zeros(nbr, dtype=np.int64)
    np.cumsum(sizes[:-1], out=starts[1:])
    entries = np.stack([np.arange(nblocks), h, r, c], axis=1).astype(np.int64)
    if shuffle_seed is not None and nblocks:
        rng = np.random.Generator(np.random.PCG64(shuffle_seed))
        row_of = h * nb + r
        order = np.lexsort((rng.random(nblocks), row_of))
        entries = entries[order]
    lut = np.empty(2 * nbr + 4 * nblocks, dtype=np.int64)
    lut[0:2 * nbr:2] = sizes
    lut[1:2 * nbr:2] = 2 * nbr + 4 * starts
    lut[2 * nbr:] = entries.reshape(-1)
    sizemax = int(sizes.max()) if nbr else 0
    return lut.astype(np.int32), nbr, nblocks, sizemax, (h * nb + r).astype(np.int64)


def make_bsr_inputs(w: BsrWorkload, device="cpu", zpad: int = 0):
    """(y, dy, lut, meta): y and dy are [Z, nblocks * block^2 + zpad] tensors of
    w.dtype (block b of item z at b * block^2), lut an int32 tensor, meta a dict
    with n_block_rows, nblocks, block, sizemax.  Draw order: the layout and the
    entry order on the CPU (numpy PCG64), then y ~ Exp(1) and dy ~ N(0, 1) with
    torch's generator on ``device``; y is divided by its row's element count."""
    lay = make_bsr_layout(w)
    lut, nbr, nblocks, sizemax, brow = make_bsr_lut(lay, w.seed + 1 if w.shuffle else None)
    bb = w.block * w.block
    g = _gen(device, w.seed)
    L = nblocks * bb
    y = torch.empty((w.Z, L), device=device, dtype=torch.float32).exponential_(generator=g)
    dy = torch.randn((w.Z, L), generator=g, device=device, dtype=torch.float32)
    sizes = torch.from_numpy(lut[0:2 * nbr:2].astype(np.int64)).to(device)
    count = (sizes[torch.from_numpy(brow).to(device)] * w.block).to(torch.float32)
    y = (y.view(w.Z, nblocks, bb) / count.view(1, nblocks, 1)).view(w.Z, L)
    if zpad:
        y = torch.cat([y, torch.full((w.Z, zpad), 7.0, device=device)], dim=1)
        dy = torch.cat([dy, torch.full((w.Z, zpad), 7.0, device=device)], dim=1)
    meta = dict(n_block_rows=nbr, nblocks=nblocks, block=w.block, sizemax=sizemax)
    return (y.to(w.dtype), dy.to(w.dtype), torch.from_numpy(lut).to(device), meta)
