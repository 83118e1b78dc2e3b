"""The seeded input generators produce the stated shapes, distributions and
structure, deterministically (CPU)."""
import math

import numpy as np

import pytest
import torch

import workloads
from workloads import IGNORE_INDEX


@pytest.mark.parametrize("name", list(workloads.CE_WORKLOADS))
def test_ce_workload_structure(name):
    w = workloads.CE_WORKLOADS[name]
    M = min(w.M, 512)
    wr = w.with_rows(M)
    x, t = workloads.make_ce_inputs(wr, "cpu")
    assert x.shape == (M, w.V) and x.dtype == w.dtype and t.dtype == torch.int64
    ign = t == IGNORE_INDEX
    assert int(ign.sum()) == int(round(w.ignore_frac * M))
    live = t[~ign]
    assert bool(((live >= 0) & (live < w.V)).all())
    xf = x.float()
    rows = torch.arange(M)
    if w.neginf_frac:
        frac = float(torch.isneginf(xf).float().mean())
        assert abs(frac - w.neginf_frac) < 0.002
        assert not bool(torch.isneginf(xf[rows[~ign], live]).any()), "-inf at a target"
    else:
        assert bool(torch.isfinite(xf).all())
    finite = xf[torch.isfinite(xf)]
    if w.spike:
        # the spike row maximum sits near spike, far above the N(0, std^2) bulk
        assert float(xf.max(dim=1).values.min()) > w.spike - 4 * w.std
    else:
        assert abs(float(finite.std()) - w.std) < 0.02 * w.std
        assert abs(float(finite.mean())) < 0.02 * w.std
    x2, t2 = workloads.make_ce_inputs(wr, "cpu")
    assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                       x2.view(torch.int16) if x2.dtype == torch.bfloat16 else x2)
    assert torch.equal(t, t2)


def test_padded_stride_layout():
    w = workloads.CE_WORKLOADS["ce_f32_64x1000"]
    x, t = workloads.make_ce_inputs(w, "cpu")
    xp, tp = workloads.make_ce_inputs(w, "cpu", stride=1005)
    assert xp.stride() == (1005, 1) and torch.equal(xp, x) and torch.equal(tp, t)
    base = xp.as_strided((64, 1005), (1005, 1))
    assert bool((base[:, 1000:] == 7.0).all())


@pytest.mark.parametrize("N", workloads.SOFTMAX_NS)
def test_softmax_inputs(N):
    x, y, dy = workloads.make_softmax_inputs(16, N)
    assert x.shape == y.shape == dy.shape == (16, N)
    assert bool((y > 0).all())
    assert torch.allclose(y.double().sum(1), torch.ones(16, dtype=torch.float64), atol=1e-5)
    assert abs(float(x.std()) - 1) < 0.1 and abs(float(dy.std()) - 1) < 0.1
    assert not math.isnan(float(x.sum()))


@pytest.mark.parametrize("name", list(workloads.BSR_WORKLOADS))
def test_bsr_layout_and_table(name):
    w = workloads.BSR_WORKLOADS[name]
    lay = workloads.make_bsr_layout(w)
    nb = w.S // w.block
    assert lay.shape == (w.H, nb, nb)
    if w.layout == "causal":
        assert (lay == np.tril(np.ones((nb, nb), dtype=bool))).all()
    else:
        assert lay[:, np.arange(nb), np.arange(nb)].all()
        off = lay.sum() - w.H * nb
        assert abs(off / (w.H * nb * (nb - 1)) - w.density) < 0.01
    lut, nbr, nblocks, sizemax, brow = workloads.make_bsr_lut(
        lay, w.seed + 1 if w.shuffle else None)
    assert nbr == w.H * nb and nblocks == int(lay.sum()) and lut.dtype == np.int32
    assert lut.size == 2 * nbr + 4 * nblocks
    sizes, offs = lut[0:2 * nbr:2], lut[1:2 * nbr:2]
    assert sizemax == sizes.max() and (sizes == lay.reshape(nbr, nb).sum(1)).all()
    seen = np.zeros(nblocks, dtype=int)
    for r in range(0, nbr, max(1, nbr // 64)):
        ent = lut[offs[r]:offs[r] + 4 * sizes[r]].reshape(-1, 4)
        h, rr = divmod(r, nb)
        assert (ent[:, 1] == h).all() and (ent[:, 2] == rr).all()
        assert lay[h, rr][ent[:, 3]].all() and len(set(ent[:, 3])) == sizes[r]
        assert (brow[ent[:, 0]] == r).all()
        seen[ent[:, 0]] += 1
    assert seen.max() <= 1
    if w.shuffle:
        ent = lut[2 * nbr:].reshape(-1, 4)
        assert not (np.diff(ent[:, 0]) > 0).all(), "entries were not shuffled"


def test_bsr_inputs_small():
    w = workloads.BSR_WORKLOADS["bsr_f32_causal_2x16x4096_b32"].with_sizes(H=2, S=256)
    y, dy, lut, meta = workloads.make_bsr_inputs(w, "cpu", zpad=24)
    L = meta["nblocks"] * 32 * 32
    assert y.shape == (2, L + 24) and dy.shape == (2, L + 24) and y.dtype == torch.float32
    assert bool((y[:, L:] == 7.0).all()) and bool((y[:, :L] > 0).all())
    # y / its row's element count: each matrix row sums to about 1
    lay = workloads.make_bsr_layout(w)
    first = y[0, :32 * 32].view(32, 32)      # block 0 = head 0, block-row 0 (size 1)
    assert abs(float(first.sum(1).mean()) - 1.0) < 0.2
    y2, dy2, lut2, _ = workloads.make_bsr_inputs(w, "cpu", zpad=24)
    assert torch.equal(y, y2) and torch.equal(dy, dy2) and torch.equal(lut, lut2)
    assert lay.sum() == meta["nblocks"]
