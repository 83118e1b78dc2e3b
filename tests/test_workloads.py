"""The seeded input generators produce the stated shapes, distributions and
structure, deterministically (CPU)."""
import math

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
