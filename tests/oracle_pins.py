"""Pins of the double-precision oracle to facts that do not come from the oracle.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with: a hand-derived worked example (tests/golden),
a closed form, an invariant of the mathematics, a library routine that
computes the same special case (torch float64), or central finite
differences of the oracle's own loss.  They are written as plain functions so
that ``test_oracle_mutations.py`` can run them against deliberately broken
copies of the oracle and check that each planted mistake is caught.
"""
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
II = workloads.IGNORE_INDEX


def _expr(s: str) -> float:
    return float(eval(s, {"__builtins__": {}}, {"ln": math.log}))


def _vec(s: str):
    return [_expr(t) for t in s.split()]


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, _, rest = line.partition(":")
                yield key.strip(), rest.strip()


def _bf16(vals) -> np.ndarray:
    return workloads_bits(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16))


def workloads_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _close(a, b, rtol, atol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    ok = np.isclose(a, b, rtol=rtol, atol=atol, equal_nan=True)
    diff = np.abs(a - b)
    worst = np.nanmax(diff) if (~np.isnan(diff)).any() else float("nan")
    assert ok.all(), f"{what}: max |diff| {worst}"


# ---------------------------------------------------------------------------
# worked examples

def pin_golden_ce(o):
    rows, targets, grads, losses = [], [], [], []
    V = ii = None
    expected_loss = None
    for key, rest in _golden_lines("ce_worked_example.txt"):
        if key == "V":
            V = int(rest)
        elif key == "ignore_index":
            ii = int(rest)
        elif key == "row":
            x, t, g, l = [p.strip() for p in rest.split("|")]
            rows.append(_vec(x))
            targets.append(int(t))
            grads.append(_vec(g))
            losses.append(_expr(l))
        elif key == "loss":
            expected_loss = _expr(rest)
    x = np.array(rows, dtype=np.float32)
    r = o.ce(x, np.array(targets), V, ii)
    assert r["n"] == 2 and r["bad"] == 0
    _close(r["grad"], grads, 1e-6, 1e-7, "golden ce gradient")
    _close(r["row_loss"], losses, 1e-6, 1e-7, "golden ce row loss")
    _close(r["loss"], expected_loss, 1e-6, 0, "golden ce mean loss")


def pin_golden_softmax(o):
    for key, rest in _golden_lines("softmax_worked_example.txt"):
        parts = [_vec(p) for p in rest.split("|")]
        if key == "fwd":
            x, y = parts
            got = o.softmax_fwd(np.array([x], dtype=np.float32))
            _close(got[0], y, 1e-6, 0, "golden softmax forward")
        elif key == "bwd":
            y, dy, dx = parts
            for arr in (lambda v: np.array([v], dtype=np.float32),
                        lambda v: _bf16([v])):
                got = o.softmax_bwd(arr(y), arr(dy))
                _close(got[0], dx, 1e-15, 1e-15, "golden softmax backward")


# ---------------------------------------------------------------------------
# closed forms

def pin_uniform_closed_form(o):
    """Equal logits: loss = ln V; gradient 1/(V n) off target, (1/V - 1)/n on it."""
    for dtype in ("f32", "bf16"):
        for V in (1, 2, 7, 1000, 32000):
            consts = [-3.5, 0.0, 1000.0, -1024.0, 2.0, 0.5]
            targets = np.array([0, V - 1, II, (V // 2), II, V // 3], dtype=np.int64)
            x32 = np.repeat(np.array(consts, dtype=np.float32)[:, None], V, axis=1)
            x = x32 if dtype == "f32" else _bf16(x32)
            r = o.ce(x, targets, V, II)
            n = 4
            assert r["n"] == n and r["bad"] == 0
            for k, t in enumerate(targets):
                if t == II:
                    assert np.all(r["grad"][k] == 0.0), "ignored row not zero"
                    assert r["row_loss"][k] == 0.0
                    continue
                _close(r["row_loss"][k], math.log(V), 1e-13, 1e-15, "uniform row loss")
                exp_g = np.full(V, 1.0 / (V * n))
                exp_g[t] = (1.0 / V - 1.0) / n
                _close(r["grad"][k], exp_g, 1e-12, 1e-18, "uniform gradient")
            _close(r["loss"], math.log(V), 1e-13, 1e-15, "uniform mean loss")


def pin_softmax_uniform(o):
    """Equal inputs: softmax = 1/N everywhere, also for large magnitudes."""
    for N in (1, 3, 1000):
        x = np.repeat(np.array([[0.0], [1000.0], [-1024.0]], dtype=np.float32), N, axis=1)
        _close(o.softmax_fwd(x), np.full((3, N), 1.0 / N), 1e-13, 0, "uniform softmax")


# ---------------------------------------------------------------------------
# invariants

def _dyadic_logits(rng, M, V):
    """fp32 logits that are multiples of 2^-10 in [-4, 4], so +4 shifts are exact."""
    return (np.round(rng.standard_normal((M, V)) * 1024.0).clip(-4096, 4096) / 1024.0
            ).astype(np.float32)


def pin_ce_invariants(o):
    rng = np.random.default_rng(7)
    M, V = 12, 97
    x = _dyadic_logits(rng, M, V)
    t = rng.integers(0, V, M)
    t[[2, 5]] = II
    r = o.ce(x, t, V, II)
    n = r["n"]
    assert n == M - 2
    for k in range(M):
        if t[k] == II:
            assert np.all(r["grad"][k] == 0.0)
            continue
        # every non-ignored gradient row sums to zero
        assert abs(r["grad"][k].sum() * n) < 1e-13, "gradient row does not sum to 0"
        # the target entry is the only negative one
        assert r["grad"][k][t[k]] < 0 and np.all(np.delete(r["grad"][k], t[k]) > 0)
        # each row loss is positive
        assert r["row_loss"][k] > 0
    # a constant shift of a row changes neither its loss nor its gradient
    x2 = x.copy()
    x2[3] += np.float32(4.0)
    x2[7] -= np.float32(4.0)
    r2 = o.ce(x2, t, V, II)
    _close(r2["grad"], r["grad"], 1e-12, 1e-18, "shift-invariant gradient")
    _close(r2["row_loss"], r["row_loss"], 1e-12, 1e-15, "shift-invariant loss")
    # permuting the columns (and the target with them) permutes the gradient
    perm = rng.permutation(V)
    inv = np.argsort(perm)
    t3 = np.where(t == II, II, inv[np.where(t == II, 0, t)])
    r3 = o.ce(np.ascontiguousarray(x[:, perm]), t3, V, II)
    _close(r3["grad"], r["grad"][:, perm], 1e-12, 1e-18, "column permutation")
    _close(r3["loss"], r["loss"], 1e-13, 0, "column permutation loss")
    # the mean over n: duplicating the batch leaves the loss unchanged
    r4 = o.ce(np.concatenate([x, x]), np.concatenate([t, t]), V, II)
    _close(r4["loss"], r["loss"], 1e-13, 0, "batch duplication loss")
    _close(r4["grad"][:M] * 2, r["grad"], 1e-12, 1e-18, "gradient scales with 1/n")


def pin_neginf_columns(o):
    """-inf logits take no probability: same loss and gradient as without them."""
    rng = np.random.default_rng(11)
    M, V = 6, 40
    x = rng.standard_normal((M, V)).astype(np.float32)
    t = rng.integers(0, V, M)
    dead = np.zeros((M, V), dtype=bool)
    for k in range(M):
        cols = rng.choice([c for c in range(V) if c != t[k]], 7, replace=False)
        dead[k, cols] = True
    xi = x.copy()
    xi[dead] = -np.inf
    r = o.ce(xi, t, V, II)
    assert np.all(r["grad"][dead] == 0.0)
    for k in range(M):
        keep = ~dead[k]
        tk = int(np.sum(keep[: t[k]]))
        g, l = o.ce_rows(np.ascontiguousarray(x[k:k + 1, keep]), np.array([tk]),
                         int(keep.sum()), r["n"], II)
        _close(r["grad"][k][keep], g[0], 1e-13, 1e-18, "-inf column removal gradient")
        _close(r["row_loss"][k], l[0], 1e-13, 0, "-inf column removal loss")


def pin_v1_and_degenerate(o):
    # V = 1: the single class always has probability 1
    r = o.ce(np.array([[3.0], [-2.0], [5.0]], dtype=np.float32), np.array([0, 0, II]), 1, II)
    assert r["n"] == 2
    assert np.all(r["grad"] == 0.0) and np.all(r["row_loss"] == 0.0) and r["loss"] == 0.0
    # every row ignored: n = 0, the mean is 0/0 and every gradient row is zero
    x = np.ones((2, 5), dtype=np.float32)
    r = o.ce(x, np.array([II, II]), 5, II)
    assert r["n"] == 0 and math.isnan(r["loss"]) and np.all(r["grad"] == 0.0)
    # a target outside [0, V): NaN loss, the row is left as it was, counted as bad
    x = np.arange(10, dtype=np.float32).reshape(2, 5)
    r = o.ce(x, np.array([5, 1]), 5, II)
    assert r["bad"] == 1 and r["n"] == 2
    assert math.isnan(r["row_loss"][0]) and not math.isnan(r["row_loss"][1])
    assert np.array_equal(r["grad"][0], x[0].astype(np.float64))
    assert math.isnan(r["loss"])


def pin_softmax_invariants(o):
    rng = np.random.default_rng(5)
    M, N = 8, 50
    x = _dyadic_logits(rng, M, N)
    y = o.softmax_fwd(x)
    assert np.all(y > 0)
    _close(y.sum(axis=1), np.ones(M), 1e-14, 0, "softmax rows sum to 1")
    x2 = x + np.float32(4.0)
    _close(o.softmax_fwd(x2), y, 1e-12, 0, "softmax shift invariance")
    # backward with y exactly on the simplex (dyadic fractions summing to 1)
    k = rng.multinomial(4096, np.full(N, 1.0 / N), size=M)
    ys = (k / 4096.0).astype(np.float32)
    dy = rng.standard_normal((M, N)).astype(np.float32)
    dx = o.softmax_bwd(ys, dy)
    _close(dx.sum(axis=1), np.zeros(M), 0, 1e-14, "softmax backward rows sum to 0")
    c = np.repeat(rng.standard_normal((M, 1)).astype(np.float32), N, axis=1)
    _close(o.softmax_bwd(ys, c), np.zeros((M, N)), 0, 1e-14, "constant dy gives zero")
    # zero probability entries get zero gradient; the map is linear in dy
    _close(o.softmax_bwd(ys, 2 * dy), 2 * dx, 1e-13, 1e-16, "linear in dy")


def pin_bf16_decoding(o):
    """bf16 inputs are exactly the fp32 values with the low 16 bits zero."""
    bits = np.array([[0x3F80, 0xC000, 0x4049, 0x0000, 0xBF00, 0x42C8]], dtype=np.uint16)
    vals = np.array([[1.0, -2.0, 3.140625, 0.0, -0.5, 100.0]], dtype=np.float32)
    _close(o.softmax_fwd(bits), o.softmax_fwd(vals), 0, 0, "bf16 decoding (softmax)")
    t = np.array([2])
    a = o.ce(bits, t, 6, II)
    b = o.ce(vals, t, 6, II)
    assert a["loss"] == b["loss"] and np.array_equal(a["grad"], b["grad"])


def pin_row_stride(o):
    """Padding columns beyond V are never read."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 33)).astype(np.float32)
    pad = np.full((5, 40), np.nan, dtype=np.float32)
    pad[:, :33] = x
    t = np.array([0, 32, II, 5, 17])
    a = o.ce(pad[:, :33], t, 33, II)
    b = o.ce(np.ascontiguousarray(x), t, 33, II)
    assert a["loss"] == b["loss"] and np.array_equal(a["grad"], b["grad"])
    _close(o.softmax_fwd(pad[:, :33]), o.softmax_fwd(x), 0, 0, "softmax stride")


# ---------------------------------------------------------------------------
# library routines that compute the same special cases (torch, float64, CPU)

def _torch_ce(x64: torch.Tensor, t: torch.Tensor):
    x = x64.clone().requires_grad_(True)
    loss = F.cross_entropy(x, t, ignore_index=II, reduction="mean")
    loss.backward()
    return loss.item(), x.grad.numpy()


def pin_torch_cross_entropy(o):
    for w in workloads.CE_WORKLOADS.values():
        M = min(w.M, 16)
        x, t = workloads.make_ce_inputs(w.with_rows(M), "cpu")
        V = w.V
        host = x.numpy() if x.dtype == torch.float32 else workloads_bits(x)
        r = o.ce(host, t.numpy(), V, II)
        ref_loss, ref_grad = _torch_ce(x.to(torch.float64), t)
        _close(r["loss"], ref_loss, 1e-12, 0, f"torch loss {w.name}")
        _close(r["grad"], ref_grad, 1e-10, 1e-18, f"torch gradient {w.name}")


def pin_torch_softmax(o):
    for dtype in (torch.float32, torch.bfloat16):
        for N in workloads.SOFTMAX_NS:
            x, y, dy = workloads.make_softmax_inputs(8, N, dtype)
            hx = x.numpy() if dtype == torch.float32 else workloads_bits(x)
            hy = y.numpy() if dtype == torch.float32 else workloads_bits(y)
            hdy = dy.numpy() if dtype == torch.float32 else workloads_bits(dy)
            ref_y = torch.softmax(x.to(torch.float64), dim=1).numpy()
            _close(o.softmax_fwd(hx), ref_y, 1e-12, 1e-300, f"torch softmax N={N}")
            ref_dx = torch._softmax_backward_data(dy.to(torch.float64), y.to(torch.float64), 1,
                                                  torch.float64).numpy()
            got = o.softmax_bwd(hy, hdy)
            scale = np.abs(y.to(torch.float64).numpy() * dy.to(torch.float64).numpy()).sum(1)
            tol = 1e-12 * (np.abs(ref_dx) + y.to(torch.float64).numpy() * scale[:, None])
            assert np.all(np.abs(got - ref_dx) <= tol + 1e-300), f"torch softmax bwd N={N}"


# ---------------------------------------------------------------------------
# finite differences of the oracle's own loss (Richardson-extrapolated)

def pin_finite_difference_ce(o):
    rng = np.random.default_rng(1)
    M, V = 3, 5
    x = _dyadic_logits(rng, M, V)
    t = np.array([1, II, 4])
    r = o.ce(x, t, V, II)

    def loss_at(xx):
        return o.ce(xx, t, V, II, want_grad=False)["loss"]

    h = 2.0 ** -6
    for i in range(M):
        for j in range(V):
            d = []
            for hh in (h, h / 2):
                xp, xm = x.copy(), x.copy()
                xp[i, j] += np.float32(hh)
                xm[i, j] -= np.float32(hh)
                d.append((loss_at(xp) - loss_at(xm)) / (2 * hh))
            fd = (4 * d[1] - d[0]) / 3
            assert abs(fd - r["grad"][i, j]) < 1e-8, f"finite difference at ({i},{j})"


def pin_finite_difference_softmax_bwd(o):
    """dx of the backward equals the gradient of sum_i dy_i softmax(x)_i."""
    rng = np.random.default_rng(2)
    N = 6
    x = _dyadic_logits(rng, 1, N)
    dy = rng.standard_normal((1, N)).astype(np.float32)
    y = o.softmax_fwd(x).astype(np.float32)
    dx = o.softmax_bwd(y, dy)[0]
    h = 2.0 ** -6
    for j in range(N):
        d = []
        for hh in (h, h / 2):
            xp, xm = x.copy(), x.copy()
            xp[0, j] += np.float32(hh)
            xm[0, j] -= np.float32(hh)
            fp = float(np.dot(o.softmax_fwd(xp)[0], dy[0].astype(np.float64)))
            fm = float(np.dot(o.softmax_fwd(xm)[0], dy[0].astype(np.float64)))
            d.append((fp - fm) / (2 * hh))
        fd = (4 * d[1] - d[0]) / 3
        assert abs(fd - dx[j]) < 1e-6, f"softmax backward finite difference at {j}"


# ---------------------------------------------------------------------------
# reductions, the incoming grad_output, fp16 inputs

def pin_decoding_exhaustive(o):
    """Every fp16 and every bf16 bit pattern widens to the value numpy / torch give."""
    h = np.arange(65536, dtype=np.uint16).view(np.float16)
    assert np.array_equal(o.widen(h), h.astype(np.float64), equal_nan=True), "fp16 decoding"
    b = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(o.widen(b), ref, equal_nan=True), "bf16 decoding"


def _as_host(t):
    if t.dtype == torch.bfloat16:
        return workloads_bits(t)
    return t.numpy()


def pin_torch_reductions(o):
    """F.cross_entropy with reduction sum / none / mean and a grad_output, float64 autograd."""
    rng = np.random.default_rng(21)
    for dtype in (torch.float32, torch.bfloat16, torch.float16):
        M, V = 9, 37
        x = (torch.from_numpy(rng.standard_normal((M, V))) * 2).to(dtype)
        t = torch.from_numpy(rng.integers(0, V, M))
        t[[1, 6]] = II
        x64 = x.to(torch.float64)
        n, _ = o.ce_count(t.numpy(), V, II)
        w = torch.from_numpy(rng.standard_normal(M))
        for reduction, go in (("mean", torch.tensor(2.5, dtype=torch.float64)),
                              ("sum", torch.tensor(-0.75, dtype=torch.float64)),
                              ("none", w)):
            xr = x64.clone().requires_grad_(True)
            out = F.cross_entropy(xr, t, ignore_index=II, reduction=reduction)
            out.backward(go)
            scale = go.numpy() if reduction == "none" else float(go)
            grad, rl = o.ce_rows_ex(_as_host(x), t.numpy(), V, n, II, reduction, scale)
            _close(grad, xr.grad.numpy(), 1e-10, 1e-18, f"torch {reduction} gradient {dtype}")
            if reduction == "none":
                _close(rl, out.detach().numpy(), 1e-12, 1e-15, f"torch none losses {dtype}")
            elif reduction == "sum":
                _close(o.ce_sum(rl), out.item(), 1e-12, 0, f"torch sum loss {dtype}")
            else:
                _close(o.ce_mean(rl, n), out.item(), 1e-12, 0, f"torch mean loss {dtype}")


def pin_reduction_invariants(o):
    rng = np.random.default_rng(22)
    M, V = 10, 29
    x = _dyadic_logits(rng, M, V)
    t = rng.integers(0, V, M)
    t[4] = II
    n, _ = o.ce_count(t, V, II)
    g_mean, l_mean = o.ce_rows_ex(x, t, V, n, II, "mean")
    g_sum, l_sum = o.ce_rows_ex(x, t, V, n, II, "sum")
    g_none, _ = o.ce_rows_ex(x, t, V, n, II, "none", np.ones(M))
    _close(g_sum, g_mean * n, 1e-13, 1e-18, "sum gradient is n times the mean gradient")
    _close(g_none, g_sum, 0, 0, "none with unit weights is the sum gradient")
    assert np.array_equal(l_mean, l_sum), "row losses do not depend on the reduction"
    g_s, _ = o.ce_rows_ex(x, t, V, n, II, "mean", 2.5)
    _close(g_s, 2.5 * g_mean, 1e-13, 1e-18, "the gradient is linear in grad_output")
    wts = rng.standard_normal(M)
    g_w, _ = o.ce_rows_ex(x, t, V, n, II, "none", wts)
    _close(g_w, wts[:, None] * g_sum, 1e-12, 1e-18, "per-row weights scale their rows")
    sel = np.array([7, 2, 9])
    g_sel, l_sel = o.ce_rows_ex(x, t, V, n, II, "none", wts, rows=sel)
    _close(g_sel, g_w[sel], 0, 0, "a row subset picks the rows' own weights")
    assert np.array_equal(l_sel, l_sum[sel])


# ---------------------------------------------------------------------------
# block-sparse softmax backward (look-up table addressing, scale)

def pin_golden_bsr(o):
    g, cases = {}, []
    for key, rest in _golden_lines("softmax_bwd_bsr_worked_example.txt"):
        if key == "case":
            sizemax, scale, dx, bad = rest.split("|")
            cases.append((int(sizemax), _expr(scale), _vec(dx), int(bad)))
        else:
            g[key] = rest
    block, nblocks, nbr = int(g["block"]), int(g["nblocks"]), int(g["n_block_rows"])
    lut = np.array([int(v) for v in g["lut"].split()], dtype=np.int32)
    y, dy = _vec(g["y"]), _vec(g["dy"])
    for sizemax, scale, want, want_bad in cases:
        for arr in (lambda v: np.array([v], dtype=np.float32), lambda v: _bf16([v])):
            got, bad = o.softmax_bwd_bsr(arr(y), arr(dy), lut, nbr, nblocks, block, sizemax,
                                         scale)
            assert bad == want_bad, f"golden bsr: bad {bad}, want {want_bad}"
            _close(got[0], want, 0, 1e-15, f"golden bsr sizemax={sizemax}")


def _bsr_host(t):
    return workloads_bits(t) if t.dtype == torch.bfloat16 else t.numpy()


def _bsr_to_dense(vals, lay, block):
    """[Z, nblocks * block^2] values -> [Z, H, S, S] float64, zero where no block is
    stored.  Blocks are numbered in the layout's (head, row, column) order."""
    Z = vals.shape[0]
    H, nb, _ = lay.shape
    v = vals[:, :int(lay.sum()) * block * block].reshape(Z, -1, block, block)
    dense = np.zeros((Z, H, nb * block, nb * block))
    for b, (h, r, c) in enumerate(zip(*np.nonzero(lay))):
        dense[:, h, r * block:(r + 1) * block, c * block:(c + 1) * block] = v[:, b]
    return dense


def _dense_to_bsr(dense, lay, block):
    out = []
    for h, r, c in zip(*np.nonzero(lay)):
        out.append(dense[:, h, r * block:(r + 1) * block, c * block:(c + 1) * block])
    return np.stack(out, axis=1).reshape(dense.shape[0], -1)


def pin_torch_bsr_softmax_bwd(o):
    """On the dense matrix with zeros where no block is stored, the row-wise
    softmax backward (torch float64) gives the block-sparse result on the stored
    blocks: a zero y contributes nothing to sum(y * dy)."""
    for dtype, block, seed in ((torch.float32, 4, 11), (torch.bfloat16, 8, 11),
                               (torch.float16, 2, 11)):
        w = workloads.BsrWorkload("pin", 2, 2, 4 * block, block, dtype, "random", 0.4, seed,
                                  shuffle=True, diagonal=False)
        lay = workloads.make_bsr_layout(w)
        assert (lay.sum(axis=2) == 0).any() and (lay.sum(axis=2) > 1).any()
        y, dy, lut, meta = workloads.make_bsr_inputs(w)
        dy_padded = torch.cat([dy, torch.full((w.Z, 8), 7.0, dtype=dtype)], dim=1)
        scale = 0.75
        got, bad = o.softmax_bwd_bsr(_bsr_host(y), _bsr_host(dy_padded), lut.numpy(),
                                     meta["n_block_rows"], meta["nblocks"], block,
                                     meta["sizemax"], scale)
        assert bad == 0
        y64 = y.to(torch.float64).numpy()
        dy64 = dy.to(torch.float64).numpy()
        yd = torch.from_numpy(_bsr_to_dense(y64, lay, block))
        dyd = torch.from_numpy(_bsr_to_dense(dy64, lay, block))
        ref = _dense_to_bsr(torch._softmax_backward_data(dyd, yd, -1, torch.float64).numpy(),
                            lay, block) * scale
        cancel = np.abs(y64) * _dense_to_bsr(
            np.broadcast_to((yd * dyd).abs().sum(-1, keepdim=True).numpy(), yd.shape), lay,
            block)
        tol = 1e-12 * (np.abs(ref) + cancel) + 1e-300
        assert np.all(np.abs(got - ref) <= tol), f"torch bsr softmax bwd {dtype}"


def pin_bsr_table_invariants(o):
    """The result does not depend on the order of a block-row's entries or on
    how the blocks are numbered; a padded batch stride changes nothing; a table
    that is wrong for a block-row leaves exactly that block-row's blocks as dy."""
    w = workloads.BsrWorkload("pin", 3, 2, 64, 8, torch.float32, "random", 0.3, 21)
    lay = workloads.make_bsr_layout(w)
    y, dy, lut, meta = workloads.make_bsr_inputs(w)
    nbr, nblocks, sizemax = meta["n_block_rows"], meta["nblocks"], meta["sizemax"]
    hy, hdy = y.numpy(), dy.numpy()
    base, bad = o.softmax_bwd_bsr(hy, hdy, lut.numpy(), nbr, nblocks, 8, sizemax, 1.5)
    assert bad == 0
    # entry order
    lut2 = workloads.make_bsr_lut(lay, 99)[0]
    got, _ = o.softmax_bwd_bsr(hy, hdy, lut2, nbr, nblocks, 8, sizemax, 1.5)
    _close(got, base, 1e-14, 1e-300, "bsr entry order")
    # block numbering: block b is stored at perm[b]
    perm = np.random.default_rng(5).permutation(nblocks)
    def move(a):
        out = np.empty_like(a).reshape(a.shape[0], nblocks, 64)
        out[:, perm] = a.reshape(a.shape[0], nblocks, 64)
        return out.reshape(a.shape)
    lut3 = lut.numpy().copy()
    lut3[2 * nbr::4] = perm[lut3[2 * nbr::4]]
    got, _ = o.softmax_bwd_bsr(move(hy), move(hdy), lut3, nbr, nblocks, 8, sizemax, 1.5)
    _close(got, move(base), 1e-14, 1e-300, "bsr block numbering")
    # padded batch stride
    pad = lambda a: np.concatenate([a, np.full((a.shape[0], 40), 7.0, a.dtype)], axis=1)
    got, _ = o.softmax_bwd_bsr(pad(hy), pad(hdy), lut.numpy(), nbr, nblocks, 8, sizemax, 1.5)
    _close(got, base, 0, 1e-300, "bsr batch stride")
    # wrong tables: one block-row each
    sizes = lut.numpy()[0:2 * nbr:2]
    rows = [r for r in range(nbr) if sizes[r] >= 2][:4]
    assert len(rows) == 4
    for how, r in zip(("size", "id_high", "id_negative", "offset"), rows):
        bad_lut = lut.numpy().copy()
        off = bad_lut[2 * r + 1]
        if how == "size":
            got, bad = o.softmax_bwd_bsr(hy, hdy, bad_lut, nbr, nblocks, 8, int(sizes[r]) - 1,
                                         1.5)
            wrong = {r2 for r2 in range(nbr) if sizes[r2] > sizes[r] - 1}
        else:
            if how == "id_high":
                bad_lut[off + 4] = nblocks
            elif how == "id_negative":
                bad_lut[off] = -1
            else:
                bad_lut[2 * r + 1] = bad_lut.size - 4 * int(sizes[r]) + 4
            got, bad = o.softmax_bwd_bsr(hy, hdy, bad_lut, nbr, nblocks, 8, sizemax, 1.5)
            wrong = {r}
        assert bad == len(wrong), f"bsr bad table ({how}): {bad} bad block-rows"
        mine = np.zeros(nblocks, dtype=bool)
        for r2 in wrong:
            ids = lut.numpy()[lut.numpy()[2 * r2 + 1]::4][:sizes[r2]]
            mine[ids] = True
        g3 = got.reshape(w.Z, nblocks, 64)
        assert np.array_equal(g3[:, mine], hdy.reshape(w.Z, nblocks, 64)[:, mine].astype(
            np.float64)), f"bsr bad table ({how}): rows were written"
        _close(g3[:, ~mine], base.reshape(w.Z, nblocks, 64)[:, ~mine], 0, 1e-300,
                f"bsr bad table ({how}): other rows")


ALL_PINS = [
    pin_golden_ce, pin_golden_softmax, pin_uniform_closed_form, pin_softmax_uniform,
    pin_ce_invariants, pin_neginf_columns, pin_v1_and_degenerate, pin_softmax_invariants,
    pin_bf16_decoding, pin_row_stride, pin_torch_cross_entropy, pin_torch_softmax,
    pin_finite_difference_ce, pin_finite_difference_softmax_bwd,
    pin_decoding_exhaustive, pin_torch_reductions, pin_reduction_invariants,
    pin_golden_bsr, pin_torch_bsr_softmax_bwd, pin_bsr_table_invariants,
]
