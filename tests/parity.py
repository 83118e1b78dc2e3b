"""Tolerances for comparing the CUDA path with the double-precision oracle.

fp32 (results computed and stored in fp32):
  gradient / softmax:   |g - o| <= 1e-5 |o| + FLOOR
  on-target gradient:   |g - o| <= 1e-5 |k| + FLOOR, k the row's factor (1/n for the mean):
                        o = (p_y - 1) k is a difference of two terms no larger than |k|, and
                        a pure relative bound on it is ill-posed as p_y -> 1 (the fp32 terms
                        carry ~1e-7 |k| of rounding), as for dy - s in the softmax backward
  softmax backward:     |dx - o| <= 1e-5 (|o| + |y_i| sum_j |y_j dy_j|) + FLOOR
                        (the second term bounds the cancellation in dy_i - s; for the
                        block-sparse form it is multiplied by |scale| and the sum runs
                        over the row's stored elements)
  loss:                 |L - Lo| <= 1e-5 |Lo| + 2^-22
                        (the floor: ln D and the other O(1) terms of a row loss carry a few
                        fp32 roundings of 2^-24, which a relative bound cannot absorb where
                        Lo = 0, e.g. V = 1)
bf16 (fp32 arithmetic, one round-to-nearest-even store):
  gradient:             |n g - n o| <= 2e-2            (the stated bound, on p - onehot)
                        |g - o| <= (2^-8 + 2e-5) |o| + FLOOR   (one bf16 rounding + fp32 error)
  on-target gradient:   the same plus 1e-5 |k|: the fp32 value carries the cancellation
                        error of (p_y - 1) k read above, which one bf16 rounding keeps
  softmax:              |y - o| <= (2^-8 + 2e-5) |o| + FLOOR
  softmax backward:     |dx - o| <= (2^-8 + 1e-5) |o| + 2e-5 |y_i| sum_j |y_j dy_j| + FLOOR
  loss:                 |L - Lo| <= 1e-3 |Lo| + 2^-22
fp16: as bf16 with 2^-10 in place of 2^-8 (an 11-bit significand), and an absolute
floor of 2^-24 (the spacing of fp16 subnormals): small gradients of a large batch
are subnormal or zero in fp16.
A 16-bit gradient scaled after it was stored (the autograd backward) is rounded
twice: twice the relative bound, the first floor amplified by the scale.
FLOOR = 1e-37 covers results below fp32's normal range, which the kernels flush to zero.
"""
import numpy as np
import torch

FLOOR = 1e-37
LOSS_FLOOR = 2.0 ** -22
BF16_REL = 2.0 ** -8 + 2e-5
F16_REL = 2.0 ** -10 + 2e-5
F16_FLOOR = 2.0 ** -24


def rel_floor(dtype):
    """(relative bound of one rounding + fp32 error, absolute floor) of a stored result."""
    if dtype == torch.float32:
        return 1e-5, FLOOR
    if dtype == torch.float16:
        return F16_REL, F16_FLOOR
    return BF16_REL, FLOOR


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def _report(bad, got, ref, tol, what):
    if bad.any():
        idx = np.argwhere(bad)[:5]
        details = ", ".join(f"{tuple(i)}: got {got[tuple(i)]!r} want {ref[tuple(i)]!r} "
                            f"tol {tol[tuple(i)]:.3g}" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; {details}")


def check_grad(got: torch.Tensor, ref: np.ndarray, n: int, dtype, what="gradient",
               targets=None):
    g = to_f64(got)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape
    check_grad_factor(got, ref, np.full(g.shape[0], 1.0 / n) if n else np.ones(g.shape[0]),
                      dtype, what, targets=targets)


def check_grad_factor(got, ref, k_rows, dtype, what="gradient", rescaled_by=None, targets=None):
    """Gradient rows (p - onehot) * k_r: for 16-bit storage the stated 2e-2 bound
    applies to (p - onehot), i.e. |g - o| <= 2e-2 |k_r|; and the relative bound
    of one rounding.  `rescaled_by` (per row) marks a gradient stored once and
    then multiplied by that factor and stored again (the autograd backward): two
    roundings, the first one's absolute floor amplified by the factor.
    `targets` (per row, optional) marks the on-target elements for the fp32
    bound on (p_y - 1) k; without it an element is on target when its value's
    sign differs from k's, which misses an exact 0 (p_y = 1: a row of one
    column, or every other logit more than ~745 below the target's)."""
    g = to_f64(got)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape
    rel, floor = rel_floor(dtype)
    amp = 1.0
    if rescaled_by is not None and dtype != torch.float32:
        rel *= 2
        amp = 1.0 + np.abs(np.asarray(rescaled_by, dtype=np.float64))[:, None]
    k = np.asarray(k_rows, dtype=np.float64)[:, None]
    if dtype != torch.float32:
        lim = 2e-2 * np.abs(k) + amp * floor
        _report(~(np.abs(g - ref) <= lim), g, ref, np.broadcast_to(lim, g.shape),
                what + " (2e-2 on p - onehot)")
    tol = rel * np.abs(ref) + amp * floor
    if targets is not None:
        t = np.asarray(targets, dtype=np.int64)[:, None]
        on_target = np.arange(g.shape[1])[None, :] == t
    else:  # the on-target element (p_y - 1) k is the one whose sign differs from k's
        on_target = ref * k < 0
    if dtype == torch.float32:
        tol = np.where(on_target, np.maximum(tol, rel * np.abs(k) + amp * floor), tol)
    else:
        tol = np.where(on_target, tol + 1e-5 * np.abs(k), tol)
    _report(~(np.abs(g - ref) <= tol), g, ref, tol, what)


def check_softmax(got: torch.Tensor, ref: np.ndarray, dtype, what="softmax"):
    y = to_f64(got)
    rel, floor = rel_floor(dtype)
    tol = rel * np.abs(ref) + floor
    _report(~(np.abs(y - ref) <= tol), y, ref, tol, what)


def check_softmax_bwd(got: torch.Tensor, ref: np.ndarray, y: torch.Tensor, dy: torch.Tensor,
                      dtype, what="softmax backward"):
    dx = to_f64(got)
    yv, dyv = to_f64(y), to_f64(dy)
    scale = np.abs(yv) * np.abs(yv * dyv).sum(axis=1, keepdims=True)
    if dtype == torch.float32:
        tol = 1e-5 * (np.abs(ref) + scale) + FLOOR
    else:
        rel, floor = rel_floor(dtype)
        tol = (rel - 1e-5) * np.abs(ref) + 2e-5 * scale + floor
    _report(~(np.abs(dx - ref) <= tol), dx, ref, tol, what)


def check_loss(got: float, ref: float, dtype, what="loss"):
    rel = 1e-5 if dtype == torch.float32 else 1e-3
    if np.isnan(ref):
        assert np.isnan(got), f"{what}: got {got}, want NaN"
        return
    assert abs(got - ref) <= rel * abs(ref) + LOSS_FLOOR, \
        f"{what}: got {got!r} want {ref!r} (rel {rel}, floor {LOSS_FLOOR})"


def ulp_distance_16(got: torch.Tensor, ref: np.ndarray, dtype) -> np.ndarray:
    """Per element, how many representable 16-bit values (bf16 or fp16) lie
    between the stored result and the oracle's value rounded to that format
    (0 = correctly rounded).  Sign-magnitude bit patterns are mapped onto a
    monotonic integer line, so +0 and -0 coincide."""
    want = torch.from_numpy(np.asarray(ref, dtype=np.float64)).to(torch.float32).to(dtype)
    a = got.detach().cpu().to(dtype).contiguous().view(torch.int16).numpy().astype(np.int32)
    b = want.contiguous().view(torch.int16).numpy().astype(np.int32)

    def line(v):
        mag = v & 0x7FFF
        return np.where(v & 0x8000, -mag, mag)

    return np.abs(line(a) - line(b))


def check_bsr(got: np.ndarray, ref: np.ndarray, y: np.ndarray, row_abs: np.ndarray, scale: float,
              dtype, what="block-sparse softmax backward"):
    """got, ref, y (float64) and row_abs = sum over the element's row of |y dy|,
    all of one shape; the bound of check_softmax_bwd with the cancellation term
    scaled by |scale|."""
    cancel = abs(scale) * np.abs(y) * row_abs
    if dtype == torch.float32:
        tol = 1e-5 * (np.abs(ref) + cancel) + FLOOR
    else:
        rel, floor = rel_floor(dtype)
        tol = (rel - 1e-5) * np.abs(ref) + 2e-5 * cancel + floor
    _report(~(np.abs(got - ref) <= tol), got, ref, tol, what)
