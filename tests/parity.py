"""Tolerances for comparing the CUDA path with the double-precision oracle.

fp32 (results computed and stored in fp32):
  gradient / softmax:   |g - o| <= 1e-5 |o| + FLOOR
  softmax backward:     |dx - o| <= 1e-5 (|o| + |y_i| sum_j |y_j dy_j|) + FLOOR
                        (the second term bounds the cancellation in dy_i - s)
  loss:                 |L - Lo| <= 1e-5 |Lo|
bf16 (fp32 arithmetic, one round-to-nearest-even store):
  gradient:             |n g - n o| <= 2e-2            (the stated bound, on p - onehot)
                        |g - o| <= (2^-8 + 2e-5) |o| + FLOOR   (one bf16 rounding + fp32 error)
  softmax:              |y - o| <= (2^-8 + 2e-5) |o| + FLOOR
  softmax backward:     |dx - o| <= (2^-8 + 1e-5) |o| + 2e-5 |y_i| sum_j |y_j dy_j| + FLOOR
  loss:                 |L - Lo| <= 1e-3 |Lo|
FLOOR = 1e-37 covers results below fp32's normal range, which the kernels flush to zero.
"""
import numpy as np
import torch

FLOOR = 1e-37
BF16_REL = 2.0 ** -8 + 2e-5


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def _report(bad, got, ref, tol, what):
    if bad.any():
        idx = np.argwhere(bad)[:5]
        details = ", ".join(f"{tuple(i)}: got {got[tuple(i)]!r} want {ref[tuple(i)]!r} "
                            f"tol {tol[tuple(i)]:.3g}" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; {details}")


def check_grad(got: torch.Tensor, ref: np.ndarray, n: int, dtype, what="gradient"):
    g = to_f64(got)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape
    if dtype == torch.float32:
        tol = 1e-5 * np.abs(ref) + FLOOR
    else:
        nabs = np.abs(n * g - n * ref)
        _report(nabs > 2e-2, n * g, n * ref, np.full_like(ref, 2e-2), what + " (n*g, 2e-2)")
        tol = BF16_REL * np.abs(ref) + FLOOR
    _report(~(np.abs(g - ref) <= tol), g, ref, tol, what)


def check_softmax(got: torch.Tensor, ref: np.ndarray, dtype, what="softmax"):
    y = to_f64(got)
    rel = 1e-5 if dtype == torch.float32 else BF16_REL
    tol = rel * np.abs(ref) + FLOOR
    _report(~(np.abs(y - ref) <= tol), y, ref, tol, what)


def check_softmax_bwd(got: torch.Tensor, ref: np.ndarray, y: torch.Tensor, dy: torch.Tensor,
                      dtype, what="softmax backward"):
    dx = to_f64(got)
    yv, dyv = to_f64(y), to_f64(dy)
    scale = np.abs(yv) * np.abs(yv * dyv).sum(axis=1, keepdims=True)
    if dtype == torch.float32:
        tol = 1e-5 * (np.abs(ref) + scale) + FLOOR
    else:
        tol = (2.0 ** -8 + 1e-5) * np.abs(ref) + 2e-5 * scale + FLOOR
    _report(~(np.abs(dx - ref) <= tol), dx, ref, tol, what)


def check_loss(got: float, ref: float, dtype, what="loss"):
    rel = 1e-5 if dtype == torch.float32 else 1e-3
    if np.isnan(ref):
        assert np.isnan(got), f"{what}: got {got}, want NaN"
        return
    assert abs(got - ref) <= rel * abs(ref), f"{what}: got {got!r} want {ref!r} (rel {rel})"
