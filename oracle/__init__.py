"""Double-precision CPU oracle for the fused cross-entropy and the row softmax.

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke()``
and by the benchmark's CPU-baseline leg.  The CUDA library and its Python
binding never import it.  The arithmetic lives in ``oracle.c`` (plain C,
double precision, the textbook definitions row by row); this module only
marshals numpy arrays through ctypes.

Inputs are numpy arrays: fp32 values as ``float32``, fp16 values as
``float16``, bf16 values as their raw bit patterns in a ``uint16`` array (see
:func:`bf16_bits`).  Outputs are float64.
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16, F16 = 0, 1, 2
MEAN, SUM, NONE = 0, 1, 2
REDUCTIONS = {"mean": MEAN, "sum": SUM, "none": NONE}


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def bf16_bits(t) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU torch bfloat16 tensor (any 2-D view), as uint16."""
    import torch
    return t.view(torch.int16).numpy().view(np.uint16)


def host_array(t) -> np.ndarray:
    """A CPU torch tensor (fp32 or bf16, possibly a strided 2-D view) as an oracle input."""
    import torch
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    if t.dtype in (torch.float32, torch.float16):
        return t.numpy()
    raise TypeError(f"oracle inputs are fp32, fp16 or bf16, not {t.dtype}")


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float16:
        return F16
    raise TypeError(f"oracle takes float32, float16 or bf16-bits (uint16) arrays, not {a.dtype}")


def _row_stride(a: np.ndarray) -> int:
    assert a.ndim == 2 and (a.shape[1] <= 1 or a.strides[1] == a.itemsize), \
        "rows must be unit-stride"
    if a.shape[0] <= 1:  # numpy leaves the stride of a length-1 axis arbitrary
        return max(a.shape[1], 1)
    return a.strides[0] // a.itemsize


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes front end of one compiled copy of oracle.c."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i64, p, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.oracle_ce_count.argtypes = [p, i64, i64, i64, p, p]
        lib.oracle_ce_rows.argtypes = [p, ci, i64, p, i64, i64, i64, p, i64, p, p, ci]
        lib.oracle_ce_rows_ex.argtypes = [p, ci, i64, p, i64, i64, i64, ci, p, p, i64, p, p, ci]
        lib.oracle_ce_mean.argtypes = [p, i64, i64]
        lib.oracle_ce_mean.restype = ctypes.c_double
        lib.oracle_ce_sum.argtypes = [p, i64]
        lib.oracle_ce_sum.restype = ctypes.c_double
        lib.oracle_widen.argtypes = [p, ci, i64, p]
        lib.oracle_softmax_fwd_rows.argtypes = [p, ci, i64, i64, p, i64, p, ci]
        lib.oracle_softmax_bwd_rows.argtypes = [p, i64, p, i64, ci, i64, p, i64, p, ci]
        lib.oracle_softmax_bwd_bsr.argtypes = [p, i64, p, i64, ci, p, i64, i64, i64, i64, i64,
                                               i64, ctypes.c_double, p, i64, p, i64, p]
        self.lib = lib

    def ce_count(self, targets, V: int, ignore_index: int = -100):
        """(n, bad): rows whose target != ignore_index, and those among them outside [0, V)."""
        t = np.ascontiguousarray(targets, dtype=np.int64)
        n, bad = ctypes.c_int64(), ctypes.c_int64()
        self.lib.oracle_ce_count(_ptr(t), t.shape[0], V, ignore_index, ctypes.byref(n),
                                 ctypes.byref(bad))
        return n.value, bad.value

    def ce_rows(self, logits: np.ndarray, targets, V: int, n: int, ignore_index: int = -100,
                rows=None, want_grad: bool = True, nthreads: int = None):
        """(grad [nrows, V] float64 or None, row_loss [nrows]) of the listed rows.

        ``logits`` is [M, >=V] with unit column stride; ``n`` is the batch-wide
        non-ignored count; ``rows`` lists input rows (all rows when None).
        """
        code = _dtype_code(logits)
        stride = _row_stride(logits)
        t = np.ascontiguousarray(targets, dtype=np.int64)
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = logits.shape[0] if rows is None else rows.shape[0]
        grad = np.empty((nrows, V), dtype=np.float64) if want_grad else None
        row_loss = np.empty((nrows,), dtype=np.float64)
        rc = self.lib.oracle_ce_rows(_ptr(logits), code, stride, _ptr(t), V, ignore_index, n,
                                     _ptr(rows), nrows, _ptr(grad), _ptr(row_loss),
                                     nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle_ce_rows rejected its arguments")
        return grad, row_loss

    def ce_rows_ex(self, logits: np.ndarray, targets, V: int, n: int, ignore_index: int = -100,
                   reduction: str = "mean", grad_scale=None, rows=None, want_grad: bool = True,
                   nthreads: int = None):
        """ce_rows with a reduction ('mean', 'sum', 'none') and the incoming
        grad_output: None (1), a scalar, or one value per input row for 'none'."""
        code = _dtype_code(logits)
        stride = _row_stride(logits)
        t = np.ascontiguousarray(targets, dtype=np.int64)
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = logits.shape[0] if rows is None else rows.shape[0]
        gs = None
        if grad_scale is not None:
            gs = np.ascontiguousarray(np.atleast_1d(grad_scale), dtype=np.float64)
            if reduction == "none":
                assert gs.shape[0] == logits.shape[0]
        grad = np.empty((nrows, V), dtype=np.float64) if want_grad else None
        row_loss = np.empty((nrows,), dtype=np.float64)
        rc = self.lib.oracle_ce_rows_ex(_ptr(logits), code, stride, _ptr(t), V, ignore_index, n,
                                        REDUCTIONS[reduction], _ptr(gs), _ptr(rows), nrows,
                                        _ptr(grad), _ptr(row_loss), nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle_ce_rows_ex rejected its arguments")
        return grad, row_loss

    def ce_sum(self, row_loss) -> float:
        rl = np.ascontiguousarray(row_loss, dtype=np.float64)
        return self.lib.oracle_ce_sum(_ptr(rl), rl.shape[0])

    def widen(self, a: np.ndarray) -> np.ndarray:
        """The exact double value of every stored element (fp32, fp16 or bf16 bits)."""
        a = np.ascontiguousarray(a)
        out = np.empty(a.size, dtype=np.float64)
        self.lib.oracle_widen(_ptr(a), _dtype_code(a), a.size, _ptr(out))
        return out.reshape(a.shape)

    def ce_mean(self, row_loss, n: int) -> float:
        rl = np.ascontiguousarray(row_loss, dtype=np.float64)
        return self.lib.oracle_ce_mean(_ptr(rl), rl.shape[0], n)

    def ce(self, logits: np.ndarray, targets, V: int = None, ignore_index: int = -100,
           want_grad: bool = True, nthreads: int = None):
        """The whole fused cross-entropy call: dict(loss, row_loss, grad, n, bad)."""
        V = logits.shape[1] if V is None else V
        n, bad = self.ce_count(targets, V, ignore_index)
        grad, row_loss = self.ce_rows(logits, targets, V, n, ignore_index, None, want_grad,
                                      nthreads)
        return dict(loss=self.ce_mean(row_loss, n), row_loss=row_loss, grad=grad, n=n, bad=bad)

    def softmax_fwd(self, x: np.ndarray, rows=None, nthreads: int = None) -> np.ndarray:
        code = _dtype_code(x)
        stride = _row_stride(x)
        N = x.shape[1]
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = x.shape[0] if rows is None else rows.shape[0]
        y = np.empty((nrows, N), dtype=np.float64)
        rc = self.lib.oracle_softmax_fwd_rows(_ptr(x), code, stride, N, _ptr(rows), nrows,
                                              _ptr(y), nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle_softmax_fwd_rows rejected its arguments")
        return y

    def softmax_bwd(self, y: np.ndarray, dy: np.ndarray, rows=None,
                    nthreads: int = None) -> np.ndarray:
        code = _dtype_code(y)
        if _dtype_code(dy) != code or y.shape != dy.shape:
            raise TypeError("y and dy must share a dtype and a shape")
        N = y.shape[1]
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = y.shape[0] if rows is None else rows.shape[0]
        dx = np.empty((nrows, N), dtype=np.float64)
        rc = self.lib.oracle_softmax_bwd_rows(_ptr(y), _row_stride(y), _ptr(dy), _row_stride(dy),
                                              code, N, _ptr(rows), nrows, _ptr(dx),
                                              nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle_softmax_bwd_rows rejected its arguments")
        return dx

    def softmax_bwd_bsr(self, y: np.ndarray, dy: np.ndarray, lut, n_block_rows: int,
                        nblocks: int, block: int, sizemax: int, scale: float = 1.0,
                        block_rows=None):
        """Block-sparse softmax backward: (dx, bad).

        ``y`` and ``dy`` are [Z, zstride] arrays (unit inner stride) whose first
        nblocks * block^2 elements per batch item hold the blocks; ``lut`` is
        the int32 table.  ``dx`` is [Z, nblocks * block^2] float64: the results
        at the positions the table names (only the listed ``block_rows`` when
        given), the widened ``dy`` elsewhere.  ``bad`` counts the block-rows the
        table describes wrongly (left as ``dy``).
        """
        code = _dtype_code(y)
        if _dtype_code(dy) != code or y.shape[0] != dy.shape[0] or y.ndim != 2 or dy.ndim != 2:
            raise TypeError("y and dy must be [Z, zstride] arrays of one dtype")
        Z = y.shape[0]
        L = nblocks * block * block
        if y.shape[1] < L or dy.shape[1] < L:
            raise ValueError("y and dy hold fewer than nblocks * block^2 elements per item")
        t = np.ascontiguousarray(lut, dtype=np.int32)
        if block_rows is not None:
            block_rows = np.ascontiguousarray(block_rows, dtype=np.int64)
        dx = np.ascontiguousarray(self.widen(np.ascontiguousarray(dy[:, :L])).reshape(Z, L))
        bad = ctypes.c_int64()
        rc = self.lib.oracle_softmax_bwd_bsr(
            _ptr(y), _row_stride(y), _ptr(dy), _row_stride(dy), code, _ptr(t), t.size,
            n_block_rows, nblocks, block, sizemax, Z, float(scale), _ptr(block_rows),
            0 if block_rows is None else block_rows.size, _ptr(dx), L, ctypes.byref(bad))
        if rc != 0:
            raise ValueError("oracle_softmax_bwd_bsr rejected its arguments")
        return dx, bad.value


_default = None


def get() -> Oracle:
    """The oracle built from oracle/oracle.c (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def ce_count(*a, **k):
    return get().ce_count(*a, **k)


def ce_rows(*a, **k):
    return get().ce_rows(*a, **k)


def ce_mean(*a, **k):
    return get().ce_mean(*a, **k)


def ce(*a, **k):
    return get().ce(*a, **k)


def softmax_fwd(*a, **k):
    return get().softmax_fwd(*a, **k)


def ce_rows_ex(*a, **k):
    return get().ce_rows_ex(*a, **k)


def ce_sum(*a, **k):
    return get().ce_sum(*a, **k)


def widen(*a, **k):
    return get().widen(*a, **k)


def softmax_bwd(*a, **k):
    return get().softmax_bwd(*a, **k)


def softmax_bwd_bsr(*a, **k):
    return get().softmax_bwd_bsr(*a, **k)
