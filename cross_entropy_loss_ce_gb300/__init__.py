"""Fused hard-label cross-entropy and row softmax on GB300 (sm_103a).

Thin ctypes binding of ``_lib/libgbce.so`` (C ABI in ``include/gbce.h``): it
checks tensor shapes, takes raw device pointers, row strides and the current
CUDA stream from torch, and calls the library.  Every step of the computation
runs in the library's own CUDA kernels; there is no CPU or PyTorch fallback.
Loading fails loudly when the library has not been built
(``python -m cross_entropy_loss_ce_gb300.build``).
"""
import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libgbce.so")

GBCE_F32, GBCE_BF16, GBCE_F16 = 0, 1, 2
DTYPES = {torch.float32: GBCE_F32, torch.bfloat16: GBCE_BF16, torch.float16: GBCE_F16}
REDUCTIONS = {"mean": 0, "sum": 1, "none": 2}

OK, ERR_NULL, ERR_SIZE, ERR_DTYPE, ERR_ALIGN, ERR_CUDA, ERR_BAD_TARGET, ERR_TIMEOUT, \
    ERR_NO_DEVICE, ERR_REDUCTION, ERR_BAD_TABLE = range(11)
# bits a call ORs into its own status word (gbce_status_bit)
STATUS_TIMEOUT, STATUS_BAD_TABLE = 1, 2

_lib = None


class GbceError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: gbce status {code}: {status_string(code)}")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgbce.so once (raises if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m cross_entropy_loss_ce_gb300.build`")
        lib = ctypes.CDLL(path)
        i64, p, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.ce_fwd_bwd.argtypes = [p, i64, p, p, i64, i64, i64, ci, p]
        lib.softmax_fwd.argtypes = [p, i64, p, i64, i64, i64, ci, p]
        lib.softmax_bwd.argtypes = [p, i64, p, i64, p, i64, i64, i64, ci, p]
        lib.softmax_fwd_ex.argtypes = [p, i64, p, i64, i64, i64, ci, p, p]
        lib.softmax_bwd_ex.argtypes = [p, i64, p, i64, p, i64, i64, i64, ci, p, p]
        lib.ce_fwd_bwd_ex.argtypes = [p, i64, p, p, p, p, i64, i64, i64, ci, ci, p]
        lib.scale_rows.argtypes = [p, i64, i64, i64, ci, p, ci, p]
        lib.gbce_plan.argtypes = [ci, i64, i64, ci, ci, ctypes.POINTER(ci)]
        lib.gbce_plan.restype = ctypes.c_char_p
        lib.gbce_last_error.argtypes = [p]
        lib.gbce_status_string.argtypes = [ci]
        lib.gbce_status_string.restype = ctypes.c_char_p
        lib.gbce_timing_enable.argtypes = [ci]
        lib.softmax_bwd_bsr.argtypes = [p, i64, p, i64, p, i64, p, i64, i64, i64, i64, i64, i64,
                                        ctypes.c_float, ci, p]
        lib.softmax_bwd_bsr_ex.argtypes = [p, i64, p, i64, p, i64, p, i64, i64, i64, i64, i64, i64,
                                           ctypes.c_float, ci, p, p]
        lib.gbce_bsr_plan.argtypes = [i64, i64, ci, ci, ctypes.POINTER(ci)]
        lib.gbce_bsr_plan.restype = ctypes.c_char_p
        lib.gbce_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double),
                                         ctypes.POINTER(ctypes.c_int64)]
        for f in ("ce_fwd_bwd", "softmax_fwd", "softmax_bwd", "gbce_last_error",
                  "gbce_timing_enable", "gbce_timing_read", "ce_fwd_bwd_ex", "scale_rows",
                  "softmax_bwd_bsr"):
            getattr(lib, f).restype = ci
        _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load_library().gbce_status_string(code).decode()


def _call_device(*named):
    """The one CUDA device that every tensor of a call lives on.

    ``named`` holds (name, tensor) pairs; None tensors are skipped.  Raises
    ValueError, before anything is launched, when a tensor is on the host or
    on another device than the first one: the library works on the current
    device, so a pointer of another GPU would be handed to the wrong one.
    """
    dev = None
    for name, t in named:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the call's other tensors on {dev}")
    return dev


class _OnDevice:
    """Makes `device` current for a library call; a no-op (no context-manager
    round trip through torch) when it already is, the common case."""
    __slots__ = ("index", "prev")

    def __init__(self, device):
        self.index = device.index if device.index is not None else torch.cuda.current_device()
        self.prev = None

    def __enter__(self):
        cur = torch.cuda.current_device()
        if cur != self.index:
            self.prev = cur
            torch.cuda.set_device(self.index)
        return self

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)
        return False


def _stream_handle(stream, device) -> ctypes.c_void_p:
    """The stream of a call on ``device``: the given one (which must belong to
    that device) or the device's current torch stream."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif stream.device != device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    return ctypes.c_void_p(stream.cuda_stream)


def _matrix(t: torch.Tensor, name: str):
    """(pointer, row stride in elements, rows, cols) of a 2-D CUDA fp32/bf16 tensor."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in DTYPES:
        raise TypeError(f"{name} must be float32, bfloat16 or float16, not {t.dtype}")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} needs unit column stride")
    stride = t.stride(0) if t.shape[0] > 1 else t.shape[1]
    return t.data_ptr(), max(stride, t.shape[1]), t.shape[0], t.shape[1]


def _check(rc: int, where: str):
    if rc != OK:
        raise GbceError(rc, where)


def ce_fwd_bwd(logits: torch.Tensor, targets: torch.Tensor, ignore_index: int = -100,
               loss: torch.Tensor = None, stream=None) -> torch.Tensor:
    """Mean cross-entropy of ``logits`` [M, V] against int64 ``targets`` [M].

    ``logits`` is overwritten in place with d(loss)/d(logits).  Returns a
    0-dim float32 CUDA tensor (``loss`` when given); nothing is synchronised.
    """
    lp, stride, M, V = _matrix(logits, "logits")
    if targets.dtype != torch.int64 or targets.dim() != 1 or targets.shape[0] != M:
        raise ValueError("targets must be int64 of shape [M]")
    if M and (not targets.is_cuda or not targets.is_contiguous()):
        raise ValueError("targets must be a contiguous CUDA tensor")
    if loss is None:
        loss = torch.empty((), dtype=torch.float32, device=logits.device)
    elif loss.dtype != torch.float32 or loss.numel() != 1 or not loss.is_cuda:
        raise ValueError("loss must be a one-element float32 CUDA tensor")
    dev = _call_device(("logits", logits), ("targets", targets if M else None), ("loss", loss))
    with _OnDevice(dev):
        rc = load_library().ce_fwd_bwd(lp, stride, targets.data_ptr(), loss.data_ptr(), M, V,
                                       int(ignore_index), DTYPES[logits.dtype],
                                       _stream_handle(stream, dev))
    _check(rc, "ce_fwd_bwd")
    return loss


def _device_floats(v, n: int, device, name: str):
    """A float32 CUDA tensor of n values on `device` from a tensor or a number."""
    if not torch.is_tensor(v):
        v = torch.full((n,), float(v), dtype=torch.float32, device=device)
    if v.dtype != torch.float32 or not v.is_cuda or v.numel() != n or not v.is_contiguous():
        raise ValueError(f"{name} must be {n} contiguous float32 CUDA value(s)")
    return v


def ce_fwd_bwd_ex(logits: torch.Tensor, targets: torch.Tensor, ignore_index: int = -100,
                  reduction: str = "mean", grad_scale=None, want_row_loss: bool = False,
                  loss: torch.Tensor = None, row_loss: torch.Tensor = None, stream=None):
    """Cross-entropy with a reduction ('mean', 'sum', 'none'), optional per-row
    losses, and grad_scale (None, a number or a float32 CUDA tensor: one value,
    or one per row for 'none') folded into the in-place gradient.

    Returns (loss, row_loss): loss is a 0-dim float32 CUDA tensor (None for
    'none'); row_loss is [M] float32 when requested or for 'none', else None.
    """
    lp, stride, M, V = _matrix(logits, "logits")
    if reduction not in REDUCTIONS:
        raise ValueError(f"reduction must be one of {sorted(REDUCTIONS)}")
    if targets.dtype != torch.int64 or targets.dim() != 1 or targets.shape[0] != M:
        raise ValueError("targets must be int64 of shape [M]")
    if M and (not targets.is_cuda or not targets.is_contiguous()):
        raise ValueError("targets must be a contiguous CUDA tensor")
    dev = logits.device
    if reduction != "none" and loss is None:
        loss = torch.empty((), dtype=torch.float32, device=dev)
    if (want_row_loss or reduction == "none") and row_loss is None:
        row_loss = torch.empty((M,), dtype=torch.float32, device=dev)
    gs = None
    if grad_scale is not None:
        gs = _device_floats(grad_scale, M if reduction == "none" else 1, dev, "grad_scale")
    dev = _call_device(("logits", logits), ("targets", targets if M else None), ("loss", loss),
                       ("row_loss", row_loss), ("grad_scale", gs))
    with _OnDevice(dev):
        rc = load_library().ce_fwd_bwd_ex(
            lp, stride, targets.data_ptr(), None if loss is None else loss.data_ptr(),
            None if row_loss is None else row_loss.data_ptr(),
            None if gs is None else gs.data_ptr(), M, V, int(ignore_index),
            DTYPES[logits.dtype], REDUCTIONS[reduction], _stream_handle(stream, dev))
    _check(rc, "ce_fwd_bwd_ex")
    return (None if reduction == "none" else loss), row_loss


def scale_rows(x: torch.Tensor, scale, stream=None) -> torch.Tensor:
    """x *= scale in place; scale is a number, a one-element float32 CUDA tensor,
    or one value per row ([M]).  A single scale of 1 costs only the launch."""
    xp, stride, M, N = _matrix(x, "x")
    per_row = torch.is_tensor(scale) and scale.numel() == M and M != 1
    sc = _device_floats(scale, M if per_row else 1, x.device, "scale")
    dev = _call_device(("x", x), ("scale", sc))
    with _OnDevice(dev):
        rc = load_library().scale_rows(xp, stride, M, N, DTYPES[x.dtype], sc.data_ptr(),
                                       1 if per_row else 0, _stream_handle(stream, dev))
    _check(rc, "scale_rows")
    return x


class FusedCrossEntropy(torch.autograd.Function):
    """Autograd form of the fused call (the behaviour of Liger-Kernel's
    LigerCrossEntropyFunction): the forward computes the loss and writes the
    gradient into the logits' storage, which it saves; the backward scales that
    gradient in place by grad_output (a device-side no-op when it is 1, so no
    host synchronisation) and returns it.  The logits' values are consumed:
    read them before this call, and call backward once.
    """

    @staticmethod
    def forward(ctx, logits, targets, ignore_index=-100, reduction="mean"):
        buf = logits.detach()
        loss, row_loss = ce_fwd_bwd_ex(buf, targets, ignore_index, reduction)
        ctx.save_for_backward(buf)
        ctx.reduction = reduction
        return row_loss if reduction == "none" else loss

    @staticmethod
    def backward(ctx, grad_output):
        (grad,) = ctx.saved_tensors
        scale_rows(grad, grad_output.detach().to(torch.float32).contiguous().reshape(-1))
        return grad, None, None, None


def cross_entropy(logits: torch.Tensor, targets: torch.Tensor, ignore_index: int = -100,
                  reduction: str = "mean", inplace: bool = True) -> torch.Tensor:
    """Hard-label cross-entropy of [M, V] logits, differentiable.  With
    inplace=True the logits' storage is reused for the gradient (no extra
    M x V buffer); with inplace=False the logits are copied first."""
    if not inplace:
        logits = logits.clone(memory_format=torch.contiguous_format)
    return FusedCrossEntropy.apply(logits, targets, ignore_index, reduction)


class CrossEntropyLoss(torch.nn.Module):
    """nn.Module form of cross_entropy (hard labels, ignore_index, reduction)."""

    def __init__(self, ignore_index: int = -100, reduction: str = "mean", inplace: bool = True):
        super().__init__()
        if reduction not in REDUCTIONS:
            raise ValueError(f"reduction must be one of {sorted(REDUCTIONS)}")
        self.ignore_index, self.reduction, self.inplace = ignore_index, reduction, inplace

    def forward(self, logits, targets):
        return cross_entropy(logits, targets, self.ignore_index, self.reduction, self.inplace)


def _status_word(status, name="status"):
    """Device address of a per-call status word: a CUDA int32 tensor of one element."""
    if status is None:
        return None
    if not status.is_cuda or status.dtype != torch.int32 or status.numel() != 1:
        raise ValueError(f"{name} must be a one-element int32 CUDA tensor")
    return status.data_ptr()


def softmax_fwd(x: torch.Tensor, y: torch.Tensor = None, stream=None) -> torch.Tensor:
    """Row softmax of ``x`` [M, N] into ``y`` (allocated when None; may be ``x``)."""
    return softmax_fwd_ex(x, y, None, stream)


def softmax_fwd_ex(x: torch.Tensor, y: torch.Tensor = None, status: torch.Tensor = None,
                   stream=None) -> torch.Tensor:
    """softmax_fwd with a status word of the call's own: ``status`` (a one-element
    int32 CUDA tensor the caller cleared) gets STATUS_TIMEOUT when one of the
    call's bounded waits gave up."""
    if y is None:
        y = torch.empty_like(x, memory_format=torch.contiguous_format)
    xp, xs, M, N = _matrix(x, "x")
    yp, ys, My, Ny = _matrix(y, "y")
    if (My, Ny) != (M, N) or y.dtype != x.dtype:
        raise ValueError("y must match x in shape and dtype")
    sp = _status_word(status)
    dev = _call_device(("x", x), ("y", y), ("status", status))
    with _OnDevice(dev):
        rc = load_library().softmax_fwd_ex(xp, xs, yp, ys, M, N, DTYPES[x.dtype], sp,
                                           _stream_handle(stream, dev))
    _check(rc, "softmax_fwd")
    return y


def softmax_bwd(y: torch.Tensor, dy: torch.Tensor, dx: torch.Tensor = None,
                stream=None) -> torch.Tensor:
    """dx = y * (dy - sum(y * dy, row)) for [M, N] operands (dx may be ``dy``)."""
    return softmax_bwd_ex(y, dy, dx, None, stream)


def softmax_bwd_ex(y: torch.Tensor, dy: torch.Tensor, dx: torch.Tensor = None,
                   status: torch.Tensor = None, stream=None) -> torch.Tensor:
    """softmax_bwd with a status word of the call's own (as softmax_fwd_ex)."""
    if dx is None:
        dx = torch.empty_like(dy, memory_format=torch.contiguous_format)
    yp, ys, M, N = _matrix(y, "y")
    dp, ds, Md, Nd = _matrix(dy, "dy")
    xp, xs, Mx, Nx = _matrix(dx, "dx")
    if (Md, Nd) != (M, N) or (Mx, Nx) != (M, N) or not (y.dtype == dy.dtype == dx.dtype):
        raise ValueError("y, dy and dx must share shape and dtype")
    sp = _status_word(status)
    dev = _call_device(("y", y), ("dy", dy), ("dx", dx), ("status", status))
    with _OnDevice(dev):
        rc = load_library().softmax_bwd_ex(yp, ys, dp, ds, xp, xs, M, N, DTYPES[y.dtype], sp,
                                           _stream_handle(stream, dev))
    _check(rc, "softmax_bwd")
    return dx


def softmax_bwd_bsr(y: torch.Tensor, dy: torch.Tensor, lut: torch.Tensor, n_block_rows: int,
                    nblocks: int, block: int, sizemax: int, scale: float = 1.0,
                    dx: torch.Tensor = None, stream=None) -> torch.Tensor:
    """Block-sparse softmax backward, dx = y * (dy - sum(y * dy)) * scale per row.

    ``y``, ``dy`` and ``dx`` are [Z, zstride] CUDA tensors (unit inner stride)
    whose first nblocks * block^2 elements per batch item hold the blocks;
    ``lut`` is the int32 look-up table (a contiguous CUDA tensor).  ``dx``
    defaults to ``dy`` (in place, as the page's kernel stores); only the
    positions the table names are written.
    """
    return softmax_bwd_bsr_ex(y, dy, lut, n_block_rows, nblocks, block, sizemax, scale, dx,
                              None, stream)


def softmax_bwd_bsr_ex(y: torch.Tensor, dy: torch.Tensor, lut: torch.Tensor, n_block_rows: int,
                       nblocks: int, block: int, sizemax: int, scale: float = 1.0,
                       dx: torch.Tensor = None, status: torch.Tensor = None,
                       stream=None) -> torch.Tensor:
    """softmax_bwd_bsr with a status word of the call's own: ``status`` (a
    one-element int32 CUDA tensor the caller cleared) gets STATUS_BAD_TABLE when
    the call finds a malformed table entry."""
    if dx is None:
        dx = dy
    yp, ys, Z, Ly = _matrix(y, "y")
    dp, ds, Zd, Ld = _matrix(dy, "dy")
    xp, xs, Zx, Lx = _matrix(dx, "dx")
    if Zd != Z or Zx != Z or not (y.dtype == dy.dtype == dx.dtype):
        raise ValueError("y, dy and dx must share the batch size and dtype")
    if min(Ly, Ld, Lx) < nblocks * block * block:
        raise ValueError("y, dy and dx must hold nblocks * block^2 elements per batch item")
    if lut.dtype != torch.int32 or lut.dim() != 1 or not lut.is_cuda or not lut.is_contiguous():
        raise ValueError("lut must be a contiguous 1-D int32 CUDA tensor")
    sp = _status_word(status)
    dev = _call_device(("y", y), ("dy", dy), ("dx", dx), ("lut", lut), ("status", status))
    with _OnDevice(dev):
        rc = load_library().softmax_bwd_bsr_ex(yp, ys, dp, ds, xp, xs, lut.data_ptr(), lut.numel(),
                                               n_block_rows, nblocks, block, sizemax, Z,
                                               float(scale), DTYPES[y.dtype], sp,
                                               _stream_handle(stream, dev))
    _check(rc, "softmax_bwd_bsr")
    return dx


def bsr_plan(block: int, sizemax: int, dtype: torch.dtype, aligned: bool = True):
    """(kernel name, rows per slab of a block-row of sizemax blocks) that
    softmax_bwd_bsr uses for this block size, longest block-row and dtype."""
    r = ctypes.c_int(0)
    name = load_library().gbce_bsr_plan(block, sizemax, DTYPES[dtype], 1 if aligned else 0,
                                        ctypes.byref(r))
    if name is None:
        raise ValueError("invalid block-sparse plan query")
    return name.decode(), r.value


def plan(op: str, M: int, cols: int, dtype: torch.dtype, same_phase: bool = True):
    """(row-kernel family, CTAs per row) the library picks for M rows of `cols`
    elements on the current device; op is 'ce', 'softmax_fwd' or 'softmax_bwd'.
    M matters only for batches of at most one row per SM (gbce_plan)."""
    c = ctypes.c_int(0)
    name = load_library().gbce_plan({"ce": 0, "softmax_fwd": 1, "softmax_bwd": 2}[op], M, cols,
                                    DTYPES[dtype], 1 if same_phase else 0, ctypes.byref(c))
    if name is None:
        raise ValueError("invalid plan query")
    return name.decode(), c.value


def last_error(stream=None) -> int:
    """Synchronise the stream and read-and-clear the error flags of its device
    (the current device when no stream is given)."""
    dev = stream.device if stream is not None else torch.device("cuda", torch.cuda.current_device())
    with _OnDevice(dev):
        return load_library().gbce_last_error(_stream_handle(stream, dev))


def timing_enable(on: bool = True):
    _check(load_library().gbce_timing_enable(1 if on else 0), "gbce_timing_enable")


def timing_read():
    """(summed row-kernel milliseconds, bracketed launches) since the last read."""
    ms, n = ctypes.c_double(), ctypes.c_int64()
    _check(load_library().gbce_timing_read(ctypes.byref(ms), ctypes.byref(n)), "gbce_timing_read")
    return ms.value, n.value


def ce_fwd_bwd_host(logits_host: torch.Tensor, targets_host: torch.Tensor,
                    ignore_index: int = -100, grad: torch.Tensor = None,
                    loss_host: torch.Tensor = None, stream=None):
    """ce_fwd_bwd from host memory: (grad, loss_host).

    ``logits_host`` [M, V] and ``targets_host`` [M] (int64) are CPU tensors
    (pinned memory makes the copies asynchronous).  ``grad`` is a CUDA tensor of
    the logits' shape and dtype (allocated when not given) that receives the
    logits and then, in place, the gradient; ``loss_host`` is a one-element
    CPU float32 tensor (pinned when allocated here) that holds the mean loss
    once the stream has reached the end of the call.
    """
    if logits_host.is_cuda or targets_host.is_cuda:
        raise ValueError("logits_host and targets_host must be CPU tensors")
    if logits_host.dim() != 2 or (logits_host.shape[1] > 1 and logits_host.stride(1) != 1):
        raise ValueError("logits_host must be 2-D with unit column stride")
    if logits_host.dtype not in DTYPES:
        raise TypeError(f"logits_host must be float32, bfloat16 or float16, not {logits_host.dtype}")
    M, V = logits_host.shape
    if targets_host.dtype != torch.int64 or targets_host.shape != (M,) or \
            not targets_host.is_contiguous():
        raise ValueError("targets_host must be a contiguous int64 tensor of shape [M]")
    hs = logits_host.stride(0) if M > 1 else V
    if grad is None:
        grad = torch.empty((M, V), dtype=logits_host.dtype, device="cuda")
    gp, gs, Mg, Vg = _matrix(grad, "grad")
    if (Mg, Vg) != (M, V) or grad.dtype != logits_host.dtype:
        raise ValueError("grad must match the logits' shape and dtype")
    if loss_host is None:
        loss_host = torch.empty((), dtype=torch.float32).pin_memory()
    elif loss_host.dtype != torch.float32 or loss_host.numel() != 1 or loss_host.is_cuda:
        raise ValueError("loss_host must be a one-element float32 CPU tensor")
    lib = load_library()
    fn = lib.ce_fwd_bwd_host
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                   ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    dev = _call_device(("grad", grad))
    with _OnDevice(dev):
        rc = fn(logits_host.data_ptr(), max(hs, V), targets_host.data_ptr(), gp, gs,
                loss_host.data_ptr(), M, V, int(ignore_index), DTYPES[logits_host.dtype],
                _stream_handle(stream, dev))
    _check(rc, "ce_fwd_bwd_host")
    return grad, loss_host


def ce_fwd_bwd_noalloc(logits: torch.Tensor, targets: torch.Tensor, ignore_index: int = -100,
                       loss: torch.Tensor = None, stream=None) -> torch.Tensor:
    """ce_fwd_bwd for callers that cannot let the library allocate device memory.

    Same results; the temporary storage is a fixed static device array inside
    the library (M <= 65536 rows), shared by every call on the device, so
    calls that overlap on the GPU must be serialised by the caller.  ``loss``
    is allocated here by torch when not given.
    """
    lp, stride, M, V = _matrix(logits, "logits")
    if targets.dtype != torch.int64 or targets.dim() != 1 or targets.shape[0] != M:
        raise ValueError("targets must be int64 of shape [M]")
    if M and (not targets.is_cuda or not targets.is_contiguous()):
        raise ValueError("targets must be a contiguous CUDA tensor")
    if loss is None:
        loss = torch.empty((), dtype=torch.float32, device=logits.device)
    elif loss.dtype != torch.float32 or loss.numel() != 1 or not loss.is_cuda:
        raise ValueError("loss must be a one-element float32 CUDA tensor")
    dev = _call_device(("logits", logits), ("targets", targets if M else None), ("loss", loss))
    fn = load_library().ce_fwd_bwd_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    with _OnDevice(dev):
        rc = fn(lp, stride, targets.data_ptr(), loss.data_ptr(), M, V, int(ignore_index),
                DTYPES[logits.dtype], _stream_handle(stream, dev))
    _check(rc, "ce_fwd_bwd_noalloc")
    return loss
