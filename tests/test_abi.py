"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
entry point declared in include/gbce.h, and rejects bad arguments on the host
(before any CUDA call, so this runs on a machine without a GPU)."""
import ctypes
import os
import re

import pytest

from cross_entropy_loss_ce_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbce.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*GBCE_API\s+(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\([^;]*\)\s*;", text, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    path = gbuild.build()
    lib = ctypes.CDLL(path)
    i64, p, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.ce_fwd_bwd.argtypes = [p, i64, p, p, i64, i64, i64, ci, p]
    lib.softmax_fwd.argtypes = [p, i64, p, i64, i64, i64, ci, p]
    lib.softmax_bwd.argtypes = [p, i64, p, i64, p, i64, i64, i64, ci, p]
    lib.softmax_fwd_ex.argtypes = [p, i64, p, i64, i64, i64, ci, p, p]
    lib.softmax_bwd_ex.argtypes = [p, i64, p, i64, p, i64, i64, i64, ci, p, p]
    lib.ce_fwd_bwd_ex.argtypes = [p, i64, p, p, p, p, i64, i64, i64, ci, ci, p]
    lib.scale_rows.argtypes = [p, i64, i64, i64, ci, p, ci, p]
    lib.gbce_status_string.restype = ctypes.c_char_p
    lib.softmax_bwd_bsr.argtypes = [p, i64, p, i64, p, i64, p, i64, i64, i64, i64, i64, i64,
                                    ctypes.c_float, ci, p]
    lib.softmax_bwd_bsr_ex.argtypes = [p, i64, p, i64, p, i64, p, i64, i64, i64, i64, i64, i64,
                                       ctypes.c_float, ci, p, p]
    lib.gbce_bsr_plan.argtypes = [i64, i64, ci, ci, ctypes.POINTER(ci)]
    lib.gbce_bsr_plan.restype = ctypes.c_char_p
    return lib


def test_header_declares_the_boundary():
    names = set(declared_functions())
    assert {"ce_fwd_bwd", "softmax_fwd", "softmax_bwd", "gbce_last_error",
            "gbce_status_string", "gbce_timing_enable", "gbce_timing_read", "ce_fwd_bwd_ex",
            "scale_rows", "softmax_bwd_bsr", "gbce_bsr_plan", "ce_fwd_bwd_noalloc",
            "ce_fwd_bwd_host", "gbce_pool_reserved", "gbce_test_failure_path",
            "softmax_fwd_ex", "softmax_bwd_ex", "softmax_bwd_bsr_ex"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in gbce.h but not exported"


def test_only_the_abi_is_exported(lib):
    # hidden visibility: nothing but the declared C names (and runtime-internal
    # symbols, if any) should be visible; spot-check a kernel name is not.
    assert not hasattr(lib, "_ZN4gbce14ce_mean_kernelILi1024EEEvPKflPKiPf")


def test_status_strings(lib):
    for code in range(11):
        s = lib.gbce_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.gbce_status_string(99).decode() == "unknown status"


FAKE = 0x10000  # never dereferenced: every call below is rejected on the host


@pytest.mark.parametrize("args,code", [
    # (logits, stride, targets, loss, M, V, ignore_index, dtype) -> status
    ((None, 10, FAKE, FAKE, 4, 10, -100, 0), 1),        # NULL logits
    ((FAKE, 10, None, FAKE, 4, 10, -100, 0), 1),        # NULL targets
    ((FAKE, 10, FAKE, None, 4, 10, -100, 0), 1),        # NULL loss
    ((FAKE, 10, FAKE, FAKE, 4, 0, -100, 0), 2),         # V < 1
    ((FAKE, 9, FAKE, FAKE, 4, 10, -100, 0), 2),         # stride < V
    ((FAKE, 10, FAKE, FAKE, -1, 10, -100, 0), 2),       # M < 0
    ((FAKE, 10, FAKE, FAKE, 4, 2**31, -100, 0), 2),     # V beyond int32
    ((FAKE, 10, FAKE, FAKE, 4, 10, -100, 3), 3),        # unknown dtype
    ((FAKE + 2, 10, FAKE, FAKE, 4, 10, -100, 0), 4),    # fp32 logits not 4-byte aligned
    ((FAKE + 1, 10, FAKE, FAKE, 4, 10, -100, 1), 4),    # bf16 logits not 2-byte aligned
    ((FAKE, 10, FAKE + 4, FAKE, 4, 10, -100, 0), 4),    # targets not 8-byte aligned
])
def test_ce_rejects_bad_arguments(lib, args, code):
    assert lib.ce_fwd_bwd(*args, None) == code


@pytest.mark.parametrize("args,code", [
    ((None, 8, FAKE, 8, 2, 8, 0), 1),
    ((FAKE, 8, None, 8, 2, 8, 0), 1),
    ((FAKE, 7, FAKE, 8, 2, 8, 0), 2),
    ((FAKE, 8, FAKE, 7, 2, 8, 0), 2),
    ((FAKE, 8, FAKE, 8, 2, 0, 0), 2),
    ((FAKE, 8, FAKE, 8, 2, 8, 5), 3),
    ((FAKE + 1, 8, FAKE, 8, 2, 8, 2), 4),      # fp16 x not 2-byte aligned
    ((FAKE + 2, 8, FAKE, 8, 2, 8, 0), 4),
])
def test_softmax_fwd_rejects_bad_arguments(lib, args, code):
    assert lib.softmax_fwd(*args, None) == code


@pytest.mark.parametrize("args,code", [
    ((None, 8, FAKE, 8, FAKE, 8, 2, 8, 0), 1),
    ((FAKE, 8, None, 8, FAKE, 8, 2, 8, 0), 1),
    ((FAKE, 8, FAKE, 8, None, 8, 2, 8, 0), 1),
    ((FAKE, 8, FAKE, 6, FAKE, 8, 2, 8, 0), 2),
    ((FAKE, 8, FAKE, 8, FAKE, 8, -3, 8, 0), 2),
    ((FAKE, 8, FAKE, 8, FAKE, 8, 2, 8, -1), 3),
    ((FAKE, 8, FAKE, 8, FAKE + 1, 8, 2, 8, 1), 4),
])
def test_softmax_bwd_rejects_bad_arguments(lib, args, code):
    assert lib.softmax_bwd(*args, None) == code


def test_softmax_ex_checks_its_status_word(lib):
    # the _ex forms take the same arguments plus a status word: checked like
    # the others, and a word off its 4-byte alignment is rejected before any launch
    assert lib.softmax_fwd_ex(None, 8, FAKE, 8, 2, 8, 0, None, None) == 1
    assert lib.softmax_fwd_ex(FAKE, 8, FAKE, 8, 2, 8, 0, FAKE + 2, None) == 4
    assert lib.softmax_bwd_ex(FAKE, 8, FAKE, 8, FAKE, 8, 2, 8, 0, FAKE + 1, None) == 4
    assert lib.softmax_bwd_ex(FAKE, 6, FAKE, 8, FAKE, 8, 2, 8, 0, FAKE, None) == 2
    assert lib.softmax_fwd_ex(None, 8, None, 8, 0, 8, 0, FAKE, None) == 0  # M = 0
    assert lib.softmax_bwd_ex(None, 8, None, 8, None, 8, 0, 8, 1, FAKE, None) == 0
    # the block-sparse form: a status word off its alignment, after the shape checks
    bsr = (FAKE, 64, FAKE, 64, FAKE, 64, FAKE, 6, 1, 4, 4, 1, 1, 1.0, 0)
    assert lib.softmax_bwd_bsr_ex(*bsr, FAKE + 2, None) == 4
    assert lib.softmax_bwd_bsr_ex(FAKE, 64, FAKE, 64, FAKE, 64, FAKE, 6, 1, 4, 3, 1, 1, 1.0, 0,
                                  FAKE, None) == 2  # block 3 is not a power of two


def test_empty_softmax_is_a_noop(lib):
    # M == 0 returns success without touching the device
    assert lib.softmax_fwd(None, 8, None, 8, 0, 8, 0, None) == 0
    assert lib.softmax_bwd(None, 8, None, 8, None, 8, 0, 8, 1, None) == 0


@pytest.mark.parametrize("args,code", [
    # (logits, stride, targets, loss, row_loss, grad_scale, M, V, ii, dtype, reduction) -> status
    ((FAKE, 10, FAKE, FAKE, None, None, 4, 10, -100, 0, 3), 9),      # unknown reduction
    ((FAKE, 10, FAKE, None, None, None, 4, 10, -100, 0, 0), 1),      # mean needs loss
    ((FAKE, 10, FAKE, None, None, None, 4, 10, -100, 0, 1), 1),      # sum needs loss
    ((FAKE, 10, FAKE, None, None, None, 4, 10, -100, 0, 2), 1),      # none needs row_loss
    ((FAKE, 10, FAKE, FAKE, FAKE + 8, None, 4, 10, -100, 0, 0), 4),  # row_loss not 16-aligned
    ((FAKE, 10, FAKE, FAKE, None, FAKE + 2, 4, 10, -100, 0, 0), 4),  # grad_scale not 4-aligned
    ((FAKE, 10, FAKE, FAKE, None, None, 4, 10, -100, 5, 0), 3),      # unknown dtype
    ((FAKE, 9, FAKE, FAKE, None, None, 4, 10, -100, 0, 0), 2),       # stride < V
])
def test_ce_ex_rejects_bad_arguments(lib, args, code):
    assert lib.ce_fwd_bwd_ex(*args, None) == code


@pytest.mark.parametrize("args,code", [
    # (x, stride, M, N, dtype, scale, per_row) -> status
    ((None, 8, 2, 8, 0, FAKE, 0), 1),
    ((FAKE, 8, 2, 8, 0, None, 0), 1),
    ((FAKE, 7, 2, 8, 0, FAKE, 0), 2),
    ((FAKE, 8, 2, 8, 4, FAKE, 0), 3),
    ((FAKE, 8, 2, 8, 0, FAKE + 1, 0), 4),
])
def test_scale_rows_rejects_bad_arguments(lib, args, code):
    assert lib.scale_rows(*args, None) == code


def test_empty_calls_are_noops(lib):
    assert lib.scale_rows(None, 8, 0, 8, 0, None, 0, None) == 0


def test_plan_picks_the_regime_by_row_length(lib):
    """Host-side plan (no device here, so no cluster split and no small-batch
    plan, whatever M): warp rows up to 8 KB per operand, resident up to 64 KB
    staged (32 KB for the softmax forward), ring beyond, streaming when
    operands' rows sit at different 16-byte phases."""
    lib.gbce_plan.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                              ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    lib.gbce_plan.restype = ctypes.c_char_p
    c = ctypes.c_int()

    def plan(op, cols, dtype, same=1, M=4096):
        return lib.gbce_plan(op, M, cols, dtype, same, ctypes.byref(c)).decode()

    assert plan(0, 1000, 0) == "rows_warp_kernel"          # 4000 B fp32
    assert plan(0, 2048, 0) == "rows_warp_kernel"          # exactly 8 KB
    assert plan(0, 2052, 0) == "rows_resident_kernel"
    assert plan(0, 32000, 1) == "rows_resident_kernel"     # 64000 B bf16
    assert plan(0, 32000, 1, M=1) == "rows_resident_kernel"
    assert plan(0, 32768, 1) == "rows_resident_kernel"     # exactly 64 KB
    assert plan(0, 32776, 1) == "rows_ring_kernel"
    assert plan(2, 8192, 0) == "rows_resident_kernel"      # two 32 KB operands: 64 KB
    assert plan(2, 8196, 0) == "rows_ring_kernel"
    assert plan(1, 8192, 0) == "rows_resident_kernel"      # softmax forward: 32 KB
    assert plan(1, 8196, 0) == "rows_ring_kernel"
    assert plan(1, 16384, 0) == "rows_ring_kernel"         # 64 KB fp32 forward rows
    assert plan(1, 8192, 0, same=0) == "rows_streaming_kernel"
    assert plan(0, 128256, 2) == "rows_ring_kernel"        # fp16
    assert plan(0, 128256, 2, M=0) == "rows_ring_kernel"
    assert c.value == 1
    assert lib.gbce_plan(3, 1, 10, 0, 1, None) is None
    assert lib.gbce_plan(0, 1, 0, 0, 1, None) is None
    assert lib.gbce_plan(0, 1, 10, 7, 1, None) is None
    assert lib.gbce_plan(0, -1, 10, 0, 1, None) is None


def test_size_limits(lib):
    # stride beyond 2^46 elements and M beyond 2^27 - 1 rows are rejected on the host
    assert lib.ce_fwd_bwd(FAKE, 2 ** 47, FAKE, FAKE, 4, 10, -100, 0, None) == 2
    assert lib.ce_fwd_bwd(FAKE, 10, FAKE, FAKE, 2 ** 27, 10, -100, 0, None) == 2
    assert lib.softmax_fwd(FAKE, 2 ** 47, FAKE, 8, 2, 8, 0, None) == 2


# softmax_bwd_bsr(y, ys, dy, dys, dx, dxs, lut, lut_len, n_block_rows, nblocks, block,
#                 sizemax, Z, scale, dtype)
BSR_OK = (FAKE, 4096, FAKE, 4096, FAKE, 4096, FAKE, 16, 4, 4, 32, 2, 2, 1.0, 0)


def _bsr(**kw):
    names = ["y", "ys", "dy", "dys", "dx", "dxs", "lut", "lut_len", "nbr", "nblocks", "block",
             "sizemax", "Z", "scale", "dtype"]
    a = dict(zip(names, BSR_OK))
    a.update(kw)
    return tuple(a[n] for n in names)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=3), 3),
    (dict(block=3), 2), (dict(block=0), 2), (dict(block=2048), 2),
    (dict(Z=-1), 2), (dict(nbr=-1), 2), (dict(nblocks=-1), 2), (dict(sizemax=-1), 2),
    (dict(lut_len=7), 2),                                # fewer than 2 ints per block-row
    (dict(ys=4095), 2), (dict(dxs=100), 2),              # batch stride < nblocks * block^2
    (dict(sizemax=2**26), 2),                            # sizemax * block >= 2^31
    (dict(Z=2**40, ys=2**20, dys=2**20, dxs=2**20), 2),  # beyond a 1-D grid
    (dict(y=None), 1), (dict(dx=None), 1), (dict(lut=None), 1),
    (dict(y=FAKE + 2), 4), (dict(lut=FAKE + 2), 4), (dict(dtype=1, dy=FAKE + 1), 4),
    (dict(Z=0, y=None, lut=None), 0), (dict(nbr=0, lut_len=0, lut=None), 0),
    (dict(sizemax=0, y=None), 0),
])
def test_bsr_rejects_bad_arguments(lib, kw, code):
    assert lib.softmax_bwd_bsr(*_bsr(**kw), None) == code


@pytest.mark.parametrize("block,sizemax,dtype,aligned,kernel,rows", [
    (32, 128, 0, 1, "bsr_bwd_staged_kernel", 1),       # causal S=4096: 32 KB per row
    (64, 25, 1, 1, "bsr_bwd_staged_kernel", 4),        # random S=8192 bf16
    (16, 2, 0, 1, "bsr_bwd_staged_kernel", 16),        # tiny rows: as many as the block has
    (128, 1, 2, 1, "bsr_bwd_staged_kernel", 64),       # capped at 64 rows per CTA
    (32, 1000, 0, 1, "bsr_bwd_unstaged_kernel", 1),    # 256 KB per row: not staged
    (32, 390, 0, 1, "bsr_bwd_staged_kernel", 1),       # two stages of 101 KB fit 200 KB
    (32, 400, 0, 1, "bsr_bwd_unstaged_kernel", 1),     # two stages of 104 KB do not
    (2, 3, 0, 1, "bsr_bwd_staged_kernel (element accesses)", 2),   # 8-byte block rows
    (32, 8, 1, 0, "bsr_bwd_staged_kernel (element accesses)", 32),
])
def test_bsr_plan(lib, block, sizemax, dtype, aligned, kernel, rows):
    r = ctypes.c_int(0)
    name = lib.gbce_bsr_plan(block, sizemax, dtype, aligned, ctypes.byref(r))
    assert name.decode() == kernel and r.value == rows
    assert lib.gbce_bsr_plan(3, 1, 0, 1, None) is None
    assert lib.gbce_bsr_plan(32, 0, 0, 1, None) is None


# ce_fwd_bwd_host(logits_host, host_stride, targets_host, grad, stride, loss_host, M, V,
#                 ignore_index, dtype)
@pytest.mark.parametrize("args,code", [
    ((FAKE, 10, FAKE, FAKE, 10, None, 4, 10, -100, 0), 1),       # NULL loss_host
    ((None, 10, FAKE, FAKE, 10, FAKE, 4, 10, -100, 0), 1),       # NULL logits_host
    ((FAKE, 10, None, FAKE, 10, FAKE, 4, 10, -100, 0), 1),       # NULL targets_host
    ((FAKE, 10, FAKE, None, 10, FAKE, 4, 10, -100, 0), 1),       # NULL grad
    ((FAKE, 9, FAKE, FAKE, 10, FAKE, 4, 10, -100, 0), 2),        # host stride < V
    ((FAKE, 10, FAKE, FAKE, 9, FAKE, 4, 10, -100, 0), 2),        # device stride < V
    ((FAKE, 10, FAKE, FAKE, 10, FAKE, -1, 10, -100, 0), 2),      # M < 0
    ((FAKE, 10, FAKE, FAKE, 10, FAKE, 4, 10, -100, 3), 3),       # unknown dtype
    ((FAKE + 2, 10, FAKE, FAKE, 10, FAKE, 4, 10, -100, 0), 4),   # host logits misaligned
    ((FAKE, 10, FAKE + 4, FAKE, 10, FAKE, 4, 10, -100, 0), 4),   # host targets misaligned
    ((FAKE, 10, FAKE, FAKE, 10, FAKE + 2, 4, 10, -100, 0), 4),   # loss_host misaligned
])
def test_ce_host_rejects_bad_arguments(lib, args, code):
    i64, p, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.ce_fwd_bwd_host.argtypes = [p, i64, p, p, i64, p, i64, i64, i64, ci, p]
    assert lib.ce_fwd_bwd_host(*args, None) == code


def test_pool_query_on_the_host(lib):
    """No call has needed the scratch pool in this process: 0 bytes, no CUDA call."""
    fn = lib.gbce_pool_reserved
    fn.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_uint64)]
    v = ctypes.c_uint64(77)
    assert fn(0, ctypes.byref(v)) == 0 and v.value == 0
    assert fn(0, None) == 1                      # NULL output
    assert fn(-1, ctypes.byref(v)) == 2          # no such device slot
    assert fn(64, ctypes.byref(v)) == 2


def test_failure_hook_arguments(lib):
    fn = lib.gbce_test_failure_path
    fn.argtypes = [ctypes.c_int64]
    assert fn(2 ** 40) == 2                      # beyond a 32-bit copy count
    assert fn(-7) == 0                           # any negative value: no copy left out
    assert fn(-1) == 0
