"""CUDA block-sparse softmax backward (look-up table, scale) against the
double-precision oracle (GPU)."""
import numpy as np
import pytest
import torch

import cross_entropy_loss_ce_gb300 as gbce
import oracle
import workloads
from gpu_util import host, require_gpu
from parity import check_bsr

pytestmark = pytest.mark.gpu

DTYPES = [torch.float32, torch.bfloat16, torch.float16]


def table_rows(lut: np.ndarray, nbr: int, nblocks: int):
    """Block-row of every block named by a (valid) table; -1 for unnamed blocks."""
    brow = np.full(nblocks, -1, dtype=np.int64)
    for r in range(nbr):
        size, off = int(lut[2 * r]), int(lut[2 * r + 1])
        brow[lut[off:off + 4 * size:4]] = r
    return brow


def row_abs_sums(y64, dy64, brow, nbr, block):
    """[Z, nblocks * block^2]: for each element, sum over its matrix row of |y dy|."""
    Z = y64.shape[0]
    nb = brow.size
    a = np.abs(y64 * dy64).reshape(Z, nb, block, block).sum(-1)       # [Z, nb, block]
    s = np.zeros((Z, nbr + 1, block))
    np.add.at(s, (slice(None), brow), a)
    per = s[:, brow, :]                                              # [Z, nb, block]
    return np.broadcast_to(per[..., None], (Z, nb, block, block)).reshape(Z, -1)


def widened(t: torch.Tensor, L: int) -> np.ndarray:
    return oracle.widen(host(t[:, :L]))


def run_and_check(y, dy, lut, meta, scale, dtype, dx=None, what="bsr"):
    """Run the CUDA op (dx defaults to dy: in place) and compare every named
    element with the oracle; returns the result on the host as float64."""
    nbr, nblocks, block, sizemax = (meta["n_block_rows"], meta["nblocks"], meta["block"],
                                    meta["sizemax"])
    L = nblocks * block * block
    lut_h = lut.cpu().numpy()
    ref, bad = oracle.softmax_bwd_bsr(host(y), host(dy), lut_h, nbr, nblocks, block, sizemax,
                                      scale)
    assert bad == 0
    y64, dy64 = widened(y, L), widened(dy, L)
    yd, dyd, lutd = y.cuda(), dy.cuda(), lut.cuda()
    out = gbce.softmax_bwd_bsr(yd, dyd, lutd, nbr, nblocks, block, sizemax, scale,
                               dx=None if dx is None else dx.cuda())
    assert gbce.last_error() == gbce.OK
    got = widened(out, L)
    brow = table_rows(lut_h, nbr, nblocks)
    named = np.repeat(brow >= 0, block * block)
    check_bsr(got[:, named], ref[:, named], y64[:, named],
              row_abs_sums(y64, dy64, brow, nbr, block)[:, named], scale, dtype, what)
    return got, out


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("name,sizes,scale", [
    ("bsr_f32_causal_2x16x4096_b32", dict(H=2, S=512), 1.0),
    ("bsr_bf16_random_4x8x8192_b64", dict(Z=2, H=2, S=1024), 0.125),
])
def test_bsr_reduced(dtype, name, sizes, scale):
    require_gpu()
    w = workloads.BSR_WORKLOADS[name].with_sizes(dtype=dtype, **sizes)
    y, dy, lut, meta = workloads.make_bsr_inputs(w)
    run_and_check(y, dy, lut, meta, scale, dtype, what=f"{name} {dtype}")


def _sub_problem(y, dy, lut_h, meta, rows):
    """The listed block-rows as a small problem of their own: their blocks
    gathered in order and a table over the new block ids."""
    block = meta["block"]
    bb = block * block
    ids, header, entries = [], [], []
    for r in rows:
        size, off = int(lut_h[2 * r]), int(lut_h[2 * r + 1])
        blocks = lut_h[off:off + 4 * size:4]
        header += [size, 2 * len(rows) + 4 * len(ids)]
        for b in blocks:
            entries += [len(ids), 0, 0, 0]
            ids.append(int(b))
    idx = (np.asarray(ids)[:, None] * bb + np.arange(bb)[None, :]).reshape(-1)
    sub_lut = np.asarray(header + entries, dtype=np.int32)
    return idx, sub_lut, len(ids)


@pytest.mark.parametrize("name", list(workloads.BSR_WORKLOADS))
def test_bsr_full_size_sampled(name):
    """The whole workload on the GPU in the benchmark's launch configuration;
    block-rows sampled for the oracle (first, last and 22 at random)."""
    require_gpu()
    w = workloads.BSR_WORKLOADS[name]
    y, dy, lut, meta = workloads.make_bsr_inputs(w, device="cuda")
    nbr, block = meta["n_block_rows"], meta["block"]
    lut_h = lut.cpu().numpy()
    rows = np.unique(np.concatenate([[0, nbr - 1],
                                     np.random.default_rng(7).choice(nbr, 22)]))
    idx, sub_lut, nsub = _sub_problem(y, dy, lut_h, meta, rows)
    it = torch.as_tensor(idx, device="cuda")
    ys, dys = y[:, it].cpu(), dy[:, it].cpu()
    ref, bad = oracle.softmax_bwd_bsr(host(ys), host(dys), sub_lut, len(rows), nsub, block,
                                      meta["sizemax"], 1.0)
    assert bad == 0
    out = gbce.softmax_bwd_bsr(y, dy, lut, nbr, meta["nblocks"], block, meta["sizemax"])
    assert gbce.last_error() == gbce.OK
    got = oracle.widen(host(out[:, it].cpu()))
    y64, dy64 = oracle.widen(host(ys)), oracle.widen(host(dys))
    brow = table_rows(sub_lut, len(rows), nsub)
    check_bsr(got, ref, y64, row_abs_sums(y64, dy64, brow, len(rows), block), 1.0, w.dtype,
              f"{name} full size")


def _layout_inputs(lay, block, dtype, Z, seed, shuffle=None, pads=(0, 0, 0)):
    """Inputs for an explicit layout: y ~ Exp(1)/row count, dy ~ N(0,1), each
    operand with its own batch padding."""
    lut, nbr, nblocks, sizemax, brow = workloads.make_bsr_lut(lay, shuffle)
    L = nblocks * block * block
    g = torch.Generator().manual_seed(seed)
    y = torch.empty((Z, L)).exponential_(generator=g)
    dy = torch.randn((Z, L), generator=g)
    sizes = torch.from_numpy(lut[0:2 * nbr:2].astype(np.int64))
    if nblocks:
        y = (y.view(Z, nblocks, -1) / (sizes[torch.from_numpy(brow)] * block).view(1, -1, 1)
             .float()).view(Z, L)

    def padded(t, pad):
        return torch.cat([t, torch.full((Z, pad), 7.0)], dim=1).to(dtype) if pad else t.to(dtype)
    meta = dict(n_block_rows=nbr, nblocks=nblocks, block=block, sizemax=sizemax)
    return padded(y, pads[0]), padded(dy, pads[1]), torch.from_numpy(lut), meta, pads[2]


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("block", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_bsr_block_sizes_strides_and_out_of_place(dtype, block):
    """Every block size, ragged and empty block-rows, shuffled entries, three
    batch items with different padded batch strides per operand, and a
    separate dx whose unnamed positions must keep their contents."""
    require_gpu()
    nb = max(2, min(12, 1024 // block))
    rng = np.random.Generator(np.random.PCG64(block))
    lay = rng.random((2, nb, nb)) < 0.35
    lay[0, 0, :] = True          # one full block-row
    lay[1, 1, :] = False         # one empty block-row
    y, dy, lut, meta, dxpad = _layout_inputs(lay, block, dtype, 3, block, shuffle=block + 1,
                                             pads=(8, 24, 40))
    L = meta["nblocks"] * block * block
    kernel, rows = gbce.bsr_plan(block, meta["sizemax"], dtype)
    assert kernel.startswith("bsr_bwd_staged_kernel")
    # in place (dx = dy, padded batch stride)
    run_and_check(y, dy, lut, meta, -0.5, dtype, what=f"block {block} in place")
    # out of place: dx with its own stride, filled with a sentinel
    dx = torch.full((3, L + dxpad), 3.0, dtype=dtype)
    got, out = run_and_check(y, dy, lut, meta, 2.0, dtype, dx=dx, what=f"block {block} dx")
    assert bool((out[:, L:] == 3.0).all()), "dx written beyond the blocks"


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
def test_bsr_misaligned_bases(dtype):
    """Operands that do not start on 16 bytes: element accesses."""
    require_gpu()
    w = workloads.BSR_WORKLOADS["bsr_f32_causal_2x16x4096_b32"].with_sizes(
        Z=2, H=1, S=256, dtype=dtype)
    y, dy, lut, meta = workloads.make_bsr_inputs(w)
    L = meta["nblocks"] * 32 * 32
    assert gbce.bsr_plan(32, meta["sizemax"], dtype, aligned=False)[0].endswith("accesses)")
    ybig = torch.zeros((2, L + 1), dtype=dtype, device="cuda")
    ybig[:, 1:] = y.cuda()
    ref, _ = oracle.softmax_bwd_bsr(host(y), host(dy), lut.numpy(), meta["n_block_rows"],
                                    meta["nblocks"], 32, meta["sizemax"], 1.0)
    out = gbce.softmax_bwd_bsr(ybig[:, 1:], dy.cuda(), lut.cuda(), meta["n_block_rows"],
                               meta["nblocks"], 32, meta["sizemax"])
    assert gbce.last_error() == gbce.OK
    y64, dy64 = widened(y, L), widened(dy, L)
    brow = table_rows(lut.numpy(), meta["n_block_rows"], meta["nblocks"])
    check_bsr(widened(out, L), ref, y64, row_abs_sums(y64, dy64, brow, meta["n_block_rows"], 32),
              1.0, dtype, "misaligned")


@pytest.mark.parametrize("dtype,block", [(torch.float32, 32), (torch.bfloat16, 64),
                                         (torch.float16, 128)])
def test_bsr_rows_too_long_to_stage(dtype, block):
    """A block-row of 1000 blocks (over 200 KB of the two operands per row):
    the unstaged kernel, vector and element accesses."""
    require_gpu()
    nb = 1000
    lay = np.zeros((1, nb, nb), dtype=bool)
    lay[0, np.arange(nb), np.arange(nb)] = True
    lay[0, 3, :] = True
    y, dy, lut, meta, _ = _layout_inputs(lay, block, dtype, 1, 3, shuffle=4)
    assert gbce.bsr_plan(block, meta["sizemax"], dtype)[0] == "bsr_bwd_unstaged_kernel"
    run_and_check(y, dy, lut, meta, 0.75, dtype, what="unstaged")
    L = meta["nblocks"] * block * block
    ybig = torch.zeros((1, L + 1), dtype=dtype)
    ybig[:, 1:] = y
    dybig = torch.zeros((1, L + 1), dtype=dtype)
    dybig[:, 1:] = dy
    ref, _ = oracle.softmax_bwd_bsr(host(y), host(dy), lut.numpy(), meta["n_block_rows"],
                                    meta["nblocks"], block, meta["sizemax"], 0.75)
    yd, dyd = ybig.cuda(), dybig.cuda()
    out = gbce.softmax_bwd_bsr(yd[:, 1:], dyd[:, 1:], lut.cuda(), meta["n_block_rows"],
                               meta["nblocks"], block, meta["sizemax"], 0.75)
    assert gbce.last_error() == gbce.OK
    y64, dy64 = widened(y, L), widened(dy, L)
    brow = table_rows(lut.numpy(), meta["n_block_rows"], meta["nblocks"])
    check_bsr(widened(out, L), ref, y64, row_abs_sums(y64, dy64, brow, meta["n_block_rows"],
                                                      block), 0.75, dtype, "unstaged misaligned")


@pytest.mark.parametrize("how", ["size", "id_high", "id_negative", "offset"])
@pytest.mark.parametrize("long_rows", [False, True], ids=["staged", "unstaged"])
def test_bsr_bad_table(how, long_rows):
    """A table wrong for one block-row: GBCE_ERR_BAD_TABLE, that block-row's
    blocks untouched (bit for bit), every other row correct."""
    require_gpu()
    block, dtype = 16, torch.float32
    nb = 1000 if long_rows else 12
    lay = np.zeros((1, nb, nb), dtype=bool)
    lay[0, np.arange(nb), np.arange(nb)] = True
    lay[0, 1, :] = True
    lay[0, 2, :nb // 2] = True
    y, dy, lut, meta, _ = _layout_inputs(lay, block, dtype, 2, 9)
    nbr, nblocks, sizemax = meta["n_block_rows"], meta["nblocks"], meta["sizemax"]
    kernel = gbce.bsr_plan(block, sizemax, dtype)[0]
    assert kernel == ("bsr_bwd_unstaged_kernel" if long_rows else "bsr_bwd_staged_kernel")
    lut_h = lut.numpy()
    bad_lut = lut_h.copy()
    r = 2
    off, size = int(lut_h[2 * r + 1]), int(lut_h[2 * r])
    bad_ids = lut_h[off:off + 4 * size:4]
    if how == "size":
        bad_lut[2 * r] = sizemax + 1
    elif how == "id_high":
        bad_lut[off + 4] = nblocks
    elif how == "id_negative":
        bad_lut[off] = -5
    else:
        bad_lut[2 * r + 1] = bad_lut.size - 4 * size + 4
    ref, bad = oracle.softmax_bwd_bsr(host(y), host(dy), bad_lut, nbr, nblocks, block, sizemax,
                                      1.0)
    assert bad == 1
    L = nblocks * block * block
    dyd = dy.cuda()
    gbce.softmax_bwd_bsr(y.cuda(), dyd, torch.from_numpy(bad_lut).cuda(), nbr, nblocks, block,
                         sizemax)
    assert gbce.last_error() == gbce.ERR_BAD_TABLE
    assert gbce.last_error() == gbce.OK, "the flag is cleared by reading it"
    got = widened(dyd, L).reshape(2, nblocks, -1)
    mine = np.zeros(nblocks, dtype=bool)
    mine[bad_ids] = True
    assert np.array_equal(got[:, mine], dy.numpy().astype(np.float64).reshape(2, nblocks, -1)[
        :, mine]), "a bad block-row was written"
    y64, dy64 = widened(y, L), widened(dy, L)
    brow = table_rows(lut_h, nbr, nblocks)
    keep = np.repeat(~mine, block * block)
    check_bsr(got.reshape(2, -1)[:, keep], ref[:, keep], y64[:, keep],
              row_abs_sums(y64, dy64, brow, nbr, block)[:, keep], 1.0, dtype, f"bad {how}")


def test_bsr_nothing_to_do():
    require_gpu()
    y = torch.zeros((0, 16), device="cuda")
    lut = torch.zeros(2, dtype=torch.int32, device="cuda")
    gbce.softmax_bwd_bsr(y, y, lut, 1, 1, 4, 1)                 # Z = 0
    y1 = torch.ones((1, 16), device="cuda")
    gbce.softmax_bwd_bsr(y1, y1, lut, 1, 1, 4, 0)               # sizemax = 0
    assert bool((y1 == 1).all())
    lut0 = torch.tensor([0, 2], dtype=torch.int32, device="cuda")  # one empty block-row
    gbce.softmax_bwd_bsr(y1, y1, lut0, 1, 1, 4, 1)
    assert bool((y1 == 1).all())
    assert gbce.last_error() == gbce.OK


@pytest.mark.parametrize("long_rows", [False, True], ids=["staged", "unstaged"])
def test_bsr_status_words_tell_calls_apart(long_rows):
    """softmax_bwd_bsr_ex: a call with a malformed table (a block id out of
    range) and a call with a good one, on two streams at once, each with its
    own status word: only the first gets STATUS_BAD_TABLE; the device flag
    reports the bad table for the device; the good call's result is the
    plain call's, bit for bit."""
    require_gpu()
    block, dtype = 16, torch.float32
    nb = 1000 if long_rows else 12
    lay = np.zeros((1, nb, nb), dtype=bool)
    lay[0, np.arange(nb), np.arange(nb)] = True
    lay[0, 1, :] = True
    y, dy, lut, meta, _ = _layout_inputs(lay, block, dtype, 2, 11)
    nbr, nblocks, sizemax = meta["n_block_rows"], meta["nblocks"], meta["sizemax"]
    bad_lut = lut.numpy().copy()
    off = int(bad_lut[2 * 1 + 1])
    bad_lut[off] = nblocks  # block-row 1's first id: out of range
    yd, dyd, lutd, badd = y.cuda(), dy.cuda(), lut.cuda(), torch.from_numpy(bad_lut).cuda()
    words = torch.zeros(2, dtype=torch.int32, device="cuda")
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(sa):
        gbce.softmax_bwd_bsr_ex(yd, dyd, badd, nbr, nblocks, block, sizemax,
                                dx=torch.empty_like(dyd), status=words[0:1])
    with torch.cuda.stream(sb):
        good = gbce.softmax_bwd_bsr_ex(yd, dyd, lutd, nbr, nblocks, block, sizemax,
                                       dx=torch.zeros_like(dyd), status=words[1:2])
    torch.cuda.synchronize()
    assert words.tolist() == [gbce.STATUS_BAD_TABLE, 0]
    assert gbce.last_error() == gbce.ERR_BAD_TABLE
    plain = gbce.softmax_bwd_bsr(yd, dyd, lutd, nbr, nblocks, block, sizemax,
                                 dx=torch.zeros_like(dyd))
    assert torch.equal(good, plain) and gbce.last_error() == gbce.OK
