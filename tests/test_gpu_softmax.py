"""CUDA row softmax forward and backward against the double-precision oracle (GPU)."""
import numpy as np
import pytest
import torch

import cross_entropy_loss_ce_gb300 as gbce
import oracle
import workloads
from gpu_util import host, require_gpu
from parity import check_softmax, check_softmax_bwd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16], ids=str)
@pytest.mark.parametrize("N", workloads.SOFTMAX_NS)
def test_softmax_reduced_rows(dtype, N):
    require_gpu()
    x, y, dy = workloads.make_softmax_inputs(64, N, dtype)
    ref_y = oracle.softmax_fwd(host(x))
    ref_dx = oracle.softmax_bwd(host(y), host(dy))
    got_y = gbce.softmax_fwd(x.cuda())
    got_dx = gbce.softmax_bwd(y.cuda(), dy.cuda())
    assert gbce.last_error() == gbce.OK
    check_softmax(got_y, ref_y, dtype, f"softmax N={N}")
    check_softmax_bwd(got_dx, ref_dx, y, dy, dtype, f"softmax bwd N={N}")


@pytest.mark.parametrize("N", workloads.SOFTMAX_NS)
def test_softmax_full_size_sampled_rows(N):
    """All 4096 rows on the GPU; rows sampled for the oracle."""
    require_gpu()
    x, y, dy = workloads.make_softmax_inputs(workloads.SOFTMAX_M, N, device="cuda")
    rows = np.unique(np.concatenate([[0, workloads.SOFTMAX_M - 1],
                                     np.random.default_rng(N).choice(workloads.SOFTMAX_M, 30)]))
    ref_y = oracle.softmax_fwd(host(x), rows=rows)
    ref_dx = oracle.softmax_bwd(host(y), host(dy), rows=rows)
    got_y = gbce.softmax_fwd(x)
    got_dx = gbce.softmax_bwd(y, dy)
    assert gbce.last_error() == gbce.OK
    r = torch.as_tensor(rows, device="cuda")
    check_softmax(got_y[r], ref_y, torch.float32)
    check_softmax_bwd(got_dx[r], ref_dx, y[r], dy[r], torch.float32)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16], ids=str)
@pytest.mark.parametrize("N", [1, 3, 7, 8, 9, 33, 1000, 65537, 300001, 1000003])
def test_softmax_shapes_strides_and_aliasing(dtype, N):
    """Ragged N, the in-place forms (y = x, dx = dy), and operands whose rows
    sit at different 16-byte phases (the streaming fallback)."""
    require_gpu()
    M = 5 if N < 500000 else 2
    g = torch.Generator().manual_seed(N)
    x = torch.randn((M, N), generator=g).to(dtype)
    e = torch.rand((M, N), generator=g) + 0.01
    y = (e / e.sum(1, keepdim=True)).to(dtype)
    dy = torch.randn((M, N), generator=g).to(dtype)
    ref_y = oracle.softmax_fwd(host(x))
    ref_dx = oracle.softmax_bwd(host(y), host(dy))
    # in place
    xd = x.cuda()
    gbce.softmax_fwd(xd, xd)
    check_softmax(xd, ref_y, dtype, f"in-place softmax N={N}")
    dyd = dy.cuda()
    gbce.softmax_bwd(y.cuda(), dyd, dyd)
    check_softmax_bwd(dyd, ref_dx, y, dy, dtype, f"in-place softmax bwd N={N}")
    # x padded by one element per row, y contiguous: different phases
    xp = torch.zeros((M, N + 1), dtype=dtype, device="cuda")
    xp[:, 1:] = x.cuda()
    yo = gbce.softmax_fwd(xp[:, 1:])
    check_softmax(yo, ref_y, dtype, f"shifted softmax N={N}")
    dyp = torch.zeros((M, N + 3), dtype=dtype, device="cuda")
    dyp[:, 3:] = dy.cuda()
    dxo = gbce.softmax_bwd(y.cuda(), dyp[:, 3:])
    check_softmax_bwd(dxo, ref_dx, y, dy, dtype, f"shifted softmax bwd N={N}")
    assert gbce.last_error() == gbce.OK


def test_softmax_empty():
    require_gpu()
    x = torch.empty((0, 16), device="cuda")
    assert gbce.softmax_fwd(x).shape == (0, 16)
    assert gbce.softmax_bwd(x, x).shape == (0, 16)


# 4 rows: warp, resident, the ring on one CTA (48 KB unaligned rows), the ring on a cluster
# (a small batch: 64 KB rows, unaligned 400 KB rows), the ring on a cluster (the L2 bound)
@pytest.mark.parametrize("N", [1000, 4096, 12001, 16384, 100003, 300001])
@pytest.mark.parametrize("offset", [50.0, -150.0, 150.0, 1e4, -1e4, 1e6, -1e6])
def test_softmax_large_inputs(N, offset):
    """Inputs far from zero (row maxima up to 2e6 in magnitude) keep the
    forward within the fp32 tolerance in every regime, the streaming fallback
    (x and y at different 16-byte phases) included."""
    require_gpu()
    g = torch.Generator().manual_seed(N)
    x = torch.randn((4, N), generator=g) * 4
    x += torch.tensor([offset, -offset, 0.5 * offset, 2 * offset])[:, None]
    ref = oracle.softmax_fwd(host(x))
    check_softmax(gbce.softmax_fwd(x.cuda()), ref, torch.float32, f"N={N} offset={offset}")
    xp = torch.zeros((4, N + 1), device="cuda")
    xp[:, 1:] = x.cuda()
    check_softmax(gbce.softmax_fwd(xp[:, 1:]), ref, torch.float32,
                  f"streaming N={N} offset={offset}")
    assert gbce.last_error() == gbce.OK


def _masked_rows(M, N, dtype, seed):
    """Rows with -inf entries as an attention mask leaves them: a short finite
    prefix (the rest -inf: whole chunks and cluster slices of -inf at the
    end), a -inf first half (the online maximum starts from -inf), a random
    half, one finite entry, an unmasked row, and only the last entry finite;
    then the same patterns again."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((M, N), generator=g) * 3
    ninf = float("-inf")
    for r in range(M):
        kind = r % 6
        if kind == 0:
            x[r, min(5, N):] = ninf
        elif kind == 1:
            x[r, : N // 2] = ninf
        elif kind == 2:
            x[r, torch.rand(N, generator=g) < 0.5] = ninf
            x[r, int(torch.randint(0, N, (1,), generator=g))] = 1.0
        elif kind == 3:
            keep = int(torch.randint(0, N, (1,), generator=g))
            v = float(x[r, keep])
            x[r] = ninf
            x[r, keep] = v
        elif kind == 5:
            x[r, : N - 1] = ninf
    return x.to(dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16], ids=str)
@pytest.mark.parametrize("N", [1000, 4096, 12001, 100003, 300001])
@pytest.mark.parametrize("M", [6, 200])
def test_softmax_masked_rows(dtype, N, M):
    """-inf entries take exactly zero probability in every regime (warp,
    resident, the ring on one CTA, clusters for small batches and for the L2
    bound), forward and backward against the oracle."""
    require_gpu()
    if M * N > 30_000_000:
        pytest.skip("large batch of long rows: covered by the 6-row case")
    x = _masked_rows(M, N, dtype, seed=N + M)
    ref = oracle.softmax_fwd(host(x))
    y = gbce.softmax_fwd(x.cuda())
    assert gbce.last_error() == gbce.OK
    check_softmax(y, ref, dtype, f"masked softmax {M}x{N}")
    assert bool(torch.all(y.cpu()[torch.isinf(x)] == 0)), "a -inf entry got probability"
    yh = y.cpu()
    g = torch.Generator().manual_seed(N)
    dy = torch.randn((M, N), generator=g).to(dtype)
    ref_dx = oracle.softmax_bwd(host(yh), host(dy))
    dx = gbce.softmax_bwd(y, dy.cuda())
    assert gbce.last_error() == gbce.OK
    check_softmax_bwd(dx, ref_dx, yh, dy, dtype, f"masked softmax backward {M}x{N}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=str)
@pytest.mark.parametrize("N", [1000, 4096, 12001, 16384, 100003, 300001])
@pytest.mark.parametrize("offset", [150.0, -150.0, 1e4, -1e4])
def test_softmax_large_inputs_16bit(dtype, N, offset):
    """bf16 and fp16 rows far from zero (row maxima up to 2e4) in every regime,
    forward and backward against the oracle at the 16-bit tolerances."""
    require_gpu()
    g = torch.Generator().manual_seed(N)
    x = torch.randn((4, N), generator=g) * 4
    x += torch.tensor([offset, -offset, 0.5 * offset, 2 * offset])[:, None]
    x = x.to(dtype)
    y = gbce.softmax_fwd(x.cuda())
    assert gbce.last_error() == gbce.OK
    check_softmax(y, oracle.softmax_fwd(host(x)), dtype, f"N={N} offset={offset}")
    yh = y.cpu()
    dy = (torch.randn((4, N), generator=g) * 3).to(dtype)
    dx = gbce.softmax_bwd(y, dy.cuda())
    assert gbce.last_error() == gbce.OK
    check_softmax_bwd(dx, oracle.softmax_bwd(host(yh), host(dy)), yh, dy, dtype,
                      f"backward N={N} offset={offset}")


@pytest.mark.parametrize("N", [1000, 4096, 16384, 300001])
def test_softmax_ex_equals_the_plain_calls(N):
    """softmax_fwd_ex / softmax_bwd_ex with a status word: bit-identical to
    softmax_fwd / softmax_bwd, and the word stays 0."""
    require_gpu()
    M = 6 if N > 100000 else 300
    x, y, dy = workloads.make_softmax_inputs(M, N, device="cuda")
    words = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert torch.equal(gbce.softmax_fwd_ex(x, status=words[0:1]), gbce.softmax_fwd(x))
    assert torch.equal(gbce.softmax_bwd_ex(y, dy, status=words[1:2]), gbce.softmax_bwd(y, dy))
    assert words.tolist() == [0, 0] and gbce.last_error() == gbce.OK
    with pytest.raises(ValueError):
        gbce.softmax_fwd_ex(x, status=torch.zeros(1, dtype=torch.int64, device="cuda"))
