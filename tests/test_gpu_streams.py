"""Calls on several streams at once, and CUDA graphs capturing ce_fwd_bwd
(stream-ordered scratch, programmatic dependent launches) and the softmax
calls, replayed on new inputs."""
import numpy as np
import pytest
import torch

import cross_entropy_loss_ce_gb300 as gbce
import oracle
import workloads
from gpu_util import oracle_ce, require_gpu
from parity import check_grad, check_loss

pytestmark = pytest.mark.gpu
II = workloads.IGNORE_INDEX


def _case(M, V, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn((M, V), generator=g) * 2).to(dtype)
    t = torch.randint(0, V, (M,), generator=g)
    t[::7] = II
    return x, t


def test_concurrent_calls_on_two_streams():
    require_gpu()
    cases = [_case(64, 50000, torch.bfloat16, 1), _case(96, 3000, torch.float32, 2),
             _case(32, 200000, torch.float32, 3)]
    refs = [oracle_ce(x, t) for x, t in cases]
    streams = [torch.cuda.Stream() for _ in cases]
    devs = [(x.cuda(), t.cuda()) for x, t in cases]
    torch.cuda.synchronize()
    losses = []
    for s, (xd, td) in zip(streams, devs):
        with torch.cuda.stream(s):
            losses.append(gbce.ce_fwd_bwd(xd, td, II))
    torch.cuda.synchronize()
    assert gbce.last_error() == gbce.OK
    for (x, t), (xd, td), ref, loss in zip(cases, devs, refs, losses):
        check_grad(xd, ref["grad"], ref["n"], x.dtype)
        check_loss(float(loss.item()), oracle.ce_mean(ref["row_loss"], ref["n"]), x.dtype)


# 64 rows each: warp, resident, the ring on one CTA (40 KB rows), the ring on a cluster of 2
# (a batch under one row per SM), the ring on a cluster of 2 (the L2 bound)
@pytest.mark.parametrize("V", [1000, 16000, 20001, 128256, 262147])
def test_graph_capture_and_replay(V):
    require_gpu()
    M = 64
    x0, t0 = _case(M, V, torch.bfloat16, V)
    x1, t1 = _case(M, V, torch.bfloat16, V + 1)
    xd = torch.empty((M, V), dtype=torch.bfloat16, device="cuda")
    td = torch.empty((M,), dtype=torch.int64, device="cuda")
    loss = torch.empty((), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        xd.copy_(x0.cuda())
        td.copy_(t0.cuda())
        gbce.ce_fwd_bwd(xd, td, II, loss)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gbce.ce_fwd_bwd(xd, td, II, loss)
    for x, t in ((x0, t0), (x1, t1), (x0, t0)):
        xd.copy_(x.cuda())
        td.copy_(t.cuda())
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle_ce(x, t)
        check_grad(xd, ref["grad"], ref["n"], torch.bfloat16, f"graph replay V={V}")
        check_loss(float(loss.item()), oracle.ce_mean(ref["row_loss"], ref["n"]), torch.bfloat16)
    assert gbce.last_error() == gbce.OK


def test_block_sparse_backward_on_two_streams():
    """Two block-sparse calls in flight on different streams (one in place,
    one into a separate dx) give the results of the calls made one at a time."""
    require_gpu()
    cases = []
    for name, sizes in (("bsr_f32_causal_2x16x4096_b32", dict(H=2, S=1024)),
                        ("bsr_bf16_random_4x8x8192_b64", dict(Z=2, H=2, S=2048))):
        w = workloads.BSR_WORKLOADS[name].with_sizes(**sizes)
        y, dy, lut, meta = workloads.make_bsr_inputs(w, device="cuda")
        cases.append((y, dy, lut, meta))
    args = lambda meta: (meta["n_block_rows"], meta["nblocks"], meta["block"], meta["sizemax"])
    refs = []
    for y, dy, lut, meta in cases:  # one at a time
        refs.append(gbce.softmax_bwd_bsr(y, dy, lut, *args(meta), 0.5, torch.empty_like(dy)))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in cases]
    outs = []
    for i, (s, (y, dy, lut, meta)) in enumerate(zip(streams, cases)):
        with torch.cuda.stream(s):
            outs.append(gbce.softmax_bwd_bsr(y, dy.clone() if i == 0 else dy, lut, *args(meta), 0.5,
                                             None if i == 0 else torch.empty_like(dy), stream=s))
    torch.cuda.synchronize()
    assert gbce.last_error() == gbce.OK
    for ref, out in zip(refs, outs):
        assert torch.equal(ref, out)


def test_host_calls_on_two_streams():
    """Two ce_fwd_bwd_host calls on different streams share the library's copy
    stream and still give the results of the device call."""
    require_gpu()
    cases = [_case(40, 64000, torch.bfloat16, 4), _case(24, 100003, torch.float32, 5)]
    refs = []
    for x, t in cases:
        xd = x.cuda()
        refs.append((xd, float(gbce.ce_fwd_bwd(xd, t.cuda(), II).item())))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in cases]
    outs = []
    for s, (x, t) in zip(streams, cases):
        with torch.cuda.stream(s):
            outs.append(gbce.ce_fwd_bwd_host(x.pin_memory(), t.pin_memory(), II, stream=s))
    torch.cuda.synchronize()
    assert gbce.last_error() == gbce.OK
    for (ref_g, ref_l), (grad, loss) in zip(refs, outs):
        assert torch.equal(grad, ref_g) and float(loss.item()) == ref_l


# warp, resident, ring on one CTA (48 KB rows), ring on a cluster (small batches of 64 KB
# rows and longer)
@pytest.mark.parametrize("N", [1000, 4096, 12001, 16384, 300001])
def test_softmax_calls_in_a_cuda_graph(N):
    """softmax_fwd, softmax_bwd and the block-sparse backward captured in one
    CUDA graph, replayed on new inputs: the results of direct calls, bit for
    bit, and the oracle's within tolerance."""
    require_gpu()
    from parity import check_softmax, check_softmax_bwd
    M = 6 if N < 100000 else 2
    w = workloads.BSR_WORKLOADS["bsr_f32_causal_2x16x4096_b32"].with_sizes(Z=1, H=1, S=256)
    x = torch.empty((M, N), device="cuda")
    yv, dy = torch.empty_like(x), torch.empty_like(x)
    y_out, dx_out = torch.empty_like(x), torch.empty_like(x)
    by, bdy, lut, meta = workloads.make_bsr_inputs(w, device="cuda")
    bdx = torch.empty_like(bdy)
    bargs = (meta["n_block_rows"], meta["nblocks"], meta["block"], meta["sizemax"])

    def calls():
        gbce.softmax_fwd(x, y_out)
        gbce.softmax_bwd(yv, dy, dx_out)
        gbce.softmax_bwd_bsr(by, bdy, lut, *bargs, 0.5, bdx)

    def fill(seed):
        xs, ys, dys = workloads.make_softmax_inputs(M, N, seed=seed)
        x.copy_(xs.cuda())
        yv.copy_(ys.cuda())
        dy.copy_(dys.cuda())
        by.copy_(torch.rand_like(by))
        bdy.copy_(torch.randn_like(bdy))
        return xs, ys, dys

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        fill(0)
        calls()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        calls()
    for seed in (1, 2):
        xs, ys, dys = fill(seed)
        graph.replay()
        torch.cuda.synchronize()
        got = (y_out.clone(), dx_out.clone(), bdx.clone())
        calls()
        torch.cuda.synchronize()
        assert torch.equal(got[0], y_out) and torch.equal(got[1], dx_out)
        assert torch.equal(got[2], bdx)
        check_softmax(got[0], oracle.softmax_fwd(oracle.host_array(xs)), torch.float32,
                      f"graph softmax N={N}")
        check_softmax_bwd(got[1], oracle.softmax_bwd(oracle.host_array(ys), oracle.host_array(dys)),
                          ys, dys, torch.float32, f"graph softmax bwd N={N}")
    assert gbce.last_error() == gbce.OK


_THREADS_CHILD = r'''
import sys, threading
import torch
import cross_entropy_loss_ce_gb300 as gbce

gbce.load_library()
torch.zeros(1, device="cuda")
II = -100
# per thread: shapes whose first use makes the library plan (small-batch cluster
# searches included), configure kernels and query occupancy
SHAPES = [[("ce", 1, 128256, torch.bfloat16), ("fwd", 3, 100003, torch.float32), ("bwd", 40, 6000, torch.float32)],
          [("ce", 8, 128256, torch.bfloat16), ("ce", 200, 32000, torch.bfloat16), ("fwd", 6, 16384, torch.float32)],
          [("ce", 33, 250007, torch.float32), ("bwd", 2, 300001, torch.bfloat16), ("ce", 64, 1000, torch.float32)],
          [("ce", 5, 130001, torch.float16), ("fwd", 152, 32000, torch.float32), ("bwd", 9, 128256, torch.float32)],
          [("ce", 16, 65537, torch.bfloat16), ("fwd", 1, 2000003, torch.bfloat16), ("ce", 7, 20001, torch.bfloat16)],
          [("bwd", 24, 20000, torch.float32), ("ce", 100, 128256, torch.bfloat16), ("fwd", 400, 3000, torch.float16)]]
ROUNDS = 6

def inputs(op, M, N, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    a = (torch.randn((M, N), generator=g) * 3).to(dtype).cuda()
    b = torch.randn((M, N), generator=g).to(dtype).cuda()
    t = torch.randint(0, N, (M,), generator=g).cuda()
    return a, b, t

def run(op, a, b, t):
    if op == "ce":
        x = a.clone()
        loss = gbce.ce_fwd_bwd(x, t, II)
        return x, loss
    if op == "fwd":
        return gbce.softmax_fwd(a), None
    return gbce.softmax_bwd(torch.softmax(a.float(), 1).to(a.dtype), b), None

results, errors = {}, []
data = {(i, j): inputs(*SHAPES[i][j], seed=100 * i + j) for i in range(len(SHAPES)) for j in range(3)}
torch.cuda.synchronize()
barrier = threading.Barrier(len(SHAPES))

def worker(i):
    try:
        s = torch.cuda.Stream()
        barrier.wait()
        with torch.cuda.stream(s):
            for r in range(ROUNDS):
                for j, (op, M, N, dtype) in enumerate(SHAPES[i]):
                    a, b, t = data[(i, j)]
                    results[(i, j, r)] = run(op, a, b, t)
        s.synchronize()
    except Exception as e:  # reported by the parent
        errors.append(f"thread {i}: {e!r}")

threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(SHAPES))]
for th in threads: th.start()
for th in threads: th.join()
torch.cuda.synchronize()
status = gbce.last_error()
if errors or status != gbce.OK:
    print("FAIL", errors, status); sys.exit(1)
# the same calls once more, one after another: every threaded result is bit-identical
bad = []
for i in range(len(SHAPES)):
    for j, (op, M, N, dtype) in enumerate(SHAPES[i]):
        ref, lref = run(op, *data[(i, j)])
        torch.cuda.synchronize()
        for r in range(ROUNDS):
            got, lgot = results[(i, j, r)]
            same = torch.equal(got.view(torch.int16) if got.dtype != torch.float32 else got.view(torch.int32),
                               ref.view(torch.int16) if ref.dtype != torch.float32 else ref.view(torch.int32))
            if lref is not None:
                same = same and torch.equal(lgot.view(torch.int32), lref.view(torch.int32))
            if not same:
                bad.append((i, j, r, op, M, N))
print("FAIL", bad) if bad else print("ok", len(results))
sys.exit(1 if bad else 0)
'''


def test_first_use_from_several_host_threads():
    """Six host threads, each on its own stream, start at once in a fresh
    process and call the library on shapes whose first use plans (small-batch
    cluster searches included), configures kernels, queries occupancy and
    creates the scratch pool: every result is bit-identical to the same call
    made afterwards from one thread, and no error flag is raised."""
    require_gpu()
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", _THREADS_CHILD], cwd=root, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]


_CAPTURE_FIRST_CHILD = r'''
import sys
import torch
import cross_entropy_loss_ce_gb300 as gbce

II = -100
torch.zeros(1, device="cuda")
g = torch.Generator(device="cuda").manual_seed(5)
x1 = torch.randn((4, 128256), generator=g, device="cuda").to(torch.bfloat16)   # small batch
x2 = torch.randn((300, 65537), generator=g, device="cuda").to(torch.bfloat16)  # ring
x3 = torch.randn((64, 3000), generator=g, device="cuda")                       # resident
t1 = torch.randint(0, 128256, (4,), generator=g, device="cuda")
t2 = torch.randint(0, 65537, (300,), generator=g, device="cuda")
x4 = torch.randn((96, 32000), generator=g, device="cuda").to(torch.bfloat16)   # no-alloc call
t4 = torch.randint(0, 32000, (96,), generator=g, device="cuda")
a1, a2, a3, a4 = x1.clone(), x2.clone(), torch.empty_like(x3), x4.clone()
l1, l2, l4 = (torch.empty((), device="cuda") for _ in range(3))
torch.cuda.synchronize()
graph = torch.cuda.CUDAGraph()
# the library's first calls in this process happen inside the capture
with torch.cuda.graph(graph):
    gbce.ce_fwd_bwd(a1, t1, II, l1)
    gbce.ce_fwd_bwd(a2, t2, II, l2)
    gbce.softmax_fwd(x3, a3)
    gbce.ce_fwd_bwd_noalloc(a4, t4, II, l4)
for _ in range(2):
    a1.copy_(x1); a2.copy_(x2); a4.copy_(x4)
    graph.replay()
    torch.cuda.synchronize()
assert gbce.last_error() == gbce.OK
b1, b2, b4 = x1.clone(), x2.clone(), x4.clone()
m1, m2 = gbce.ce_fwd_bwd(b1, t1, II), gbce.ce_fwd_bwd(b2, t2, II)
m4 = gbce.ce_fwd_bwd(b4, t4, II)
b3 = gbce.softmax_fwd(x3)
torch.cuda.synchronize()
ok = (torch.equal(a1.view(torch.int16), b1.view(torch.int16)) and
      torch.equal(a2.view(torch.int16), b2.view(torch.int16)) and torch.equal(a3, b3) and
      torch.equal(a4.view(torch.int16), b4.view(torch.int16)) and
      float(l1) == float(m1) and float(l2) == float(m2) and float(l4) == float(m4))
print("ok" if ok else "FAIL mismatch")
sys.exit(0 if ok else 1)
'''


def test_first_calls_inside_a_graph_capture():
    """In a fresh process, the library's very first calls are made inside a
    CUDA graph capture: library load, plans (a small-batch cluster search
    included), kernel configuration, occupancy queries, the scratch pool and
    the allocation-free call's static array all happen during capture (in
    the default, global capture mode); replays equal later direct calls bit
    for bit."""
    require_gpu()
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", _CAPTURE_FIRST_CHILD], cwd=root, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout[-2000:] + r.stderr[-3000:]
