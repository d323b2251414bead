"""GPU parity of the allreduce, reduce-scatter and all-gather kernels against
the CPU oracle, through the C ABI. Ring and fused results must equal the
oracle's literal ring simulation bit for bit, tree results the oracle's
recursive-halving order bit for bit; every output buffer is canary-guarded."""
import numpy as np
import pytest
import torch

import gradient_allreduce_collective_gb300 as gar
import oracle
import synthgen
from tests import _golden as G
from tests._dev import ESIZE, TORCH, Guarded, from_dev, to_dev

pytestmark = pytest.mark.gpu

ALL_DT = ("f32", "bf16", "f16", "i32")
OPS = ("sum", "avg", "min", "max")


@pytest.fixture(scope="module", autouse=True)
def _built():
    gar.build()
    gar.lib()


def _rand(dtype, n, count, seed=0, sigma=1.0):
    if dtype == "i32":
        return synthgen.ranks_int(n, count, -(2**20), 2**20, base_seed=seed)
    return synthgen.ranks_normal(n, count, sigma, base_seed=seed, dtype=dtype)


def _gpu_allreduce(send_np, dtype, op, algo, offset=0, in_offset=0):
    n, count = len(send_np), send_np[0].size
    if in_offset:
        gin = Guarded(n, count, dtype, in_offset)
        for v, a in zip(gin.views, send_np):
            v.copy_(to_dev(a, dtype))
        send = gin.views
    else:
        send = [to_dev(a, dtype) for a in send_np]
    out = Guarded(n, count, dtype, offset)
    if algo.startswith("step") and ESIZE[dtype] == 2:  # binary32 partials in a workspace
        wsb = gar.ar_stepwise_workspace_bytes(n, count, dtype)
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
        gar.ar_allreduce_stepwise(send, out.views, ws, op, algo)
    else:
        gar.ar_allreduce(send, out.views, op, algo)
    out.check()
    return [from_dev(v) for v in out.views]


def _expect(send_np, dtype, op, algo):
    if algo in ("tree", "step_tree"):
        return oracle.tree_allreduce(send_np, dtype, op)[0]
    return oracle.ring_allreduce(send_np, dtype, op)[0]


def _same_bits(a, b):
    return np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


def _algos(n, dtype="f32"):
    """Orders to check: the one-pass ones, AUTO, and the stepwise executors (16-bit
    types through ar_allreduce_stepwise with binary32 partials)."""
    pow2 = n & (n - 1) == 0
    algos = ["ring", "fused", "auto"] + (["tree"] if pow2 else [])
    algos += ["step_ring"] + (["step_tree"] if pow2 else [])
    return tuple(algos)


def test_worked_example_every_algo():
    g = G.load("worked_example_allreduce.txt")
    for dtype in ("i32", "f32"):
        send = [np.array(G.nums(g[f"rank{r}"]), dtype=np.int32 if dtype == "i32" else np.float32) for r in range(4)]
        for algo in ("ring", "fused", "tree"):
            for y in _gpu_allreduce(send, dtype, "sum", algo):
                assert y.tolist() == G.nums(g["expect"], int if dtype == "i32" else float)


def test_page_placement_examples():
    g = G.load("all_gather_rank_order.txt")
    send = [to_dev(np.array(G.nums(g[f"rank{r}"], int), dtype=np.int32), "i32") for r in range(4)]
    recv = [torch.empty(4, dtype=torch.int32, device="cuda") for _ in range(4)]
    gar.ar_all_gather(send, recv)
    for y in recv:
        assert y.cpu().tolist() == G.nums(g["expect"], int)
    g = G.load("reduce_scatter_placement.txt")
    send = [to_dev(np.array(G.nums(g[f"rank{r}"], int), dtype=np.int32), "i32") for r in range(2)]
    recv = [torch.empty(1, dtype=torch.int32, device="cuda") for _ in range(2)]
    gar.ar_reduce_scatter(send, recv, "sum")
    assert recv[0].cpu().tolist() == G.nums(g["expect_rank0"], int)
    assert recv[1].cpu().tolist() == G.nums(g["expect_rank1"], int)


def test_ring_start_rank_and_tree_order_pins():
    g = G.load("ring_start_rank.txt")
    send = [np.full(int(g["count"]), float(g[f"rank{r}"]), dtype=np.float32) for r in range(3)]
    for algo in ("ring", "fused"):
        for y in _gpu_allreduce(send, "f32", "sum", algo):
            assert y.tolist() == G.nums(g["expect"])
    g = G.load("tree_order.txt")
    send = [np.array([float(g[f"rank{r}"])], dtype=np.float32) for r in range(4)]
    assert _gpu_allreduce(send, "f32", "sum", "tree")[0].tolist() == G.nums(g["expect_tree"])
    assert _gpu_allreduce(send, "f32", "sum", "fused")[0].tolist() == G.nums(g["expect_ring"])


@pytest.mark.parametrize("dtype", ALL_DT)
@pytest.mark.parametrize("op", OPS)
def test_tiny_brute_force(dtype, op):
    counts = (0, 1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 33, 127, 129, 1000)
    for n in (1, 2, 3, 4, 5, 6, 7, 8, 16):
        for count in counts:
            send = _rand(dtype, n, count, seed=1000 * n + count)
            for algo in _algos(n, dtype):
                want = _expect(send, dtype, op, algo)
                for y in _gpu_allreduce(send, dtype, op, algo):
                    assert _same_bits(y, want), (n, count, algo)


@pytest.mark.parametrize("dtype", ALL_DT)
@pytest.mark.parametrize("op", OPS)
def test_multi_tile_ragged(dtype, op):
    n, count = 8, 3 * (1 << 20) + 12345
    send = _rand(dtype, n, count, seed=7)
    for algo in _algos(n, dtype):
        want = _expect(send, dtype, op, algo)
        ys = _gpu_allreduce(send, dtype, op, algo)
        for y in ys:
            assert _same_bits(y, want), algo


@pytest.mark.parametrize("n", [9, 16, 33, 64])
def test_many_ranks(n):
    count = 50_003
    for dtype in ("f32", "bf16"):
        send = _rand(dtype, n, count, seed=n)
        for algo in _algos(n, dtype):
            want = _expect(send, dtype, "sum", algo)
            for y in _gpu_allreduce(send, dtype, "sum", algo):
                assert _same_bits(y, want), (n, dtype, algo)


def test_config1_four_ranks():
    send = synthgen.ranks_normal(4, 65_536, 1.0, base_seed=0)
    for algo in ("ring", "fused", "tree"):
        want = _expect(send, "f32", "sum", algo)
        for y in _gpu_allreduce(send, "f32", "sum", algo):
            assert _same_bits(y, want)


def test_config2_full_size_bucket():
    # one 25 MiB fp32 bucket on 8 ranks, average: ring (RS+AG) and fused are bit-identical
    n, count = 8, 6_553_600
    send_np = synthgen.ranks_normal(n, count, 1e-3, base_seed=0)
    want = oracle.ring_allreduce(send_np, "f32", "avg")[0]
    send = [to_dev(a, "f32") for a in send_np]
    outs = {}
    for algo in ("ring", "fused"):
        recv = [torch.empty(count, dtype=torch.float32, device="cuda") for _ in range(n)]
        gar.ar_allreduce(send, recv, "avg", algo)
        torch.cuda.synchronize()
        for r in range(1, n):
            assert torch.equal(recv[r].view(torch.int32), recv[0].view(torch.int32))
        outs[algo] = from_dev(recv[0])
        assert _same_bits(outs[algo], want), algo
    ystar, S = oracle.reference_f64(send_np, "f32", "avg")
    err = np.abs(outs["fused"].astype(np.float64) - ystar) / S
    assert err.max() <= 1e-6


@pytest.mark.parametrize("dtype", ALL_DT)
def test_reduce_scatter_and_all_gather(dtype):
    n = 6
    for rc in (1, 3, 8, 64, 1001, 65_536):
        send_np = _rand(dtype, n, n * rc, seed=rc)
        send = [to_dev(a, dtype) for a in send_np]
        rs = Guarded(n, rc, dtype)
        gar.ar_reduce_scatter(send, rs.views, "sum")
        rs.check()
        want = oracle.ring_reduce_scatter(send_np, dtype, "sum")
        for c in range(n):
            assert _same_bits(from_dev(rs.views[c]), want[c])
        ag = Guarded(n, n * rc, dtype)
        gar.ar_all_gather(rs.views, ag.views)
        ag.check()
        want_ag = oracle.ring_all_gather([from_dev(v) for v in rs.views], dtype)
        ar = oracle.ring_allreduce(send_np, dtype, "sum")[0] if (rc * ESIZE[dtype]) % 16 == 0 else None
        for q in range(n):
            got = from_dev(ag.views[q])
            assert _same_bits(got, want_ag[q])
            if ar is not None:  # chunk length equals the allreduce's: RS then AG is the allreduce
                assert _same_bits(got, ar)


def test_in_place_forms():
    n, count = 8, 100_000
    for dtype in ("f32", "bf16", "i32"):
        send_np = _rand(dtype, n, count, seed=3)
        for algo in _algos(n, dtype):
            bufs = [to_dev(a, dtype) for a in send_np]
            if algo.startswith("step") and ESIZE[dtype] == 2:
                ws = torch.empty(gar.ar_stepwise_workspace_bytes(n, count, dtype), dtype=torch.uint8, device="cuda")
                gar.ar_allreduce_stepwise(bufs, bufs, ws, "sum", algo)
            else:
                gar.ar_allreduce(bufs, bufs, "sum", algo)
            want = _expect(send_np, dtype, "sum", algo)
            for b in bufs:
                assert _same_bits(from_dev(b), want)
        rc = 1000
        send_np = _rand(dtype, n, n * rc, seed=4)
        bufs = [to_dev(a, dtype) for a in send_np]
        gar.ar_reduce_scatter(bufs, [bufs[c][c * rc:(c + 1) * rc] for c in range(n)], "max")
        want = oracle.ring_reduce_scatter(send_np, dtype, "max")
        for c in range(n):
            assert _same_bits(from_dev(bufs[c][c * rc:(c + 1) * rc]), want[c])
        gar.ar_all_gather([bufs[r][r * rc:(r + 1) * rc] for r in range(n)], bufs)
        full = np.concatenate(want)
        for b in bufs:
            assert _same_bits(from_dev(b), full)


def test_unaligned_buffers_take_the_element_path():
    n, count = 5, 70_001
    for dtype in ("f32", "bf16", "f16", "i32"):
        send = _rand(dtype, n, count, seed=9)
        es = ESIZE[dtype]
        for algo in _algos(n, dtype):
            want = _expect(send, dtype, "avg", algo)
            for y in _gpu_allreduce(send, dtype, "avg", algo, offset=es, in_offset=3 * es):
                assert _same_bits(y, want)


def test_nan_and_signed_zero():
    pz, nz = np.float32(0.0), np.float32(-0.0)
    base = [np.array([pz, nz, 1.0, np.nan] * 5, dtype=np.float32),
            np.array([nz, pz, np.nan, 2.0] * 5, dtype=np.float32)]
    for dtype in ("f32", "bf16", "f16"):
        send = [a if dtype == "f32" else synthgen.to_dtype(a, dtype) for a in base]
        for op in ("min", "max"):
            for algo in ("ring", "fused", "tree"):
                want = _expect(send, dtype, op, algo)
                for y in _gpu_allreduce(send, dtype, op, algo):
                    assert _same_bits(y, want), (dtype, op, algo)
        # SUM with NaN input: the result is some NaN
        y = _gpu_allreduce(send, dtype, "sum", "fused")[0]
        f = y if dtype == "f32" else oracle.bf16_to_f32(y) if dtype == "bf16" else oracle.f16_to_f32(y)
        assert np.isnan(f[2]) and np.isnan(f[3])


def test_errors_write_nothing():
    n, count = 4, 4096
    send = [to_dev(a, "f32") for a in _rand("f32", n, count)]
    out = Guarded(n, count, "f32")
    for v in out.views:
        v.view(torch.int32).fill_(0x5A5A5A5A)
    with pytest.raises(gar.ArError):
        gar.ar_allreduce(send[:3], out.views[:3], "sum", "tree")  # 3 ranks: tree unsupported
    with pytest.raises(gar.ArError):
        gar.ar_allreduce(send, [out.views[0]] * n, "sum", "fused")  # outputs alias
    out.check()
    for v in out.views:
        assert bool((v.view(torch.int32) == 0x5A5A5A5A).all())


def test_cuda_graph_capture_and_side_stream():
    n, count = 8, 1 << 16
    send_np = _rand("f32", n, count, seed=11)
    send = [to_dev(a, "f32") for a in send_np]
    recv = [torch.zeros(count, device="cuda") for _ in range(n)]
    want = oracle.ring_allreduce(send_np, "f32", "sum")[0]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        gar.ar_allreduce(send, recv, "sum", "fused")
    torch.cuda.current_stream().wait_stream(side)
    assert _same_bits(from_dev(recv[3]), want)
    for r in recv:
        r.zero_()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    with torch.cuda.stream(cap):
        graph.capture_begin()
        gar.ar_allreduce(send, recv, "sum", "ring")
        graph.capture_end()
    torch.cuda.synchronize()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for r in recv:
        assert _same_bits(from_dev(r), want)


def test_communicator_threads_launch_one_allreduce():
    import threading
    n, count = 8, 1 << 20
    send_np = _rand("f32", n, count, seed=33)
    send = [to_dev(a, "f32") for a in send_np]
    recv = [torch.empty_like(x) for x in send]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    comm = gar.Comm(n, 10_000)
    st = [None] * n

    def go(r):
        st[r] = comm.allreduce(r, send[r], recv[r], op="avg", algo="fused", stream=stream)

    ts = [threading.Thread(target=go, args=(r,)) for r in range(n)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(timeout=60)
    assert st == [0] * n
    stream.synchronize()
    want = oracle.ring_allreduce(send_np, "f32", "avg")[0]
    for r in range(n):
        assert _same_bits(from_dev(recv[r]), want)
    rec = comm.last_record(0)
    assert rec.seq == 1 and rec.arrived_mask == (1 << n) - 1


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("n", [3, 8])
def test_slices_reassemble_the_allreduce(dtype, n):
    # G "GPUs" each hold a contiguous slice of every rank's buffer (separate
    # allocations, boundaries anywhere); their slice results concatenated are
    # the whole problem's allreduce, bit for bit, in the ring and tree orders
    count = 100_003
    send_np = _rand(dtype, n, count, seed=77 + n)
    rng = np.random.default_rng(n)
    for op in ("sum", "avg", "max"):
        for algo in ["fused", "ring", "auto", "step_ring"] + (["tree", "step_tree"] if n & (n - 1) == 0 else []):
            want = _expect(send_np, dtype, op, algo)
            for G in (1, 2, 3, 5):
                cuts = [0] + sorted(int(x) for x in rng.integers(1, count, G - 1)) + [count]
                got = []
                for lo, hi in zip(cuts[:-1], cuts[1:]):
                    send = [to_dev(a[lo:hi].copy(), dtype) for a in send_np]
                    recv = [torch.empty_like(x) for x in send]
                    gar.ar_allreduce_slice(send, recv, count, lo, op, algo)
                    got.append([from_dev(x) for x in recv])
                for r in range(n):
                    assert _same_bits(np.concatenate([g[r] for g in got]), want), (op, algo, G, r)
