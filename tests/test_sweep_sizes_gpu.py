"""Parity at the message-size sweep's large sizes (8 ranks, fp32 uniform(-1,1)
sum; int32 uniform[-2^20, 2^20] min and max), through the C ABI.

The vasteelab page ("All-Reduce・All-Gather・All-to-Allとは？", §負荷試験)
asks for the message size to be varied from small to large, and the
AllReduce glossary's algorithm table (§主要なAllReduceアルゴリズム) defines
the orders compared. Two per-rank sizes are checked here: 16 MiB, the first
size of the doubling sweep whose 2·N·M bytes no longer fit in L2, and the
sweep's largest, 1 GiB per rank (8 GiB of inputs and 8 GiB of outputs; 256 MiB
per rank when the device or the host has no room for that).

The outputs are too large for the oracle to recompute in full, so each case
gathers about 10^6 points on the device and compares them bit for bit with
the oracle's per-element fold in the same order: every chunk boundary and its
neighbours, the first and last 64 elements, and random points. All 8 replicas
are compared with each other in full on the device.
"""
import os

import numpy as np
import pytest
import torch

import gradient_allreduce_collective_gb300 as gar
import oracle
import synthgen

pytestmark = pytest.mark.gpu

N = 8
LO_I, HI_I = -(2**20), 2**20
SMALL = 16 << 20
NRAND = 1_000_000


@pytest.fixture(scope="module", autouse=True)
def _built():
    gar.build()
    gar.lib()


def _large_bytes() -> int:
    """1 GiB per rank if 2 x 8 GiB fit on the device with room to spare and
    2 GiB of host memory is free, else 256 MiB."""
    free, _ = torch.cuda.mem_get_info()
    try:
        host_free = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError):  # pragma: no cover
        host_free = 0
    if free >= 2 * N * (1 << 30) + (4 << 30) and host_free >= 4 << 30:
        return 1 << 30
    return 256 << 20


def _points(count: int, seed: int) -> np.ndarray:
    """Chunk boundaries +-1 (chunk length of the allreduce's plan), the first
    and last 64 elements, and random points; sorted, unique, int64."""
    L = oracle.chunk_len(count, N, 4)
    pts = [np.arange(min(64, count)), np.arange(max(0, count - 64), count)]
    for c in range(1, N + 1):
        b = c * L
        pts.append(np.array([b - 2, b - 1, b, b + 1]))
    pts.append(np.random.default_rng(seed).integers(0, count, NRAND))
    idx = np.unique(np.concatenate(pts).astype(np.int64))
    return idx[(idx >= 0) & (idx < count)]


def _ranks(dtype: str, count: int, idx: np.ndarray):
    """Rank r's inputs (seed r) on the device, one rank at a time through the
    host, and the inputs at the sampled points: vals[j, r]."""
    vals = np.empty((idx.size, N), dtype=np.int32 if dtype == "i32" else np.float32)
    send = []
    for r in range(N):
        host = (synthgen.uniform_i32(count, r, LO_I, HI_I) if dtype == "i32"
                else synthgen.uniform_f32(count, r, -1.0, 1.0))
        vals[:, r] = host[idx]
        send.append(torch.from_numpy(host).cuda())
        del host
    return send, vals


def _run(dtype: str, ops_algos, count: int):
    idx = _points(count, seed=count % 9973)
    send, vals = _ranks(dtype, count, idx)
    recv = [torch.empty_like(s) for s in send]
    idx_dev = torch.from_numpy(idx).cuda()
    try:
        for op, algo in ops_algos:
            for r in recv:  # stale results from the previous case must not pass
                r.view(torch.int32).fill_(0x7FA5A5A5)
            gar.ar_allreduce(send, recv, op, algo)
            torch.cuda.synchronize()
            for r in range(1, N):
                assert torch.equal(recv[r].view(torch.int32), recv[0].view(torch.int32)), (op, algo, r)
            got = recv[0][idx_dev].cpu().numpy()
            if algo == "tree":
                want = oracle.tree_points(vals, dtype, op)
            else:  # the fused pass and reduce-scatter + all-gather fold in the ring's order
                want = oracle.fold_points(vals, idx, count, dtype, op)
            bad = np.flatnonzero(got.view(np.uint32) != want.view(np.uint32))
            assert bad.size == 0, (op, algo, count, idx[bad[:5]], got[bad[:5]], want[bad[:5]])
            if dtype == "i32":  # min and max are order-free: the plain definition as well
                ref = vals.min(axis=1) if op == "min" else vals.max(axis=1)
                assert np.array_equal(got, ref), (op, algo)
            else:  # within the recursive-summation bound of the fp64 sum
                x = vals.astype(np.float64)
                err = np.abs(got.astype(np.float64) - x.sum(axis=1)) / np.abs(x).sum(axis=1)
                assert err.max() <= 1e-6, (algo, err.max())
    finally:
        del send, recv, idx_dev
        torch.cuda.empty_cache()


F32_CASES = [("sum", "fused"), ("sum", "ring"), ("sum", "tree")]
I32_CASES = [(op, algo) for op in ("min", "max") for algo in ("fused", "tree", "ring")]


def test_f32_sum_16MiB_per_rank():
    _run("f32", F32_CASES, SMALL // 4)


def test_i32_min_max_16MiB_per_rank():
    _run("i32", I32_CASES, SMALL // 4)


def test_f32_sum_largest_size():
    _run("f32", F32_CASES, _large_bytes() // 4)


def test_i32_min_max_largest_size():
    _run("i32", I32_CASES, _large_bytes() // 4)
