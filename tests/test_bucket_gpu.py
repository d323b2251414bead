"""GPU parity of DDP-style bucketing: flatten -> allreduce (avg, bf16 in/out,
binary32 accumulation) -> unflatten, against the oracle's bucket plan and
ring allreduce. Full comparison on a reduced decoder; the 124M-parameter
GPT-2-small shape set on sampled elements."""
import math

import numpy as np
import pytest
import torch

import gradient_allreduce_collective_gb300 as gar
import oracle
import synthgen
from tests._dev import from_dev, to_dev

pytestmark = pytest.mark.gpu

CAP = 25 * 1024 * 1024


@pytest.fixture(scope="module", autouse=True)
def _built():
    gar.build()
    gar.lib()


def _same_bits(a, b):
    return np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


def test_flatten_unflatten_roundtrip():
    rng = np.random.default_rng(0)
    counts = [int(c) for c in rng.integers(0, 40_000, size=300)] + [0, 1, 3, 777_777]
    for dt, npdt in ((torch.float32, np.float32), (torch.bfloat16, np.uint16)):
        es = 4 if dt == torch.float32 else 2
        arena = torch.empty(sum(counts) + 8 * len(counts), dtype=dt, device="cuda")
        tensors, pos = [], 1  # odd start: some tensors are not 16-byte aligned
        for c in counts:
            tensors.append(arena[pos:pos + c])
            pos += c + int(rng.integers(0, 3))
        for t in tensors:
            t.view(torch.int16 if es == 2 else torch.int32).copy_(
                torch.randint(-30000, 30000, (t.numel(),), dtype=torch.int16 if es == 2 else torch.int32))
        bucket_of, offset_of, bcounts = gar.ar_bucket_plan(counts, dt, 1 << 20)
        for b, bc in enumerate(bcounts):
            ids = [t for t in range(len(counts)) if bucket_of[t] == b]
            bucket = torch.zeros(bc, dtype=dt, device="cuda")
            gar.ar_bucket_flatten([tensors[t] for t in ids], [offset_of[t] for t in ids], bucket)
            host = from_dev(bucket)
            for t in ids:
                assert _same_bits(host[offset_of[t]:offset_of[t] + counts[t]], from_dev(tensors[t]))
            back = [torch.empty_like(tensors[t]) for t in ids]
            gar.ar_bucket_unflatten(bucket, back, [offset_of[t] for t in ids])
            for t, x in zip(ids, back):
                assert _same_bits(from_dev(x), from_dev(tensors[t]))


def _model_shapes(d, vocab, ctx, layers):
    shapes = [(vocab, d), (ctx, d)]
    for _ in range(layers):
        shapes += [(d,), (d,), (d, 3 * d), (3 * d,), (d, d), (d,), (d,), (d,), (d, 4 * d), (4 * d,), (4 * d, d), (d,)]
    return shapes + [(d,), (d,)]


def _ddp_sync(shapes, nranks, cap, algo, seed=0):
    counts = [math.prod(s) for s in shapes]
    total = sum(counts)
    grads_np = synthgen.ranks_normal(nranks, total, 1e-4, base_seed=seed, dtype="bf16")
    arenas = [to_dev(g, "bf16") for g in grads_np]
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    views = [[arenas[r][int(s):int(s) + c] for s, c in zip(starts, counts)] for r in range(nranks)]
    bucket_of, offset_of, bcounts = gar.ar_bucket_plan(counts, torch.bfloat16, cap)
    for b, bc in enumerate(bcounts):
        ids = [t for t in range(len(counts)) if bucket_of[t] == b]
        # all ranks' buckets back to back: one flatten and one unflatten call per bucket
        flat = torch.empty(nranks * bc, dtype=torch.bfloat16, device="cuda")
        tens = [views[r][t] for r in range(nranks) for t in ids]
        offs = [r * bc + offset_of[t] for r in range(nranks) for t in ids]
        gar.ar_bucket_flatten(tens, offs, flat)
        ranks = [flat[r * bc:(r + 1) * bc] for r in range(nranks)]
        gar.ar_allreduce(ranks, ranks, "avg", algo)
        gar.ar_bucket_unflatten(flat, tens, offs)
    torch.cuda.synchronize()
    return grads_np, arenas, counts, starts, bucket_of, offset_of, bcounts


@pytest.mark.parametrize("algo", ["fused", "ring", "tree"])
def test_reduced_decoder_full_comparison(algo):
    shapes = _model_shapes(d=128, vocab=5003, ctx=256, layers=3)
    grads_np, arenas, counts, starts, bucket_of, offset_of, bcounts = _ddp_sync(shapes, 8, 1 << 20, algo)
    assert len(bcounts) > 2
    want_flat = np.empty(sum(counts), dtype=np.uint16)
    for b, bc in enumerate(bcounts):
        ids = [t for t in range(len(counts)) if bucket_of[t] == b]
        buckets = []
        for r in range(8):
            x = np.zeros(bc, dtype=np.uint16)
            for t in ids:
                x[offset_of[t]:offset_of[t] + counts[t]] = grads_np[r][starts[t]:starts[t] + counts[t]]
            buckets.append(x)
        fn = oracle.tree_allreduce if algo == "tree" else oracle.ring_allreduce
        y = fn(buckets, "bf16", "avg")[0]
        for t in ids:
            want_flat[starts[t]:starts[t] + counts[t]] = y[offset_of[t]:offset_of[t] + counts[t]]
    for r in range(8):
        assert _same_bits(from_dev(arenas[r]), want_flat)


def test_gpt2_small_sampled():
    shapes = [s for _, s in synthgen.gpt2_small_param_shapes()]
    grads_np, arenas, counts, starts, bucket_of, offset_of, bcounts = _ddp_sync(shapes, 8, CAP, "fused", seed=0)
    assert len(bcounts) == 9
    for r in range(1, 8):
        assert torch.equal(arenas[r].view(torch.int16), arenas[0].view(torch.int16))
    rng = np.random.default_rng(1)
    idx = np.sort(rng.choice(sum(counts), 200_000, replace=False))
    t_of = np.searchsorted(starts, idx, side="right") - 1
    bidx = np.array([offset_of[t] for t in t_of]) + (idx - starts[t_of])
    got = from_dev(arenas[0])[idx]
    vals = np.stack([g[idx] for g in grads_np], axis=1)
    for b, bc in enumerate(bcounts):
        m = np.array([bucket_of[t] == b for t in t_of])
        want = oracle.fold_points(vals[m], bidx[m], bc, "bf16", "avg")
        assert _same_bits(got[m], want), b
    # tolerance against fp64
    x = vals.astype(np.uint32) << 16
    xf = x.view(np.float32).astype(np.float64)
    ystar = xf.mean(axis=1)
    S = np.abs(xf).mean(axis=1)
    y = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ok = S > 0
    assert np.max(np.abs(y - ystar)[ok] / S[ok]) <= 1e-2


def _rank_views(grads, counts, starts):
    return [[g[int(s):int(s) + c] for s, c in zip(starts, counts)] for g in grads]


@pytest.mark.parametrize("algo", ["fused", "ring", "tree"])
@pytest.mark.parametrize("inplace", [True, False])
def test_bucket_allreduce_matches_three_step_path(algo, inplace):
    # ar_bucket_allreduce reads the tensors where they live; it must give the
    # bits of flatten -> allreduce -> unflatten (which the test above pins to the oracle)
    shapes = _model_shapes(d=128, vocab=5003, ctx=256, layers=3)
    counts = [math.prod(s) for s in shapes]
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    n = 8
    grads_np = synthgen.ranks_normal(n, sum(counts), 1e-4, base_seed=1, dtype="bf16")
    ref = [to_dev(g, "bf16") for g in grads_np]
    work = [to_dev(g, "bf16") for g in grads_np]
    outs = [torch.empty_like(w) for w in work]
    bucket_of, offset_of, bcounts = gar.ar_bucket_plan(counts, torch.bfloat16, 1 << 20)
    rv, wv, ov = _rank_views(ref, counts, starts), _rank_views(work, counts, starts), _rank_views(outs, counts, starts)
    for b, bc in enumerate(bcounts):
        ids = [t for t in range(len(counts)) if bucket_of[t] == b]
        flat = torch.empty(n * bc, dtype=torch.bfloat16, device="cuda")
        tens = [rv[r][t] for r in range(n) for t in ids]
        offs = [r * bc + offset_of[t] for r in range(n) for t in ids]
        gar.ar_bucket_flatten(tens, offs, flat)
        ranks = [flat[r * bc:(r + 1) * bc] for r in range(n)]
        gar.ar_allreduce(ranks, ranks, "avg", algo)
        gar.ar_bucket_unflatten(flat, tens, offs)
        src = [[wv[r][t] for t in ids] for r in range(n)]
        dst = src if inplace else [[ov[r][t] for t in ids] for r in range(n)]
        gar.ar_bucket_allreduce(src, dst, [offset_of[t] for t in ids], bc, "avg", algo)
    torch.cuda.synchronize()
    got = work if inplace else outs
    for r in range(n):
        assert torch.equal(got[r].view(torch.int16), ref[r].view(torch.int16))
    if not inplace:  # inputs untouched
        for r in range(n):
            assert _same_bits(from_dev(work[r]), grads_np[r])


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
def test_bucket_allreduce_against_oracle_ragged_unaligned(dtype):
    rng = np.random.default_rng(5)
    n = 5
    counts = [int(c) for c in rng.integers(1, 3000, size=40)] + [1, 7, 13]
    es = {"f32": 4, "bf16": 2, "i32": 4}[dtype]
    _, offset_of, bcounts = gar.ar_bucket_plan(counts, {"f32": torch.float32, "bf16": torch.bfloat16,
                                                        "i32": torch.int32}[dtype], 1 << 30)
    assert len(bcounts) == 1
    bc = bcounts[0]
    gen = (lambda k, s: synthgen.ranks_int(n, k, -(2**20), 2**20, base_seed=s)) if dtype == "i32" else \
        (lambda k, s: synthgen.ranks_normal(n, k, 1.0, base_seed=s, dtype=dtype))
    total = sum(counts)
    data = gen(total, 9)
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    for shift in (0, 1):  # shift 1: tensors off 16-byte alignment -> element path
        arenas = []
        for r in range(n):
            a = torch.zeros(total + 64, dtype={"f32": torch.float32, "bf16": torch.bfloat16,
                                               "i32": torch.int32}[dtype], device="cuda")
            a[shift:shift + total].copy_(to_dev(data[r], dtype))
            arenas.append(a)
        views = [[a[shift + int(s):shift + int(s) + c] for s, c in zip(starts, counts)] for a in arenas]
        gar.ar_bucket_allreduce(views, views, offset_of, bc, "sum", "fused")
        buckets = []
        for r in range(n):
            x = np.zeros(bc, dtype=data[r].dtype)
            for t, c in enumerate(counts):
                x[offset_of[t]:offset_of[t] + c] = data[r][starts[t]:starts[t] + c]
            buckets.append(x)
        y = oracle.ring_allreduce(buckets, dtype, "sum")[0]
        want = np.concatenate([y[offset_of[t]:offset_of[t] + c] for t, c in enumerate(counts)])
        for r in range(n):
            assert _same_bits(from_dev(arenas[r][shift:shift + total]), want), (shift, r)


@pytest.mark.parametrize("n", [16, 64])
def test_bucket_allreduce_many_ranks_batches_launches(n):
    # 1024 pointer slots per launch: 64 ranks -> 16 tensors per launch
    counts = [1000 + 8 * t for t in range(70)]
    _, offset_of, bcounts = gar.ar_bucket_plan(counts, torch.float32, 1 << 30)
    bc = bcounts[0]
    data = synthgen.ranks_normal(n, sum(counts), 1.0, base_seed=n)
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    dev = [to_dev(d, "f32") for d in data]
    views = [[g[int(s):int(s) + c] for s, c in zip(starts, counts)] for g in dev]
    outs = [torch.empty_like(g) for g in dev]
    oviews = [[g[int(s):int(s) + c] for s, c in zip(starts, counts)] for g in outs]
    gar.ar_bucket_allreduce(views, oviews, offset_of, bc, "sum", "tree")
    buckets = []
    for r in range(n):
        x = np.zeros(bc, dtype=np.float32)
        for t, c in enumerate(counts):
            x[offset_of[t]:offset_of[t] + c] = data[r][starts[t]:starts[t] + c]
        buckets.append(x)
    y = oracle.tree_allreduce(buckets, "f32", "sum")[0]
    want = np.concatenate([y[offset_of[t]:offset_of[t] + c] for t, c in enumerate(counts)])
    for r in range(n):
        assert _same_bits(from_dev(outs[r]), want)
