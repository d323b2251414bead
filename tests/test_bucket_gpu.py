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
