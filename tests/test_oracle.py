"""Pins of the CPU oracle against what the pages and mathematics fix (no GPU).

Each test pins the oracle to something other than itself: values the pages
print, hand-computed cases, closed forms, invariants, library routines,
error bounds, or an independent algorithm (literal ring simulator vs the
per-element fold).
"""
import math

import numpy as np
import pytest

import oracle
import synthgen
from tests import _golden as G

ALL_DT = ("f32", "bf16", "f16", "i32")
FLOAT_DT = ("f32", "bf16", "f16")


def _as(dtype, vals):
    if dtype == "i32":
        return np.array(vals, dtype=np.int32)
    x = np.array(vals, dtype=np.float32)
    return x if dtype == "f32" else synthgen.to_dtype(x, dtype)


def _to_f32(dtype, a):
    if dtype == "bf16":
        return oracle.bf16_to_f32(a)
    if dtype == "f16":
        return oracle.f16_to_f32(a)
    return a.astype(np.float32)


def _rand(dtype, n, count, seed=0, sigma=1.0):
    if dtype == "i32":
        return synthgen.ranks_int(n, count, -(2**20), 2**20, base_seed=seed)
    return synthgen.ranks_normal(n, count, sigma, base_seed=seed, dtype=dtype)


# ---------------------------------------------------------------- page values

@pytest.mark.parametrize("dtype", ["i32", "f32", "bf16", "f16"])
@pytest.mark.parametrize("fn", ["ring", "fold", "tree"])
def test_worked_example(dtype, fn):
    g = G.load("worked_example_allreduce.txt")
    send = [_as(dtype, G.nums(g[f"rank{r}"])) for r in range(4)]
    out = getattr(oracle, f"{fn}_allreduce")(send, dtype, g["op"])
    want = G.nums(g["expect"])
    if dtype == "bf16":
        # the inputs are exact in bf16 but 1111 and 2222 are not (8 significant bits):
        # the page's exact result, rounded once by the library's conversion
        import torch
        want = torch.tensor(want).to(torch.bfloat16).float().tolist()
    for y in out:
        assert _to_f32(dtype, y).tolist() == want


def test_all_gather_rank_order():
    g = G.load("all_gather_rank_order.txt")
    send = [_as("i32", G.nums(g[f"rank{r}"], int)) for r in range(4)]
    for y in oracle.ring_all_gather(send, "i32"):
        assert y.tolist() == G.nums(g["expect"], int)


def test_reduce_scatter_placement():
    g = G.load("reduce_scatter_placement.txt")
    send = [_as("i32", G.nums(g[f"rank{r}"], int)) for r in range(2)]
    out = oracle.ring_reduce_scatter(send, "i32", g["op"])
    assert out[0].tolist() == G.nums(g["expect_rank0"], int)
    assert out[1].tolist() == G.nums(g["expect_rank1"], int)


# ---------------------------------------------------------- hand-computed pins

def test_ring_start_rank():
    g = G.load("ring_start_rank.txt")
    n = int(g["count"])
    send = [np.full(n, float(g[f"rank{r}"]), dtype=np.float32) for r in range(3)]
    for fn in (oracle.ring_allreduce, oracle.fold_allreduce):
        for y in fn(send, "f32", g["op"]):
            assert y.tolist() == G.nums(g["expect"])


def test_tree_order():
    g = G.load("tree_order.txt")
    send = [np.array([float(g[f"rank{r}"])], dtype=np.float32) for r in range(4)]
    assert oracle.tree_allreduce(send, "f32", "sum")[0].tolist() == G.nums(g["expect_tree"])
    assert oracle.ring_allreduce(send, "f32", "sum")[0].tolist() == G.nums(g["expect_ring"])


def test_gpt2_buckets():
    g = G.load("gpt2_buckets.txt")
    shapes = synthgen.gpt2_small_param_shapes()
    counts = [math.prod(s) for _, s in shapes]
    assert len(counts) == 148 and sum(counts) == 124_439_808
    esize = int(g["esize"])
    bucket_of, offset_of, bucket_counts = oracle.bucket_plan(counts, esize, int(g["cap_bytes"]))
    assert (bucket_counts * esize).tolist() == G.nums(g["expect_bytes"], int)
    # every tensor lies inside its bucket, 16-byte aligned, tensors do not overlap,
    # and bucket b holds tensors later in registration order than bucket b+1
    for b in range(len(bucket_counts)):
        ts = sorted((int(offset_of[t]), counts[t], t) for t in range(148) if bucket_of[t] == b)
        end = 0
        for off, c, t in ts:
            assert off % (16 // esize) == 0 and off >= end
            end = off + c
        assert end == bucket_counts[b]
    assert all(bucket_of[t] >= bucket_of[t + 1] for t in range(147))


def test_fp8_block_example():
    g = G.load("fp8_block_example.txt")
    send = [_as("bf16", G.nums(g[f"rank{r}"])) for r in range(2)]
    for op in ("sum", "avg"):
        for y in oracle.fp8_ring_allreduce(send, "bf16", "bf16", op):
            assert oracle.bf16_to_f32(y).tolist() == G.nums(g[f"expect_{op}"])


def test_nan_and_signed_zero_min_max():
    pz, nz = np.float32(0.0), np.float32(-0.0)
    send = [np.array([pz, nz, 1.0, np.nan], dtype=np.float32),
            np.array([nz, pz, np.nan, 2.0], dtype=np.float32)]
    for fn in (oracle.ring_allreduce, oracle.tree_allreduce):
        mn = fn(send, "f32", "min")[0].view(np.uint32).tolist()
        mx = fn(send, "f32", "max")[0].view(np.uint32).tolist()
        assert mn == [0x80000000, 0x80000000, 0x7FC00000, 0x7FC00000]
        assert mx == [0x00000000, 0x00000000, 0x7FC00000, 0x7FC00000]
    for dt, canon in (("bf16", 0x7FC0), ("f16", 0x7E00)):
        s2 = [synthgen.to_dtype(a, dt) for a in send]
        assert oracle.ring_allreduce(s2, dt, "min")[0].tolist() == [0x8000, 0x8000, canon, canon]
        assert oracle.ring_allreduce(s2, dt, "max")[0].tolist() == [0x0000, 0x0000, canon, canon]


def test_single_rank_nan_is_canonical():
    x = np.array([np.float32(np.nan), 1.0], dtype=np.float32)
    x.view(np.uint32)[0] = 0x7FA00001  # a NaN with a payload
    for op in ("min", "max"):
        assert oracle.ring_allreduce([x], "f32", op)[0].view(np.uint32).tolist() == [0x7FC00000, 0x3F800000]


def test_int32_wrap_and_truncating_average():
    send = [np.array([2**31 - 1, -7, 7, -8], dtype=np.int32), np.array([1, 0, 0, 1], dtype=np.int32)]
    assert oracle.ring_allreduce(send, "i32", "sum")[0].tolist() == [-(2**31), -7, 7, -7]
    assert oracle.ring_allreduce(send, "i32", "avg")[0].tolist() == [-(2**30), -3, 3, -3]


# ------------------------------------------------------------------ closed form

@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("op", ["sum", "avg"])
def test_sum_closed_form(n, op):
    count = 2 * 1024 + 37
    i = np.arange(count)
    send = [(r * 1024 + (i % 1024)).astype(np.float32) for r in range(n)]
    exact = 1024 * n * (n - 1) // 2 + n * (i % 1024)
    want = exact / n if op == "avg" else exact
    fns = [oracle.ring_allreduce, oracle.fold_allreduce] + ([oracle.tree_allreduce] if n & (n - 1) == 0 else [])
    for fn in fns:
        for y in fn(send, "f32", op):
            assert np.array_equal(y.astype(np.float64), want.astype(np.float64))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_low_precision_closed_form(dtype):
    # small integers are exact in both formats and their sum is exact in binary32, so the
    # result is the library's rounding of the exact sum (torch for bf16, numpy for fp16)
    import torch
    n, count = 8, 1000
    i = np.arange(count)
    send = [synthgen.to_dtype((r * 16 + (i % 8)).astype(np.float32) * 3, dtype) for r in range(n)]
    exact = (3 * (16 * n * (n - 1) // 2 + n * (i % 8))).astype(np.float32)
    if dtype == "bf16":
        want = torch.from_numpy(exact).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    else:
        want = exact.astype(np.float16).view(np.uint16)
    for y in oracle.ring_allreduce(send, dtype, "sum"):
        assert np.array_equal(y, want)


# -------------------------------------------------------------------- invariants

@pytest.mark.parametrize("dtype", ALL_DT)
@pytest.mark.parametrize("op", ["sum", "avg", "min", "max"])
@pytest.mark.parametrize("n", [1, 2, 3, 5, 8, 16])
def test_simulator_equals_fold(dtype, op, n):
    for count in (0, 1, 7, 33, 1021):
        send = _rand(dtype, n, count, seed=11 * n + count)
        ring = oracle.ring_allreduce(send, dtype, op)
        fold = oracle.fold_allreduce(send, dtype, op)
        for r in range(n):
            assert np.array_equal(ring[r].view(np.uint8), ring[0].view(np.uint8))  # replicas identical
            assert np.array_equal(fold[r].view(np.uint8), ring[0].view(np.uint8))


@pytest.mark.parametrize("dtype", ALL_DT)
@pytest.mark.parametrize("n", [1, 2, 4, 7, 8])
def test_reduce_scatter_then_all_gather_is_allreduce(dtype, n):
    v = 16 // (4 if dtype in ("f32", "i32") else 2)
    for per in (v, 5 * v):
        count = n * per
        send = _rand(dtype, n, count, seed=3 + n)
        for op in ("sum", "avg", "max"):
            rs = oracle.ring_reduce_scatter(send, dtype, op)
            ag = oracle.ring_all_gather(rs, dtype)
            ar = oracle.ring_allreduce(send, dtype, op)
            for r in range(n):
                assert np.array_equal(ag[r].view(np.uint8), ar[r].view(np.uint8))


@pytest.mark.parametrize("dtype", ALL_DT)
def test_min_max_match_numpy_and_are_order_free(dtype):
    n, count = 8, 4099
    send = _rand(dtype, n, count, seed=5)
    f = np.stack([_to_f32(dtype, a) if dtype != "i32" else a for a in send])
    for op, ref in (("min", f.min(axis=0)), ("max", f.max(axis=0))):
        outs = [oracle.ring_allreduce(send, dtype, op)[0], oracle.tree_allreduce(send, dtype, op)[0],
                oracle.fold_allreduce(send, dtype, op)[0]]
        for y in outs:
            assert np.array_equal(y.view(np.uint8), outs[0].view(np.uint8))
        got = _to_f32(dtype, outs[0]) if dtype != "i32" else outs[0]
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("dtype", ALL_DT)
@pytest.mark.parametrize("op", ["sum", "avg", "min", "max"])
def test_single_rank_is_identity(dtype, op):
    x = _rand(dtype, 1, 777, seed=9)  # finite values
    for fn in (oracle.ring_allreduce, oracle.tree_allreduce):
        assert np.array_equal(fn(x, dtype, op)[0], x[0])


def test_points_match_full_problem():
    n, count = 8, 50_003
    for dtype in ("f32", "bf16", "i32"):
        send = _rand(dtype, n, count, seed=21)
        full = oracle.ring_allreduce(send, dtype, "sum")[0]
        idx = np.random.default_rng(0).choice(count, 500, replace=False)
        vals = np.stack([a[idx] for a in send], axis=1)
        assert np.array_equal(oracle.fold_points(vals, idx, count, dtype, "sum"), full[idx])
        tfull = oracle.tree_allreduce(send, dtype, "sum")[0]
        assert np.array_equal(oracle.tree_points(vals, dtype, "sum"), tfull[idx])


# ------------------------------------------------------------------ error bounds

def _gamma(k):
    u = 2.0**-24
    return k * u / (1 - k * u)


@pytest.mark.parametrize("n", [2, 4, 8, 16])
@pytest.mark.parametrize("op", ["sum", "avg"])
def test_f32_error_bound(n, op):
    # recursive summation: |fl(sum) - sum| <= gamma_{n-1} * sum|x| (Higham, Accuracy and
    # Stability of Numerical Algorithms, 2nd ed., §4.2); a pairwise tree needs gamma_{log2 n};
    # the final division adds one more rounding
    count = 20_011
    send = synthgen.ranks_normal(n, count, 1e-3, base_seed=n)
    ystar, S = oracle.reference_f64(send, "f32", op)
    extra = 1 if op == "avg" else 0
    for fn, k in ((oracle.ring_allreduce, n - 1), (oracle.tree_allreduce, int(math.log2(n)))):
        y = fn(send, "f32", op)[0].astype(np.float64)
        bound = _gamma(k + extra) * S
        assert np.all(np.abs(y - ystar) <= bound + 1e-300)
        assert np.max(np.abs(y - ystar) / S) <= 1e-6


def test_bf16_output_error_bound():
    n, count = 8, 30_000
    send = synthgen.ranks_normal(n, count, 1e-4, base_seed=100, dtype="bf16")
    ystar, S = oracle.reference_f64(send, "bf16", "avg")
    y = oracle.bf16_to_f32(oracle.ring_allreduce(send, "bf16", "avg")[0]).astype(np.float64)
    # one bf16 rounding (relative 2^-8) on top of the binary32 sum and division
    bound = 2.0**-8 * np.abs(ystar) + (1 + 2.0**-8) * _gamma(n) * S
    assert np.all(np.abs(y - ystar) <= bound)
    assert np.max(np.abs(y - ystar) / S) <= 1e-2


def test_fp8_error_bounds():
    n, count = 16, 128 * 300 + 77
    send = synthgen.ranks_normal(n, count, 1e-3, base_seed=0, dtype="bf16", outlier_p=1e-3, outlier_scale=100.0)
    ystar, S = oracle.reference_f64(send, "bf16", "sum")
    y = oracle.bf16_to_f32(oracle.fp8_ring_allreduce(send, "bf16", "bf16", "sum")[0]).astype(np.float64)
    # a-priori bound: E4M3 rounding (relative 2^-4 for normals, so u/(1+u) of |x|) plus
    # half an E4M3 subnormal step s*2^-10 per element, the dequantise multiply, the
    # binary32 sum and one bf16 rounding
    x = np.stack([oracle.bf16_to_f32(a).astype(np.float64) for a in send])
    sc = np.stack([np.repeat(oracle.fp8_quantize(a, "bf16")[1].astype(np.float64), 128)[:count] for a in send])
    per = (0.0589 * np.abs(x) + sc * 2.0**-10).sum(axis=0)
    bound = per * (1 + 2.0**-23) + _gamma(n) * (S + per) + 2.0**-8 * (np.abs(ystar) + per + _gamma(n) * S)
    assert np.all(np.abs(y - ystar) <= bound)
    assert np.linalg.norm(y - ystar) / np.linalg.norm(ystar) <= 6e-2


def test_fp8_quantize_block_rules():
    # zero block -> scale 0, codes 0; block max maps to 448 (0x7E); partial last block
    x = np.zeros(128 + 5, dtype=np.float32)
    x[128:] = [3.0, -1.0, 0.5, 0.0, 6.0]
    q, s = oracle.fp8_quantize(x, "f32")
    assert s.tolist()[0] == 0.0 and not q[:128].any()
    assert s[1] == np.float32(6.0) / np.float32(448.0)
    assert q[132] == 0x7E and oracle.e4m3_to_f32(q[128:133]).tolist()[4] == 448.0
    # codes are the E4M3 rounding of x/s
    assert np.array_equal(q[128:], oracle.f32_to_e4m3(x[128:] / s[1]))


def test_fp8_blocks_match_full():
    n, count = 4, 128 * 40 + 50
    send = synthgen.ranks_normal(n, count, 1e-3, base_seed=3, dtype="bf16", outlier_p=1e-2, outlier_scale=100.0)
    full = oracle.fp8_ring_allreduce(send, "bf16", "bf16", "sum")[0]
    blocks_idx = [0, 7, 20, 39, 40]
    blk = np.zeros((len(blocks_idx), n, 128), dtype=np.uint16)
    first, blen = [], []
    for j, b in enumerate(blocks_idx):
        lo, hi = b * 128, min(b * 128 + 128, count)
        for r in range(n):
            blk[j, r, : hi - lo] = send[r][lo:hi]
        first.append(lo)
        blen.append(hi - lo)
    out = oracle.fp8_ring_blocks(blk, np.array(first), np.array(blen), count, "bf16", "bf16", "sum")
    for j, b in enumerate(blocks_idx):
        assert np.array_equal(out[j, : blen[j]], full[first[j]: first[j] + blen[j]])


def test_fp8_nan_makes_its_block_nan():
    # the block amax is the NaN-propagating maximum: a NaN anywhere in a block
    # (here the last element, after every larger magnitude, and a block of
    # zeros) makes its scale NaN and the whole block NaN; an infinity makes
    # the scale inf and the block NaN (inf/inf, 0*inf); other blocks unchanged
    # 2 ranks x 768 values: chunks of 384 = 3 blocks, so the per-hop path's
    # blocks (counted from each chunk's start) are the same 128-value blocks
    x = np.zeros(6 * 128, dtype=np.float32)
    x[128:] = np.linspace(-3, 3, 5 * 128, dtype=np.float32)
    x[127] = np.nan           # block 0: zeros and a NaN
    x[255] = np.nan           # block 1: values, the NaN last
    x[300] = np.inf           # block 2: an infinity
    q, s = oracle.fp8_quantize(x, "f32")
    assert np.isnan(s[0]) and np.isnan(s[1]) and np.isinf(s[2]) and np.isfinite(s[3:]).all()
    other = np.zeros_like(x)
    for fn in (oracle.fp8_ring_allreduce, oracle.fp8_hop_ring_allreduce):
        y = fn([x, other], "f32", "f32", "sum")[0]
        assert np.isnan(y[:384]).all() and not np.isnan(y[384:]).any(), fn.__name__
    y = oracle.fp8_ring_allreduce([x, other], "f32", "f32", "sum")[0]
    assert np.array_equal(y[384:], oracle.fp8_ring_allreduce([x[384:], other[384:]], "f32", "f32", "sum")[0])


def test_fp8_tree_example():
    # hand-computed: the recursive-halving pairing (x0 + x2) + (x1 + x3) after E4M3 quantisation,
    # distinct from the ring order and from the adjacent pairing
    g = G.load("fp8_tree_example.txt")
    send = [_as("bf16", G.nums(g[f"rank{r}"])) for r in range(4)]
    for op in ("sum", "avg"):
        for y in oracle.fp8_tree_allreduce(send, "bf16", "bf16", op):
            assert oracle.bf16_to_f32(y).tolist() == G.nums(g[f"expect_tree_{op}"])
        for y in oracle.fp8_ring_allreduce(send, "bf16", "bf16", op):
            assert oracle.bf16_to_f32(y).tolist() == G.nums(g[f"expect_ring_{op}"])


def test_fp8_tree_and_ring_agree_up_to_order():
    n, count = 8, 4096
    send = synthgen.ranks_normal(n, count, 1e-3, base_seed=8, dtype="bf16")
    a = oracle.bf16_to_f32(oracle.fp8_ring_allreduce(send, "bf16", "bf16", "avg")[0])
    b = oracle.bf16_to_f32(oracle.fp8_tree_allreduce(send, "bf16", "bf16", "avg")[0])
    assert np.max(np.abs(a - b)) <= 2.0**-7 * np.max(np.abs(a)) + 1e-12


def test_empty_inputs():
    for dtype in ALL_DT:
        send = _rand(dtype, 4, 0)
        assert all(y.size == 0 for y in oracle.ring_allreduce(send, dtype, "sum"))
        assert all(y.size == 0 for y in oracle.tree_allreduce(send, dtype, "sum"))
    assert oracle.bucket_plan([], 2, 1 << 20)[2].size == 0


# ------------------------------------------------------------------ FP8 per hop

def test_fp8_hop_example():
    g = G.load("fp8_hop_example.txt")
    send = [_as("bf16", G.nums(g[f"rank{r}"])) for r in range(2)]
    for op in ("sum", "avg"):
        for fn in (oracle.fp8_hop_ring_allreduce, oracle.fp8_hop_blocks_allreduce):
            for y in fn(send, "bf16", "bf16", op):
                assert oracle.bf16_to_f32(y).tolist() == G.nums(g[f"expect_{op}"])
    once = oracle.fp8_ring_allreduce(send, "bf16", "bf16", "sum")[0]
    assert oracle.bf16_to_f32(once).tolist() == G.nums(g["expect_once_sum"])


@pytest.mark.parametrize("n", [1, 2, 3, 5, 8, 16])
def test_fp8_hop_simulator_equals_block_fold(n):
    for count in (1, 100, 128 * 9 + 7, 128 * 40):
        send = synthgen.ranks_normal(n, count, 1e-3, base_seed=n * 7 + count, dtype="bf16", outlier_p=1e-2,
                                     outlier_scale=100.0)
        for op in ("sum", "avg"):
            a = oracle.fp8_hop_ring_allreduce(send, "bf16", "bf16", op)
            b = oracle.fp8_hop_blocks_allreduce(send, "bf16", "bf16", op)
            for r in range(n):
                assert np.array_equal(a[r], a[0]) and np.array_equal(b[r], a[0])


def test_fp8_hop_single_rank_equals_quantise_once():
    x = synthgen.ranks_normal(1, 128 * 50 + 3, 1e-3, base_seed=2, dtype="bf16", outlier_p=1e-2, outlier_scale=100.0)
    for op in ("sum", "avg"):
        assert np.array_equal(oracle.fp8_hop_ring_allreduce(x, "bf16", "bf16", op)[0],
                              oracle.fp8_ring_allreduce(x, "bf16", "bf16", op)[0])


def test_fp8_hop_error_bound_and_growth():
    # each hop's E4M3 rounding is at most u = 2^-4 relative to the block's magnitude
    # (u/(1+u) for normals) plus half a subnormal step s*2^-10; the bound below sums
    # those over the N-1 hops and the final quantisation, then the bf16 output rounding
    n, count = 16, 128 * 200
    send = synthgen.ranks_normal(n, count, 1e-3, base_seed=0, dtype="bf16", outlier_p=1e-3, outlier_scale=100.0)
    ystar, S = oracle.reference_f64(send, "bf16", "sum")
    hop = oracle.bf16_to_f32(oracle.fp8_hop_ring_allreduce(send, "bf16", "bf16", "sum")[0]).astype(np.float64)
    once = oracle.bf16_to_f32(oracle.fp8_ring_allreduce(send, "bf16", "bf16", "sum")[0]).astype(np.float64)
    e_hop = np.linalg.norm(hop - ystar) / np.linalg.norm(ystar)
    e_once = np.linalg.norm(once - ystar) / np.linalg.norm(ystar)
    # per-element: |partial error| grows at most by 0.0589*|partial| + 2^-10 * blockmax/448 per hop
    x = np.stack([oracle.bf16_to_f32(a).astype(np.float64) for a in send])
    blockmax = np.abs(np.cumsum(x, axis=0)).reshape(n, -1, 128).max(axis=2).repeat(128, axis=1)
    partial = np.abs(np.cumsum(x, axis=0))
    per = (0.0589 * (partial + S) + blockmax / 448 * 2.0**-10 * 2).sum(axis=0)
    assert np.all(np.abs(hop - ystar) <= per + 2.0**-8 * (np.abs(ystar) + per))
    assert e_hop <= 6e-2 * 4 and e_once <= 6e-2
    assert e_hop > e_once  # re-quantising partials on every hop loses more than quantising inputs once


# ------------------------------------------------------------- Top-K sparsification

def test_topk_hand_ties():
    g = G.load("topk_ties.txt")
    grad = np.array(G.nums(g["grad"]), dtype=np.float32)
    res = np.array(G.nums(g["residual"]), dtype=np.float32)
    idx, val, e = oracle.topk_compress(grad, res, 3)
    assert idx.tolist() == G.nums(g["k3_idx"], int) and val.tolist() == G.nums(g["k3_val"])
    idx, val, e = oracle.topk_compress(grad, res, 2)
    assert idx.tolist() == G.nums(g["k2_idx"], int) and val.tolist() == G.nums(g["k2_val"])
    assert e.tolist() == G.nums(g["k2_residual"])


def _nan_class_equal(got, want):
    """Bit-equal where `want` is a number, NaN where it is NaN (NaN payloads
    are unspecified, reading nan-order)."""
    got, want = np.asarray(got, dtype=np.float32), np.asarray(want, dtype=np.float32)
    nan = np.isnan(want)
    return np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_topk_nans_rank_above_every_number_and_tie():
    # Worked by hand: a NaN ranks above every number, +-inf included, and all
    # NaNs tie whatever their sign and payload (the lower index first); -0 + 0
    # is +0. Ranking: NaN (1), NaN (4), NaN (7), -inf (2), 3 (6), 2 (3), 1 (0), +0 (5).
    bits = [0x3F800000, 0x7FC00001, 0xFF800000, 0x40000000, 0xFFC12345, 0x80000000, 0x40400000, 0x7FA00000]
    grad = np.array(bits, dtype=np.uint32).view(np.float32)
    res = np.zeros(8, dtype=np.float32)
    nan = np.float32("nan")
    cases = {
        2: ([1, 4], [nan, nan], [1.0, 0.0, -np.inf, 2.0, 0.0, 0.0, 3.0, nan]),
        4: ([1, 2, 4, 7], [nan, -np.inf, nan, nan], [1.0, 0.0, 0.0, 2.0, 0.0, 0.0, 3.0, 0.0]),
        6: ([1, 2, 3, 4, 6, 7], [nan, -np.inf, 2.0, nan, 3.0, nan], [1.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0]),
    }
    for k, (want_idx, want_val, want_res) in cases.items():
        idx, val, e = oracle.topk_compress(grad, res, k)
        assert idx.tolist() == want_idx, k
        assert _nan_class_equal(val, want_val), k
        assert _nan_class_equal(e, want_res), k
        assert not np.any(e.view(np.uint32) == 0x80000000)  # the kept entries and -0 + 0 are +0


def test_topk_extremes_partition_and_brute_force():
    rng = np.random.default_rng(4)
    for count in (1, 7, 300, 5000):
        grad = synthgen.normal_f32(count, seed=count, sigma=1e-3)
        res = synthgen.normal_f32(count, seed=count + 1, sigma=1e-4)
        # ties on purpose: repeat some magnitudes
        grad[rng.integers(0, count, size=count // 10)] = np.float32(2e-3)
        a = (grad + res).astype(np.float32)
        for k in sorted({0, 1, count // 3, count}):
            idx, val, e = oracle.topk_compress(grad, res, k)
            assert idx.size == k and np.all(np.diff(idx.astype(np.int64)) > 0)
            dense = oracle.sparse_to_dense(idx, val, count)
            assert np.array_equal((dense + e).view(np.uint32), a.view(np.uint32))  # a = s + e, bitwise
            assert np.all(dense[e != 0] == 0)
            # brute force: the kept set is the k smallest (-|a|, index) pairs
            order = sorted(range(count), key=lambda i: (-abs(float(a[i])), i))[:k]
            assert sorted(order) == idx.tolist()


def test_sparse_allreduce_is_dense_allreduce_of_sparse_vectors():
    n, count, k = 8, 20_000, 2_000
    grads = synthgen.ranks_normal(n, count, 1e-3, base_seed=2)
    res = [np.zeros(count, dtype=np.float32) for _ in range(n)]
    sp = [oracle.topk_compress(g, e, k) for g, e in zip(grads, res)]
    y = oracle.sparse_ring_allreduce([s[0] for s in sp], [s[1] for s in sp], count, "avg")[0]
    dense = [oracle.sparse_to_dense(s[0], s[1], count) for s in sp]
    assert np.array_equal(y, oracle.ring_allreduce(dense, "f32", "avg")[0])
    # every kept value appears in the sum (at most n contributions per element)
    support = np.zeros(count, dtype=bool)
    for s in sp:
        support[s[0]] = True
    assert np.all(y[~support] == 0)


def test_error_feedback_conserves_the_gradient_mass():
    # over T steps, sent + final residual = sum of gradients (up to the rounding of g + e)
    count, k, T = 4000, 200, 6
    e = np.zeros(count, dtype=np.float32)
    sent = np.zeros(count, dtype=np.float64)
    total = np.zeros(count, dtype=np.float64)
    for t in range(T):
        g = synthgen.normal_f32(count, seed=100 + t, sigma=1e-3)
        idx, val, e = oracle.topk_compress(g, e, k)
        sent[idx] += val
        total += g
    err = np.abs(sent + e - total)
    assert np.all(err <= T * 2.0**-23 * (np.abs(total) + np.abs(sent) + 1e-3))


@pytest.mark.parametrize("threads", [1, 3, 8])
def test_threaded_fold_equals_the_ring_simulator(threads):
    # disjoint element ranges on host threads keep the whole problem's chunk plan
    for dtype in ("f32", "bf16", "i32"):
        for n, count in ((8, 100_003), (5, 4_099), (3, 7)):
            send = _rand(dtype, n, count, seed=31 * n)
            want = oracle.ring_allreduce(send, dtype, "sum")
            got = oracle.fold_allreduce_threads(send, dtype, "sum", threads)
            for g, w in zip(got, want):
                assert np.array_equal(np.asarray(g).view(np.uint8), np.asarray(w).view(np.uint8))
