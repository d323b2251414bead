"""GPU parity of Top-K sparsification with error feedback and of the sparse
allreduce, against the oracle: bit-exact indices, values and residuals on
seeded inputs (ragged sizes, heavy ties, signed zeros, k = 0 and k = count,
unaligned buffers, several steps of error feedback), and in full at the size
of one 25 MiB f32 gradient per rank on 8 ranks."""
import numpy as np
import pytest
import torch

import gradient_allreduce_collective_gb300 as gar
import oracle
import synthgen
from tests._dev import from_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gar.build()
    gar.lib()


def _bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


def _dev_f32(a: np.ndarray, offset: int) -> tuple[torch.Tensor, torch.Tensor]:
    """(base, view): a device copy of `a` starting `offset` elements into its allocation."""
    base = torch.empty(a.size + offset + 1, dtype=torch.float32, device="cuda")
    base.fill_(float("nan"))
    v = base[offset: offset + a.size]
    v.copy_(torch.from_numpy(np.ascontiguousarray(a)))
    return base, v


def _gpu_topk(g: np.ndarray, e: np.ndarray, k: int, offset: int = 0):
    count = g.size
    gb, gd = _dev_f32(g, offset)
    eb, ed = _dev_f32(e, offset)
    idx = torch.full((k + 8,), -1, dtype=torch.int32, device="cuda")
    val = torch.full((k + 8,), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(gar.ar_topk_workspace_bytes(1, count, k), 1), dtype=torch.uint8, device="cuda")
    ws.fill_(0x5A)  # the workspace needs no initialisation
    gar.ar_topk_compress([gd], [ed], k, [idx], [val], ws)
    torch.cuda.synchronize()
    i = from_dev(idx).view(np.uint32)
    v = from_dev(val)
    # nothing beyond k written, grad untouched, nothing outside the residual written
    assert np.all(i[k:] == 0xFFFFFFFF) and np.all(v[k:] == 7.0)
    assert np.array_equal(_bits(from_dev(gd)), _bits(g))
    eb_host = from_dev(eb)
    assert np.all(np.isnan(eb_host[:offset])) and np.all(np.isnan(eb_host[offset + count:]))
    return i[:k].copy(), v[:k].copy(), from_dev(ed).copy()


def _check_against_oracle(g, e, k, offset=0):
    gi, gv, ge = _gpu_topk(g, e, k, offset)
    oi, ov, oe = oracle.topk_compress(g, e, k)
    assert np.array_equal(gi, oi), "indices differ"
    assert np.array_equal(_bits(gv), _bits(ov)), "values differ"
    assert np.array_equal(_bits(ge), _bits(oe)), "residuals differ"


@pytest.mark.parametrize("count", [0, 1, 7, 4095, 4096, 4097, 100_003, (1 << 20) + 13])
def test_topk_matches_oracle_ragged(count):
    g = synthgen.normal_f32(count, 11, 1e-3)
    e = synthgen.normal_f32(count, 12, 1e-4)
    for k in sorted({0, min(1, count), max(min(1, count), count // 100), count // 2, count}):
        _check_against_oracle(g, e, k)


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_topk_unaligned_buffers_take_the_element_path(offset):
    count = 50_001
    g = synthgen.normal_f32(count, 21, 1.0)
    e = synthgen.normal_f32(count, 22, 0.1)
    for k in (1, 500, 25_000):
        _check_against_oracle(g, e, k, offset)


@pytest.mark.parametrize("unaligned_rank", [None, 3])
def test_topk_many_ranks_in_one_call(unaligned_rank):
    # 5 ranks with different data, scales and residuals; one unaligned rank
    # sends the whole call down the element path
    n, count, k = 5, 70_001, 700
    g_np = [synthgen.normal_f32(count, 500 + r, 10.0 ** -r) for r in range(n)]
    e_np = [synthgen.normal_f32(count, 600 + r, 10.0 ** (-r - 1)) for r in range(n)]
    keep = []
    grads, res = [], []
    for r in range(n):
        off = 1 if r == unaligned_rank else 0
        gb, gd = _dev_f32(g_np[r], off)
        eb, ed = _dev_f32(e_np[r], off)
        keep += [gb, eb]
        grads.append(gd)
        res.append(ed)
    idx = [torch.empty(k, dtype=torch.int32, device="cuda") for _ in range(n)]
    val = [torch.empty(k, dtype=torch.float32, device="cuda") for _ in range(n)]
    ws = torch.full((gar.ar_topk_workspace_bytes(n, count, k),), 0xC3, dtype=torch.uint8, device="cuda")
    gar.ar_topk_compress(grads, res, k, idx, val, ws)
    torch.cuda.synchronize()
    for r in range(n):
        oi, ov, oe = oracle.topk_compress(g_np[r], e_np[r], k)
        assert np.array_equal(from_dev(idx[r]).view(np.uint32), oi), r
        assert np.array_equal(_bits(from_dev(val[r])), _bits(ov)), r
        assert np.array_equal(_bits(from_dev(res[r])), _bits(oe)), r


@pytest.mark.parametrize("offset", [0, 1])
def test_topk_heavy_ties_and_signed_zeros(offset):
    # magnitudes from {0, 1, 2, 3}, both signs, both zeros: every threshold is
    # a tie that the lower indices win; the candidate slots overflow, so the
    # passes after the second read the data
    count = 30_011
    ints = synthgen.uniform_i32(count, 31, -3, 3)
    g = ints.astype(np.float32)
    g[ints == 0] = np.where(np.arange(count)[ints == 0] % 2 == 0, 0.0, -0.0).astype(np.float32)
    e = np.zeros(count, dtype=np.float32)
    e[::7] = -0.0
    nz3 = int(np.sum(np.abs(g) == 3))
    for k in (1, nz3 - 1, nz3, nz3 + 1, count // 2, count - 1, count):
        _check_against_oracle(g, e, k, offset)


@pytest.mark.parametrize("every,k,listed", [(600, 200, True), (40, 2000, False)])
def test_topk_match_list_with_ties(every, k, listed):
    # Ties at +-0.5 spread over every tile hold the threshold, all else is
    # small: the keys equal to T's two-digit prefix are the ties. With 334 of
    # them pass 3 lists them and derives the per-tile counts itself (the ties
    # kept in index order across tiles); with 5,000 the list overflows while
    # the slots still fit, and the count pass reads the slots instead.
    count = 200_000
    g = synthgen.normal_f32(count, 61, 1e-3)
    pos = np.arange(0, count, every)
    g[pos] = np.where(pos % 3 == 0, -0.5, 0.5).astype(np.float32)
    e = np.zeros(count, dtype=np.float32)
    ws = torch.full((gar.ar_topk_workspace_bytes(1, count, k),), 0x5A, dtype=torch.uint8, device="cuda")
    res = [to_dev(e, "f32")]
    idx = [torch.empty(k, dtype=torch.int32, device="cuda")]
    val = [torch.empty(k, dtype=torch.float32, device="cuda")]
    gar.ar_topk_compress([to_dev(g, "f32")], res, k, idx, val, ws)
    torch.cuda.synchronize()
    words = ws.view(torch.int32)
    assert int(words[2048 + 8]) == 0  # no slot overflow
    assert int(words[2048 + 16]) == pos.size and int(words[2048 + 17]) == int(listed)
    oi, ov, oe = oracle.topk_compress(g, e, k)
    assert np.array_equal(from_dev(idx[0]).view(np.uint32), oi)
    assert np.array_equal(_bits(from_dev(val[0])), _bits(ov))
    assert np.array_equal(_bits(from_dev(res[0])), _bits(oe))


def test_topk_one_overflowing_tile():
    # a block of equal magnitudes inside one tile holds the threshold: that
    # tile's candidates overflow their slots while every other tile's fit
    count = 200_000
    g = synthgen.normal_f32(count, 51, 1e-3)
    g[40_000:46_000] = np.where(np.arange(6_000) % 3 == 0, -0.5, 0.5).astype(np.float32)
    e = np.zeros(count, dtype=np.float32)
    for k in (100, 3_000, 6_000, 6_001, 8_000):
        _check_against_oracle(g, e, k)


def test_topk_special_values():
    count = 9000
    g = synthgen.normal_f32(count, 41, 1.0)
    g[5] = np.inf
    g[17] = -np.inf
    g[100:200] = np.float32(1e-45)  # subnormals
    g[300] = np.finfo(np.float32).max
    e = np.zeros(count, dtype=np.float32)
    e[300] = np.finfo(np.float32).max  # overflows to +inf in a = g + e
    for k in (1, 2, 3, 4, 50, 8950, count):
        _check_against_oracle(g, e, k)


def _nan_class_equal(got, want):
    """Bit-equal where `want` is a number, NaN where it is NaN (NaN payloads
    are unspecified: the device's add returns its own canonical NaN)."""
    got, want = np.asarray(got, dtype=np.float32), np.asarray(want, dtype=np.float32)
    nan = np.isnan(want)
    return np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def _nan_inputs(count, seed, n_nan, n_inf):
    g = synthgen.normal_f32(count, seed, 1e-3)
    rng = np.random.default_rng(seed)
    pos = rng.choice(count, size=n_nan + n_inf, replace=False)
    payload = rng.integers(1, 1 << 22, size=n_nan, dtype=np.uint32) | np.uint32(0x7F800000)
    sign = rng.integers(0, 2, size=n_nan, dtype=np.uint32) << np.uint32(31)
    g[pos[:n_nan]] = (payload | sign).view(np.float32)  # quiet and signalling, both signs
    g[pos[n_nan:]] = np.where(rng.integers(0, 2, size=n_inf) == 1, np.inf, -np.inf).astype(np.float32)
    return g


@pytest.mark.parametrize("k", [50, 299, 300, 301, 2000])
def test_topk_nans_rank_above_every_number(k):
    # 300 NaNs (random payloads and signs, some signalling) and 40 infinities
    # among small values: the NaNs tie above every number, the lower index
    # first; k below, at and above the NaN count.
    count = 50_000
    g = _nan_inputs(count, 71, 300, 40)
    e = np.zeros(count, dtype=np.float32)
    gi, gv, ge = _gpu_topk(g, e, k)
    oi, ov, oe = oracle.topk_compress(g, e, k)
    assert np.array_equal(gi, oi)
    assert _nan_class_equal(gv, ov) and _nan_class_equal(ge, oe)


def test_topk_nans_on_the_speculative_path():
    # Eight ranks large enough for the speculative pass 1, two calls on one
    # workspace: rank 0 with fewer NaNs than k (T a number), rank 1 with more
    # (T a NaN: the next hint is the infinity's key), the rest without.
    n, count, k = 8, 5_242_880, 52_428
    g_np = [synthgen.normal_f32(count, 500 + r, 1e-3) for r in range(n)]
    g_np[0] = _nan_inputs(count, 501, 10_000, 100)
    g_np[1] = _nan_inputs(count, 502, 60_000, 100)
    grads = [to_dev(x, "f32") for x in g_np]
    ws = torch.full((gar.ar_topk_workspace_bytes(n, count, k),), 0x5A, dtype=torch.uint8, device="cuda")
    e_np = [np.zeros(count, dtype=np.float32) for _ in range(n)]
    res = [torch.zeros(count, dtype=torch.float32, device="cuda") for _ in range(n)]
    idx = [torch.empty(k, dtype=torch.int32, device="cuda") for _ in range(n)]
    val = [torch.empty(k, dtype=torch.float32, device="cuda") for _ in range(n)]
    for call in range(2):
        gar.ar_topk_compress(grads, res, k, idx, val, ws)
        torch.cuda.synchronize()
        for r in (0, 1, 2):
            oi, ov, e_np[r] = oracle.topk_compress(g_np[r], e_np[r], k)
            assert np.array_equal(from_dev(idx[r]).view(np.uint32), oi), (call, r)
            assert _nan_class_equal(from_dev(val[r]), ov), (call, r)
            assert _nan_class_equal(from_dev(res[r]), e_np[r]), (call, r)


def test_error_feedback_over_several_steps():
    count, k = 200_000, 2_000
    e_host = np.zeros(count, dtype=np.float32)
    ed = torch.zeros(count, dtype=torch.float32, device="cuda")
    idx = torch.empty(k, dtype=torch.int32, device="cuda")
    val = torch.empty(k, dtype=torch.float32, device="cuda")
    ws = torch.empty(gar.ar_topk_workspace_bytes(1, count, k), dtype=torch.uint8, device="cuda")
    for step in range(4):
        g = synthgen.normal_f32(count, 100 + step, 1e-3)
        gar.ar_topk_compress([to_dev(g, "f32")], [ed], k, [idx], [val], ws)
        oi, ov, e_host = oracle.topk_compress(g, e_host, k)
        torch.cuda.synchronize()
        assert np.array_equal(from_dev(idx).view(np.uint32), oi)
        assert np.array_equal(_bits(from_dev(val)), _bits(ov))
        assert np.array_equal(_bits(from_dev(ed)), _bits(e_host))


def _algos(n):
    pow2 = n & (n - 1) == 0
    return ["ring", "fused", "auto", "step_ring"] + (["tree", "step_tree"] if pow2 else [])


@pytest.mark.parametrize("n", [1, 3, 4, 8])
def test_sparse_allreduce_matches_oracle(n):
    count = 40_009
    idx_np, val_np = [], []
    for r in range(n):
        g = synthgen.normal_f32(count, 200 + r, 1.0)
        k = [count // 100, 0, count, 517, 3, 1, 4000, count // 2][r % 8]
        i, v, _ = oracle.topk_compress(g, np.zeros(count, dtype=np.float32), k)
        idx_np.append(i)
        val_np.append(v)
    idx = [torch.from_numpy(i.view(np.int32)).cuda() if i.size else torch.empty(0, dtype=torch.int32, device="cuda")
           for i in idx_np]
    val = [to_dev(v, "f32") if v.size else torch.empty(0, dtype=torch.float32, device="cuda") for v in val_np]
    nnz = [i.size for i in idx_np]
    for op in ("sum", "avg", "max"):
        for algo in _algos(n):
            out = [torch.full((count,), float("nan"), device="cuda") for _ in range(n)]
            ws = torch.empty(gar.ar_sparse_workspace_bytes(n, count), dtype=torch.uint8, device="cuda")
            ws.fill_(0x77)  # needs no initialisation
            gar.ar_sparse_allreduce(idx, val, nnz, out, op, algo, ws)
            torch.cuda.synchronize()
            dense = [oracle.sparse_to_dense(i, v, count) for i, v in zip(idx_np, val_np)]
            if algo in ("tree", "step_tree"):
                want = oracle.tree_allreduce(dense, "f32", op)[0]
            else:
                want = oracle.sparse_ring_allreduce(idx_np, val_np, count, op)[0]
            for r in range(n):
                assert np.array_equal(_bits(from_dev(out[r])), _bits(want)), (op, algo, r)


@pytest.mark.parametrize("n", [3, 4])
def test_sparse_allreduce_signed_zeros_and_overlaps(n):
    # Values with signed zeros, opposite signs and rounding-sensitive
    # magnitudes on indices that several ranks share: the fold reads only the
    # present values, an absent one counting as +0 in the same order, so the
    # bits (-0 only where every rank holds -0) must equal the dense forms'.
    count = 9_001
    pick = np.array([-0.0, 0.0, 1.0, -1.0, 1e-8, -1e-8, 3.0e38, -3.0e38, 0.1, -0.3], dtype=np.float32)
    rng = np.random.default_rng(5)
    idx_np, val_np = [], []
    for r in range(n):
        i = np.union1d([0], np.arange(r % 2, count, 1 + r % 3)).astype(np.uint32)
        v = pick[rng.integers(0, pick.size, i.size)]
        v[0] = np.float32(-0.0)  # every rank holds -0 at index 0
        idx_np.append(i)
        val_np.append(v)
    idx = [torch.from_numpy(i.view(np.int32)).cuda() for i in idx_np]
    val = [to_dev(v, "f32") for v in val_np]
    nnz = [i.size for i in idx_np]
    dense = [oracle.sparse_to_dense(i, v, count) for i, v in zip(idx_np, val_np)]
    for op in ("sum", "avg"):
        for algo in _algos(n):
            out = [torch.full((count,), float("nan"), device="cuda") for _ in range(n)]
            ws = torch.empty(gar.ar_sparse_workspace_bytes(n, count), dtype=torch.uint8, device="cuda")
            gar.ar_sparse_allreduce(idx, val, nnz, out, op, algo, ws)
            torch.cuda.synchronize()
            if algo in ("tree", "step_tree"):
                want = oracle.tree_allreduce(dense, "f32", op)[0]
            else:
                want = oracle.sparse_ring_allreduce(idx_np, val_np, count, op)[0]
            for r in range(n):
                assert np.array_equal(_bits(from_dev(out[r])), _bits(want)), (op, algo, r)


def test_sparse_allreduce_drops_out_of_range_indices():
    count = 1000
    idx = torch.tensor([0, 999, 1000, 5000], dtype=torch.int32, device="cuda")
    val = torch.tensor([1.0, 2.0, 3.0, 4.0], device="cuda")
    out = [torch.full((count + 64,), 9.0, device="cuda")]
    ws = torch.empty(gar.ar_sparse_workspace_bytes(1, count), dtype=torch.uint8, device="cuda")
    gar.ar_sparse_allreduce([idx], [val], [4], [out[0][:count]], "sum", "fused", ws)
    torch.cuda.synchronize()
    h = from_dev(out[0])
    assert h[0] == 1.0 and h[999] == 2.0 and np.all(h[1:999] == 0.0) and np.all(h[count:] == 9.0)


def test_topk_full_size_eight_ranks():
    """8 ranks x 6,553,600 f32 (25 MiB each), k = 1%: every rank's indices,
    values and residual against the oracle in full, the defining properties
    checked on the device, and the sparse allreduce of the oracle's pairs on
    sampled elements against the oracle's ring-order fold."""
    n, count = 8, 6_553_600
    k = count // 100
    g_np = synthgen.ranks_normal(n, count, 1e-3, base_seed=300)
    e_np = synthgen.ranks_normal(n, count, 1e-4, base_seed=400)
    grads = [to_dev(x, "f32") for x in g_np]
    res = [to_dev(x, "f32") for x in e_np]
    idx = [torch.empty(k, dtype=torch.int32, device="cuda") for _ in range(n)]
    val = [torch.empty(k, dtype=torch.float32, device="cuda") for _ in range(n)]
    ws = torch.empty(gar.ar_topk_workspace_bytes(n, count, k), dtype=torch.uint8, device="cuda")
    gar.ar_topk_compress(grads, res, k, idx, val, ws)
    torch.cuda.synchronize()
    o_idx, o_val = [], []
    for r in range(n):
        oi, ov, oe = oracle.topk_compress(g_np[r], e_np[r], k)
        assert np.array_equal(from_dev(idx[r]).view(np.uint32), oi), r
        assert np.array_equal(_bits(from_dev(val[r])), _bits(ov)), r
        assert np.array_equal(_bits(from_dev(res[r])), _bits(oe)), r
        o_idx.append(oi)
        o_val.append(ov)
        # the defining properties: ascending indices, kept magnitudes never below dropped ones
        i = idx[r].long()
        assert bool((i[1:] > i[:-1]).all())
        assert float(res[r].abs().max()) <= float(val[r].abs().min())
    # sparse allreduce of the oracle's pairs
    d_idx = [torch.from_numpy(i.view(np.int32)).cuda() for i in o_idx]
    d_val = [to_dev(v, "f32") for v in o_val]
    out = [torch.empty(count, device="cuda") for _ in range(n)]
    sws = torch.empty(gar.ar_sparse_workspace_bytes(n, count), dtype=torch.uint8, device="cuda")
    gar.ar_sparse_allreduce(d_idx, d_val, [k] * n, out, "avg", "fused", sws)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    sample = np.unique(np.concatenate([rng.integers(0, count, 4000)] + [i[:64].astype(np.int64) for i in o_idx]))
    vals = np.stack([oracle.sparse_to_dense(i, v, count)[sample] for i, v in zip(o_idx, o_val)], axis=1)
    want = oracle.fold_points(vals, sample, count, "f32", "avg")
    for r in range(n):
        assert np.array_equal(_bits(from_dev(out[r])[sample]), _bits(want)), r


def test_sparse_allreduce_unsorted_indices_stay_in_bounds():
    # out-of-order indices give an unspecified sum but never an access outside
    # the buffers: the canaries around every output stay intact
    from tests._dev import Guarded
    n, count, k = 4, 30_011, 3_000
    rng = np.random.default_rng(7)
    idx, val = [], []
    for r in range(n):
        i = rng.permutation(count)[:k].astype(np.int32)
        idx.append(torch.from_numpy(i).cuda())
        val.append(torch.from_numpy(rng.standard_normal(k).astype(np.float32)).cuda())
    out = Guarded(n, count, "f32")
    ws = torch.empty(gar.ar_sparse_workspace_bytes(n, count), dtype=torch.uint8, device="cuda")
    gar.ar_sparse_allreduce(idx, val, [k] * n, out.views, "sum", "fused", ws)
    out.check()
    # sorted, the same pairs give the oracle's bits
    order = [torch.argsort(i) for i in idx]
    idx_s = [i[o].contiguous() for i, o in zip(idx, order)]
    val_s = [v[o].contiguous() for v, o in zip(val, order)]
    gar.ar_sparse_allreduce(idx_s, val_s, [k] * n, out.views, "sum", "fused", ws)
    out.check()
    want = oracle.sparse_ring_allreduce([from_dev(i).view(np.uint32) for i in idx_s], [from_dev(v) for v in val_s],
                                        count, "sum")[0]
    for r in range(n):
        assert np.array_equal(_bits(from_dev(out.views[r])), _bits(want))


@pytest.mark.parametrize("offset", [0, 1])
def test_topk_workspace_reused_across_steps(offset):
    # One workspace for eight steps of error feedback while the gradient scale
    # holds still, jumps up by 1e3 and drops by 1e6: the oracle's bits every
    # step; unaligned buffers take the element path.
    n, count, k = 3, 300_007, 3_000
    ws = torch.full((gar.ar_topk_workspace_bytes(n, count, k),), 0x5A, dtype=torch.uint8, device="cuda")
    e_np = [np.zeros(count, dtype=np.float32) for _ in range(n)]
    keep = []
    res = []
    for r in range(n):
        eb, ed = _dev_f32(e_np[r], offset)
        keep.append(eb)
        res.append(ed)
    idx = [torch.empty(k, dtype=torch.int32, device="cuda") for _ in range(n)]
    val = [torch.empty(k, dtype=torch.float32, device="cuda") for _ in range(n)]
    for step, scale in enumerate([1.0, 1.0, 1.05, 1e3, 1e3, 1e-3, 1.0, 1.0]):
        g_np = [synthgen.normal_f32(count, 800 + 10 * step + r, 1e-3 * scale) for r in range(n)]
        grads = []
        for r in range(n):
            gb, gd = _dev_f32(g_np[r], offset)
            keep.append(gb)
            grads.append(gd)
        gar.ar_topk_compress(grads, res, k, idx, val, ws)
        torch.cuda.synchronize()
        for r in range(n):
            oi, ov, e_np[r] = oracle.topk_compress(g_np[r], e_np[r], k)
            assert np.array_equal(from_dev(idx[r]).view(np.uint32), oi), (step, r)
            assert np.array_equal(_bits(from_dev(val[r])), _bits(ov)), (step, r)
            assert np.array_equal(_bits(from_dev(res[r])), _bits(e_np[r])), (step, r)


HINT_SCALES = np.array([0.99, 0.98, 0.95, 0.9, 0.8, 0.5], dtype=np.float32)  # by margin level


def _spec_decision(a: np.ndarray, hint: int, k: int, slots: int):
    """Whether pass 1's speculative slots serve the split pass for values a,
    whether fewer than k keys (bits 30..0 of a) lie at or above the hint, and
    T, the k-th largest key: the slots serve when at least k keys are at or
    above the hint (so T is one of them) and no tile of 16,384 values has
    more of them than its slots hold."""
    key = a.view(np.uint32) & 0x7FFFFFFF
    nb = -(-key.size // 16384)
    above = np.zeros(nb * 16384, dtype=bool)  # padding past the end never counts
    above[:key.size] = key >= np.uint32(hint)
    cand = np.count_nonzero(above.reshape(nb, 16384), axis=1)
    short = int(cand.sum()) < k
    ok = not short and int(cand.max()) <= slots
    return ok, short, int(np.sort(key)[key.size - k])


def _next_hint(T: int, margin: int, ok: bool, short: bool):
    """The hint and margin word a call leaves: the margin level (bits 0..7;
    outside the table it counts as 2, with an empty run) widens by one after
    a call whose candidates fell short of k, and narrows by one after 16
    calls in a row whose slots served (the run, bits 8..); the hint is the
    key of T's magnitude times the level's factor, rounded to nearest (the
    infinity's key for an infinite or NaN T)."""
    level, run = margin & 0xFF, margin >> 8
    if level >= HINT_SCALES.size:
        level, run = 2, 0
    if ok:
        run += 1
        if run >= 16:
            if level > 0:
                level, run = level - 1, 0
            else:
                run = 16
    else:
        run = 0
        if short and level + 1 < HINT_SCALES.size:
            level += 1
    if T >= 0x7F800000:
        return 0x7F800000, level | run << 8
    return int((np.uint32(T).view(np.float32) * HINT_SCALES[level]).view(np.uint32)), level | run << 8


def test_topk_speculative_first_pass_across_steps():
    # Large enough for pass 1 to compact its candidates speculatively (a warp
    # per tile of 16,384 values). The hint it uses comes from the previous
    # call on the same workspace: garbage on the first call (too high: the
    # margin widens), far too low (every tile overflowing) when the gradient
    # scale jumps by 1e3, valid while the residual that jump left decays and
    # once the scale holds. The bits must equal the oracle's every step
    # whichever path ran; the path taken (rank 0's spec_ok word in the
    # workspace) and the hint left for the next call must be the ones the
    # rule gives.
    n, count, k = 8, 5_242_880, 52_428
    share = -(-k * 16384 // count)
    slots = min(8192, -(-(16 * share + 1024) // 32) * 32)
    ws = torch.full((gar.ar_topk_workspace_bytes(n, count, k),), 0x5A, dtype=torch.uint8, device="cuda")
    state_hint, state_spec_ok, state_pre2 = 2048 + 9, 2048 + 10, 2048 + 14  # words of rank 0's workspace
    t_prev = margin = 0x5A5A5A5A
    hint = 0x5A5A5A5A
    e_np = [np.zeros(count, dtype=np.float32) for _ in range(n)]
    res = [torch.zeros(count, dtype=torch.float32, device="cuda") for _ in range(n)]
    idx = [torch.empty(k, dtype=torch.int32, device="cuda") for _ in range(n)]
    val = [torch.empty(k, dtype=torch.float32, device="cuda") for _ in range(n)]
    spec_steps = 0
    for step, scale in enumerate([1.0, 1.0, 1.0, 1e3, 1e-3, 1.0, 1.0, 1.0]):
        g_np = [synthgen.normal_f32(count, 900 + 10 * step + r, 1e-3 * scale) for r in range(n)]
        want_ok, short, T = _spec_decision(g_np[0] + e_np[0], hint, k, slots)
        want_pre2 = want_ok and (T >> 20) == (t_prev >> 20)  # the previous T's first digit held
        hint, margin = _next_hint(T, margin, want_ok, short)
        t_prev = T
        grads = [to_dev(x, "f32") for x in g_np]
        gar.ar_topk_compress(grads, res, k, idx, val, ws)
        torch.cuda.synchronize()
        assert int(ws.view(torch.int32)[state_spec_ok]) == int(want_ok), step
        assert int(ws.view(torch.int32)[state_hint]) == hint, step
        assert int(ws.view(torch.int32)[state_pre2]) == int(want_pre2), step
        spec_steps += int(want_ok)
        for r in range(n):
            oi, ov, e_np[r] = oracle.topk_compress(g_np[r], e_np[r], k)
            assert np.array_equal(from_dev(idx[r]).view(np.uint32), oi), (step, r)
            assert np.array_equal(_bits(from_dev(val[r])), _bits(ov)), (step, r)
            assert np.array_equal(_bits(from_dev(res[r])), _bits(e_np[r])), (step, r)
    assert spec_steps >= 3


def test_topk_first_digit_guess_skips_the_split_pass():
    # The same gradients and a zero residual on every call: from the second
    # call on the hint holds and T's first digit is the previous call's, so
    # pass 1 finds the second digit from its own histogram of the candidates
    # in that bin and the split pass returns at once. The bits must not
    # change.
    n, count, k = 8, 5_242_880, 52_428
    g_np = [synthgen.normal_f32(count, 700 + r, 1e-3) for r in range(n)]
    want = [oracle.topk_compress(g, np.zeros(count, dtype=np.float32), k) for g in g_np]
    ws = torch.full((gar.ar_topk_workspace_bytes(n, count, k),), 0x5A, dtype=torch.uint8, device="cuda")
    grads = [to_dev(x, "f32") for x in g_np]
    idx = [torch.empty(k, dtype=torch.int32, device="cuda") for _ in range(n)]
    val = [torch.empty(k, dtype=torch.float32, device="cuda") for _ in range(n)]
    for call in range(3):
        res = [torch.zeros(count, dtype=torch.float32, device="cuda") for _ in range(n)]
        gar.ar_topk_compress(grads, res, k, idx, val, ws)
        torch.cuda.synchronize()
        words = ws.view(torch.int32)
        assert int(words[2048 + 10]) == int(call > 0) and int(words[2048 + 14]) == int(call > 0), call
        assert int(words[2048 + 17]) == 1, call  # pass 3 derived the counts
        for r in range(n):
            wi, wv, we = want[r]
            assert np.array_equal(from_dev(idx[r]).view(np.uint32), wi), (call, r)
            assert np.array_equal(_bits(from_dev(val[r])), _bits(wv)), (call, r)
            assert np.array_equal(_bits(from_dev(res[r])), _bits(we)), (call, r)


def test_topk_hint_margin_widens_and_narrows():
    # The margin word of rank 0's state is set by hand between calls to reach
    # every transition: a run of 16 served calls narrows the level, a run at
    # the narrowest level stays capped, and a threshold that falls by 3 %
    # below a 0.99 hint (fewer than k candidates) costs that call the pass
    # over the data and widens the level. The residual is reset each call, so
    # a = g * scale; the bits must equal the oracle's on every call.
    n, count, k = 8, 5_242_880, 52_428
    share = -(-k * 16384 // count)
    slots = min(8192, -(-(16 * share + 1024) // 32) * 32)
    g1 = [synthgen.normal_f32(count, 800 + r, 1e-3) for r in range(n)]
    inputs = {1.0: g1, 0.97: [x * np.float32(0.97) for x in g1]}
    zero = np.zeros(count, dtype=np.float32)
    want = {sc: [oracle.topk_compress(x, zero, k) for x in xs] for sc, xs in inputs.items()}
    dev = {sc: [to_dev(x, "f32") for x in xs] for sc, xs in inputs.items()}
    ws = torch.full((gar.ar_topk_workspace_bytes(n, count, k),), 0x5A, dtype=torch.uint8, device="cuda")
    words = ws.view(torch.int32)
    idx = [torch.empty(k, dtype=torch.int32, device="cuda") for _ in range(n)]
    val = [torch.empty(k, dtype=torch.float32, device="cuda") for _ in range(n)]
    hint, margin = 0x5A5A5A5A, 0x5A5A5A5A
    # (input scale, margin word written before the call or None, expected spec_ok)
    plan = [(1.0, None, False), (1.0, 2 | 15 << 8, True), (1.0, 0, True), (0.97, None, False),
            (0.97, None, True), (0.97, 0 | 15 << 8, True)]
    for call, (sc, set_margin, want_ok) in enumerate(plan):
        if set_margin is not None:
            words[2048 + 15] = set_margin
            margin = set_margin
        ok, short, T = _spec_decision(inputs[sc][0], hint, k, slots)
        assert ok == want_ok, call  # the plan itself follows the rule
        hint, margin = _next_hint(T, margin, ok, short)
        res = [torch.zeros(count, dtype=torch.float32, device="cuda") for _ in range(n)]
        gar.ar_topk_compress(dev[sc], res, k, idx, val, ws)
        torch.cuda.synchronize()
        assert int(words[2048 + 10]) == int(ok), call
        assert int(words[2048 + 9]) == hint and int(words[2048 + 15]) == margin, (call, hex(margin))
        for r in range(n):
            wi, wv, we = want[sc][r]
            assert np.array_equal(from_dev(idx[r]).view(np.uint32), wi), (call, r)
            assert np.array_equal(_bits(from_dev(val[r])), _bits(wv)), (call, r)
            assert np.array_equal(_bits(from_dev(res[r])), _bits(we)), (call, r)
    assert margin == 0 | 16 << 8  # the last call capped the run at the narrowest level


@pytest.mark.parametrize("n", [16, 64])
def test_topk_and_sparse_allreduce_many_ranks(n):
    # the most ranks one call takes: a shared-memory fold tile of 8192 / N values
    count, k = 20_011, 150
    g_np = [synthgen.normal_f32(count, 900 + r, 1.0) for r in range(n)]
    e_np = [synthgen.normal_f32(count, 1900 + r, 0.1) for r in range(n)]
    grads = [to_dev(x, "f32") for x in g_np]
    res = [to_dev(x, "f32") for x in e_np]
    idx = [torch.empty(k, dtype=torch.int32, device="cuda") for _ in range(n)]
    val = [torch.empty(k, dtype=torch.float32, device="cuda") for _ in range(n)]
    ws = torch.empty(gar.ar_topk_workspace_bytes(n, count, k), dtype=torch.uint8, device="cuda")
    gar.ar_topk_compress(grads, res, k, idx, val, ws)
    out = [torch.empty(count, device="cuda") for _ in range(n)]
    sws = torch.empty(gar.ar_sparse_workspace_bytes(n, count), dtype=torch.uint8, device="cuda")
    algo = "tree" if n & (n - 1) == 0 else "fused"
    gar.ar_sparse_allreduce(idx, val, [k] * n, out, "avg", algo, sws)
    torch.cuda.synchronize()
    o_idx, o_val = [], []
    for r in range(n):
        oi, ov, oe = oracle.topk_compress(g_np[r], e_np[r], k)
        assert np.array_equal(from_dev(idx[r]).view(np.uint32), oi), r
        assert np.array_equal(_bits(from_dev(val[r])), _bits(ov)), r
        assert np.array_equal(_bits(from_dev(res[r])), _bits(oe)), r
        o_idx.append(oi)
        o_val.append(ov)
    dense = [oracle.sparse_to_dense(i, v, count) for i, v in zip(o_idx, o_val)]
    want = oracle.tree_allreduce(dense, "f32", "avg")[0]
    for r in range(n):
        assert np.array_equal(_bits(from_dev(out[r])), _bits(want)), r


def test_topk_step_captured_in_a_cuda_graph():
    # the launches of one step (programmatic dependent launches included)
    # replay from a CUDA graph with the same bits as eager calls
    n, count, k = 4, 100_003, 1_000
    g_np = [synthgen.normal_f32(count, 950 + r, 1.0) for r in range(n)]
    grads = [to_dev(x, "f32") for x in g_np]
    res = [torch.zeros(count, device="cuda") for _ in range(n)]
    idx = [torch.empty(k, dtype=torch.int32, device="cuda") for _ in range(n)]
    val = [torch.empty(k, dtype=torch.float32, device="cuda") for _ in range(n)]
    out = [torch.empty(count, device="cuda") for _ in range(n)]
    ws = torch.empty(gar.ar_topk_workspace_bytes(n, count, k), dtype=torch.uint8, device="cuda")
    sws = torch.empty(gar.ar_sparse_workspace_bytes(n, count), dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        g.capture_begin()
        gar.ar_topk_compress(grads, res, k, idx, val, ws, side)
        gar.ar_sparse_allreduce(idx, val, [k] * n, out, "sum", "fused", sws, side)
        g.capture_end()
    torch.cuda.current_stream().wait_stream(side)
    e_np = [np.zeros(count, dtype=np.float32) for _ in range(n)]
    for step in range(3):  # capture itself ran nothing; three replays are three steps of feedback
        g.replay()
        torch.cuda.synchronize()
        pairs = []
        for r in range(n):
            oi, ov, e_np[r] = oracle.topk_compress(g_np[r], e_np[r], k)
            assert np.array_equal(from_dev(idx[r]).view(np.uint32), oi), (step, r)
            assert np.array_equal(_bits(from_dev(res[r])), _bits(e_np[r])), (step, r)
            pairs.append((oi, ov))
        want = oracle.sparse_ring_allreduce([p[0] for p in pairs], [p[1] for p in pairs], count, "sum")[0]
        assert np.array_equal(_bits(from_dev(out[0])), _bits(want)), step


def test_sparse_allreduce_unaligned_outputs_and_ragged_tiles():
    # outputs one float off 16-byte alignment take the element stores; a count
    # that is not a multiple of the fold tile or of 4 leaves a ragged last tile
    from tests._dev import Guarded
    n, count = 6, 9_999
    rng = np.random.default_rng(3)
    idx_np, val_np = [], []
    for r in range(n):
        i = np.sort(rng.choice(count, size=[0, 1, 57, 999, count, 5][r], replace=False)).astype(np.uint32)
        idx_np.append(i)
        val_np.append(rng.standard_normal(i.size).astype(np.float32))
    idx = [torch.from_numpy(i.view(np.int32)).cuda() if i.size else torch.empty(0, dtype=torch.int32, device="cuda")
           for i in idx_np]
    val = [to_dev(v, "f32") if v.size else torch.empty(0, dtype=torch.float32, device="cuda") for v in val_np]
    ws = torch.empty(gar.ar_sparse_workspace_bytes(n, count), dtype=torch.uint8, device="cuda")
    for op in ("sum", "avg"):
        out = Guarded(n, count, "f32", offset_bytes=4)
        gar.ar_sparse_allreduce(idx, val, [i.size for i in idx_np], out.views, op, "fused", ws)
        out.check()
        want = oracle.sparse_ring_allreduce(idx_np, val_np, count, op)[0]
        for r in range(n):
            assert np.array_equal(_bits(from_dev(out.views[r])), _bits(want)), (op, r)
