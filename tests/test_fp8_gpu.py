"""GPU parity of the FP8 (E4M3, per-128-element block scale) path against the
oracle, bit for bit, plus the tolerance against the fp64 reference. The full
16 x 134,217,728 bf16 workload is checked on sampled whole blocks, which the
oracle evaluates one by one, and by properties (replicas identical, ring ==
fused bitwise, normwise error)."""
import numpy as np
import pytest
import torch

import gradient_allreduce_collective_gb300 as gar
import oracle
import synthgen
from tests import _golden as G
from tests._dev import ESIZE, TORCH, Guarded, from_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gar.build()
    gar.lib()


def _same_bits(a, b):
    return np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


def _ws(n, count):
    return torch.empty(gar.ar_fp8_workspace_bytes(n, count), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("in_dtype", ["bf16", "f16", "f32"])
def test_quantize_matches_oracle(in_dtype):
    for count in (1, 5, 127, 128, 129, 128 * 1000 + 77):
        x = synthgen.ranks_normal(1, count, 1e-3, base_seed=count, dtype=in_dtype, outlier_p=1e-2,
                                  outlier_scale=100.0)[0]
        x[: min(count, 128)] = 0  # an all-zero block (scale 0)
        for off in (0, ESIZE[in_dtype]):  # aligned, and the element path
            g = Guarded(1, count, in_dtype, off)
            g.views[0].copy_(to_dev(x, in_dtype))
            q = torch.empty(count, dtype=torch.uint8, device="cuda")
            s = torch.empty((count + 127) // 128, dtype=torch.float32, device="cuda")
            gar.ar_quantize_fp8_blocks(g.views[0], q, s)
            wq, ws = oracle.fp8_quantize(x, in_dtype)
            assert _same_bits(from_dev(q), wq) and _same_bits(from_dev(s), ws), (count, off)


@pytest.mark.parametrize("offset", [0, 4])
def test_block_scales_over_the_binary32_range(offset):
    # one block per amax: amax = random binary32 patterns over the whole
    # positive range (the division-free scale's domain, its edges, subnormals,
    # FLT_MAX) in slot 0 and zeros elsewhere; every scale and code bit-exact
    rng = np.random.default_rng(11)
    bits = rng.integers(0x00000001, 0x7F800000, size=1 << 18, dtype=np.uint32)
    edges = np.array([0x05800000, 0x057FFFFF, 0x05800001, 0x7F7FFFFF, 0x7F7FFFFE, 0x00800000, 0x007FFFFF,
                      0x3F800000, 0x43E00000, 0x43E00001, 0x3B124925, 0x3B124924], dtype=np.uint32)
    amax = np.concatenate([edges, bits]).view(np.float32)
    x = np.zeros(amax.size * 128, dtype=np.float32)
    x[::128] = amax
    x[1::128] = -amax / np.float32(3.0)  # a second value per block (its code depends on the scale too)
    g = Guarded(1, x.size, "f32", offset)
    g.views[0].copy_(to_dev(x, "f32"))
    q = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    sc = torch.empty(amax.size, dtype=torch.float32, device="cuda")
    gar.ar_quantize_fp8_blocks(g.views[0], q, sc)
    wq, ws = oracle.fp8_quantize(x, "f32")
    assert _same_bits(from_dev(sc), ws)
    assert _same_bits(from_dev(q), wq)
    g.check()


def _e4m3_midpoints():
    codes = np.arange(0x7F, dtype=np.uint8)
    v = np.sort(oracle.e4m3_to_f32(codes).astype(np.float64))
    return (v[1:] + v[:-1]) / 2  # 126 rounding boundaries between magnitudes


def test_quantize_rounding_boundaries():
    # every block: x[0] = amax (so s = amax/448), then values whose x/s fall on
    # and within a few binary32 ulps of every E4M3 midpoint, both signs
    mids = _e4m3_midpoints()
    blocks = []
    for amax in (1.0, 3.0, 0.7, 1e-3, 123456.0, 1e-36, 2.0**-127, 2.0**-140):
        a = np.float32(amax)
        s = np.float32(a / np.float32(448.0))
        vals = []
        for m in mids:
            x = np.float32(m * np.float64(s))
            for j in range(-3, 4):
                y = x
                for _ in range(abs(j)):
                    y = np.nextafter(y, np.float32(np.inf) if j > 0 else np.float32(0))
                if abs(y) <= a:
                    vals.append(y)
        vals = np.array(vals, dtype=np.float32)
        vals = np.concatenate([vals, -vals])
        for i in range(0, len(vals), 127):
            blk = np.zeros(128, dtype=np.float32)
            blk[0] = a
            part = vals[i:i + 127]
            blk[1:1 + len(part)] = part
            blocks.append(blk)
    blocks.append(np.zeros(128, dtype=np.float32))
    x = np.concatenate(blocks)
    q = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    sc = torch.empty(x.size // 128, dtype=torch.float32, device="cuda")
    gar.ar_quantize_fp8_blocks(to_dev(x, "f32"), q, sc)
    wq, ws = oracle.fp8_quantize(x, "f32")
    assert _same_bits(from_dev(sc), ws)
    got = from_dev(q)
    bad = np.nonzero(got != wq)[0]
    assert bad.size == 0, (bad[:10], got[bad[:10]], wq[bad[:10]], x[bad[:10]])


def _every_bf16_blocks():
    pats = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    f = oracle.bf16_to_f32(pats)
    fin = np.isfinite(f) & (f >= 0)
    pos = pats[fin]
    posf = f[fin]
    rng = np.random.default_rng(17)
    amaxes = [1.0, 448.0, 3.0, 0.0078125, 1e-3, 65504.0, 1e30, 3e38, 1e-24, 1e-26, 1e-30, 2.0**-120,
              2.0**-133, 5e29, 3.7e-25]
    amaxes += list(oracle.bf16_to_f32(rng.choice(pos[posf > 0], 25)).astype(float))
    blocks = []
    for amax in amaxes:
        a = synthgen.to_dtype(np.array([amax], dtype=np.float32), "bf16")[0]
        af = oracle.bf16_to_f32(np.array([a]))[0]
        vals = pos[posf <= af]
        vals = np.concatenate([vals, vals | np.uint16(0x8000)])
        for i in range(0, len(vals), 127):
            part = vals[i:i + 127]
            blk = np.full(128, a, dtype=np.uint16)
            blk[1:1 + len(part)] = part
            blocks.append(blk)
    return np.concatenate(blocks)


def test_quantize_every_bf16_value():
    # every finite bf16 x with |x| <= amax, for ~40 block maxima spanning the
    # reciprocal path and the division fallback (s < 2^-90, s > 2^90)
    x = _every_bf16_blocks()
    q = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    sc = torch.empty(x.size // 128, dtype=torch.float32, device="cuda")
    gar.ar_quantize_fp8_blocks(to_dev(x, "bf16"), q, sc)
    wq, ws = oracle.fp8_quantize(x, "bf16")
    assert _same_bits(from_dev(sc), ws)
    got = from_dev(q)
    bad = np.nonzero(got != wq)[0]
    assert bad.size == 0, (bad[:8], got[bad[:8]], wq[bad[:8]], oracle.bf16_to_f32(x[bad[:8]]))
    # the same values through both allreduce paths (one rank: the dequantised values, rounded to bf16)
    want = oracle.fp8_ring_allreduce([x], "bf16", "bf16", "sum")[0]
    xin = [to_dev(x, "bf16")]
    for fn in ("materialised", "fused"):
        out = [torch.empty(x.size, dtype=torch.bfloat16, device="cuda")]
        if fn == "fused":
            gar.ar_allreduce_fp8_fused(xin, out, "sum", "fused")
        else:
            gar.ar_allreduce_fp8(xin, out, _ws(1, x.size), "sum", "fused")
        assert _same_bits(from_dev(out[0]), want), fn


def test_fp8_block_example():
    g = G.load("fp8_block_example.txt")
    send = [to_dev(synthgen.to_dtype(np.array(G.nums(g[f"rank{r}"]), dtype=np.float32), "bf16"), "bf16")
            for r in range(2)]
    for op in ("sum", "avg"):
        for algo in ("ring", "fused", "tree"):
            recv = [torch.empty(4, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
            gar.ar_allreduce_fp8(send, recv, _ws(2, 4), op, algo)
            for y in recv:
                assert y.float().cpu().tolist() == G.nums(g[f"expect_{op}"]), (op, algo)


def test_fp8_tree_example():
    # the hand-computed recursive-halving pairing after E4M3 quantisation, on
    # the materialised and the fused paths (the ring order gives other values)
    g = G.load("fp8_tree_example.txt")
    send = [to_dev(synthgen.to_dtype(np.array(G.nums(g[f"rank{r}"]), dtype=np.float32), "bf16"), "bf16")
            for r in range(4)]
    for op in ("sum", "avg"):
        for algo, key in (("tree", "tree"), ("fused", "ring"), ("ring", "ring")):
            for path in ("materialised", "fused"):
                recv = [torch.empty(4, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
                if path == "materialised":
                    gar.ar_allreduce_fp8(send, recv, _ws(4, 4), op, algo)
                else:
                    gar.ar_allreduce_fp8_fused(send, recv, op, algo)
                for y in recv:
                    assert y.float().cpu().tolist() == G.nums(g[f"expect_{key}_{op}"]), (op, algo, path)


def _nan_blocks(n, nblk, seed, dtype):
    """Ranks of nblk blocks: block 0 of every rank all zeros but one NaN,
    block 1 normal values with one NaN, the rest normal values."""
    x = synthgen.ranks_normal(n, nblk * 128, 1e-3, base_seed=seed)
    for r, a in enumerate(x):
        a[:128] = 0.0
        a[5 + r] = np.nan
        a[128 + 17 * r] = np.nan
    return [a if dtype == "f32" else synthgen.to_dtype(a, dtype) for a in x]


@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
def test_fp8_nan_blocks_agree_on_every_path(in_dtype):
    # the block amax propagates a NaN: a block holding one (among zeros or among
    # normal values) has a NaN scale and dequantises to NaN throughout, on the
    # materialised, fused and per-hop paths alike, as in the oracle; the other
    # blocks are bit-exact
    n, nblk = 4, 8  # chunks of 2 blocks: the per-hop path's blocks are the same
    send_np = _nan_blocks(n, nblk, 21, in_dtype)
    send = [to_dev(a, in_dtype) for a in send_np]
    count = nblk * 128
    want_once = oracle.fp8_ring_allreduce(send_np, in_dtype, "bf16", "sum")[0]
    want_hops = oracle.fp8_hop_ring_allreduce(send_np, in_dtype, "bf16", "sum")[0]
    for w in (want_once, want_hops):
        f = oracle.bf16_to_f32(w)
        assert np.isnan(f[:256]).all() and not np.isnan(f[256:]).any()
    runs = {
        "materialised": lambda out: gar.ar_allreduce_fp8(send, out, _ws(n, count), "sum", "fused"),
        "fused": lambda out: gar.ar_allreduce_fp8_fused(send, out, "sum", "fused"),
        "hops": lambda out: gar.ar_allreduce_fp8_hops(send, out, "sum"),
    }
    for name, run in runs.items():
        out = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
        run(out)
        want = want_hops if name == "hops" else want_once
        wf = oracle.bf16_to_f32(want)
        for o in out:
            got = from_dev(o)
            gf = oracle.bf16_to_f32(got)
            nan = np.isnan(wf)
            assert np.array_equal(np.isnan(gf), nan), name
            assert np.array_equal(got[~nan], want[~nan]), name


@pytest.mark.parametrize("in_dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("out_dtype", ["bf16", "f16", "f32"])
def test_fp8_allreduce_matches_oracle(in_dtype, out_dtype):
    for n in (1, 2, 3, 4, 8, 16):
        for count in (1, 100, 128 * 50 + 3, 128 * 300):
            send_np = synthgen.ranks_normal(n, count, 1e-3, base_seed=n + count, dtype=in_dtype, outlier_p=1e-2,
                                            outlier_scale=100.0)
            send = [to_dev(a, in_dtype) for a in send_np]
            for op in ("sum", "avg"):
                algos = ("ring", "fused", "tree") if n & (n - 1) == 0 else ("ring", "fused")
                for algo in algos:
                    if algo == "tree":
                        want = oracle.fp8_tree_allreduce(send_np, in_dtype, out_dtype, op)[0]
                    else:
                        want = oracle.fp8_ring_allreduce(send_np, in_dtype, out_dtype, op)[0]
                    out = Guarded(n, count, out_dtype)
                    gar.ar_allreduce_fp8(send, out.views, _ws(n, count), op, algo)
                    out.check()
                    for v in out.views:
                        assert _same_bits(from_dev(v), want), (n, count, op, algo)


FUSED_IO = [("bf16", "bf16"), ("bf16", "f16"), ("f16", "f16"), ("f16", "bf16"), ("f32", "f32"), ("f32", "bf16"),
            ("f32", "f16")]


def test_fp8_fused_many_ranks():
    # 33 ranks: the kernels' largest rank tier (batches of eight ranks in a loop)
    n = 33
    for in_dtype in ("bf16", "f32"):
        for count in (128 * 66 + 24, 128 * 200):
            send_np = synthgen.ranks_normal(n, count, 1e-3, base_seed=count, dtype=in_dtype, outlier_p=1e-2,
                                            outlier_scale=100.0)
            send = [to_dev(a, in_dtype) for a in send_np]
            for op in ("sum", "avg"):
                want = oracle.fp8_ring_allreduce(send_np, in_dtype, "bf16", op)[0]
                out = Guarded(n, count, "bf16")
                gar.ar_allreduce_fp8_fused(send, out.views, op, "fused")
                out.check()
                for v in out.views:
                    assert _same_bits(from_dev(v), want), (in_dtype, count, op)


@pytest.mark.parametrize("in_dtype,out_dtype", FUSED_IO)
def test_fp8_fused_matches_oracle(in_dtype, out_dtype):
    # counts put chunk boundaries inside vector-kernel warps (element-wise path),
    # on warp edges, and leave short last blocks
    for n in (1, 2, 3, 5, 8, 16):
        for count in (1, 100, 128 * 97 + 24, 128 * 300, 128 * 1000 + 72):
            send_np = synthgen.ranks_normal(n, count, 1e-3, base_seed=3 * n + count, dtype=in_dtype,
                                            outlier_p=1e-2, outlier_scale=100.0)
            send = [to_dev(a, in_dtype) for a in send_np]
            for op in ("sum", "avg"):
                algos = ("ring", "fused", "tree") if n & (n - 1) == 0 else ("ring", "fused")
                for algo in algos:
                    if algo == "tree":
                        want = oracle.fp8_tree_allreduce(send_np, in_dtype, out_dtype, op)[0]
                    else:
                        want = oracle.fp8_ring_allreduce(send_np, in_dtype, out_dtype, op)[0]
                    out = Guarded(n, count, out_dtype)
                    gar.ar_allreduce_fp8_fused(send, out.views, op, algo)
                    out.check()
                    for v in out.views:
                        assert _same_bits(from_dev(v), want), (n, count, op, algo)


def test_fp8_fused_unaligned_and_unsupported():
    n, count = 4, 128 * 20 + 9
    send_np = synthgen.ranks_normal(n, count, 1e-3, base_seed=6, dtype="bf16")
    want = oracle.fp8_ring_allreduce(send_np, "bf16", "bf16", "sum")[0]
    gin = Guarded(n, count, "bf16", 2)
    for v, a in zip(gin.views, send_np):
        v.copy_(to_dev(a, "bf16"))
    out = Guarded(n, count, "bf16", 6)
    gar.ar_allreduce_fp8_fused(gin.views, out.views, "sum", "fused")
    out.check()
    for v in out.views:
        assert _same_bits(from_dev(v), want)
    f32_out = [torch.empty(count, dtype=torch.float32, device="cuda") for _ in range(n)]
    with pytest.raises(gar.ArError) as ei:
        gar.ar_allreduce_fp8_fused(gin.views, f32_out, "sum", "fused")
    assert ei.value.status == gar.AR_ERR_UNSUPPORTED


@pytest.mark.parametrize("in_dtype,out_dtype", [("bf16", "bf16"), ("bf16", "f32"), ("f16", "f16"), ("f32", "f32"),
                                               ("f32", "bf16")])
def test_fp8_hops_matches_oracle(in_dtype, out_dtype):
    for n in (1, 2, 3, 5, 8, 16, 33):
        for count in (1, 100, 128 * 9 + 7, 128 * 40, 128 * 300 + 72):
            send_np = synthgen.ranks_normal(n, count, 1e-3, base_seed=5 * n + count, dtype=in_dtype,
                                            outlier_p=1e-2, outlier_scale=100.0)
            send = [to_dev(a, in_dtype) for a in send_np]
            for op in ("sum", "avg"):
                want = oracle.fp8_hop_ring_allreduce(send_np, in_dtype, out_dtype, op)[0]
                out = Guarded(n, count, out_dtype, ESIZE[out_dtype] if n == 3 else 0)
                gar.ar_allreduce_fp8_hops(send, out.views, op)
                out.check()
                for v in out.views:
                    assert _same_bits(from_dev(v), want), (n, count, op)


def _wide_scale_ranks(n, nblk, seed, dtype):
    # every block of every rank at its own magnitude, 2^-140 .. 2^100 (block
    # scales below, inside and above the range of the kernels' division-free
    # path, subnormal values), some blocks zero
    rng = np.random.default_rng(seed)
    count = 128 * nblk + 40
    out = []
    for r in range(n):
        x = rng.standard_normal(count)
        e = rng.integers(-140, 100, size=nblk + 1)
        scale = np.exp2(e.astype(np.float64))
        scale[rng.random(nblk + 1) < 0.1] = 0.0
        out.append(synthgen.to_dtype((x * np.repeat(scale, 128)[:count]).astype(np.float32), dtype))
    return out


def _signed_zero_ranks(n, nblk, seed, dtype):
    # normal blocks with a fifth of their elements set to -0 or +0, blocks of
    # mixed -0 / +0 only, and blocks of -0 only
    rng = np.random.default_rng(seed)
    count = 128 * nblk + 40
    out = []
    for r in range(n):
        x = (rng.standard_normal(count) * 1e-3).astype(np.float32)
        x[rng.random(count) < 0.1] = np.float32(-0.0)
        x[rng.random(count) < 0.1] = np.float32(0.0)
        kind = rng.integers(0, 4, size=nblk + 1)
        for b in range(nblk + 1):
            if kind[b] == 1:
                x[128 * b:128 * (b + 1)] = np.where(rng.random(min(128, count - 128 * b)) < 0.5, -0.0, 0.0)
            elif kind[b] == 2:
                x[128 * b:128 * (b + 1)] = -0.0
        out.append(synthgen.to_dtype(x, dtype))
    return out


@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
def test_fp8_signed_zeros(in_dtype):
    # the sign of zero through quantisation, the fold and the output, on the
    # fused, per-hop and materialised paths (every rank's block kinds differ,
    # so some chunks fold only zeros)
    for n in (3, 4):
        send_np = _signed_zero_ranks(n, 120, 21 + n, in_dtype)
        count = send_np[0].size
        send = [to_dev(a, in_dtype) for a in send_np]
        for op in ("sum", "avg"):
            want = oracle.fp8_ring_allreduce(send_np, in_dtype, "bf16", op)[0]
            out = Guarded(n, count, "bf16")
            gar.ar_allreduce_fp8_fused(send, out.views, op, "fused")
            out.check()
            for v in out.views:
                assert _same_bits(from_dev(v), want), ("fused", n, op)
            gar.ar_allreduce_fp8(send, out.views, _ws(n, count), op, "fused")
            for v in out.views:
                assert _same_bits(from_dev(v), want), ("materialised", n, op)
            want_hop = oracle.fp8_hop_ring_allreduce(send_np, in_dtype, "bf16", op)[0]
            gar.ar_allreduce_fp8_hops(send, out.views, op)
            out.check()
            for v in out.views:
                assert _same_bits(from_dev(v), want_hop), ("hops", n, op)


@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
def test_fp8_fused_scales_over_the_binary32_range(in_dtype):
    for n in (3, 4):
        send_np = _wide_scale_ranks(n, 300, 13 + n, in_dtype)
        count = send_np[0].size
        send = [to_dev(a, in_dtype) for a in send_np]
        for op in ("sum", "avg"):
            for algo in (("fused", "tree") if n == 4 else ("fused",)):
                if algo == "tree":
                    want = oracle.fp8_tree_allreduce(send_np, in_dtype, "bf16", op)[0]
                else:
                    want = oracle.fp8_ring_allreduce(send_np, in_dtype, "bf16", op)[0]
                out = Guarded(n, count, "bf16")
                gar.ar_allreduce_fp8_fused(send, out.views, op, algo)
                out.check()
                for v in out.views:
                    assert _same_bits(from_dev(v), want), (n, op, algo)


@pytest.mark.parametrize("in_dtype,out_dtype", [("f32", "f32"), ("f32", "bf16"), ("bf16", "bf16")])
def test_fp8_hops_scales_over_the_binary32_range(in_dtype, out_dtype):
    # both blocks of a pair, one or neither on the general path (binary32
    # inputs fold four ranks per batch, 16-bit inputs eight)
    n = 3 if in_dtype == "f32" else 10
    send_np = _wide_scale_ranks(n, 200, 12, in_dtype)
    count = send_np[0].size
    send = [to_dev(a, in_dtype) for a in send_np]
    for op in ("sum", "avg"):
        want = oracle.fp8_hop_ring_allreduce(send_np, in_dtype, out_dtype, op)[0]
        out = Guarded(n, count, out_dtype, 0)
        gar.ar_allreduce_fp8_hops(send, out.views, op)
        out.check()
        for v in out.views:
            assert _same_bits(from_dev(v), want), op


def test_fp8_hops_example():
    g = G.load("fp8_hop_example.txt")
    send = [to_dev(synthgen.to_dtype(np.array(G.nums(g[f"rank{r}"]), dtype=np.float32), "bf16"), "bf16")
            for r in range(2)]
    for op in ("sum", "avg"):
        recv = [torch.empty(4, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        gar.ar_allreduce_fp8_hops(send, recv, op)
        for y in recv:
            assert y.float().cpu().tolist() == G.nums(g[f"expect_{op}"])


def test_fp8_unaligned_outputs():
    n, count = 4, 128 * 20 + 9
    send_np = synthgen.ranks_normal(n, count, 1e-3, base_seed=5, dtype="bf16")
    send = [to_dev(a, "bf16") for a in send_np]
    want = oracle.fp8_ring_allreduce(send_np, "bf16", "bf16", "sum")[0]
    for algo in ("ring", "fused"):
        out = Guarded(n, count, "bf16", 2)
        gar.ar_allreduce_fp8(send, out.views, _ws(n, count), "sum", algo)
        out.check()
        for v in out.views:
            assert _same_bits(from_dev(v), want)


def test_config5_full_size_sampled():
    n, count = 16, 134_217_728
    send_np = synthgen.ranks_normal(n, count, 1e-3, base_seed=0, dtype="bf16", outlier_p=1e-3, outlier_scale=100.0)
    send = [to_dev(a, "bf16") for a in send_np]
    ws = _ws(n, count)
    fused = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    gar.ar_allreduce_fp8(send, fused, ws, "sum", "fused")
    ring = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    gar.ar_allreduce_fp8(send, ring, ws, "sum", "ring")
    torch.cuda.synchronize()
    f0 = fused[0].view(torch.int16)
    for r in range(n):
        assert torch.equal(fused[r].view(torch.int16), f0)
        assert torch.equal(ring[r].view(torch.int16), f0)
    del ws
    # the quantisation fused into the reduction gives the same bits
    gar.ar_allreduce_fp8_fused(send, ring, "sum", "fused")
    torch.cuda.synchronize()
    for r in range(n):
        assert torch.equal(ring[r].view(torch.int16), f0)
    del ring
    rng = np.random.default_rng(0)
    nblocks = count // 128
    blocks = np.unique(np.concatenate([rng.choice(nblocks, 3000, replace=False), [0, nblocks - 1],
                                       # blocks at every chunk boundary
                                       [(c * (count // n)) // 128 for c in range(n)]]))
    blk = np.stack([np.stack([send_np[r][b * 128:(b + 1) * 128] for r in range(n)]) for b in blocks])
    want = oracle.fp8_ring_blocks(blk, blocks * 128, np.full(len(blocks), 128), count, "bf16", "bf16", "sum")
    got = from_dev(fused[0]).reshape(-1, 128)[blocks]
    assert _same_bits(got, want)
    # tolerance against fp64 on the sample (normwise, as the FP8 bound is stated)
    x = np.stack([oracle.bf16_to_f32(blk[:, r, :].ravel()).astype(np.float64) for r in range(n)])
    ystar = x.sum(axis=0)
    y = oracle.bf16_to_f32(got.ravel()).astype(np.float64)
    assert np.linalg.norm(y - ystar) / np.linalg.norm(ystar) <= 6e-2
