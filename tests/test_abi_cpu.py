"""The C ABI without a GPU: the library loads, exports every symbol that
include/ar.h declares, and its host-only logic (status text, bucket plan,
argument and aliasing checks that return before anything is enqueued)
behaves as documented. Fake device addresses are used where a check must
fire before any pointer is dereferenced."""
import ctypes
import math
import re
from pathlib import Path

import numpy as np
import pytest

import gradient_allreduce_collective_gb300 as gar
import oracle
import synthgen
from tests import _golden as G

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "ar.h"


@pytest.fixture(scope="module")
def L():
    gar.build()
    return gar.lib()


def _declared():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(encoding="utf-8"), flags=re.S)
    return sorted(set(re.findall(r"\b(ar_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(L):
    for st in range(7):
        assert gar.ar_status_string(st)
    assert gar.ar_status_string(99) == "unknown status"
    assert "sm_103a" in gar.ar_version()


P = ctypes.POINTER(ctypes.c_void_p)


def _arr(addrs):
    return (ctypes.c_void_p * len(addrs))(*addrs)


def _ar(L, send, recv, n, count, dt=0, op=0, algo=1):
    return L.ar_allreduce(_arr(send), _arr(recv), n, count, dt, op, algo, None)


def test_allreduce_argument_errors(L):
    s = [0x100000 * (r + 1) for r in range(8)]
    d = [0x8000000 + 0x100000 * r for r in range(8)]
    assert L.ar_allreduce(None, _arr(d), 8, 16, 0, 0, 1, None) == gar.AR_ERR_INVALID_ARGUMENT
    assert _ar(L, s, d, 0, 16) == gar.AR_ERR_INVALID_ARGUMENT
    assert L.ar_allreduce(_arr(s * 9), _arr(d * 9), 65, 16, 0, 0, 1, None) == gar.AR_ERR_INVALID_ARGUMENT
    assert _ar(L, s, d, 8, 16, dt=7) == gar.AR_ERR_INVALID_ARGUMENT
    assert _ar(L, s, d, 8, 16, op=9) == gar.AR_ERR_INVALID_ARGUMENT
    assert _ar(L, s, d, 8, 16, algo=9) == gar.AR_ERR_INVALID_ARGUMENT
    # stepwise orders keep partials in the element type: 4-byte types only; tree needs 2^k ranks
    assert _ar(L, s, d, 8, 16, dt=2, algo=3) == gar.AR_ERR_UNSUPPORTED
    assert _ar(L, s[:3], d[:3], 3, 16, algo=4) == gar.AR_ERR_UNSUPPORTED
    assert _ar(L, s[:3], d[:3], 3, 0, algo=5) == gar.AR_SUCCESS
    assert _ar(L, s[:3], d[:3], 3, 16, algo=2) == gar.AR_ERR_UNSUPPORTED
    assert "power of two" in gar.ar_last_error()
    assert _ar(L, s[:3], d[:3], 3, 0, algo=1) == gar.AR_SUCCESS  # count 0: no-op
    bad = list(s)
    bad[2] = 0
    assert _ar(L, bad, d, 8, 16) == gar.AR_ERR_INVALID_ARGUMENT
    assert "sendbufs[2] is null" in gar.ar_last_error()
    mis = list(d)
    mis[5] += 2  # not 4-byte aligned for f32
    assert _ar(L, s, mis, 8, 16) == gar.AR_ERR_INVALID_ARGUMENT


def test_allreduce_alias_rules(L):
    n, count = 4, 1024
    s = [0x1000000 * (r + 1) for r in range(n)]
    d = [0x20000000 + 0x1000000 * r for r in range(n)]
    over = list(d)
    over[1] = d[0] + 8  # two outputs overlap
    assert _ar(L, s, over, n, count) == gar.AR_ERR_ALIAS
    cross = list(d)
    cross[1] = s[0]  # an output on another rank's input
    assert _ar(L, s, cross, n, count) == gar.AR_ERR_ALIAS
    shifted = list(d)
    shifted[2] = s[2] + 16  # overlaps its own input but not exactly
    assert _ar(L, s, shifted, n, count) == gar.AR_ERR_ALIAS


def test_reduce_scatter_and_all_gather_alias_rules(L):
    n, rc = 4, 64
    s = [0x1000000 * (r + 1) for r in range(n)]
    # in place is recvbufs[c] == sendbufs[c] + c*recvcount; recvbufs[c] == sendbufs[c] is not
    wrong = [s[c] for c in range(n)]
    wrong[0] = 0x30000000
    assert L.ar_reduce_scatter(_arr(s), _arr(wrong), n, rc, 0, 0, None) == gar.AR_ERR_ALIAS
    d = [0x20000000 + 0x1000000 * r for r in range(n)]
    assert L.ar_all_gather(_arr([d[0] + 4] + s[1:]), _arr(d), n, rc, 0, None) == gar.AR_ERR_ALIAS


def test_fp8_argument_errors(L):
    n, count = 4, 1000
    s = [0x1000000 * (r + 1) for r in range(n)]
    d = [0x20000000 + 0x1000000 * r for r in range(n)]
    need = gar.ar_fp8_workspace_bytes(n, count)
    qs = math.ceil(count / 256) * 256
    ss = math.ceil(math.ceil(count / 128) / 64) * 64 * 4
    assert need == n * (qs + ss)
    ws = 0x40000000
    f = L.ar_allreduce_fp8
    assert f(_arr(s), _arr(d), n, count, 2, 2, 2, 1, ws, need, None) == gar.AR_ERR_UNSUPPORTED  # MIN
    assert f(_arr(s), _arr(d), n, count, 3, 2, 0, 1, ws, need, None) == gar.AR_ERR_UNSUPPORTED  # int input
    assert f(_arr(s), _arr(d), n, count, 2, 2, 0, 1, ws, need - 1, None) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(_arr(s), _arr(d), n, count, 2, 2, 0, 1, ws + 8, need, None) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(_arr(s[:3]), _arr(d[:3]), 3, count, 2, 2, 0, 2, ws, need, None) == gar.AR_ERR_UNSUPPORTED
    assert f(_arr(s), _arr(d), n, count, 2, 2, 0, 1, d[1] + 64, need, None) == gar.AR_ERR_ALIAS
    assert f(_arr(s), _arr(d), n, count, 2, 2, 0, 3, ws, need, None) == gar.AR_ERR_UNSUPPORTED  # stepwise
    assert gar.ar_fp8_workspace_bytes(0, 10) == 0


def test_stepwise_workspace_and_argument_errors(L):
    n, count = 8, 1000
    s = [0x1000000 * (r + 1) for r in range(n)]
    d = [0x20000000 + 0x1000000 * r for r in range(n)]
    per = (count * 4 + 255) // 256 * 256
    assert gar.ar_stepwise_workspace_bytes(n, count, "bf16") == n * per
    assert gar.ar_stepwise_workspace_bytes(n, count, "f16") == n * per
    assert gar.ar_stepwise_workspace_bytes(n, count, "f32") == 0  # partials in the outputs
    assert gar.ar_stepwise_workspace_bytes(0, count, "bf16") == 0
    f = L.ar_allreduce_stepwise
    ws = 0x40000000
    need = n * per
    assert f(_arr(s), _arr(d), n, count, 2, 0, 1, ws, need, None) == gar.AR_ERR_INVALID_ARGUMENT  # FUSED
    assert "STEP_RING or STEP_TREE" in gar.ar_last_error()
    assert f(_arr(s[:3]), _arr(d[:3]), 3, count, 2, 0, 4, ws, need, None) == gar.AR_ERR_UNSUPPORTED  # tree, 3 ranks
    assert f(_arr(s), _arr(d), n, count, 2, 0, 3, None, 0, None) == gar.AR_ERR_INVALID_ARGUMENT  # no workspace
    assert f(_arr(s), _arr(d), n, count, 2, 0, 3, ws, need - 1, None) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(_arr(s), _arr(d), n, count, 2, 0, 3, ws + 8, need, None) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(_arr(s), _arr(d), n, count, 2, 0, 3, d[2] + 64, need, None) == gar.AR_ERR_ALIAS
    assert f(_arr(s), _arr(d), n, 0, 2, 0, 3, None, 0, None) == gar.AR_SUCCESS  # count 0: no-op
    # through ar_allreduce the 16-bit stepwise orders point to this entry point
    assert _ar(L, s, d, n, 16, dt=2, algo=3) == gar.AR_ERR_UNSUPPORTED
    assert "ar_allreduce_stepwise" in gar.ar_last_error()


def test_fp8_noalloc_reports_argument_errors_before_its_size_limit(L):
    # every case returns before any CUDA call: fake device addresses suffice
    n, big = 8, 2_100_000  # big: needs more than the library's 16 MiB array
    s = [0x1000000 * (r + 1) for r in range(n)]
    d = [0x20000000 + 0x1000000 * r for r in range(n)]
    f = L.ar_allreduce_fp8_noalloc
    assert gar.ar_fp8_workspace_bytes(n, big) > 16 * 1024 * 1024
    assert f(_arr(s), _arr(d), n, big, 7, 2, 0, 1, None) == gar.AR_ERR_INVALID_ARGUMENT
    assert "unknown dtype" in gar.ar_last_error()
    assert f(_arr(s), _arr(d), n, big, 2, 2, 9, 1, None) == gar.AR_ERR_INVALID_ARGUMENT
    assert "unknown op" in gar.ar_last_error()
    assert f(_arr(s), _arr(d), n, big, 2, 2, 2, 1, None) == gar.AR_ERR_UNSUPPORTED  # MIN
    assert f(_arr(s), _arr(d), n, big, 2, 2, 0, 9, None) == gar.AR_ERR_INVALID_ARGUMENT
    assert "unknown algo" in gar.ar_last_error()
    assert f(_arr(s[:3]), _arr(d[:3]), 3, big, 2, 2, 0, 2, None) == gar.AR_ERR_UNSUPPORTED  # tree, 3 ranks
    assert f(None, _arr(d), n, big, 2, 2, 0, 1, None) == gar.AR_ERR_INVALID_ARGUMENT
    # a count whose workspace size overflows is "count too large", not "needs 0 bytes"
    assert f(_arr(s), _arr(d), n, 1 << 62, 2, 2, 0, 1, None) == gar.AR_ERR_INVALID_ARGUMENT
    assert "count too large" in gar.ar_last_error()
    # valid arguments beyond the array: the size limit, with the sizes in the message
    assert f(_arr(s), _arr(d), n, big, 2, 2, 0, 1, None) == gar.AR_ERR_INVALID_ARGUMENT
    assert "static FP8 workspace holds 16777216 bytes" in gar.ar_last_error()
    assert str(gar.ar_fp8_workspace_bytes(n, big)) in gar.ar_last_error()
    assert f(_arr(s), _arr(d), n, 0, 2, 2, 0, 1, None) == gar.AR_SUCCESS  # count 0: no-op


def test_bucket_plan_matches_hand_derivation(L):
    import torch
    g = G.load("gpt2_buckets.txt")
    counts = [math.prod(s) for _, s in synthgen.gpt2_small_param_shapes()]
    bucket_of, offset_of, bucket_counts = gar.ar_bucket_plan(counts, torch.bfloat16, int(g["cap_bytes"]))
    assert [b * 2 for b in bucket_counts] == G.nums(g["expect_bytes"], int)


@pytest.mark.parametrize("seed", range(5))
def test_bucket_plan_matches_oracle(L, seed):
    import torch
    rng = np.random.default_rng(seed)
    counts = [int(x) for x in rng.integers(0, 5000, size=int(rng.integers(1, 60)))]
    for dt, es in ((torch.float32, 4), (torch.bfloat16, 2)):
        for cap in (1, 64, 4096, 40000):
            b1, o1, c1 = gar.ar_bucket_plan(counts, dt, cap)
            b2, o2, c2 = oracle.bucket_plan(counts, es, cap)
            assert b1 == b2.tolist() and o1 == o2.tolist() and c1 == c2.tolist()


def test_bucket_copy_errors(L):
    import torch
    t = [0x1000000, 0x2000000]
    counts = (ctypes.c_size_t * 2)(100, 100)
    offs = (ctypes.c_size_t * 2)(0, 50)  # the two tensors overlap inside the bucket
    assert L.ar_bucket_flatten(_arr(t), counts, offs, 2, 2, 0x4000000, None) == gar.AR_ERR_ALIAS
    offs_ok = (ctypes.c_size_t * 2)(0, 100)
    assert L.ar_bucket_flatten(_arr(t), counts, offs_ok, 2, 2, 0, None) == gar.AR_ERR_INVALID_ARGUMENT
    assert L.ar_bucket_flatten(_arr(t), counts, offs_ok, 0, 2, 0x4000000, None) == gar.AR_SUCCESS
    del torch


def test_bucket_allreduce_argument_errors(L):
    n, nt = 4, 3
    ins = [0x1000000 * (1 + r * nt + t) for r in range(n) for t in range(nt)]
    outs = [0x40000000 + 0x1000000 * (r * nt + t) for r in range(n) for t in range(nt)]
    counts = (ctypes.c_size_t * nt)(100, 200, 300)
    offs = (ctypes.c_size_t * nt)(0, 104, 304)
    f = L.ar_bucket_allreduce
    bad_offs = (ctypes.c_size_t * nt)(0, 104, 400)  # last tensor ends beyond the bucket
    assert f(_arr(ins), _arr(outs), n, nt, counts, bad_offs, 600, 2, 1, 1, None) == gar.AR_ERR_INVALID_ARGUMENT
    assert "outside the bucket" in gar.ar_last_error()
    over = list(outs)
    over[5] = outs[4] + 2  # two outputs overlap
    assert f(_arr(ins), _arr(over), n, nt, counts, offs, 604, 2, 1, 1, None) == gar.AR_ERR_ALIAS
    assert f(_arr(ins[:9]), _arr(outs[:9]), 3, nt, counts, offs, 604, 2, 1, 2, None) == gar.AR_ERR_UNSUPPORTED
    assert f(_arr(ins), _arr(outs), n, 0, counts, offs, 604, 2, 1, 1, None) == gar.AR_SUCCESS


def test_topk_workspace_and_argument_errors(L):
    n, count, k10 = 3, 100_000, 1000
    need = gar.ar_topk_workspace_bytes(n, count, k10)
    nb = math.ceil(count / 16384)
    share = math.ceil(k10 * 16384 / count)
    slots = min(16384, 8192, math.ceil((16 * share + 1024) / 32) * 32)
    assert need == n * math.ceil((2048 + 32 + (5 + 1024) * nb + 2 * slots * nb) / 64) * 64 * 4
    assert gar.ar_topk_workspace_bytes(1, 1 << 32, 1) == 0 and gar.ar_topk_workspace_bytes(0, 10, 1) == 0
    assert gar.ar_topk_workspace_bytes(1, 10, 11) == 0
    # at most about 4.25 bytes per value plus the fixed part, whatever k is
    assert gar.ar_topk_workspace_bytes(1, count, count) <= 4.25 * count + 3 * 16384 * 4 + 9 * 1024
    g = [0x1000000 * (r + 1) for r in range(n)]
    e = [0x10000000 + 0x1000000 * r for r in range(n)]
    i = [0x20000000 + 0x1000000 * r for r in range(n)]
    v = [0x30000000 + 0x1000000 * r for r in range(n)]
    ws = 0x40000000

    need = gar.ar_topk_workspace_bytes(n, count, 10)

    def f(g=g, e=e, count=count, k=10, i=i, v=v, ws=ws, wsb=need, n=n):
        return L.ar_topk_compress(_arr(g), _arr(e), n, count, k, _arr(i), _arr(v), ws, wsb, None)

    assert f(k=count + 1) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(count=1 << 32) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(wsb=need - 1) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(ws=ws + 8) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(e=[e[0] + 2] + e[1:]) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(i=[None] + i[1:]) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(n=0) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(e=[g[1] + 200] + e[1:]) == gar.AR_ERR_ALIAS          # a residual inside another rank's grad
    assert f(v=[i[0] + 8] + v[1:]) == gar.AR_ERR_ALIAS            # idx and val overlap
    assert f(ws=e[2] + 64) == gar.AR_ERR_ALIAS                    # workspace inside a residual
    assert f(count=0, k=0, ws=None, wsb=0) == gar.AR_SUCCESS      # empty


def test_sparse_allreduce_argument_errors(L):
    n, count = 4, 1000
    idx = [0x1000000 * (r + 1) for r in range(n)]
    val = [0x10000000 + 0x1000000 * r for r in range(n)]
    out = [0x20000000 + 0x1000000 * r for r in range(n)]
    ws = 0x30000000
    need = gar.ar_sparse_workspace_bytes(n, count)
    # one boundary word per rank and output tile; the tile keeps N x tile
    # floats of shared memory at most 24 KiB (within 128..4096 values)
    for nn, cc in [(n, count), (1, 5), (2, 10**6), (3, 6145), (8, 6_553_600), (16, 767), (48, 10**5), (49, 129),
                   (64, 10**7 + 3)]:
        tile = max(128, min(4096, 6144 // nn // 128 * 128))
        assert gar.ar_sparse_workspace_bytes(nn, cc) == math.ceil(nn * (math.ceil(cc / tile) + 1) * 4 / 256) * 256
    assert gar.ar_sparse_workspace_bytes(8, 6_553_600) == 273_152  # 8 x 8,534 words: 768-value tiles
    assert gar.ar_sparse_workspace_bytes(0, 10) == 0 and gar.ar_sparse_workspace_bytes(1, 1 << 32) == 0
    nnz = (ctypes.c_size_t * n)(10, 0, 1000, 5)

    def f(idx=idx, val=val, nnz=nnz, n=n, count=count, op=0, algo=1, out=out, ws=ws, wsb=need):
        return L.ar_sparse_allreduce(_arr(idx), _arr(val), nnz, n, count, op, algo, _arr(out), ws, wsb, None)

    assert f(nnz=(ctypes.c_size_t * n)(10, 0, 1001, 5)) == gar.AR_ERR_INVALID_ARGUMENT  # nnz > count
    assert f(n=3, algo=2, out=out[:3]) == gar.AR_ERR_UNSUPPORTED                        # tree, N=3
    assert f(op=7) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(algo=9) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(ws=None) == gar.AR_ERR_INVALID_ARGUMENT                                    # SUM needs a workspace
    assert f(wsb=need - 1) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(ws=ws + 4) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(ws=out[1] + 64) == gar.AR_ERR_ALIAS                                        # workspace inside an output
    assert f(out=[out[0], out[0] + 400, out[2], out[3]]) == gar.AR_ERR_ALIAS
    assert f(idx=idx[:3] + [out[0] + 8]) == gar.AR_ERR_ALIAS                            # an index array inside an output
    assert f(count=1 << 32) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(count=0) == gar.AR_SUCCESS


def test_allreduce_slice_argument_errors(L):
    n, count = 4, 1000
    s = [0x1000000 * (r + 1) for r in range(n)]
    d = [0x20000000 + 0x1000000 * r for r in range(n)]
    f = L.ar_allreduce_slice
    assert f(_arr(s), _arr(d), n, count, 990, 11, 0, 0, 1, None) == gar.AR_ERR_INVALID_ARGUMENT  # past the end
    assert f(_arr(s), _arr(d), n, count, 1001, 0, 0, 0, 1, None) == gar.AR_ERR_INVALID_ARGUMENT
    assert f(_arr(s), _arr(d), n, count, 10, 0, 0, 0, 1, None) == gar.AR_SUCCESS                  # empty slice
    assert f(_arr(s[:3]), _arr(d[:3]), 3, count, 0, 10, 0, 0, 2, None) == gar.AR_ERR_UNSUPPORTED  # tree, N=3
    assert f(_arr(s[:3]), _arr(d[:3]), 3, count, 0, 10, 0, 0, 4, None) == gar.AR_ERR_UNSUPPORTED  # step tree, N=3
    assert f(_arr(s), _arr(d), n, count, 0, 10, 0, 7, 1, None) == gar.AR_ERR_INVALID_ARGUMENT     # op
    assert f(_arr(s), _arr(d), n, count, 0, 10, 0, 0, 9, None) == gar.AR_ERR_INVALID_ARGUMENT     # algo
    over = list(d)
    over[1] = d[0] + 8
    assert f(_arr(s), _arr(over), n, count, 0, 10, 0, 0, 1, None) == gar.AR_ERR_ALIAS
