"""ar_allreduce_fp8_noalloc: the FP8 allreduce for callers that cannot
allocate device memory (code running inside an allocator's or memory pool's
callbacks, on a path where allocation is forbidden, or without the CUDA
allocation API). It keeps its quantised codes and scales in a fixed array
inside the library instead of a caller workspace.

Its results must equal the oracle's FP8 ring allreduce bit for bit, and those
of ar_allreduce_fp8 with a caller-provided workspace on two calls in a row
with different shapes, so the second call runs on the array the first one
left filled. A call that needs more than the built-in array is refused with a
clear error.

This file is collected last, so a run that stops at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import gradient_allreduce_collective_gb300 as gar
import oracle
import synthgen
from tests._dev import from_dev, to_dev

pytestmark = pytest.mark.gpu

LIMIT = 16 * 1024 * 1024


@pytest.fixture(scope="module", autouse=True)
def _built():
    gar.build()
    gar.lib()


def _case(n, count, in_dtype, out_dtype, seed):
    send_np = synthgen.ranks_normal(n, count, 1e-3, base_seed=seed, dtype=in_dtype, outlier_p=1e-3,
                                    outlier_scale=100.0)
    send = [to_dev(a, in_dtype) for a in send_np]
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[out_dtype]
    return send, tdt


@pytest.mark.parametrize("n,count,idt,odt,op,algo", [
    (8, 128 * 700 + 77, "bf16", "bf16", "sum", "fused"),
    (4, 128 * 300 + 5, "f32", "f16", "avg", "ring"),
    (3, 128 * 41 + 100, "f16", "f32", "sum", "fused"),
])
def test_noalloc_matches_the_oracle(n, count, idt, odt, op, algo):
    send_np = synthgen.ranks_normal(n, count, 1e-3, base_seed=300 + n, dtype=idt, outlier_p=1e-3, outlier_scale=100.0)
    send = [to_dev(a, idt) for a in send_np]
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[odt]
    out = [torch.full((count,), float("nan"), dtype=tdt, device="cuda") for _ in range(n)]
    gar.ar_allreduce_fp8_noalloc(send, out, op, algo)
    torch.cuda.synchronize()
    want = oracle.fp8_ring_allreduce(send_np, idt, odt, op)[0]
    for o in out:
        got = from_dev(o)
        assert got.tobytes() == np.ascontiguousarray(want).tobytes(), (n, count, op, algo)


def test_noalloc_matches_caller_workspace_on_two_calls_in_a_row():
    cases = [  # (nranks, count, in, out, op, algo)
        (8, 128 * 5000 + 77, "bf16", "bf16", "sum", "fused"),
        (4, 128 * 300 + 5, "f32", "f16", "avg", "ring"),
    ]
    prepared = []
    for i, (n, count, idt, odt, op, algo) in enumerate(cases):
        assert gar.ar_fp8_workspace_bytes(n, count) <= LIMIT
        send, tdt = _case(n, count, idt, odt, seed=10 * i)
        ws = torch.empty(gar.ar_fp8_workspace_bytes(n, count), dtype=torch.uint8, device="cuda")
        ref = [torch.empty(count, dtype=tdt, device="cuda") for _ in range(n)]
        gar.ar_allreduce_fp8(send, ref, ws, op, algo)
        prepared.append((send, ref, tdt, op, algo))
    torch.cuda.synchronize()
    outs = []
    for send, ref, tdt, op, algo in prepared:  # two calls in a row on the library's array
        out = [torch.full_like(r, float("nan")) for r in ref]
        gar.ar_allreduce_fp8_noalloc(send, out, op, algo)
        outs.append(out)
    torch.cuda.synchronize()
    for (send, ref, tdt, op, algo), out in zip(prepared, outs):
        for r, o in zip(ref, out):
            assert np.array_equal(from_dev(o), from_dev(r)), (op, algo)
    # and once more, repeating the first case after the second overwrote the array
    send, ref, tdt, op, algo = prepared[0]
    out = [torch.empty_like(r) for r in ref]
    gar.ar_allreduce_fp8_noalloc(send, out, op, algo)
    torch.cuda.synchronize()
    for r, o in zip(ref, out):
        assert np.array_equal(from_dev(o), from_dev(r))


def test_noalloc_refuses_calls_beyond_its_array():
    n, count = 8, 2_100_000
    assert gar.ar_fp8_workspace_bytes(n, count) > LIMIT
    send, tdt = _case(n, count, "bf16", "bf16", seed=3)
    out = [torch.zeros(count, dtype=tdt, device="cuda") for _ in range(n)]
    with pytest.raises(gar.ArError) as ei:
        gar.ar_allreduce_fp8_noalloc(send, out, "sum", "fused")
    assert ei.value.status == gar.AR_ERR_INVALID_ARGUMENT
    assert "static FP8 workspace" in ei.value.detail
    torch.cuda.synchronize()
    assert all(bool((o == 0).all()) for o in out)  # nothing was written
