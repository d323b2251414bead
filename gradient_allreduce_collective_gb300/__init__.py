"""GB300-native gradient allreduce: thin Python binding of libar.so.

Each function here has the name of the C entry point it calls (include/ar.h)
and only marshals arguments: tensor -> device pointer, dtype -> enum, the
current PyTorch stream -> cudaStream_t. All work runs in the library's sm_103a
kernels; there is no fallback path. PyTorch supplies device memory and
streams, and must be imported before the library is loaded so that both use
one CUDA runtime (and one current device).
"""
from __future__ import annotations

import ctypes
from typing import Sequence

import torch  # noqa: F401  (loads the shared CUDA runtime first)

from ._build import build, lib_path

__all__ = [
    "ArError", "build", "lib", "lib_path", "ar_allreduce", "ar_allreduce_slice", "ar_reduce_scatter", "ar_all_gather",
    "ar_bucket_plan", "ar_bucket_flatten", "ar_bucket_unflatten", "ar_bucket_allreduce", "ar_fp8_workspace_bytes",
    "ar_quantize_fp8_blocks", "ar_allreduce_fp8", "ar_allreduce_fp8_fused", "ar_allreduce_fp8_hops", "ar_allreduce_fp8_noalloc",
    "ar_stepwise_workspace_bytes", "ar_allreduce_stepwise", "ar_topk_workspace_bytes", "ar_topk_compress", "ar_sparse_workspace_bytes", "ar_sparse_allreduce",
    "ar_status_string", "ar_last_error", "ar_version",
    "DTYPES", "OPS", "ALGOS", "Comm", "CallRecord",
]

AR_SUCCESS, AR_ERR_INVALID_ARGUMENT, AR_ERR_UNSUPPORTED, AR_ERR_ALIAS, AR_ERR_CUDA, AR_ERR_TIMEOUT, \
    AR_ERR_MISMATCH = range(7)
DTYPES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2, torch.int32: 3}
DTYPE_NAMES = {"f32": 0, "f16": 1, "bf16": 2, "i32": 3}
OPS = {"sum": 0, "avg": 1, "min": 2, "max": 3}
ALGOS = {"ring": 0, "fused": 1, "tree": 2, "step_ring": 3, "step_tree": 4, "auto": 5}
FP8_BLOCK = 128


class ArError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        self.detail = detail
        super().__init__(f"{_status_text(status)} ({status}): {detail}")


class CallRecord(ctypes.Structure):
    """ar_call_record_t: what a rank last did on a communicator."""
    _fields_ = [("comm_id", ctypes.c_uint64), ("seq", ctypes.c_uint64), ("collective", ctypes.c_int),
                ("count", ctypes.c_size_t), ("dtype", ctypes.c_int), ("op", ctypes.c_int), ("algo", ctypes.c_int),
                ("status", ctypes.c_int), ("arrived_mask", ctypes.c_uint64), ("mismatch_mask", ctypes.c_uint64),
                ("arrival_skew_ms", ctypes.c_double)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libar.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not path.exists():
        raise ImportError(f"libar.so is not built ({path}); run gradient_allreduce_collective_gb300.build()")
    L = ctypes.CDLL(str(path))
    vp, sz, ci = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    pp = ctypes.POINTER(ctypes.c_void_p)
    L.ar_allreduce.argtypes = [pp, pp, ci, sz, ci, ci, ci, vp]
    L.ar_reduce_scatter.argtypes = [pp, pp, ci, sz, ci, ci, vp]
    L.ar_allreduce_slice.argtypes = [pp, pp, ci, sz, sz, sz, ci, ci, ci, vp]
    L.ar_all_gather.argtypes = [pp, pp, ci, sz, ci, vp]
    L.ar_bucket_plan.argtypes = [vp, ci, ci, sz, vp, vp, vp, vp]
    L.ar_bucket_flatten.argtypes = [pp, vp, vp, ci, ci, vp, vp]
    L.ar_bucket_unflatten.argtypes = [vp, pp, vp, vp, ci, ci, vp]
    L.ar_bucket_allreduce.argtypes = [pp, pp, ci, ci, vp, vp, sz, ci, ci, ci, vp]
    L.ar_fp8_workspace_bytes.argtypes = [ci, sz]
    L.ar_fp8_workspace_bytes.restype = sz
    L.ar_quantize_fp8_blocks.argtypes = [vp, ci, sz, vp, vp, vp]
    L.ar_allreduce_fp8.argtypes = [pp, pp, ci, sz, ci, ci, ci, ci, vp, sz, vp]
    L.ar_allreduce_fp8_noalloc.argtypes = [pp, pp, ci, sz, ci, ci, ci, ci, vp]
    L.ar_allreduce_fp8_fused.argtypes = [pp, pp, ci, sz, ci, ci, ci, ci, vp]
    L.ar_allreduce_fp8_hops.argtypes = [pp, pp, ci, sz, ci, ci, ci, vp]
    L.ar_stepwise_workspace_bytes.argtypes = [ci, sz, ci]
    L.ar_stepwise_workspace_bytes.restype = sz
    L.ar_allreduce_stepwise.argtypes = [pp, pp, ci, sz, ci, ci, ci, vp, sz, vp]
    L.ar_topk_workspace_bytes.argtypes = [ci, sz, sz]
    L.ar_topk_workspace_bytes.restype = sz
    L.ar_topk_compress.argtypes = [pp, pp, ci, sz, sz, pp, pp, vp, sz, vp]
    L.ar_sparse_workspace_bytes.argtypes = [ci, sz]
    L.ar_sparse_workspace_bytes.restype = sz
    L.ar_sparse_allreduce.argtypes = [pp, pp, vp, ci, sz, ci, ci, pp, vp, sz, vp]
    for name in ("ar_allreduce", "ar_allreduce_stepwise", "ar_allreduce_slice", "ar_reduce_scatter", "ar_all_gather", "ar_bucket_plan", "ar_bucket_flatten",
                 "ar_bucket_unflatten", "ar_bucket_allreduce", "ar_quantize_fp8_blocks", "ar_allreduce_fp8", "ar_allreduce_fp8_noalloc", "ar_allreduce_fp8_fused", "ar_allreduce_fp8_hops",
                 "ar_topk_compress", "ar_sparse_allreduce"):
        getattr(L, name).restype = ci
    L.ar_comm_create.argtypes = [ci, ci, ctypes.POINTER(ctypes.c_void_p)]
    L.ar_comm_destroy.argtypes = [vp]
    L.ar_comm_allreduce.argtypes = [vp, ci, vp, vp, sz, ci, ci, ci, vp]
    L.ar_comm_last_record.argtypes = [vp, ci, ctypes.POINTER(CallRecord)]
    for name in ("ar_comm_create", "ar_comm_destroy", "ar_comm_allreduce", "ar_comm_last_record"):
        getattr(L, name).restype = ci
    L.ar_status_string.argtypes = [ci]
    L.ar_status_string.restype = ctypes.c_char_p
    L.ar_last_error.argtypes = []
    L.ar_last_error.restype = ctypes.c_char_p
    L.ar_version.argtypes = []
    L.ar_version.restype = ctypes.c_char_p
    _lib = L
    return L


def _status_text(st: int) -> str:
    try:
        return lib().ar_status_string(st).decode()
    except Exception:  # pragma: no cover
        return "status"


def ar_status_string(st: int) -> str:
    return lib().ar_status_string(st).decode()


def ar_last_error() -> str:
    return lib().ar_last_error().decode()


def ar_version() -> str:
    return lib().ar_version().decode()


def _check(st: int) -> None:
    if st != AR_SUCCESS:
        raise ArError(st, ar_last_error())


def _ptrs(ts: Sequence) -> ctypes.Array:
    return (ctypes.c_void_p * len(ts))(*[t if isinstance(t, int) else t.data_ptr() for t in ts])


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream if isinstance(stream, int) else stream.cuda_stream


def _same(ts: Sequence[torch.Tensor], what: str):
    if len(ts) == 0:
        raise ValueError(f"{what}: empty list")
    t0 = ts[0]
    for t in ts:
        if t.dtype != t0.dtype or t.numel() != t0.numel() or not t.is_contiguous():
            raise ValueError(f"{what}: tensors must be contiguous with one dtype and size")
    return t0.dtype, t0.numel()


def ar_allreduce(sendbufs: Sequence[torch.Tensor], recvbufs: Sequence[torch.Tensor], op: str = "sum",
                 algo: str = "fused", stream=None) -> None:
    dt, n = _same(sendbufs, "sendbufs")
    if len(recvbufs) != len(sendbufs):
        raise ValueError("one output per rank")
    _same(recvbufs, "recvbufs")
    _check(lib().ar_allreduce(_ptrs(sendbufs), _ptrs(recvbufs), len(sendbufs), n, DTYPES[dt], OPS[op],
                              ALGOS[algo], _stream(stream)))


def ar_stepwise_workspace_bytes(nranks: int, count: int, dtype) -> int:
    dt = DTYPES[dtype] if isinstance(dtype, torch.dtype) else DTYPE_NAMES[dtype]
    return int(lib().ar_stepwise_workspace_bytes(nranks, count, dt))


def ar_allreduce_stepwise(sendbufs: Sequence[torch.Tensor], recvbufs: Sequence[torch.Tensor], workspace,
                          op: str = "sum", algo: str = "step_ring", stream=None) -> None:
    """The stepwise ring / recursive halving-doubling for every element type;
    `workspace` (a device tensor or None) holds the binary32 partials of
    16-bit inputs (ar_stepwise_workspace_bytes)."""
    dt, n = _same(sendbufs, "sendbufs")
    if len(recvbufs) != len(sendbufs):
        raise ValueError("one output per rank")
    _same(recvbufs, "recvbufs")
    ws, wsb = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    _check(lib().ar_allreduce_stepwise(_ptrs(sendbufs), _ptrs(recvbufs), len(sendbufs), n, DTYPES[dt], OPS[op],
                                       ALGOS[algo], ws, wsb, _stream(stream)))


def ar_allreduce_slice(sendbufs: Sequence[torch.Tensor], recvbufs: Sequence[torch.Tensor], count: int, first: int,
                       op: str = "sum", algo: str = "fused", stream=None) -> None:
    """Elements [first, first + n) of the allreduce of `count` elements per rank,
    from each rank's slice of n elements (see include/ar.h)."""
    dt, n = _same(sendbufs, "sendbufs")
    if len(recvbufs) != len(sendbufs):
        raise ValueError("one output per rank")
    _same(recvbufs, "recvbufs")
    _check(lib().ar_allreduce_slice(_ptrs(sendbufs), _ptrs(recvbufs), len(sendbufs), count, first, n, DTYPES[dt],
                                    OPS[op], ALGOS[algo], _stream(stream)))


def ar_reduce_scatter(sendbufs: Sequence[torch.Tensor], recvbufs: Sequence[torch.Tensor], op: str = "sum",
                      stream=None) -> None:
    dt, n = _same(sendbufs, "sendbufs")
    _, rc = _same(recvbufs, "recvbufs")
    _check(lib().ar_reduce_scatter(_ptrs(sendbufs), _ptrs(recvbufs), len(sendbufs), rc, DTYPES[dt], OPS[op],
                                   _stream(stream)))


def ar_all_gather(sendbufs: Sequence[torch.Tensor], recvbufs: Sequence[torch.Tensor], stream=None) -> None:
    dt, sc = _same(sendbufs, "sendbufs")
    _same(recvbufs, "recvbufs")
    _check(lib().ar_all_gather(_ptrs(sendbufs), _ptrs(recvbufs), len(sendbufs), sc, DTYPES[dt], _stream(stream)))


def ar_bucket_plan(counts: Sequence[int], dtype: torch.dtype, cap_bytes: int):
    """Host-only: (bucket_of, offset_of, bucket_counts) lists."""
    t = len(counts)
    c = (ctypes.c_size_t * max(t, 1))(*counts)
    bucket_of = (ctypes.c_int * max(t, 1))()
    offset_of = (ctypes.c_size_t * max(t, 1))()
    bucket_counts = (ctypes.c_size_t * max(t, 1))()
    nb = ctypes.c_int(0)
    _check(lib().ar_bucket_plan(c, t, DTYPES[dtype], cap_bytes, bucket_of, offset_of, bucket_counts,
                                ctypes.byref(nb)))
    return list(bucket_of)[:t], list(offset_of)[:t], list(bucket_counts)[: nb.value]


def ar_bucket_flatten(tensors: Sequence[torch.Tensor], offsets: Sequence[int], bucket: torch.Tensor,
                      stream=None) -> None:
    t = len(tensors)
    counts = (ctypes.c_size_t * max(t, 1))(*[x.numel() for x in tensors])
    offs = (ctypes.c_size_t * max(t, 1))(*offsets)
    _check(lib().ar_bucket_flatten(_ptrs(tensors), counts, offs, t, DTYPES[bucket.dtype], bucket.data_ptr(),
                                   _stream(stream)))


def ar_bucket_unflatten(bucket: torch.Tensor, tensors: Sequence[torch.Tensor], offsets: Sequence[int],
                        stream=None) -> None:
    t = len(tensors)
    counts = (ctypes.c_size_t * max(t, 1))(*[x.numel() for x in tensors])
    offs = (ctypes.c_size_t * max(t, 1))(*offsets)
    _check(lib().ar_bucket_unflatten(bucket.data_ptr(), _ptrs(tensors), counts, offs, t, DTYPES[bucket.dtype],
                                     _stream(stream)))


def ar_bucket_allreduce(tensors: Sequence[Sequence[torch.Tensor]], out_tensors: Sequence[Sequence[torch.Tensor]],
                        offsets: Sequence[int], bucket_count: int, op: str = "avg", algo: str = "fused",
                        stream=None) -> None:
    """tensors[r][t] / out_tensors[r][t]: rank r's tensor t; offsets[t]: its
    element offset in the bucket layout of bucket_count elements."""
    n = len(tensors)
    t = len(tensors[0]) if n else 0
    flat_in = [x for rank in tensors for x in rank]
    flat_out = [x for rank in out_tensors for x in rank]
    if len(flat_in) != n * t or len(flat_out) != n * t:
        raise ValueError("every rank needs the same tensors")
    dt = flat_in[0].dtype
    counts = (ctypes.c_size_t * max(t, 1))(*[x.numel() for x in tensors[0]])
    offs = (ctypes.c_size_t * max(t, 1))(*offsets)
    _check(lib().ar_bucket_allreduce(_ptrs(flat_in), _ptrs(flat_out), n, t, counts, offs, bucket_count, DTYPES[dt],
                                     OPS[op], ALGOS[algo], _stream(stream)))


def ar_fp8_workspace_bytes(nranks: int, count: int) -> int:
    return int(lib().ar_fp8_workspace_bytes(nranks, count))


def ar_quantize_fp8_blocks(x: torch.Tensor, q: torch.Tensor, scales: torch.Tensor, stream=None) -> None:
    _check(lib().ar_quantize_fp8_blocks(x.data_ptr(), DTYPES[x.dtype], x.numel(), q.data_ptr(), scales.data_ptr(),
                                        _stream(stream)))


def ar_allreduce_fp8(sendbufs: Sequence[torch.Tensor], recvbufs: Sequence[torch.Tensor], workspace: torch.Tensor,
                     op: str = "sum", algo: str = "fused", stream=None) -> None:
    dt, n = _same(sendbufs, "sendbufs")
    odt, _ = _same(recvbufs, "recvbufs")
    _check(lib().ar_allreduce_fp8(_ptrs(sendbufs), _ptrs(recvbufs), len(sendbufs), n, DTYPES[dt], DTYPES[odt],
                                  OPS[op], ALGOS[algo], workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def ar_allreduce_fp8_fused(sendbufs: Sequence[torch.Tensor], recvbufs: Sequence[torch.Tensor], op: str = "sum",
                           algo: str = "fused", stream=None) -> None:
    """ar_allreduce_fp8's result with the quantisation fused into the reduction (no workspace)."""
    dt, n = _same(sendbufs, "sendbufs")
    odt, _ = _same(recvbufs, "recvbufs")
    _check(lib().ar_allreduce_fp8_fused(_ptrs(sendbufs), _ptrs(recvbufs), len(sendbufs), n, DTYPES[dt], DTYPES[odt],
                                        OPS[op], ALGOS[algo], _stream(stream)))


def ar_allreduce_fp8_hops(sendbufs: Sequence[torch.Tensor], recvbufs: Sequence[torch.Tensor], op: str = "sum",
                          stream=None) -> None:
    """FP8 re-quantised on every ring hop (see include/ar.h)."""
    dt, n = _same(sendbufs, "sendbufs")
    odt, _ = _same(recvbufs, "recvbufs")
    _check(lib().ar_allreduce_fp8_hops(_ptrs(sendbufs), _ptrs(recvbufs), len(sendbufs), n, DTYPES[dt], DTYPES[odt],
                                       OPS[op], _stream(stream)))


FP8_STATIC_WS_BYTES = 16 * 1024 * 1024


def ar_allreduce_fp8_noalloc(sendbufs: Sequence[torch.Tensor], recvbufs: Sequence[torch.Tensor], op: str = "sum",
                             algo: str = "fused", stream=None) -> None:
    """ar_allreduce_fp8 without a caller workspace, for callers that cannot
    allocate device memory: the library's own fixed FP8_STATIC_WS_BYTES array
    holds the codes and scales (see include/ar.h for the limit and sharing)."""
    dt, n = _same(sendbufs, "sendbufs")
    odt, _ = _same(recvbufs, "recvbufs")
    _check(lib().ar_allreduce_fp8_noalloc(_ptrs(sendbufs), _ptrs(recvbufs), len(sendbufs), n, DTYPES[dt],
                                          DTYPES[odt], OPS[op], ALGOS[algo], _stream(stream)))


def ar_topk_workspace_bytes(nranks: int, count: int, k: int) -> int:
    return int(lib().ar_topk_workspace_bytes(nranks, count, k))


def _idx_ok(t: torch.Tensor, what: str) -> None:
    if t.dtype not in (torch.int32, torch.uint32) or not t.is_contiguous():
        raise ValueError(f"{what}: contiguous 32-bit index tensor expected")


def ar_topk_compress(grads: Sequence[torch.Tensor], residuals: Sequence[torch.Tensor], k: int,
                     idx: Sequence[torch.Tensor], val: Sequence[torch.Tensor], workspace: torch.Tensor,
                     stream=None) -> None:
    """Every rank's Top-K step with error feedback (see include/ar.h):
    residuals[r] becomes grads[r] + residuals[r] with the kept entries zeroed;
    idx[r][:k] / val[r][:k] the kept (index, value) pairs in ascending index order."""
    n = len(grads)
    if len(residuals) != n or len(idx) != n or len(val) != n:
        raise ValueError("one grad, residual, idx and val per rank")
    dt, count = _same(grads, "grads")
    rdt, rcount = _same(residuals, "residuals")
    if dt != torch.float32 or rdt != torch.float32 or rcount != count:
        raise ValueError("grads and residuals: float32 tensors of one size")
    for r in range(n):
        _idx_ok(idx[r], "idx")
        if val[r].dtype != torch.float32 or not val[r].is_contiguous():
            raise ValueError("val: contiguous float32 tensor expected")
        if idx[r].numel() < k or val[r].numel() < k:
            raise ValueError("idx and val need k entries")
    _check(lib().ar_topk_compress(_ptrs(grads), _ptrs(residuals), n, count, k, _ptrs(idx), _ptrs(val),
                                  workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                  _stream(stream)))


def ar_sparse_workspace_bytes(nranks: int, count: int) -> int:
    return int(lib().ar_sparse_workspace_bytes(nranks, count))


def ar_sparse_allreduce(idx: Sequence[torch.Tensor], val: Sequence[torch.Tensor], nnz: Sequence[int],
                        recvbufs: Sequence[torch.Tensor], op: str = "sum", algo: str = "fused",
                        workspace: torch.Tensor | None = None, stream=None) -> None:
    """Allreduce of each rank's sparse vector (idx[r][:nnz[r]], val[r][:nnz[r]])
    into the dense float32 recvbufs (see include/ar.h); SUM and AVG need a
    workspace of ar_sparse_workspace_bytes(nranks, count) bytes and ascending
    indices."""
    n = len(recvbufs)
    if len(idx) != n or len(val) != n or len(nnz) != n:
        raise ValueError("one idx, val, nnz and output per rank")
    _, count = _same(recvbufs, "recvbufs")
    for r in range(n):
        _idx_ok(idx[r], "idx")
        if recvbufs[r].dtype != torch.float32 or val[r].dtype != torch.float32:
            raise ValueError("values and outputs are float32")
        if idx[r].numel() < nnz[r] or val[r].numel() < nnz[r]:
            raise ValueError("idx and val need nnz entries")
    counts = (ctypes.c_size_t * n)(*nnz)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().ar_sparse_allreduce(_ptrs(idx), _ptrs(val), counts, n, count, OPS[op], ALGOS[algo],
                                     _ptrs(recvbufs), ws_ptr, ws_len, _stream(stream)))


class Comm:
    """ar_comm_t: host-side communicator of `nranks` virtual ranks (one host thread per rank)."""

    def __init__(self, nranks: int, timeout_ms: int):
        h = ctypes.c_void_p()
        _check(lib().ar_comm_create(nranks, timeout_ms, ctypes.byref(h)))
        self.handle = h
        self.nranks = nranks

    def allreduce(self, rank: int, sendbuf, recvbuf, count: int | None = None, dtype=None, op: str = "sum",
                  algo: str = "fused", stream=None) -> int:
        """Rank `rank`'s half of an allreduce; returns the status (0 = success). Tensors or raw addresses."""
        if count is None:
            count = sendbuf.numel()
        if dtype is None:
            dtype = sendbuf.dtype
        sp = sendbuf if isinstance(sendbuf, int) else sendbuf.data_ptr()
        rp = recvbuf if isinstance(recvbuf, int) else recvbuf.data_ptr()
        dt = DTYPES[dtype] if not isinstance(dtype, int) else dtype
        st = stream if isinstance(stream, int) else (0 if stream is None else stream.cuda_stream)
        return int(lib().ar_comm_allreduce(self.handle, rank, sp, rp, count, dt, OPS[op], ALGOS[algo], st))

    def last_record(self, rank: int) -> CallRecord:
        rec = CallRecord()
        _check(lib().ar_comm_last_record(self.handle, rank, ctypes.byref(rec)))
        return rec

    def close(self) -> None:
        if self.handle:
            lib().ar_comm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
