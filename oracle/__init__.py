"""CPU oracle of the gradient AllReduce -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference arms may import this package. It wraps ``ar_oracle.c`` (plain C,
built with gcc, no FMA contraction, no fast-math) through ctypes; it shares no
code with the CUDA library or its binding, and the library never calls it.

Arrays are numpy arrays in their storage type: ``float32``, ``int32``, or
``uint16`` bit patterns for bf16 / fp16. Every function follows the page
passages cited in ``ar_oracle.c``. The FP8 block semantics (block of 128,
scale amax/448) come from the workload statement, not from the pages; the
arithmetic is pinned by format anchors, brute-force rounding and bounds.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sysconfig
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "ar_oracle.c"
_LIB_DIR = _HERE / "_build"
_lib = None

DTYPES = {"f32": 0, "f16": 1, "bf16": 2, "i32": 3}
OPS = {"sum": 0, "avg": 1, "min": 2, "max": 3}
NP_STORAGE = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16, "i32": np.int32}
FP8_BLOCK = 128


def _lib_path() -> Path:
    tag = sysconfig.get_platform().replace("-", "_")
    return _LIB_DIR / f"liboracle_{tag}.so"


def build(force: bool = False) -> Path:
    """Compile ar_oracle.c with gcc (-O2 -std=c11 -ffp-contract=off)."""
    out = _lib_path()
    if out.exists() and not force and out.stat().st_mtime >= _SRC.stat().st_mtime:
        return out
    _LIB_DIR.mkdir(exist_ok=True)
    tmp = out.with_suffix(f".{os.getpid()}.tmp")
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           str(_SRC), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(str(build()))
    vp, sz, ci = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    pp = ctypes.POINTER(ctypes.c_void_p)
    for name in ("or_ring_allreduce", "or_fold_allreduce", "or_tree_allreduce"):
        getattr(lib, name).argtypes = [pp, pp, ci, sz, ci, ci]
        getattr(lib, name).restype = ci
    lib.or_ring_reduce_scatter.argtypes = [pp, pp, ci, sz, ci, ci]
    lib.or_ring_all_gather.argtypes = [pp, pp, ci, sz, ci]
    lib.or_fold_points.argtypes = [vp, vp, sz, sz, ci, ci, ci, vp]
    lib.or_fold_allreduce_range.argtypes = [pp, pp, ci, sz, sz, sz, ci, ci]
    lib.or_tree_points.argtypes = [vp, sz, ci, ci, ci, vp]
    lib.or_reference_f64.argtypes = [pp, ci, sz, ci, ci, vp, vp]
    lib.or_fp8_quantize.argtypes = [vp, ci, sz, vp, vp]
    lib.or_fp8_quantize.restype = None
    lib.or_fp8_ring_allreduce.argtypes = [pp, pp, ci, sz, ci, ci, ci]
    lib.or_fp8_tree_allreduce.argtypes = [pp, pp, ci, sz, ci, ci, ci]
    lib.or_fp8_ring_blocks.argtypes = [vp, vp, vp, sz, sz, ci, ci, ci, ci, vp]
    lib.or_topk_compress.argtypes = [vp, vp, sz, sz, vp, vp]
    lib.or_sparse_to_dense.argtypes = [vp, vp, sz, sz, vp]
    lib.or_fp8_hop_ring_allreduce.argtypes = [pp, pp, ci, sz, ci, ci, ci]
    lib.or_fp8_hop_blocks_allreduce.argtypes = [pp, pp, ci, sz, ci, ci, ci]
    lib.or_bucket_plan.argtypes = [vp, ci, ci, ctypes.c_uint64, vp, vp, vp, vp]
    lib.or_chunk_len.argtypes = [sz, ci, sz]
    lib.or_chunk_len.restype = sz
    for name, t_in, t_out in (("or_f32_to_bf16_n", vp, vp), ("or_f32_to_f16_n", vp, vp),
                              ("or_f32_to_e4m3_n", vp, vp), ("or_bf16_to_f32_n", vp, vp),
                              ("or_f16_to_f32_n", vp, vp), ("or_e4m3_to_f32_n", vp, vp)):
        getattr(lib, name).argtypes = [t_in, t_out, sz]
        getattr(lib, name).restype = None
    _lib = lib
    return lib


def _ptrs(arrays) -> ctypes.Array:
    return (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def _contig(arrays, dtype):
    out = []
    for a in arrays:
        a = np.ascontiguousarray(a)
        if a.dtype != np.dtype(NP_STORAGE[dtype]):
            raise TypeError(f"expected storage {NP_STORAGE[dtype]} for {dtype}, got {a.dtype}")
        out.append(a)
    return out


def chunk_len(count: int, nranks: int, vec_elems: int) -> int:
    return int(_load().or_chunk_len(count, nranks, vec_elems))


def _allreduce(fn: str, send, dtype: str, op: str):
    send = _contig(send, dtype)
    recv = [np.empty_like(send[0]) for _ in send]
    rc = getattr(_load(), fn)(_ptrs(send), _ptrs(recv), len(send), send[0].size, DTYPES[dtype], OPS[op])
    _check(rc, fn)
    return recv


def ring_allreduce(send, dtype: str, op: str):
    """Literal ring: reduce-scatter then all-gather, chunk by chunk."""
    return _allreduce("or_ring_allreduce", send, dtype, op)


def fold_allreduce(send, dtype: str, op: str):
    """Per-element fold in the ring order (cross-check of the simulator)."""
    return _allreduce("or_fold_allreduce", send, dtype, op)


def fold_allreduce_threads(send, dtype: str, op: str, threads: int):
    """The per-element fold over `threads` disjoint element ranges run on
    host threads at once (the C code releases the interpreter lock); the
    chunk plan is the whole problem's, so the result equals fold_allreduce."""
    from concurrent.futures import ThreadPoolExecutor
    send = _contig(send, dtype)
    recv = [np.empty_like(send[0]) for _ in send]
    count = send[0].size
    sp, rp = _ptrs(send), _ptrs(recv)
    lib = _load()
    bounds = [count * k // threads for k in range(threads + 1)]

    def run(k):
        return lib.or_fold_allreduce_range(sp, rp, len(send), count, bounds[k], bounds[k + 1], DTYPES[dtype],
                                           OPS[op])

    with ThreadPoolExecutor(max_workers=threads) as ex:
        for rc in ex.map(run, range(threads)):
            _check(rc, "or_fold_allreduce_range")
    return recv


def tree_allreduce(send, dtype: str, op: str):
    """Recursive-halving order; len(send) must be a power of two."""
    return _allreduce("or_tree_allreduce", send, dtype, op)


def ring_reduce_scatter(send, dtype: str, op: str):
    send = _contig(send, dtype)
    n = len(send)
    recvcount = send[0].size // n
    recv = [np.empty(recvcount, dtype=send[0].dtype) for _ in send]
    _check(_load().or_ring_reduce_scatter(_ptrs(send), _ptrs(recv), n, recvcount, DTYPES[dtype], OPS[op]),
           "reduce_scatter")
    return recv


def ring_all_gather(send, dtype: str):
    send = _contig(send, dtype)
    n = len(send)
    recv = [np.empty(n * send[0].size, dtype=send[0].dtype) for _ in send]
    _check(_load().or_ring_all_gather(_ptrs(send), _ptrs(recv), n, send[0].size, DTYPES[dtype]), "all_gather")
    return recv


def fold_points(vals: np.ndarray, gidx: np.ndarray, count: int, dtype: str, op: str) -> np.ndarray:
    """vals[j, r] = rank r's value at global element gidx[j] (of `count` per rank)."""
    vals = np.ascontiguousarray(vals, dtype=NP_STORAGE[dtype])
    gidx = np.ascontiguousarray(gidx, dtype=np.int64)
    out = np.empty(vals.shape[0], dtype=vals.dtype)
    _check(_load().or_fold_points(vals.ctypes.data, gidx.ctypes.data, vals.shape[0], count, vals.shape[1],
                                  DTYPES[dtype], OPS[op], out.ctypes.data), "fold_points")
    return out


def tree_points(vals: np.ndarray, dtype: str, op: str) -> np.ndarray:
    vals = np.ascontiguousarray(vals, dtype=NP_STORAGE[dtype])
    out = np.empty(vals.shape[0], dtype=vals.dtype)
    _check(_load().or_tree_points(vals.ctypes.data, vals.shape[0], vals.shape[1], DTYPES[dtype], OPS[op],
                                  out.ctypes.data), "tree_points")
    return out


def reference_f64(send, dtype: str, op: str):
    """(y*, S): fp64 sum (or average) and conditioning scale sum|x| (/N for avg)."""
    send = _contig(send, dtype)
    n = send[0].size
    y = np.empty(n, dtype=np.float64)
    s = np.empty(n, dtype=np.float64)
    _check(_load().or_reference_f64(_ptrs(send), len(send), n, DTYPES[dtype], OPS[op], y.ctypes.data,
                                    s.ctypes.data), "reference_f64")
    return y, s


def fp8_quantize(x: np.ndarray, in_dtype: str):
    x = np.ascontiguousarray(x, dtype=NP_STORAGE[in_dtype])
    nb = (x.size + FP8_BLOCK - 1) // FP8_BLOCK
    q = np.empty(x.size, dtype=np.uint8)
    s = np.empty(nb, dtype=np.float32)
    _load().or_fp8_quantize(x.ctypes.data, DTYPES[in_dtype], x.size, q.ctypes.data, s.ctypes.data)
    return q, s


def fp8_ring_allreduce(send, in_dtype: str, out_dtype: str, op: str):
    send = _contig(send, in_dtype)
    recv = [np.empty(send[0].size, dtype=NP_STORAGE[out_dtype]) for _ in send]
    _check(_load().or_fp8_ring_allreduce(_ptrs(send), _ptrs(recv), len(send), send[0].size, DTYPES[in_dtype],
                                         DTYPES[out_dtype], OPS[op]), "fp8_ring_allreduce")
    return recv


def fp8_tree_allreduce(send, in_dtype: str, out_dtype: str, op: str):
    send = _contig(send, in_dtype)
    recv = [np.empty(send[0].size, dtype=NP_STORAGE[out_dtype]) for _ in send]
    _check(_load().or_fp8_tree_allreduce(_ptrs(send), _ptrs(recv), len(send), send[0].size, DTYPES[in_dtype],
                                         DTYPES[out_dtype], OPS[op]), "fp8_tree_allreduce")
    return recv


def _fp8_hop(fn: str, send, in_dtype: str, out_dtype: str, op: str):
    send = _contig(send, in_dtype)
    recv = [np.empty(send[0].size, dtype=NP_STORAGE[out_dtype]) for _ in send]
    _check(getattr(_load(), fn)(_ptrs(send), _ptrs(recv), len(send), send[0].size, DTYPES[in_dtype],
                                DTYPES[out_dtype], OPS[op]), fn)
    return recv


def fp8_hop_ring_allreduce(send, in_dtype: str, out_dtype: str, op: str):
    """FP8 on every ring hop: literal ring simulation with quantised wire buffers."""
    return _fp8_hop("or_fp8_hop_ring_allreduce", send, in_dtype, out_dtype, op)


def fp8_hop_blocks_allreduce(send, in_dtype: str, out_dtype: str, op: str):
    """The same computation written per block (cross-check)."""
    return _fp8_hop("or_fp8_hop_blocks_allreduce", send, in_dtype, out_dtype, op)


def fp8_ring_blocks(blocks: np.ndarray, first: np.ndarray, blen: np.ndarray, count: int, in_dtype: str,
                    out_dtype: str, op: str) -> np.ndarray:
    """blocks[j, r, :blen[j]] = rank r's quantisation block j, starting at element first[j]."""
    blocks = np.ascontiguousarray(blocks, dtype=NP_STORAGE[in_dtype])
    assert blocks.ndim == 3 and blocks.shape[2] == FP8_BLOCK
    first = np.ascontiguousarray(first, dtype=np.int64)
    blen = np.ascontiguousarray(blen, dtype=np.int32)
    out = np.zeros((blocks.shape[0], FP8_BLOCK), dtype=NP_STORAGE[out_dtype])
    _check(_load().or_fp8_ring_blocks(blocks.ctypes.data, first.ctypes.data, blen.ctypes.data, blocks.shape[0],
                                      count, blocks.shape[1], DTYPES[in_dtype], DTYPES[out_dtype], OPS[op],
                                      out.ctypes.data), "fp8_ring_blocks")
    return out


def topk_compress(grad, residual, k: int):
    """(idx, val, new_residual): a = grad + residual; the k largest |a| (ties: lower
    index first) as ascending (index, value) pairs; residual = a with those zeroed."""
    g = np.ascontiguousarray(grad, dtype=np.float32)
    e = np.array(residual, dtype=np.float32, copy=True)
    idx = np.empty(max(k, 1), dtype=np.uint32)
    val = np.empty(max(k, 1), dtype=np.float32)
    _check(_load().or_topk_compress(g.ctypes.data, e.ctypes.data, g.size, k, idx.ctypes.data, val.ctypes.data),
           "topk_compress")
    return idx[:k].copy(), val[:k].copy(), e


def sparse_to_dense(idx, val, count: int):
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    val = np.ascontiguousarray(val, dtype=np.float32)
    out = np.empty(count, dtype=np.float32)
    _check(_load().or_sparse_to_dense(idx.ctypes.data, val.ctypes.data, idx.size, count, out.ctypes.data),
           "sparse_to_dense")
    return out


def sparse_ring_allreduce(idx_list, val_list, count: int, op: str):
    """Allreduce of sparse vectors: the ring allreduce of their dense forms."""
    dense = [sparse_to_dense(i, v, count) for i, v in zip(idx_list, val_list)]
    return ring_allreduce(dense, "f32", op)


def bucket_plan(counts, esize: int, cap_bytes: int):
    """(bucket_of, offset_of, bucket_counts) under the reverse-order greedy rule."""
    c = np.ascontiguousarray(counts, dtype=np.uint64)
    t = c.size
    bucket_of = np.empty(t, dtype=np.int32)
    offset_of = np.empty(t, dtype=np.uint64)
    bucket_counts = np.empty(max(t, 1), dtype=np.uint64)
    nb = np.zeros(1, dtype=np.int32)
    _check(_load().or_bucket_plan(c.ctypes.data, t, esize, cap_bytes, bucket_of.ctypes.data,
                                  offset_of.ctypes.data, bucket_counts.ctypes.data, nb.ctypes.data), "bucket_plan")
    return bucket_of, offset_of, bucket_counts[: int(nb[0])].copy()


def _conv(fn: str, x: np.ndarray, out_dtype) -> np.ndarray:
    x = np.ascontiguousarray(x)
    y = np.empty(x.size, dtype=out_dtype)
    getattr(_load(), fn)(x.ctypes.data, y.ctypes.data, x.size)
    return y


def f32_to_bf16(x):
    return _conv("or_f32_to_bf16_n", np.asarray(x, dtype=np.float32), np.uint16)


def f32_to_f16(x):
    return _conv("or_f32_to_f16_n", np.asarray(x, dtype=np.float32), np.uint16)


def f32_to_e4m3(x):
    return _conv("or_f32_to_e4m3_n", np.asarray(x, dtype=np.float32), np.uint8)


def bf16_to_f32(x):
    return _conv("or_bf16_to_f32_n", np.asarray(x, dtype=np.uint16), np.float32)


def f16_to_f32(x):
    return _conv("or_f16_to_f32_n", np.asarray(x, dtype=np.uint16), np.float32)


def e4m3_to_f32(x):
    return _conv("or_e4m3_to_f32_n", np.asarray(x, dtype=np.uint8), np.float32)
