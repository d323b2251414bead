"""Seeded synthetic inputs shared by the tests and the benchmark.

This module draws values only: it holds none of the allreduce arithmetic and
imports neither the CUDA library nor the oracle. Every value is a pure
function of (seed, element index) -- a SplitMix64 counter hash feeding a
Box-Muller normal, a uniform or a bounded integer (the exact definition is in
``synth.c``) -- so a rank's buffer, or any slice of it, regenerates
identically anywhere. Rank ``r`` of a workload uses ``seed = base + r``.

Reduced-precision inputs (bf16, fp16) are the fp32 draw rounded by PyTorch's
CPU conversion (round to nearest even); they are returned as raw ``uint16``
bit patterns so that both sides see the same bytes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sysconfig
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "synth.c"
_LIB_DIR = _HERE / "_build"
_lib = None


def _lib_path() -> Path:
    tag = sysconfig.get_platform().replace("-", "_")
    return _LIB_DIR / f"libsynth_{tag}.so"


def build(force: bool = False) -> Path:
    """Compile synth.c with gcc into a shared library next to it."""
    out = _lib_path()
    if out.exists() and not force and out.stat().st_mtime >= _SRC.stat().st_mtime:
        return out
    _LIB_DIR.mkdir(exist_ok=True)
    tmp = out.with_suffix(f".{os.getpid()}.tmp")
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           str(_SRC), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(str(build()))
        u64, sz, dbl, ci = ctypes.c_uint64, ctypes.c_size_t, ctypes.c_double, ctypes.c_int
        lib.synth_normal_f32.argtypes = [ctypes.c_void_p, u64, sz, u64, dbl, dbl, dbl, ci]
        lib.synth_uniform_f32.argtypes = [ctypes.c_void_p, u64, sz, u64, dbl, dbl, ci]
        lib.synth_uniform_i32.argtypes = [ctypes.c_void_p, u64, sz, u64, ctypes.c_int64,
                                          ctypes.c_int64, ci]
        lib.synth_splitmix64.argtypes = [u64]
        lib.synth_splitmix64.restype = u64
        _lib = lib
    return _lib


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def splitmix64(state: int) -> int:
    return int(_load().synth_splitmix64(state & (2**64 - 1)))


def normal_f32(n: int, seed: int, sigma: float, outlier_p: float = 0.0,
               outlier_scale: float = 1.0, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _load().synth_normal_f32(out.ctypes.data, first, n, seed, sigma, outlier_p, outlier_scale,
                             _threads())
    return out


def uniform_f32(n: int, seed: int, lo: float, hi: float, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _load().synth_uniform_f32(out.ctypes.data, first, n, seed, lo, hi, _threads())
    return out


def uniform_i32(n: int, seed: int, lo: int, hi: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _load().synth_uniform_i32(out.ctypes.data, first, n, seed, lo, hi, _threads())
    return out


def to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 draw -> storage dtype ('f32', 'bf16', 'f16'); bf16/f16 as uint16 bits."""
    if dtype == "f32":
        return x
    import torch  # conversion only
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype == "bf16":
        return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if dtype == "f16":
        return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    raise ValueError(dtype)


def ranks_normal(nranks: int, count: int, sigma: float, base_seed: int = 0, dtype: str = "f32",
                 outlier_p: float = 0.0, outlier_scale: float = 1.0) -> list[np.ndarray]:
    return [to_dtype(normal_f32(count, base_seed + r, sigma, outlier_p, outlier_scale), dtype)
            for r in range(nranks)]


def ranks_uniform(nranks: int, count: int, lo: float, hi: float, base_seed: int = 0,
                  dtype: str = "f32") -> list[np.ndarray]:
    return [to_dtype(uniform_f32(count, base_seed + r, lo, hi), dtype) for r in range(nranks)]


def ranks_int(nranks: int, count: int, lo: int, hi: int, base_seed: int = 0) -> list[np.ndarray]:
    return [uniform_i32(count, base_seed + r, lo, hi) for r in range(nranks)]


def gpt2_small_param_shapes() -> list[tuple[str, tuple[int, ...]]]:
    """Parameter shapes, in registration order, of a 12-layer decoder transformer
    with d_model 768, 12 heads, vocabulary 50,257 and context 1,024 (GPT-2 small
    layout: token and position embeddings, 12 blocks of {ln_1, c_attn, c_proj,
    ln_2, c_fc, mlp c_proj}, final layer norm). 148 tensors, 124,439,808 values."""
    d, v, ctx, L = 768, 50257, 1024, 12
    shapes: list[tuple[str, tuple[int, ...]]] = [("wte", (v, d)), ("wpe", (ctx, d))]
    for i in range(L):
        p = f"h.{i}."
        shapes += [
            (p + "ln_1.weight", (d,)), (p + "ln_1.bias", (d,)),
            (p + "attn.c_attn.weight", (d, 3 * d)), (p + "attn.c_attn.bias", (3 * d,)),
            (p + "attn.c_proj.weight", (d, d)), (p + "attn.c_proj.bias", (d,)),
            (p + "ln_2.weight", (d,)), (p + "ln_2.bias", (d,)),
            (p + "mlp.c_fc.weight", (d, 4 * d)), (p + "mlp.c_fc.bias", (4 * d,)),
            (p + "mlp.c_proj.weight", (4 * d, d)), (p + "mlp.c_proj.bias", (d,)),
        ]
    shapes += [("ln_f.weight", (d,)), ("ln_f.bias", (d,))]
    return shapes
