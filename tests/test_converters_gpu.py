"""The oracle's binary32 -> E4M3 (nearest even, saturating to +-448) and
binary32 -> bf16 (nearest even) conversions against the GPU's hardware
conversions, the ones the kernels use, for all 2^32 binary32 bit patterns.
E4M3 codes are identical for every non-NaN input, and bf16 patterns are
identical for every non-NaN input; a NaN input gives a NaN on both sides
(payloads are not part of the contract). A small helper compiled against the
library's own device header converts chunks of 2^24 patterns on the GPU; the
oracle converts the same chunks on the host cores."""
import ctypes
import os
import shutil
import subprocess
import tempfile
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

import numpy as np
import pytest

import oracle

CSRC = Path(__file__).resolve().parent.parent / "gradient_allreduce_collective_gb300" / "csrc"
INCLUDE = Path(__file__).resolve().parent.parent / "include"

SRC = r"""
#include <cstdint>
#include <cuda_runtime.h>
#include "ar_fp8_common.cuh"

__global__ void conv(uint32_t lo, uint32_t n, uint8_t* e, uint16_t* b) {
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float x = __uint_as_float(lo + i);
    e[i] = (uint8_t)gar::f32_to_e4m3(x);
    b[i] = (uint16_t)gar::from_f32<gar::DT_BF16>(x);
  }
}

static uint8_t* de = nullptr;
static uint16_t* db = nullptr;
static uint32_t cap = 0;

extern "C" int convert_chunk(uint32_t lo, uint32_t n, uint8_t* e, uint16_t* b) {
  if (n > cap) {
    if (de) cudaFree(de);
    if (db) cudaFree(db);
    de = nullptr;
    db = nullptr;
    cap = 0;
    if (cudaMalloc(&de, n) != cudaSuccess || cudaMalloc(&db, 2ull * n) != cudaSuccess) return 1;
    cap = n;
  }
  conv<<<1024, 256>>>(lo, n, de, db);
  if (cudaGetLastError() != cudaSuccess) return 2;
  if (cudaMemcpy(e, de, n, cudaMemcpyDeviceToHost) != cudaSuccess) return 3;
  if (cudaMemcpy(b, db, 2ull * n, cudaMemcpyDeviceToHost) != cudaSuccess) return 4;
  return 0;
}
"""

CHUNK = 1 << 24


def _nvcc():
    for cand in ("/usr/local/cuda/bin/nvcc", shutil.which("nvcc") or ""):
        if cand and Path(cand).exists():
            return cand
    pytest.skip("nvcc not available")


def _check_chunk(lo, e_gpu, b_gpu):
    x = (np.arange(CHUNK, dtype=np.uint64) + lo).astype(np.uint32).view(np.float32)
    nan = np.isnan(x)
    e_or = oracle.f32_to_e4m3(x)
    b_or = oracle.f32_to_bf16(x)
    bad_e = int(np.count_nonzero((e_or != e_gpu) & ~nan))
    bad_e += int(np.count_nonzero(((e_gpu[nan] & 0x7F) != 0x7F) | ((e_or[nan] & 0x7F) != 0x7F)))
    bad_b = int(np.count_nonzero((b_or != b_gpu) & ~nan))
    b_nan = ((b_gpu[nan] & 0x7F80) == 0x7F80) & ((b_gpu[nan] & 0x7F) != 0)
    o_nan = ((b_or[nan] & 0x7F80) == 0x7F80) & ((b_or[nan] & 0x7F) != 0)
    bad_b += int(np.count_nonzero(~b_nan | ~o_nan))
    return bad_e, bad_b


@pytest.mark.gpu
def test_oracle_converters_match_the_hardware_for_every_binary32():
    with tempfile.TemporaryDirectory() as d:
        cu, so = Path(d) / "conv.cu", Path(d) / "libconv.so"
        cu.write_text(SRC)
        subprocess.run([_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-shared",
                        "-Xcompiler", "-fPIC", f"-I{CSRC}", f"-I{INCLUDE}", str(cu), "-o", str(so)], check=True)
        lib = ctypes.CDLL(str(so))
        lib.convert_chunk.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p]
        lib.convert_chunk.restype = ctypes.c_int
        bad = [0, 0]
        workers = max(1, min(16, os.cpu_count() or 1))
        with ThreadPoolExecutor(max_workers=workers) as pool:
            pending = []

            def drain(keep):
                while len(pending) > keep:  # bounds the host memory held by chunks in flight
                    be, bb = pending.pop(0).result()
                    bad[0] += be
                    bad[1] += bb

            for c in range((1 << 32) // CHUNK):
                lo = c * CHUNK
                e = np.empty(CHUNK, dtype=np.uint8)
                b = np.empty(CHUNK, dtype=np.uint16)
                assert lib.convert_chunk(lo, CHUNK, e.ctypes.data, b.ctypes.data) == 0
                pending.append(pool.submit(_check_chunk, lo, e, b))
                drain(2 * workers)
            drain(0)
    assert bad == [0, 0], bad
