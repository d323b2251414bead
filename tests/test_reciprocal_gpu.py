"""The per-hop FP8 kernel's inline reciprocal (the hardware approximation plus
one Newton-Raphson step in fused multiply-adds) must equal the correctly
rounded reciprocal __frcp_rn for every binary32 scale it is used on, every
s in [2^-90, 2^90]: the Markstein quotient that follows needs RN(1/s). This
compiles a small checker against the library's own device header and runs it
over all 1,275,068,417 such bit patterns on the GPU."""
import shutil
import subprocess
import tempfile
from pathlib import Path

import pytest

CSRC = Path(__file__).resolve().parent.parent / "gradient_allreduce_collective_gb300" / "csrc"

SRC = r"""
#include <cstdio>
#include "ar_fp8_common.cuh"

__global__ void check(uint32_t lo, uint32_t hi, unsigned long long* bad, uint32_t* first) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t u = lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; u <= hi; u += stride) {
    const float s = __uint_as_float((uint32_t)u);
    const float got = gar::recip_in_range(s), want = __frcp_rn(s);
    if (__float_as_uint(got) != __float_as_uint(want)) {
      const unsigned long long k = atomicAdd(bad, 1ull);
      if (k < 8) first[k] = (uint32_t)u;
    }
  }
}

int main() {
  unsigned long long* bad;
  uint32_t* first;
  if (cudaMalloc(&bad, 8) != cudaSuccess || cudaMalloc(&first, 32) != cudaSuccess) return 2;
  cudaMemset(bad, 0, 8);
  cudaMemset(first, 0, 32);
  check<<<152 * 8, 256>>>(0x1A800000u, 0x66800000u, bad, first);  // 2^-90 .. 2^90
  if (cudaDeviceSynchronize() != cudaSuccess) return 3;
  unsigned long long h = 0;
  uint32_t f[8];
  cudaMemcpy(&h, bad, 8, cudaMemcpyDeviceToHost);
  cudaMemcpy(f, first, 32, cudaMemcpyDeviceToHost);
  printf("%llu", h);
  for (int i = 0; i < 8 && i < (int)h; ++i) printf(" 0x%08x", f[i]);
  printf("\n");
  return 0;
}
"""


def _nvcc():
    for cand in ("/usr/local/cuda/bin/nvcc", shutil.which("nvcc") or ""):
        if cand and Path(cand).exists():
            return cand
    pytest.skip("nvcc not available")


@pytest.mark.gpu
def test_inline_reciprocal_is_correctly_rounded_over_the_scale_range():
    with tempfile.TemporaryDirectory() as d:
        cu, exe = Path(d) / "r.cu", Path(d) / "r"
        cu.write_text(SRC)
        subprocess.run([_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", f"-I{CSRC}",
                        str(cu), "-o", str(exe)], check=True)
        out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=120).stdout.split()
    assert out[0] == "0", "mismatching scales: " + " ".join(out[1:])
