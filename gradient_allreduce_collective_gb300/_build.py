"""In-tree build of libar.so: every CUDA/C++ translation unit under csrc/ is
compiled by nvcc for sm_103a only (one -gencode), in parallel, and linked
against the shared CUDA runtime so the library uses the same runtime (and the
same current device) as the process that loads it."""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sysconfig
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = PKG / "_build"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", "") + "/bin/nvcc", "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libar.so")
    return found


def _tag() -> str:
    return sysconfig.get_platform().replace("-", "_")


def lib_path() -> Path:
    return BUILD / f"libar_{_tag()}.so"


def _sources() -> list[Path]:
    return sorted(list(CSRC.glob("*.cu")) + list(CSRC.glob("*.cpp")))


def _fingerprint(extra: list[str]) -> str:
    h = hashlib.sha256()
    for p in sorted(list(CSRC.iterdir()) + [INCLUDE / "ar.h"]):
        if p.is_file():
            h.update(p.name.encode())
            h.update(p.read_bytes())
    h.update(" ".join(ARCH + CUDA_FLAGS + extra).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, jobs: int | None = None) -> Path:
    """Compile and link libar.so (skipped when sources and flags are unchanged)."""
    out = lib_path()
    stamp = out.with_suffix(".sha256")
    fp = _fingerprint([])
    if not force and out.exists() and stamp.exists() and stamp.read_text() == fp:
        return out
    nvcc = _nvcc()
    objdir = BUILD / f"obj_{_tag()}"
    objdir.mkdir(parents=True, exist_ok=True)
    srcs = _sources()

    def compile_one(src: Path) -> Path:
        obj = objdir / (src.name + ".o")
        cmd = [nvcc, *ARCH, *CUDA_FLAGS, "-c", str(src), "-o", str(obj)]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src.name}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr)
        return obj

    n = jobs or min(len(srcs), max(1, os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=n) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = out.with_suffix(f".{os.getpid()}.tmp")
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", str(tmp), *map(str, objs)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, out)
    stamp.write_text(fp)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))
