"""Helpers for GPU tests: numpy storage arrays <-> CUDA tensors, canary-guarded
buffers. Test infrastructure only."""
import numpy as np
import torch

TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "i32": torch.int32}
NPSTORE = {"f32": np.float32, "bf16": np.uint16, "f16": np.uint16, "i32": np.int32}
ESIZE = {"f32": 4, "bf16": 2, "f16": 2, "i32": 4}


def to_dev(a: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype in ("bf16", "f16"):
        t = t.view(torch.int16).view(TORCH[dtype])
    return t.cuda()


def from_dev(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


class Guarded:
    """`n` tensors of `count` elements carved from one allocation with a
    4 KiB canary before and after each; check() asserts no canary byte changed."""

    GUARD = 4096

    def __init__(self, n: int, count: int, dtype: str, offset_bytes: int = 0):
        es = ESIZE[dtype]
        self.nbytes = count * es
        self.slot = self.GUARD + ((self.nbytes + offset_bytes + 255) // 256) * 256 + self.GUARD
        self.raw = torch.empty(n * self.slot + 256, dtype=torch.uint8, device="cuda")
        self.raw.fill_(0xA5)
        self.views = []
        for r in range(n):
            start = r * self.slot + self.GUARD + offset_bytes
            v = self.raw[start: start + self.nbytes]
            self.views.append(v.view(TORCH[dtype]) if count else torch.empty(0, dtype=TORCH[dtype], device="cuda"))
        self.offset = offset_bytes
        self.n = n

    def check(self):
        torch.cuda.synchronize()
        host = self.raw.cpu().numpy()
        for r in range(self.n):
            a = r * self.slot
            pre = host[a: a + self.GUARD + self.offset]
            post = host[a + self.GUARD + self.offset + self.nbytes: (r + 1) * self.slot]
            assert np.all(pre == 0xA5) and np.all(post == 0xA5), f"canary of buffer {r} overwritten"
