"""Helpers for the GPU tests: rank buffers in device memory (with guard
bands), calls through the C ABI, and sampled comparison with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import reducescatter_reduction_gb300 as ccl
from reducescatter_reduction_gb300 import build as ccl_build

GUARD = 256           # guard-band bytes before and after every buffer
CANARY = 0x5A


def ensure_built():
    ccl_build.build()
    ccl.load_library()


def to_torch(arr: np.ndarray) -> torch.Tensor:
    """Raw element storage as a torch tensor of the same width."""
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16))
    return torch.from_numpy(arr)


def to_numpy(t: torch.Tensor, storage) -> np.ndarray:
    a = t.cpu().numpy()
    return a.view(storage) if a.dtype != storage else a


class RankBuffers:
    """p device buffers of n elements, each inside its own allocation with a
    canary-filled guard band on both sides (offset shifts the data start by
    that many bytes, for misaligned-pointer tests).  device="pinned" puts
    them in page-locked host memory instead, which the kernels address
    directly."""

    def __init__(self, host: list[np.ndarray] | None, n: int, storage, p: int | None = None,
                 offset: int = 0, device="cuda"):
        self.storage = np.dtype(storage)
        self.s = self.storage.itemsize
        self.n = n
        self.p = len(host) if host is not None else p
        self.offset = offset
        nbytes = n * self.s
        self.raw = []
        self.views = []
        pinned = device == "pinned"
        where = "cpu" if pinned else device
        for r in range(self.p):
            raw = torch.full((GUARD + offset + nbytes + GUARD,), CANARY, dtype=torch.uint8, device=where)
            if pinned:
                raw = raw.pin_memory()
            body = raw[GUARD + offset: GUARD + offset + nbytes]
            if host is not None:
                body.copy_(torch.from_numpy(host[r].view(np.uint8).reshape(-1)).to(where))
            self.raw.append(raw)
            self.views.append(body)

    def ptrs(self):
        return [v.data_ptr() if v.numel() else r.data_ptr() + GUARD + self.offset
                for v, r in zip(self.views, self.raw)]

    def ptr(self, r, elem_offset=0):
        return self.ptrs()[r] + elem_offset * self.s

    def host(self, r) -> np.ndarray:
        return self.views[r].cpu().numpy().view(self.storage).copy()

    def at(self, r, idx: np.ndarray) -> np.ndarray:
        """Elements idx of rank r, gathered on the device."""
        t = self.views[r].view(torch.int16 if self.s == 2 else torch.int32)
        sel = t[torch.from_numpy(idx.astype(np.int64)).to(t.device)]
        return sel.cpu().numpy().view(self.storage)

    def guards_intact(self) -> bool:
        for raw in self.raw:
            head = raw[:GUARD + self.offset]
            tail = raw[GUARD + self.offset + self.n * self.s:]
            if not (bool((head == CANARY).all()) and bool((tail == CANARY).all())):
                return False
        return True

    def identical_across_ranks(self) -> bool:
        return all(torch.equal(self.views[0], v) for v in self.views[1:])


class Comm:
    """A communicator over RankBuffers (inputs) and optional outputs."""

    def __init__(self, bufs: RankBuffers, outs=None, out_ptrs=None):
        self.h = ccl.ccl_comm_create(bufs.p, bufs.ptrs())
        if outs is not None:
            ccl.ccl_comm_set_outputs(self.h, outs.ptrs())
        elif out_ptrs is not None:
            ccl.ccl_comm_set_outputs(self.h, out_ptrs)

    def __enter__(self):
        return self

    def __exit__(self, *a):
        ccl.ccl_comm_destroy(self.h)


def stream_ptr():
    return torch.cuda.current_stream().cuda_stream


def sample_indices(p: int, n: int, count: int = 100000, seed: int = 0) -> np.ndarray:
    """Every chunk's first and last elements (and their neighbours), the
    buffer ends, and random elements."""
    idx = set()
    for c in range(p):
        b, e = oracle.chunk_bounds(p, n, c)
        for v in (b - 1, b, b + 1, b + 7, b + 8, e - 9, e - 8, e - 1, e):
            if 0 <= v < n:
                idx.add(v)
    for v in list(range(min(n, 64))) + list(range(max(0, n - 64), n)):
        idx.add(v)
    rng = np.random.default_rng(seed)
    if n:
        idx.update(rng.integers(0, n, min(count, n)).tolist())
    return np.array(sorted(idx), dtype=np.uint64)


def bits_equal(a: np.ndarray, b: np.ndarray) -> bool:
    return a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8))
