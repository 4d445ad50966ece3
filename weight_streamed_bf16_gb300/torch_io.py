"""PyTorch plumbing around the C ABI: device memory, pinned host memory and
streams come from torch; every operator call goes to libpsi.

Nothing here computes any part of an operator.
"""
from __future__ import annotations

import torch

from . import psi

MiB = 1 << 20


def ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def pinned_like(t: torch.Tensor) -> torch.Tensor:
    """A pinned host copy of a CPU tensor (host weights stream from here)."""
    out = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    out.copy_(t)
    return out


def heads_view(t: torch.Tensor) -> psi.psi_heads:
    """psi_heads of a [heads x tokens x dh] view (strides in elements)."""
    assert t.dtype == torch.bfloat16 and t.dim() == 3 and t.stride(2) == 1
    return psi.psi_heads(t.data_ptr(), t.stride(1), t.stride(0))


class Arena:
    """An arena over a torch-allocated device buffer of `slots * page_bytes`."""

    def __init__(self, page_bytes: int, slots: int, device="cuda",
                 compute: torch.cuda.Stream | None = None,
                 copy: torch.cuda.Stream | None = None):
        dev = torch.device(device)
        self.page_bytes = page_bytes
        # 1024 extra bytes so the base can be aligned to 1024
        self.buf = torch.empty(page_bytes * slots + 1024, dtype=torch.uint8, device=dev)
        base = self.buf.data_ptr()
        self.base = (base + 1023) // 1024 * 1024
        self.compute = compute or torch.cuda.current_stream(dev)
        self.copy = copy or torch.cuda.Stream(dev)
        self.handle = psi.psi_arena_create(self.base, page_bytes * slots, page_bytes,
                                           self.compute.cuda_stream, self.copy.cuda_stream)

    @property
    def slots(self) -> int:
        return psi.psi_arena_slots(self.handle)

    def sync(self, timeout_ms: int = 120000):
        psi.psi_sync(self.handle, timeout_ms)

    def stats(self) -> dict:
        return psi.psi_arena_stats(self.handle)

    def close(self):
        if self.handle:
            psi.psi_arena_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Journal:
    """A host state journal over a pinned region of `slots * slot_bytes`,
    ordered against `arena`'s compute stream."""

    def __init__(self, arena: Arena, slot_bytes: int, slots: int):
        self.arena = arena
        self.slot_bytes = slot_bytes
        self.host = torch.empty(slot_bytes * slots, dtype=torch.uint8, pin_memory=True)
        self.handle = psi.psi_journal_create(arena.handle, self.host.data_ptr(),
                                             slot_bytes * slots, slot_bytes)

    def commit(self, key, t: torch.Tensor):
        psi.psi_journal_commit(self.handle, key, t.data_ptr(), t.numel() * t.element_size())

    def reload(self, key, t: torch.Tensor):
        psi.psi_journal_reload(self.handle, key, t.data_ptr(), t.numel() * t.element_size())

    def acquire(self, key):
        psi.psi_journal_acquire(self.handle, key)

    def fence(self, t: torch.Tensor):
        psi.psi_journal_fence(self.handle, t.data_ptr(), t.numel() * t.element_size())

    def drop(self, key):
        psi.psi_journal_drop(self.handle, key)

    def host_tensor(self, key, like: torch.Tensor, timeout_ms: int = 10000) -> torch.Tensor:
        """A CPU copy of the committed entry, viewed with `like`'s dtype and
        shape (waits for the entry's D2H copy)."""
        addr, n = psi.psi_journal_host_view(self.handle, key, timeout_ms)
        off = addr - self.host.data_ptr()
        raw = self.host[off:off + n].clone()
        return raw.view(like.dtype).view(like.shape)

    def stats(self) -> dict:
        return psi.psi_journal_get_stats(self.handle)

    def close(self):
        if self.handle:
            psi.psi_journal_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class LinearWeight:
    """Host (pinned) and optional resident copies of W [rows x cols]."""

    def __init__(self, W: torch.Tensor, page_bytes: int, page_rows: int | None = None,
                 resident: bool = False, device="cuda"):
        assert W.dtype == torch.bfloat16 and W.dim() == 2
        self.host = W if W.is_pinned() else pinned_like(W.contiguous())
        self.rows, self.cols = W.shape
        self.page_rows = page_rows or psi.psi_plan_linear(self.rows, self.cols, page_bytes)
        self.dev = self.host.to(device) if resident else None

    def desc(self) -> psi.psi_linear_weight:
        return psi.psi_linear_weight(self.host.data_ptr(), ptr(self.dev), self.rows, self.cols,
                                     self.page_rows)


class FfnWeight:
    """Packed page image of U [h x d], V [r x h] in pinned memory (+ resident copy)."""

    def __init__(self, U: torch.Tensor, V: torch.Tensor, slice_: int, resident: bool = False,
                 device="cuda", host_image: torch.Tensor | None = None):
        self.h, self.d = U.shape
        self.r = V.shape[0]
        assert V.shape[1] == self.h
        self.slice = slice_
        self.page_bytes = psi.psi_ffn_page_bytes(self.d, self.r, slice_)
        n = (self.h // slice_) * self.page_bytes
        if host_image is None:
            host_image = torch.empty(n, dtype=torch.uint8, pin_memory=True)
            Uc, Vc = U.contiguous(), V.contiguous()
            psi.psi_ffn_pack(Uc.data_ptr(), Vc.data_ptr(), self.d, self.h, self.r, slice_,
                             host_image.data_ptr())
        self.host = host_image
        self.dev = self.host.to(device) if resident else None

    def desc(self) -> psi.psi_ffn_weight:
        return psi.psi_ffn_weight(self.host.data_ptr(), ptr(self.dev), self.d, self.h, self.r,
                                  self.slice)


def ffn_workspace(N: int, r: int, slice_: int, device="cuda"):
    hb, ab = psi.psi_ffn_workspace(N, r, slice_)
    hid = torch.empty(hb // 2, dtype=torch.bfloat16, device=device)
    acc = torch.empty(ab // 4, dtype=torch.float32, device=device)
    return hid, acc
