"""Canary guard regions around device buffers (a debugging aid for tests).

A guarded buffer is one allocation of ``guard + nbytes + guard`` bytes whose
two guard regions hold a fixed byte pattern; the caller uses the middle.  A
kernel or copy that writes past either end of the middle changes a guard,
which ``corrupted`` reports.  Works on any torch device (the CPU included).
"""
from __future__ import annotations

GUARD_BYTES = 256


def _pattern(n: int, device):
    import torch
    # bytes 0xA5 ^ (i mod 256): no run of zeros, no single repeated value
    return (torch.arange(n, dtype=torch.int32, device=device) % 256 ^ 0xA5).to(torch.uint8)


class Guarded:
    """One guarded allocation; ``view`` is the usable middle."""

    def __init__(self, nbytes: int, device, guard: int = GUARD_BYTES, name: str = ""):
        import torch
        self.guard, self.nbytes, self.name = guard, nbytes, name
        self.raw = torch.empty(nbytes + 2 * guard, dtype=torch.uint8, device=device)
        pat = _pattern(guard, device)
        self.raw[:guard] = pat
        self.raw[guard + nbytes:] = pat
        self.view = self.raw[guard:guard + nbytes]

    def corrupted(self) -> list:
        """[(name, 'head' | 'tail', first changed byte offset)] for each changed guard."""
        import torch
        pat = _pattern(self.guard, self.raw.device)
        out = []
        for side, reg in (("head", self.raw[:self.guard]), ("tail", self.raw[self.guard + self.nbytes:])):
            bad = torch.nonzero(reg != pat)
            if bad.numel():
                out.append((self.name, side, int(bad[0].item())))
        return out


class GuardSet:
    """Every guarded buffer of one owner, checked together."""

    def __init__(self, guard: int = GUARD_BYTES):
        self.guard = guard
        self.items = []

    def alloc(self, nbytes: int, device, name: str = ""):
        g = Guarded(nbytes, device, self.guard, name)
        self.items.append(g)
        return g.view

    def corrupted(self) -> list:
        out = []
        for g in self.items:
            out.extend(g.corrupted())
        return out
