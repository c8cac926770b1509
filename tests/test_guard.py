"""The canary checker the GPU tests run after each test, exercised on the CPU:
an untouched guarded buffer reports nothing, a write one byte past either end
of the usable middle is reported with its side and offset, and writes inside
the middle are not."""
import torch

from any_precision_weight_gb300.guard import GuardSet, Guarded


def test_untouched_and_inside_writes_are_clean():
    g = Guarded(1000, "cpu", guard=64, name="buf")
    assert g.view.numel() == 1000
    g.view.fill_(0)
    g.view[0] = 7
    g.view[-1] = 9
    assert g.corrupted() == []


def test_overrun_and_underrun_are_reported():
    gs = GuardSet(guard=32)
    a = gs.alloc(100, "cpu", "a")
    b = gs.alloc(50, "cpu", "b")
    assert gs.corrupted() == []
    a.view(torch.uint8)  # the middle is a plain tensor view
    ga, gb = gs.items
    ga.raw[32 + 100 + 3] ^= 0xFF        # 4th byte past the end of a
    gb.raw[31] ^= 0x01                   # the byte just before b
    assert gs.corrupted() == [("a", "tail", 3), ("b", "head", 31)]


def test_guard_pattern_is_not_a_constant():
    g = Guarded(16, "cpu", guard=256)
    head = g.raw[:256]
    assert len(set(head.tolist())) == 256    # every byte value once: a zero fill is caught
