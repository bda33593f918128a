"""Canary-guarded device buffers for the GPU tests (a substitute for a memory
checker, which is not available on the GPU pool).

``guarded(shape, dtype)`` returns a tensor that lives inside a larger
allocation whose 4 KiB before and after it hold the byte 0xA5.  A kernel that
writes past either end of the buffer changes those bytes; ``check_guards()``
(run after every test by an autouse fixture in conftest.py) asserts that every
guard allocated since the last check is intact, then forgets them."""
from __future__ import annotations

GUARD_BYTES = 4096   # also keeps the interior 4 KiB-aligned (the workspace needs 256)
PATTERN = 0xA5
_LIVE = []           # (raw buffer, interior bytes, label)


def guarded(shape, dtype, device="cuda", fill=None, label: str = ""):
    import torch
    shape = tuple(shape) if isinstance(shape, (tuple, list)) else (shape,)
    n = 1
    for v in shape:
        n *= int(v)
    itemsize = torch.empty(0, dtype=dtype).element_size()
    nbytes = n * itemsize
    raw = torch.full((GUARD_BYTES + nbytes + GUARD_BYTES,), PATTERN, dtype=torch.uint8,
                     device=device)
    inner = raw[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(shape)
    if fill is not None:
        inner.fill_(fill)
    _LIVE.append((raw, nbytes, label or f"{dtype} {shape}"))
    return inner


def guarded_like(t, fill=None, label: str = ""):
    return guarded(tuple(t.shape), t.dtype, t.device, fill, label)


def check_guards():
    """Asserts that no guard byte changed; forgets every guarded buffer."""
    global _LIVE
    live, _LIVE = _LIVE, []
    bad = []
    for raw, nbytes, label in live:
        head = raw[:GUARD_BYTES]
        tail = raw[GUARD_BYTES + nbytes:]
        if not bool((head == PATTERN).all()) or not bool((tail == PATTERN).all()):
            bad.append(label)
    assert not bad, f"writes outside the buffer (guard bytes changed): {bad}"
