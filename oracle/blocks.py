"""Block-management oracle: a reference-counted block allocator with
copy-on-write, and block copy / swap on a ``PoolMirror``.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU legs of ``bench.py`` may import this module; the product never does,
and this module never imports the product.

What it follows: "KV cache, PagedAttention and FlashAttention", Problem 4,
"The idea" -- physical blocks are handed out on demand and listed in each
sequence's block table; several tables may point at one block, which then
carries a reference count; a shared block is copied before it is written
(copy-on-write); when memory runs out a sequence's blocks may be swapped to
CPU memory and back.  "Memory Management in LLM Serving Systems",
"Eviction: recompute or offload?" gives the reload-from-CPU path.

Everything is written one operation at a time over plain Python lists, in
the order the library documents: free blocks are handed out lowest id
first, and every call checks its whole argument before changing anything.
"""
from __future__ import annotations

import numpy as np


class AllocatorModel:
    """``ref[i]`` is the number of block-table entries that point at block i;
    a block is free exactly when ``ref[i] == 0``."""

    def __init__(self, num_blocks: int):
        if num_blocks <= 0:
            raise ValueError("num_blocks must be positive")
        self.ref = [0] * int(num_blocks)

    def free_blocks(self) -> int:
        return sum(1 for r in self.ref if r == 0)

    def _lowest_free(self) -> int:
        for i, r in enumerate(self.ref):
            if r == 0:
                return i
        raise MemoryError("no free block")

    def _check_held(self, ids, count_repeats: bool):
        for i in ids:
            if not 0 <= i < len(self.ref):
                raise IndexError(f"block {i} out of range")
            if self.ref[i] == 0:
                raise ValueError(f"block {i} is not allocated")
        if count_repeats:
            for i in set(ids):
                if list(ids).count(i) > self.ref[i]:
                    raise ValueError(f"block {i} released more often than it is referenced")

    def take(self, n: int) -> list[int]:
        """n fresh blocks, each referenced once."""
        if self.free_blocks() < n:
            raise MemoryError(f"{n} blocks wanted, {self.free_blocks()} free")
        out = []
        for _ in range(n):
            i = self._lowest_free()
            self.ref[i] = 1
            out.append(i)
        return out

    def share(self, ids) -> None:
        """One more table entry points at each listed block."""
        ids = [int(i) for i in ids]
        self._check_held(ids, count_repeats=False)
        for i in ids:
            self.ref[i] += 1

    def release(self, ids) -> None:
        """One table entry per listed block stops pointing at it."""
        ids = [int(i) for i in ids]
        self._check_held(ids, count_repeats=True)
        for i in ids:
            self.ref[i] -= 1

    def prepare_write(self, ids):
        """Copy-on-write before writing through the entries ``ids``: an entry
        whose block is also referenced elsewhere moves to a fresh block, and
        (old, fresh) is a copy to make.  Returns (new_ids, copies)."""
        ids = [int(i) for i in ids]
        self._check_held(ids, count_repeats=False)
        # enough free blocks for every copy this list will need?
        ref = list(self.ref)
        need = 0
        for i in ids:
            if ref[i] > 1:
                need += 1
                ref[i] -= 1
        if self.free_blocks() < need:
            raise MemoryError(f"{need} copies needed, {self.free_blocks()} free")
        copies = []
        for k, i in enumerate(ids):
            if self.ref[i] > 1:
                fresh = self._lowest_free()
                self.ref[fresh] = 1
                self.ref[i] -= 1
                copies.append((i, fresh))
                ids[k] = fresh
        return ids, copies


def copy_blocks(mirror, src, dst) -> None:
    """Block dst[i] of the mirror gets block src[i]'s K and V rows (all heads)
    and, in a 4-bit mirror, its value rows' (scale, zero point)."""
    for s, d in zip((int(x) for x in src), (int(x) for x in dst)):
        mirror.k[d] = mirror.k[s]
        mirror.v[d] = mirror.v[s]
        if mirror.v_params is not None:
            mirror.v_params[d] = mirror.v_params[s]


def _parts(mirror):
    """The arrays one block owns, in host-entry order: K, V, then (4-bit) the value parameters."""
    return [mirror.k, mirror.v] + ([mirror.v_params] if mirror.v_params is not None else [])


def swap_out(mirror, ids) -> bytes:
    """The host image of blocks ``ids``: per block, its K bytes, its V bytes and,
    in a 4-bit mirror, its value parameters' bytes."""
    parts = []
    for i in (int(x) for x in ids):
        for arr in _parts(mirror):
            parts.append(np.ascontiguousarray(arr[i]).tobytes())
    return b"".join(parts)


def swap_in(mirror, image: bytes, ids) -> None:
    """Blocks ``ids`` of the mirror get the bytes of ``image`` (as swap_out lays it out)."""
    arrs = _parts(mirror)
    entry = sum(arr[0].nbytes for arr in arrs)
    for n, i in enumerate(int(x) for x in ids):
        off = n * entry
        for arr in arrs:
            arr[i] = np.frombuffer(image, dtype=arr.dtype, count=arr[0].size, offset=off).reshape(arr[0].shape)
            off += arr[0].nbytes
