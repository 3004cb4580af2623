"""Python binding of the host KV block manager in libpagedkv.so (see include/pagedkv.h).

The manager decides where every token's K/V lives: fresh blocks on demand, sharing by
fork, copy-on-write when a sharer writes into a shared block, reuse of a finished
sequence's blocks.  Its output feeds the device calls directly: the slots go to
paged_kv_append, the copy-on-write pairs to paged_block_copy, the tables and lengths
to paged_attention_decode.
"""
from __future__ import annotations

import ctypes

import torch

from . import PagedKVError, _check, library


class BlockStats(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("free_blocks", ctypes.c_int32), ("used_blocks", ctypes.c_int32),
                ("num_sequences", ctypes.c_int32), ("shared_blocks", ctypes.c_int32),
                ("stored_tokens", ctypes.c_int64), ("logical_tokens", ctypes.c_int64),
                ("allocated_slots", ctypes.c_int64), ("max_len", ctypes.c_int64), ("copies", ctypes.c_int64),
                ("swapped", ctypes.c_int64)]


def _lib():
    lib = library()
    if not getattr(lib, "_bm_bound", False):
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.pkv_bm_create.argtypes = [i32, i32, ctypes.POINTER(vp)]
        lib.pkv_bm_destroy.argtypes = [vp]
        lib.pkv_bm_destroy.restype = None
        lib.pkv_bm_add_sequence.argtypes = [vp, i64, i64]
        lib.pkv_bm_fork.argtypes = [vp, i64, i64]
        lib.pkv_bm_append.argtypes = [vp, vp, i32, vp, vp, ctypes.POINTER(i32)]
        lib.pkv_bm_free_sequence.argtypes = [vp, i64]
        lib.pkv_bm_block_tables.argtypes = [vp, vp, i32, i32, vp, vp]
        lib.pkv_bm_stats.argtypes = [vp, ctypes.POINTER(BlockStats)]
        lib.pkv_bm_swap_out.argtypes = [vp, i64, vp, i32, ctypes.POINTER(i32)]
        lib.pkv_bm_swap_in.argtypes = [vp, i64, vp, i32, ctypes.POINTER(i32)]
        for n in ("pkv_bm_create", "pkv_bm_add_sequence", "pkv_bm_fork", "pkv_bm_append",
                  "pkv_bm_free_sequence", "pkv_bm_block_tables", "pkv_bm_stats", "pkv_bm_swap_out",
                  "pkv_bm_swap_in"):
            getattr(lib, n).restype = ctypes.c_int
        lib._bm_bound = True
    return lib


class BlockManager:
    """A pool of num_blocks blocks of block_size tokens, tracked on the host."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = _lib()
        h = ctypes.c_void_p()
        _check(self._lib.pkv_bm_create(num_blocks, block_size, ctypes.byref(h)))
        self._h = h
        self.num_blocks, self.block_size = num_blocks, block_size

    def close(self) -> None:
        if self._h:
            self._lib.pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_sequence(self, seq_id: int, num_tokens: int) -> None:
        _check(self._lib.pkv_bm_add_sequence(self._h, seq_id, num_tokens))

    def fork(self, parent: int, child: int) -> None:
        _check(self._lib.pkv_bm_fork(self._h, parent, child))

    def append(self, seq_ids):
        """Slots (int64 [n]) for one new token per sequence and copy-on-write pairs (int64 [k, 2])."""
        ids = torch.tensor(list(seq_ids), dtype=torch.int64)
        n = ids.numel()
        slots = torch.empty(n, dtype=torch.int64)
        pairs = torch.empty((max(n, 1), 2), dtype=torch.int64)
        k = ctypes.c_int32(0)
        _check(self._lib.pkv_bm_append(self._h, ids.data_ptr(), n, slots.data_ptr(), pairs.data_ptr(),
                                       ctypes.byref(k)))
        return slots, pairs[:k.value].clone()

    def free_sequence(self, seq_id: int) -> None:
        _check(self._lib.pkv_bm_free_sequence(self._h, seq_id))

    def _blocks_call(self, fn, seq_id):
        cap = self.num_blocks
        out = torch.empty(cap, dtype=torch.int32)
        n = ctypes.c_int32(0)
        _check(fn(self._h, seq_id, out.data_ptr(), cap, ctypes.byref(n)))
        return out[:n.value].tolist()

    def swap_out(self, seq_id: int) -> list:
        """Preempt: the sequence's blocks (copy them out with paged_block_swap_out), released."""
        return self._blocks_call(self._lib.pkv_bm_swap_out, seq_id)

    def swap_in(self, seq_id: int) -> list:
        """Restore into fresh blocks (copy the data back with paged_block_swap_in)."""
        return self._blocks_call(self._lib.pkv_bm_swap_in, seq_id)

    def block_tables(self, seq_ids, max_blocks: int | None = None):
        """(block_tables int32 [n, max_blocks] padded with -1, context_lens int32 [n])."""
        ids = torch.tensor(list(seq_ids), dtype=torch.int64)
        n = ids.numel()
        if max_blocks is None:
            max_blocks = max(1, -(-self.stats()["max_len"] // self.block_size))
        tables = torch.empty((n, max_blocks), dtype=torch.int32)
        lens = torch.empty(n, dtype=torch.int32)
        _check(self._lib.pkv_bm_block_tables(self._h, ids.data_ptr(), n, max_blocks, tables.data_ptr(),
                                             lens.data_ptr()))
        return tables, lens

    def stats(self) -> dict:
        st = BlockStats()
        _check(self._lib.pkv_bm_stats(self._h, ctypes.byref(st)))
        return {f: getattr(st, f) for f, _ in BlockStats._fields_}


def waste_report(lengths, block_size: int, max_len: int) -> dict:
    """KV memory waste of paged storage against a contiguous reservation of max_len
    tokens per sequence (how earlier servers allocated), for the given lengths.

    paged: 1 - tokens / (blocks * block_size), the unused tails of last blocks.
    contiguous: 1 - tokens / (sequences * max_len).
    """
    lengths = [int(x) for x in lengths]
    need = sum(-(-n // block_size) for n in lengths)
    bm = BlockManager(max(1, need), block_size)
    for i, n in enumerate(lengths):
        bm.add_sequence(i, n)
    st = bm.stats()
    bm.close()
    tokens = st["stored_tokens"]
    return dict(sequences=len(lengths), tokens=tokens, block_size=block_size, max_len=max_len,
                allocated_slots=st["allocated_slots"],
                paged_waste=1.0 - tokens / st["allocated_slots"] if st["allocated_slots"] else 0.0,
                contiguous_waste=1.0 - tokens / (len(lengths) * max_len) if lengths else 0.0)
